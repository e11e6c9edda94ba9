"""GPU parity of the attention side of a decode step (per-head Q/K RMSNorm +
RoPE + KV-cache write) through the C ABI, against the fp64 CPU oracle.

Bar, element by element:
  - q_out and the written key rows: |got - ref| <= 2^-8 |ref| + 1e-4.  The
    kernel computes in fp32 (the rotation angles in fp64) and rounds once to
    bf16 (half an ulp is 2^-9 relative); the absolute term covers fp32 rounding
    where a rotation cancels (|terms| ~ 4 for unit-RMS heads with gains ~ 1);
  - the written value rows: bit for bit the input value heads;
  - every cache row whose slot no token maps to (and every row of a padding
    token, slot -1, or of a slot beyond the cache): bit for bit unchanged.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import flint_synth as fs
import oracle

pytestmark = pytest.mark.gpu

NQ, NKV, HD = 32, 4, 128
RTOL, ATOL = 2.0 ** -8, 1e-4


@pytest.fixture(scope="module")
def m():
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as mod
    mod.lib()
    return mod


def _f64(t):
    return t.cpu().float().double().numpy()


def _run(m, inp, theta, eps=1e-6):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inp.items()}
    B = g["qkv"].shape[0]
    q = torch.full((B, NQ, HD), float("nan"), dtype=torch.bfloat16, device=dev)
    m.flint_qk_norm_rope_kv_bf16(g["qkv"], g["q_norm"], g["k_norm"], g["positions"],
                                 g["slot_mapping"], q, g["k_cache"], g["v_cache"], theta, eps)
    torch.cuda.synchronize()
    return q.cpu(), g["k_cache"].cpu(), g["v_cache"].cpu()


def _check(inp, theta, q, kc, vc, eps=1e-6):
    qr, kr, vr = oracle.qk_norm_rope(inp["qkv"], inp["q_norm"], inp["k_norm"], inp["positions"],
                                     NQ, NKV, theta, eps=eps)
    np.testing.assert_allclose(_f64(q), qr, rtol=RTOL, atol=ATOL)
    slots = inp["slot_mapping"].tolist()
    n = inp["k_cache"].shape[0]
    written = set()
    for t, s in enumerate(slots):
        if 0 <= s < n:
            written.add(s)
            np.testing.assert_allclose(_f64(kc[s]), kr[t], rtol=RTOL, atol=ATOL)
            assert torch.equal(vc[s].view(torch.int16),
                               inp["qkv"][t, (NQ + NKV) * HD:].reshape(NKV, HD).view(torch.int16))
    keep = [s for s in range(n) if s not in written]
    assert torch.equal(kc[keep].view(torch.int16), inp["k_cache"][keep].view(torch.int16))
    assert torch.equal(vc[keep].view(torch.int16), inp["v_cache"][keep].view(torch.int16))


@pytest.mark.parametrize("batch,theta", [(1, 1.0e6), (8, 1.0e6), (37, 1.0e4), (256, 1.0e6),
                                         (8, 0.0), (100, 0.0)])
def test_qk_norm_rope_kv_matches_oracle(m, batch, theta):
    inp = fs.attn_inputs(700 + batch, batch, cache_slots=batch + 61)
    q, kc, vc = _run(m, inp, theta)
    _check(inp, theta, q, kc, vc)


def test_positions_at_the_ends_and_slots_beyond_the_cache(m):
    inp = fs.attn_inputs(811, 9, cache_slots=16)
    inp["positions"] = torch.tensor([0, 1, 2, (1 << 18) - 1, (1 << 31) - 1, -5, 513, 512, 7],
                                    dtype=torch.int32)
    inp["slot_mapping"] = torch.tensor([3, -1, 16, 15, 0, 1000, 8, -7, 2], dtype=torch.int32)
    q, kc, vc = _run(m, inp, 1.0e6)
    _check(inp, 1.0e6, q, kc, vc)


def test_scaled_and_zero_rows_and_large_eps(m):
    inp = fs.attn_inputs(812, 6, cache_slots=8)
    qkv = inp["qkv"].float()
    qkv[0] *= 300.0            # far above unit RMS: the norm removes the scale
    qkv[1] *= 1.0 / 256.0      # far below
    qkv[2] = 0.0               # all zero: every head normalises to 0 (eps > 0)
    inp["qkv"] = qkv.to(torch.bfloat16)
    for eps in (1e-6, 0.25):
        case = {k: v.clone() for k, v in inp.items()}
        q, kc, vc = _run(m, case, 1.0e6, eps=eps)
        _check(case, 1.0e6, q, kc, vc, eps=eps)
        assert torch.count_nonzero(q[2].float()) == 0


def test_repeat_is_bitwise_identical(m):
    inp = fs.attn_inputs(813, 64, cache_slots=80)
    a = _run(m, {k: v.clone() for k, v in inp.items()}, 1.0e6)
    b = _run(m, {k: v.clone() for k, v in inp.items()}, 1.0e6)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
