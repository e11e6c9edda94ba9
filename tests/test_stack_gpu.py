"""GPU parity of the 47-layer stack: 47 distinct resident BF16 MoE layers
(~76 GB) applied in sequence, each taking the RMSNorm of the previous layer's
output as its input (folded into the layer call, flint_moe_decode_bf16_prenorm),
launched exactly as bench.py times it.  Checked teacher-forced: each sampled
layer's oracle consumes the GPU's own bf16 residual stream of that layer (and
its own RMSNorm of it, rounded to bf16, as the layer input), so bf16 drift
cannot flip later routing.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import flint_synth as fs
import oracle
from tests._util import REL_TOL, bf16_bits_to_f64, rel_err, rel_err_delta, topk_margin, TAU

pytestmark = pytest.mark.gpu

D = fs.FULL
LAYERS = 47
SAMPLED = (0, 1, 23, 46)


@pytest.fixture(scope="module")
def m():
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as mod
    mod.lib()
    return mod


@pytest.fixture(scope="module")
def stack():
    free, _ = torch.cuda.mem_get_info()
    if free < LAYERS * 1.62e9 + 8e9:
        pytest.skip("the 47-layer stack needs ~85 GB of free device memory")
    layers = [fs.layer_weights(5000 + l, D, device="cuda") for l in range(LAYERS)]
    yield layers
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [1, 8, 32])
def test_stack_teacher_forced(m, stack, B):
    _, r0 = fs.tokens(6000 + B, B, device="cuda")
    outs = [torch.empty_like(r0) for _ in range(LAYERS)]
    idx = torch.empty((LAYERS, B, 6), dtype=torch.int32, device="cuda")
    wts = torch.empty((LAYERS, B, 6), dtype=torch.float32, device="cuda")
    ws = m.new_workspace(B)
    res = r0
    for l, W in enumerate(stack):
        m.flint_moe_decode_bf16_prenorm(res, W["wr"], None, W["w13"], W["w2"], W["ws13"],
                                        W["ws2"], outs[l], ws, 1e-6, idx[l], wts[l])
        res = outs[l]
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    for l in SAMPLED:
        W = {k: v.cpu() for k, v in stack[l].items()}
        r_l = (r0 if l == 0 else outs[l - 1]).cpu()
        x_l = torch.from_numpy(oracle.rmsnorm(r_l, 1e-6)).to(torch.bfloat16)
        gi = idx[l].cpu().numpy()
        ref_idx, _, logits = oracle.route(D, x_l, W["wr"], None)
        clear = topk_margin(logits, 6) >= TAU
        np.testing.assert_array_equal(gi[clear], ref_idx[clear])
        L = np.take_along_axis(logits, gi.astype(np.int64), axis=1)
        s = 1.0 / (1.0 + np.exp(-L))
        w_ref = s / s.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(wts[l].cpu().numpy(), w_ref, rtol=1e-5)
        ref = oracle.moe_bf16_given_routing(D, x_l, r_l, gi, w_ref, W["w13"], W["w2"], W["ws13"],
                                            W["ws2"])
        got = bf16_bits_to_f64(outs[l])
        r = bf16_bits_to_f64(r_l)
        assert rel_err(got, ref) <= REL_TOL, l
        assert rel_err_delta(got, ref, r) <= REL_TOL, l
