"""GPU parity of the decode layer with its input RMSNorm folded in
(flint_moe_decode_bf16_prenorm), through the C ABI.

Bar:
  - bit for bit the two-launch path it replaces (flint_moe_rmsnorm_bf16 into a
    separate x, then flint_moe_decode_bf16): out, expert indices and routing
    weights, in the persistent kernel (batch <= 8) and the chained kernels;
  - against the fp64 oracle (its RMSNorm rounded to bf16, then its layer) under
    the decode parity bar of test_parity_gpu.py;
  - in place (out aliasing the residual) bit for bit the out-of-place result.
"""
from __future__ import annotations

import pytest
import torch

import flint_synth as fs
import oracle
from tests.test_parity_gpu import check_layer, run_decode

pytestmark = pytest.mark.gpu

D = fs.FULL
K = D.top_k
EPS = 1e-6


@pytest.fixture(scope="module")
def m():
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as mod
    mod.lib()
    return mod


@pytest.fixture(scope="module")
def layer():
    W = fs.layer_weights(1001, D, device=torch.device("cuda:0"))
    return W, {k: v.cpu() for k, v in W.items()}


@pytest.fixture(scope="module")
def ws(m):
    return m.new_workspace(256)


def pre_norm(seed, B):
    """A residual stream as a layer of a pre-norm stack sees it: scaled,
    non-unit RMS rows (the tokens' pre-norm draw times 3)."""
    _, res = fs.tokens(seed, B, device="cuda")
    return (res.float() * 3.0).to(torch.bfloat16)


def run_prenorm(m, W, res, ws, eps=EPS, out=None):
    B = res.shape[0]
    out = torch.empty_like(res) if out is None else out
    idx = torch.full((B, K), -1, dtype=torch.int32, device=res.device)
    w = torch.zeros((B, K), dtype=torch.float32, device=res.device)
    m.flint_moe_decode_bf16_prenorm(res, W["wr"], None, W["w13"], W["w2"], W["ws13"], W["ws2"],
                                    out, ws, eps, idx, w)
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    return out, idx, w


def same_bits(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("B,eps", [(1, EPS), (3, EPS), (4, EPS), (5, EPS), (8, EPS), (8, 0.25),
                                   (13, EPS), (32, EPS), (128, EPS)])
def test_prenorm_equals_norm_then_decode_bitwise(m, layer, ws, B, eps):
    W, _ = layer
    res = pre_norm(400 + B, B)
    x = torch.empty_like(res)
    m.flint_moe_rmsnorm_bf16(res, x, eps)
    out_a, idx_a, w_a = run_decode(m, W, x, res, None, ws)
    out_b, idx_b, w_b = run_prenorm(m, W, res, ws, eps)
    assert torch.equal(idx_a, idx_b)
    assert same_bits(w_a, w_b)
    assert same_bits(out_a, out_b)


@pytest.mark.parametrize("B", [1, 5, 8, 24])
def test_prenorm_matches_oracle(m, layer, ws, B):
    W, host = layer
    res = pre_norm(500 + B, B)
    out, idx, w = run_prenorm(m, W, res, ws)
    x_ref = torch.from_numpy(oracle.rmsnorm(res.cpu(), EPS)).to(torch.bfloat16)
    check_layer(host, x_ref.cuda(), res, None, out, idx, w)


@pytest.mark.parametrize("B", [2, 5, 20])
def test_prenorm_in_place(m, layer, ws, B):
    W, _ = layer
    res = pre_norm(600 + B, B)
    out, _, _ = run_prenorm(m, W, res, ws)
    inplace = res.clone()
    run_prenorm(m, W, inplace, ws, out=inplace)
    assert same_bits(out, inplace)
