"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Bar (applied to every case):
  - expert indices bit-exact on every token whose fp64 gap between the 6th and
    7th logit is >= TAU; on the rare near-tie token the GPU's set must be a
    valid top-6 within TAU of the boundary;
  - routing weights within 1e-5 relative of the oracle's for the GPU's set;
  - out and the MoE delta (out - residual) within REL_TOL under the error rule
    of tests/_util.py, against the oracle evaluated on the GPU's expert set.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import flint_synth as fs
import oracle
from tests._util import REL_TOL, TAU, bf16_bits_to_f64, rel_err, rel_err_delta, topk_margin

pytestmark = pytest.mark.gpu

D = fs.FULL
K = D.top_k


@pytest.fixture(scope="module")
def m():
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as mod
    mod.lib()
    return mod


@pytest.fixture(scope="module")
def layer():
    dev = torch.device("cuda:0")
    W = fs.layer_weights(1001, D, device=dev)
    host = {k: v.cpu() for k, v in W.items()}
    return W, host


@pytest.fixture(scope="module")
def ws(m):
    return m.new_workspace(256)


def run_decode(m, W, x, res, bias, ws, out=None):
    B = x.shape[0]
    out = torch.empty_like(res) if out is None else out
    idx = torch.full((B, K), -1, dtype=torch.int32, device=x.device)
    w = torch.zeros((B, K), dtype=torch.float32, device=x.device)
    m.flint_moe_decode_bf16(x, res, W["wr"], bias, W["w13"], W["w2"], W["ws13"], W["ws2"], out,
                            ws, idx, w)
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    return out, idx, w


def check_routing(host, x, bias, idx, w):
    """Returns the oracle weights for the GPU's expert set (f64 [B,k])."""
    ref_idx, _, logits = oracle.route(D, x.cpu(), host["wr"], None if bias is None else bias.cpu())
    gi = idx.cpu().numpy().astype(np.int64)
    margin = topk_margin(logits, K)
    clear = margin >= TAU
    np.testing.assert_array_equal(gi[clear], ref_idx[clear])
    for t in np.nonzero(~clear)[0]:   # near-tie tokens: a valid top-k within TAU
        s = -np.sort(-logits[t])
        sel = logits[t, gi[t]]
        assert len(set(gi[t].tolist())) == K
        assert sel.min() >= s[K - 1] - TAU
        assert np.all(np.diff(sel) <= TAU)
    L = np.take_along_axis(logits, gi, axis=1)
    s = 1.0 / (1.0 + np.exp(-L))
    w_ref = s / s.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-5, atol=0)
    return gi.astype(np.int32), w_ref


def check_layer(host, x, res, bias, out, idx, w):
    gi, w_ref = check_routing(host, x, bias, idx, w)
    ref = oracle.moe_bf16_given_routing(D, x.cpu(), res.cpu(), gi, w_ref, host["w13"], host["w2"],
                                        host["ws13"], host["ws2"])
    got = bf16_bits_to_f64(out)
    r = bf16_bits_to_f64(res)
    e_out = rel_err(got, ref)
    e_delta = rel_err_delta(got, ref, r)
    assert e_out <= REL_TOL and e_delta <= REL_TOL, (e_out, e_delta)
    return e_out, e_delta


ROUTE_CASES = [(1, False), (5, False), (8, False), (64, True), (128, True), (256, False)]


@pytest.mark.parametrize("B,with_bias", ROUTE_CASES)
def test_route_matches_oracle(m, layer, ws, B, with_bias):
    W, host = layer
    x, _ = fs.tokens(3000 + B, B, device="cuda")
    bias = fs.logit_offsets(1003, device="cuda") if with_bias else None
    idx = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((B, K), dtype=torch.float32, device="cuda")
    m.flint_moe_route(x, W["wr"], bias, idx, w, ws)
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    check_routing(host, x, bias, idx, w)


@pytest.mark.parametrize("B", [1, 8, 37, 128, 256])
def test_bucket_matches_oracle(m, layer, ws, B):
    W, host = layer
    x, _ = fs.tokens(3100 + B, B, device="cuda")
    bias = fs.logit_offsets(1003, device="cuda")
    ref_idx, _, _ = oracle.route(D, x.cpu(), host["wr"], bias.cpu())
    u_ref, off_ref, pairs_ref = oracle.bucket(ref_idx, D.n_experts)
    dev_idx = torch.from_numpy(ref_idx).cuda()
    uniq = torch.full((256,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((257,), -7, dtype=torch.int32, device="cuda")
    pairs = torch.full((B * K,), -7, dtype=torch.int32, device="cuda")
    n = torch.zeros((4,), dtype=torch.int32, device="cuda")
    m.flint_moe_bucket(dev_idx, uniq, offsets, pairs, n, ws)
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    U = int(n[0])
    assert U == len(u_ref)
    np.testing.assert_array_equal(uniq[:U].cpu().numpy(), u_ref)
    np.testing.assert_array_equal(offsets[:U + 1].cpu().numpy(), off_ref)
    np.testing.assert_array_equal(pairs.cpu().numpy(), pairs_ref)


DECODE_CASES = [(1, False), (2, False), (3, False), (5, False), (8, False), (13, False),
                (31, True), (32, True), (77, True), (128, True), (128, False), (129, True),
                (160, True), (200, False), (255, True), (256, True), (256, False)]


@pytest.mark.parametrize("B,with_bias", DECODE_CASES)
def test_decode_bf16_matches_oracle(m, layer, ws, B, with_bias):
    W, host = layer
    x, res = fs.tokens(2000 + B, B, device="cuda")
    bias = fs.logit_offsets(1003, device="cuda") if with_bias else None
    out, idx, w = run_decode(m, W, x, res, bias, ws)
    check_layer(host, x, res, bias, out, idx, w)


@pytest.mark.parametrize("B,with_bias", [(1, False), (4, False), (8, False), (24, False),
                                          (64, True)])
def test_decode_bf16_zero_residual_pins_expert_path(m, layer, ws, B, with_bias):
    """residual = 0: out = bf16(MoE delta), so the expert path's own error is
    visible without the residual's rounding (CUDA-core groups at B <= 4, the
    tensor-core path for the shared expert from B = 5, both above)."""
    W, host = layer
    x, _ = fs.tokens(2100 + B, B, device="cuda")
    res = torch.zeros_like(x)
    bias = fs.logit_offsets(1003, device="cuda") if with_bias else None
    out, idx, w = run_decode(m, W, x, res, bias, ws)
    e_out, _ = check_layer(host, x, res, bias, out, idx, w)
    assert e_out <= 8e-3, e_out    # bf16 output rounding is <= 2^-8 relative


def test_zero_input_gives_lowest_experts_and_residual_bitwise(m, layer, ws):
    W, _ = layer
    B = 4
    _, res = fs.tokens(11, B, device="cuda")
    x = torch.zeros_like(res)
    out, idx, w = run_decode(m, W, x, res, None, ws)
    assert torch.equal(idx.cpu(), torch.arange(K, dtype=torch.int32).repeat(B, 1))
    assert torch.all(w.cpu() == 1.0 / K)
    assert torch.equal(out.view(torch.int16), res.view(torch.int16))


def test_planted_router_ties_pick_lower_index(m, layer, ws):
    """x = sqrt(H) e_0 (45.25, exact in bf16) and a router whose column 0 holds
    planted duplicates at the 6/7 boundary: logits are single exact products, so
    both sides see exact ties and the lower index must win."""
    W, host = layer
    H, E = D.hidden, D.n_experts
    col = torch.zeros(E)
    col[[200, 13, 77, 5]] = torch.tensor([4.0, 3.0, 2.5, 2.0])
    col[[250, 9, 130, 64]] = 1.5      # four-way tie for the last two slots
    wr = torch.zeros((E, H))
    wr[:, 0] = col
    wr = wr.to(torch.bfloat16)
    x = torch.zeros((2, H))
    x[:, 0] = 45.25
    x = x.to(torch.bfloat16)
    _, res = fs.tokens(12, 2)
    Wt = dict(W)
    Wt["wr"] = wr.cuda()
    out, idx, w = run_decode(m, Wt, x.cuda(), res.cuda(), None, ws)
    expect = [200, 13, 77, 5, 9, 64]
    assert idx.cpu().tolist() == [expect, expect]
    ref_idx, _, _ = oracle.route(D, x, wr, None)
    assert ref_idx.tolist() == [expect, expect]
    hostt = dict(host)
    hostt["wr"] = wr
    check_layer(hostt, x.cuda(), res.cuda(), None, out, idx, w)


def test_token_permutation_permutes_outputs_bitwise(m, layer, ws):
    W, _ = layer
    B = 24
    x, res = fs.tokens(13, B, device="cuda")
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(0)).cuda()
    out, idx, _ = run_decode(m, W, x, res, None, ws)
    out_p, idx_p, _ = run_decode(m, W, x[perm].contiguous(), res[perm].contiguous(), None, ws)
    assert torch.equal(idx_p, idx[perm])
    assert torch.equal(out_p.view(torch.int16), out[perm].view(torch.int16))


def test_batch_invariance(m, layer, ws):
    W, host = layer
    B = 16
    x, res = fs.tokens(14, B, device="cuda")
    out, idx, _ = run_decode(m, W, x, res, None, ws)
    for t in (0, 7, 15):
        o1, i1, _ = run_decode(m, W, x[t:t + 1].contiguous(), res[t:t + 1].contiguous(), None, ws)
        assert torch.equal(i1[0], idx[t])
        ref = bf16_bits_to_f64(out[t:t + 1])
        assert rel_err(bf16_bits_to_f64(o1), ref) <= REL_TOL


def test_in_place_residual_and_repeat_determinism(m, layer, ws):
    W, _ = layer
    B = 8
    x, res = fs.tokens(15, B, device="cuda")
    out1, _, _ = run_decode(m, W, x, res, None, ws)
    out2, _, _ = run_decode(m, W, x, res, None, ws)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    buf = res.clone()
    run_decode(m, W, x, buf, None, ws, out=buf)   # out aliases residual exactly
    assert torch.equal(buf.view(torch.int16), out1.view(torch.int16))


def test_cuda_graph_replay_matches_eager(m, layer):
    W, _ = layer
    B = 8
    ws = m.new_workspace(B)
    x, res = fs.tokens(16, B, device="cuda")
    out_e, _, _ = run_decode(m, W, x, res, None, ws)
    out = torch.empty_like(res)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        m.flint_moe_decode_bf16(x, res, W["wr"], None, W["w13"], W["w2"], W["ws13"], W["ws2"],
                                out, ws, stream=s)   # warm-up outside capture
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            m.flint_moe_decode_bf16(x, res, W["wr"], None, W["w13"], W["w2"], W["ws13"], W["ws2"],
                                    out, ws, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    assert torch.equal(out.view(torch.int16), out_e.view(torch.int16))


def test_stuck_wait_reports_timeout_and_workspace_recovers(m, layer):
    """The stall hook makes one device wait on a flag nothing sets; the wait
    runs out after the (short) limit, the call reports a timeout instead of
    hanging, and after re-initialisation the next call is correct."""
    W, host = layer
    B = 2
    ws = m.new_workspace(B, wait_limit_ns=20_000_000)   # 20 ms
    x, res = fs.tokens(17, B, device="cuda")
    m.flint_moe_debug_arm_stall(ws)
    out = torch.empty_like(res)
    m.flint_moe_decode_bf16(x, res, W["wr"], None, W["w13"], W["w2"], W["ws13"], W["ws2"], out, ws)
    assert m.flint_moe_get_device_status(ws) == m.FLINT_ERR_DEVICE_TIMEOUT
    m.flint_moe_workspace_init(ws)
    out, idx, w = run_decode(m, W, x, res, None, ws)
    check_layer(host, x, res, None, out, idx, w)


def test_bucket_reports_bad_routing(m, ws):
    B = 2
    bad = torch.tensor([[0, 1, 2, 3, 4, 4], [0, 1, 2, 3, 4, 300]], dtype=torch.int32).cuda()
    z = lambda n: torch.zeros((n,), dtype=torch.int32, device="cuda")  # noqa: E731
    m.flint_moe_bucket(bad, z(256), z(257), z(B * K), z(4), ws)
    assert m.flint_moe_get_device_status(ws) == m.FLINT_ERR_INVALID_ARG
    m.flint_moe_workspace_init(ws)


def test_rmsnorm_matches_oracle(m):
    B = 37
    x, _ = fs.tokens(18, B, device="cuda")
    y = (x.float() * 3.0).to(torch.bfloat16)
    out = torch.empty_like(y)
    m.flint_moe_rmsnorm_bf16(y, out, 1e-6)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(y.cpu(), 1e-6)
    got = bf16_bits_to_f64(out)
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)) <= 2 ** -8


# ---------------------------------------------------------------- NVFP4 (W4A16)

@pytest.fixture(scope="module")
def nv_layer(layer):
    W, _ = layer
    nv = fs.nvfp4_layer(W)
    torch.cuda.synchronize()
    return nv, {k: v.cpu() for k, v in nv.items()}


def run_nvfp4(m, W, nv, x, res, bias, ws):
    B = x.shape[0]
    out = torch.empty_like(res)
    idx = torch.full((B, K), -1, dtype=torch.int32, device=x.device)
    w = torch.zeros((B, K), dtype=torch.float32, device=x.device)
    m.flint_moe_decode_nvfp4_w4a16(x, res, W["wr"], bias, nv, out, ws, idx, w)
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    return out, idx, w


@pytest.mark.parametrize("B,with_bias", [(1, False), (2, False), (3, False), (5, False),
                                          (8, False), (13, False), (32, True), (128, True),
                                          (160, True), (200, False), (256, True), (256, False)])
def test_decode_nvfp4_matches_oracle(m, layer, nv_layer, ws, B, with_bias):
    W, host = layer
    nv, nv_host = nv_layer
    x, res = fs.tokens(4000 + B, B, device="cuda")
    bias = fs.logit_offsets(1003, device="cuda") if with_bias else None
    out, idx, w = run_nvfp4(m, W, nv, x, res, bias, ws)
    gi, w_ref = check_routing(host, x, bias, idx, w)
    ref = oracle.moe_nvfp4_given_routing(D, x.cpu(), res.cpu(), gi, w_ref, nv_host)
    got = bf16_bits_to_f64(out)
    r = bf16_bits_to_f64(res)
    e_out, e_delta = rel_err(got, ref), rel_err_delta(got, ref, r)
    assert e_out <= REL_TOL and e_delta <= REL_TOL, (e_out, e_delta)


def test_nvfp4_zero_input_residual_bitwise(m, layer, nv_layer, ws):
    W, _ = layer
    nv, _ = nv_layer
    _, res = fs.tokens(19, 3, device="cuda")
    out, idx, _ = run_nvfp4(m, W, nv, torch.zeros_like(res), res, None, ws)
    assert torch.equal(idx.cpu(), torch.arange(K, dtype=torch.int32).repeat(3, 1))
    assert torch.equal(out.view(torch.int16), res.view(torch.int16))


@pytest.mark.parametrize("B", [8, 40])
def test_nvfp4_repeat_and_token_permutation_bitwise(m, layer, nv_layer, ws, B):
    """The NVFP4 down kernel adds each token's partial sums in a fixed order
    (ascending pair index, i.e. expert order), so a repeat gives the same bits
    and permuting the tokens permutes the output bits."""
    W, _ = layer
    nv, _ = nv_layer
    x, res = fs.tokens(4200 + B, B, device="cuda")
    out1, idx1, _ = run_nvfp4(m, W, nv, x, res, None, ws)
    out2, idx2, _ = run_nvfp4(m, W, nv, x, res, None, ws)
    assert torch.equal(idx1, idx2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(7)).cuda()
    out_p, idx_p, _ = run_nvfp4(m, W, nv, x[perm].contiguous(), res[perm].contiguous(), None, ws)
    assert torch.equal(idx_p, idx1[perm])
    assert torch.equal(out_p.view(torch.int16), out1[perm].view(torch.int16))


@pytest.mark.parametrize("B", [1, 3, 8, 13, 32])
def test_workspace_sized_for_the_batch(m, layer, nv_layer, ws, B):
    """A workspace sized for exactly B tokens gives the same bits as a larger
    one on both paths (the offsets of every array but h and the per-pair
    partials do not depend on the size), and the BF16 output matches the
    oracle (seed 2001 at batch 3 is the smoke case)."""
    W, host = layer
    nv, _ = nv_layer
    x, res = fs.tokens(2001 if B == 3 else 2300 + B, B, device="cuda")
    tight = m.new_workspace(B)
    assert tight.numel() == m.flint_moe_workspace_bytes(B) < ws.numel()
    out_t, idx_t, w_t = run_decode(m, W, x, res, None, tight)
    out_l, idx_l, _ = run_decode(m, W, x, res, None, ws)
    assert torch.equal(idx_t, idx_l)
    assert torch.equal(out_t.view(torch.int16), out_l.view(torch.int16))
    check_layer(host, x, res, None, out_t, idx_t, w_t)
    nv_t, _, _ = run_nvfp4(m, W, nv, x, res, None, tight)
    nv_l, _, _ = run_nvfp4(m, W, nv, x, res, None, ws)
    assert torch.equal(nv_t.view(torch.int16), nv_l.view(torch.int16))


@pytest.mark.parametrize("B", [3, 8, 32])
def test_stage_calls_match_oracle(m, layer, ws, B):
    """route -> gate/up -> down through their own entry points computes the
    layer (the three-kernel path, also at batches the decode call fuses); above
    8 tokens the decode call runs the same kernels, so the bits agree."""
    W, host = layer
    x, res = fs.tokens(2400 + B, B, device="cuda")
    bias = fs.logit_offsets(1003, device="cuda") if B > 8 else None
    idx = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((B, K), dtype=torch.float32, device="cuda")
    out = torch.empty_like(res)
    m.flint_moe_route(x, W["wr"], bias, idx, w, ws)
    m.flint_moe_gateup_bf16(x, W["w13"], W["ws13"], ws)
    m.flint_moe_down_bf16(res, W["w2"], W["ws2"], out, ws)
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    check_layer(host, x, res, bias, out, idx, w)
    if B > 8:
        out_d, idx_d, _ = run_decode(m, W, x, res, bias, ws)
        assert torch.equal(idx_d, idx)
        assert torch.equal(out_d.view(torch.int16), out.view(torch.int16))


@pytest.mark.parametrize("B", [3, 8, 13, 40])
def test_large_h_beyond_f16_range_matches_oracle(m, layer, nv_layer, ws, B):
    """Gate and up scaled by 256 (a power of two, so the NVFP4 codes and the
    bf16 weights stay exact): g and u grow 256x and h ~65536x, far beyond
    f16's 65504, on both formats, at batches of both the fused and the
    three-kernel path.  The outputs must still match the oracle."""
    W, host = layer
    nv, nv_host = nv_layer
    x, res = fs.tokens(4600 + B, B, device="cuda")
    # BF16: w13 x 256 (exact in bf16)
    Wb = dict(W)
    Wb["w13"] = (W["w13"].float() * 256.0).to(torch.bfloat16)
    Wb["ws13"] = (W["ws13"].float() * 256.0).to(torch.bfloat16)
    out, idx, w = run_decode(m, Wb, x, res, None, ws)
    hostb = dict(host)
    hostb["w13"] = Wb["w13"].cpu()
    hostb["ws13"] = Wb["ws13"].cpu()
    gi, w_ref = check_routing(host, x, None, idx, w)
    ref = oracle.moe_bf16_given_routing(D, x.cpu(), res.cpu(), gi, w_ref, hostb["w13"], hostb["w2"],
                                        hostb["ws13"], hostb["ws2"])
    assert np.max(np.abs(ref - bf16_bits_to_f64(res))) > 1e3   # the delta really is large
    got = bf16_bits_to_f64(out)
    assert rel_err(got, ref) <= REL_TOL
    assert rel_err_delta(got, ref, bf16_bits_to_f64(res)) <= REL_TOL
    # NVFP4: tensor scales of gate and up x 256
    nvb = dict(nv)
    nvb["w13_ts"] = nv["w13_ts"] * 256.0
    nvb["ws13_ts"] = nv["ws13_ts"] * 256.0
    nvh = {k: v.cpu() for k, v in nvb.items()}
    out4, idx4, w4 = run_nvfp4(m, W, nvb, x, res, None, ws)
    gi4, w_ref4 = check_routing(host, x, None, idx4, w4)
    ref4 = oracle.moe_nvfp4_given_routing(D, x.cpu(), res.cpu(), gi4, w_ref4, nvh)
    got4 = bf16_bits_to_f64(out4)
    assert rel_err(got4, ref4) <= REL_TOL
    assert rel_err_delta(got4, ref4, bf16_bits_to_f64(res)) <= REL_TOL


@pytest.mark.parametrize("B", [2, 13])
def test_nvfp4_reports_activations_beyond_f16(m, layer, nv_layer, B):
    """The NVFP4 path multiplies f16 activations: a value beyond f16's range
    makes the call report FLINT_ERR_INVALID_ARG on the device instead of
    returning infinities; after re-initialisation the workspace works again
    (at 2 tokens, where each gate/up CTA selects locally, and at 13)."""
    W, host = layer
    nv, nv_host = nv_layer
    ws = m.new_workspace(B)
    x, res = fs.tokens(4700, B, device="cuda")
    xb = x.clone()
    xb[B // 2, 100] = 70000.0
    out = torch.empty_like(res)
    m.flint_moe_decode_nvfp4_w4a16(xb, res, W["wr"], None, nv, out, ws)
    assert m.flint_moe_get_device_status(ws) == m.FLINT_ERR_INVALID_ARG
    m.flint_moe_workspace_init(ws)
    out, idx, w = run_nvfp4(m, W, nv, x, res, None, ws)
    gi, w_ref = check_routing(host, x, None, idx, w)
    ref = oracle.moe_nvfp4_given_routing(D, x.cpu(), res.cpu(), gi, w_ref, nv_host)
    assert rel_err(bf16_bits_to_f64(out), ref) <= REL_TOL


@pytest.mark.parametrize("B", [1, 3, 13])
def test_nvfp4_reports_h_beyond_its_f16_pair(m, layer, nv_layer, B):
    """The NVFP4 path keeps h / 256 as an f16 pair: gate and up
    tensor scales times 2^16 put |h| far beyond 65520 * 256, which the call
    reports as FLINT_ERR_INVALID_ARG on the device instead of returning
    infinities; after re-initialisation the workspace works again."""
    W, host = layer
    nv, nv_host = nv_layer
    ws = m.new_workspace(B)
    x, res = fs.tokens(4800 + B, B, device="cuda")
    nvb = dict(nv)
    nvb["w13_ts"] = nv["w13_ts"] * 65536.0
    nvb["ws13_ts"] = nv["ws13_ts"] * 65536.0
    out = torch.empty_like(res)
    m.flint_moe_decode_nvfp4_w4a16(x, res, W["wr"], None, nvb, out, ws)
    assert m.flint_moe_get_device_status(ws) == m.FLINT_ERR_INVALID_ARG
    m.flint_moe_workspace_init(ws)
    out, idx, w = run_nvfp4(m, W, nv, x, res, None, ws)
    gi, w_ref = check_routing(host, x, None, idx, w)
    ref = oracle.moe_nvfp4_given_routing(D, x.cpu(), res.cpu(), gi, w_ref, nv_host)
    assert rel_err(bf16_bits_to_f64(out), ref) <= REL_TOL


def test_calls_of_mixed_batches_on_one_workspace_match_fresh_workspaces(m, layer):
    """The batch <= 8 kernel tells this call's exchanged data from older data
    by a call tag; calls of different batches (and of the three-kernel path)
    on one workspace must give exactly what a fresh workspace gives."""
    W, _ = layer
    shared = m.new_workspace(16)
    for i, B in enumerate([8, 1, 8, 3, 13, 8, 1, 1, 5, 8]):
        x, res = fs.tokens(4800 + i, B, device="cuda")
        out_s, idx_s, w_s = run_decode(m, W, x, res, None, shared)
        out_f, idx_f, w_f = run_decode(m, W, x, res, None, m.new_workspace(B))
        assert torch.equal(idx_s, idx_f), (i, B)
        assert torch.equal(w_s, w_f), (i, B)
        assert torch.equal(out_s.view(torch.int16), out_f.view(torch.int16)), (i, B)


def test_claimed_units_reset_between_calls_of_both_formats(m, layer, nv_layer):
    """The chained gate/up and down kernels hand out units from workspace
    counters that the last CTA of each call resets: BF16 and NVFP4 calls of
    claimed (32+ tokens) and equal-share batches in any order on one workspace
    give exactly what fresh workspaces give."""
    W, _ = layer
    nv, _ = nv_layer
    shared = m.new_workspace(64)
    seq = [(40, "nvfp4"), (13, "bf16"), (64, "nvfp4"), (40, "bf16"), (8, "nvfp4"),
           (64, "bf16"), (3, "nvfp4"), (40, "nvfp4")]
    for i, (B, fmt) in enumerate(seq):
        x, res = fs.tokens(4900 + i, B, device="cuda")
        run = (lambda ws: run_decode(m, W, x, res, None, ws)) if fmt == "bf16" else \
              (lambda ws: run_nvfp4(m, W, nv, x, res, None, ws))
        out_s, idx_s, w_s = run(shared)
        out_f, idx_f, w_f = run(m.new_workspace(B))
        assert torch.equal(idx_s, idx_f), (i, B, fmt)
        assert torch.equal(w_s, w_f), (i, B, fmt)
        assert torch.equal(out_s.view(torch.int16), out_f.view(torch.int16)), (i, B, fmt)


@pytest.mark.parametrize("B,fmt", [(1, "bf16"), (5, "bf16"), (8, "bf16"), (13, "bf16"),
                                   (64, "bf16"), (3, "nvfp4"), (40, "nvfp4"), (8, "route"),
                                   (128, "route")])
def test_select_only_offsets_match_oracle(m, layer, nv_layer, ws, B, fmt):
    """Logit offsets used for the selection only (FLINT_OFFSET_SELECT): the
    ranking uses score + offset, the weights the sigmoid of the score alone."""
    W, host = layer
    nv, nv_host = nv_layer
    Dsel = dataclasses.replace(D, offset_mode=1)
    x, res = fs.tokens(4900 + B, B, device="cuda")
    bias = fs.logit_offsets(1003, device="cuda")
    idx = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((B, K), dtype=torch.float32, device="cuda")
    out = torch.empty_like(res)
    if fmt == "route":
        m.flint_moe_route(x, W["wr"], bias, idx, w, ws, dims=m.SELECT_DIMS)
    elif fmt == "bf16":
        m.flint_moe_decode_bf16(x, res, W["wr"], bias, W["w13"], W["w2"], W["ws13"], W["ws2"],
                                out, ws, idx, w, dims=m.SELECT_DIMS)
    else:
        m.flint_moe_decode_nvfp4_w4a16(x, res, W["wr"], bias, nv, out, ws, idx, w,
                                       dims=m.SELECT_DIMS)
    torch.cuda.synchronize()
    assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
    ref_idx, _, keys = oracle.route(Dsel, x.cpu(), host["wr"], bias.cpu())
    raw_logits = oracle.route(D, x.cpu(), host["wr"], None)[2]   # scores without offsets
    gi = idx.cpu().numpy().astype(np.int64)
    clear = topk_margin(keys, K) >= TAU
    np.testing.assert_array_equal(gi[clear], ref_idx[clear])
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(raw_logits, gi, axis=1)))
    w_ref = s / s.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-5, atol=0)
    if fmt == "route":
        return
    if fmt == "bf16":
        ref = oracle.moe_bf16_given_routing(D, x.cpu(), res.cpu(), gi.astype(np.int32), w_ref,
                                            host["w13"], host["w2"], host["ws13"], host["ws2"])
    else:
        ref = oracle.moe_nvfp4_given_routing(D, x.cpu(), res.cpu(), gi.astype(np.int32), w_ref,
                                             nv_host)
    got = bf16_bits_to_f64(out)
    assert rel_err(got, ref) <= REL_TOL
    assert rel_err_delta(got, ref, bf16_bits_to_f64(res)) <= REL_TOL
