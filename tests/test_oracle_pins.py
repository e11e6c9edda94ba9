"""Pins the fp64 CPU oracle to things other than itself (no GPU needed).

Each test targets a plausible mistake: a dropped term (shared expert,
residual), a wrong sign (sigmoid), a wrong index or order (tie rule, gate/up
swap, down-projection transpose, nibble order, block-scale index), or a wrong
renormalisation.
"""
from __future__ import annotations

import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import flint_synth as fs
import oracle
from oracle import brute
from tests._util import topk_margin

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _f64(t) -> np.ndarray:
    return brute.bf16_to_f64(t)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed,batch,with_bias,select_only",
                         [(1, 1, False, False), (2, 3, False, False), (3, 8, True, False),
                          (4, 17, False, False), (5, 33, True, False), (6, 8, True, True),
                          (7, 33, True, True)])
def test_matches_dense_brute_force_tiny(seed, batch, with_bias, select_only):
    d = dataclasses.replace(fs.TINY, offset_mode=1 if select_only else 0)
    W = fs.layer_weights(seed, d)
    x, r = fs.tokens(seed + 100, batch, d.hidden)
    bias = fs.logit_offsets(seed + 200, d.n_experts) if with_bias else None
    out, idx, w = oracle.moe_bf16(d, x, r, W["wr"], bias, W["w13"], W["w2"], W["ws13"], W["ws2"])
    o2, i2, w2 = brute.dense_moe_bf16(x, r, W["wr"], bias, W["w13"], W["w2"], W["ws13"],
                                      W["ws2"], d.top_k, select_only)
    np.testing.assert_array_equal(idx, i2)
    np.testing.assert_allclose(w, w2, rtol=1e-13, atol=0)
    scale = np.abs(o2).max()
    assert np.abs(out - o2).max() <= 1e-12 * scale


@pytest.mark.slow
@pytest.mark.parametrize("batch,with_bias", [(1, False), (8, False), (8, True)])
def test_matches_dense_brute_force_full_size(batch, with_bias):
    d = fs.FULL
    W = fs.layer_weights(1001, d)
    x, r = fs.tokens(2001 + batch, batch, d.hidden)
    bias = fs.logit_offsets(3001, d.n_experts) if with_bias else None
    out, idx, w = oracle.moe_bf16(d, x, r, W["wr"], bias, W["w13"], W["w2"], W["ws13"], W["ws2"])
    o2, i2, w2 = brute.dense_moe_bf16(x, r, W["wr"], bias, W["w13"], W["w2"], W["ws13"],
                                      W["ws2"], d.top_k)
    np.testing.assert_array_equal(idx, i2)
    np.testing.assert_allclose(w, w2, rtol=1e-13, atol=0)
    assert np.abs(out - o2).max() <= 1e-12 * np.abs(o2).max()


# ---------------------------------------------------------------- invariants

def test_selection_is_first_k_of_full_sort_and_weights_sum_to_one():
    d = fs.TINY
    W = fs.layer_weights(11, d)
    x, _ = fs.tokens(12, 64, d.hidden)
    bias = fs.logit_offsets(13, d.n_experts)
    idx, w, logits = oracle.route(d, x, W["wr"], bias)
    E = d.n_experts
    for t in range(x.shape[0]):
        order = np.lexsort((np.arange(E), -logits[t]))  # key: (-logit, index)
        np.testing.assert_array_equal(idx[t], order[:d.top_k])
    assert np.all(w > 0)
    assert np.max(np.abs(w.sum(axis=1) - 1.0)) <= 1e-12
    for t in range(x.shape[0]):
        assert len(set(idx[t].tolist())) == d.top_k
        assert idx[t].min() >= 0 and idx[t].max() < E
    # Weights follow the sigmoid of the selected logits (ratio check).
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(logits, idx.astype(np.int64), axis=1)))
    np.testing.assert_allclose(w / w[:, :1], s / s[:, :1], rtol=1e-13)
    # Rank order: selected logits are non-increasing along the slots.
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    assert np.all(np.diff(sel, axis=1) <= 0)


def test_token_permutation_permutes_outputs_exactly():
    d = fs.TINY
    W = fs.layer_weights(21, d)
    x, r = fs.tokens(22, 9, d.hidden)
    perm = np.random.default_rng(0).permutation(9)
    out, idx, w = oracle.moe_bf16(d, x, r, W["wr"], None, W["w13"], W["w2"], W["ws13"], W["ws2"])
    op, ip, wp = oracle.moe_bf16(d, x[perm], r[perm], W["wr"], None, W["w13"], W["w2"],
                                 W["ws13"], W["ws2"])
    np.testing.assert_array_equal(op, out[perm])
    np.testing.assert_array_equal(ip, idx[perm])
    np.testing.assert_array_equal(wp, w[perm])


def test_batch_invariance_row_alone_equals_row_in_batch():
    d = fs.TINY
    W = fs.layer_weights(31, d)
    x, r = fs.tokens(32, 5, d.hidden)
    out, idx, _ = oracle.moe_bf16(d, x, r, W["wr"], None, W["w13"], W["w2"], W["ws13"], W["ws2"])
    for t in range(5):
        o1, i1, _ = oracle.moe_bf16(d, x[t:t + 1], r[t:t + 1], W["wr"], None, W["w13"], W["w2"],
                                    W["ws13"], W["ws2"])
        np.testing.assert_array_equal(o1[0], out[t])
        np.testing.assert_array_equal(i1[0], idx[t])


# ---------------------------------------------------------------- closed forms

def test_zero_input_gives_lowest_indices_equal_weights_and_residual():
    """x = 0: every logit is 0, a full tie, so experts 0..k-1 win; each weight
    is sigma(0) / (k sigma(0)) = 1/k; every projection of 0 is 0, so out is the
    residual exactly."""
    for d in (fs.TINY, fs.FULL):
        W = fs.layer_weights(41, d)
        _, r = fs.tokens(42, 3, d.hidden)
        x = torch.zeros((3, d.hidden), dtype=torch.bfloat16)
        out, idx, w = oracle.moe_bf16(d, x, r, W["wr"], None, W["w13"], W["w2"], W["ws13"],
                                      W["ws2"])
        np.testing.assert_array_equal(idx, np.tile(np.arange(d.top_k), (3, 1)))
        assert np.all(w == 1.0 / d.top_k)
        np.testing.assert_array_equal(out, _f64(r))


def test_zero_input_with_offsets_ranks_by_offsets():
    d = fs.TINY
    W = fs.layer_weights(43, d)
    bias = fs.logit_offsets(44, d.n_experts)
    x = torch.zeros((2, d.hidden), dtype=torch.bfloat16)
    idx, w, logits = oracle.route(d, x, W["wr"], bias)
    b = bias.double().numpy()
    expect = np.argsort(-b, kind="stable")[:d.top_k]
    np.testing.assert_array_equal(idx[0], expect)
    np.testing.assert_array_equal(logits[0], b)


def test_zero_input_select_only_offsets_rank_and_weights_are_equal():
    """x = 0 with offsets used for selection only: every router score is 0, so
    the offsets alone rank the experts and every kept weight is
    sigmoid(0) / (6 sigmoid(0)) = 1/6 exactly; with the offsets in the logit
    (mode 0) the weights follow the offsets instead."""
    d = dataclasses.replace(fs.TINY, offset_mode=1)
    W = fs.layer_weights(45, d)
    bias = fs.logit_offsets(46, d.n_experts)
    x = torch.zeros((2, d.hidden), dtype=torch.bfloat16)
    idx, w, logits = oracle.route(d, x, W["wr"], bias)
    b = bias.double().numpy()
    expect = np.argsort(-b, kind="stable")[:d.top_k]
    np.testing.assert_array_equal(idx[0], expect)
    assert np.all(w == 1.0 / d.top_k)
    idx0, w0, _ = oracle.route(fs.TINY, x, W["wr"], bias)
    np.testing.assert_array_equal(idx0, idx)
    s = 1.0 / (1.0 + np.exp(-b[expect]))
    np.testing.assert_allclose(w0[0], s / s.sum(), rtol=1e-14)


def _embedded_layer(d, shared_up=3.0):
    """Identity-embedded SwiGLU experts (see tests/golden/crafted_router.json):
    Wg_e = [I | 0], Wu_e = s_e [I | 0] with s_e = 1 + e/8, Wd_e = cyclic shift
    (row i picks column (i+1) mod I) in the first I rows; shared expert with
    Wu = shared_up [I | 0] and Wd = identity in the first I rows."""
    H, E, I = d.hidden, d.n_experts, d.inter
    eye = np.zeros((I, H), np.float32)
    eye[np.arange(I), np.arange(I)] = 1.0
    w13 = np.zeros((E, 2 * I, H), np.float32)
    w2 = np.zeros((E, H, I), np.float32)
    for e in range(E):
        w13[e, :I] = eye
        w13[e, I:] = (1.0 + e / 8.0) * eye
        w2[e, np.arange(I), (np.arange(I) + 1) % I] = 1.0
    ws13 = np.zeros((1, 2 * I, H), np.float32)
    ws2 = np.zeros((1, H, I), np.float32)
    ws13[0, :I] = eye
    ws13[0, I:] = shared_up * eye
    ws2[0, np.arange(I), np.arange(I)] = 1.0
    return _bf16(w13), _bf16(w2), _bf16(ws13), _bf16(ws2)


def test_crafted_router_and_identity_embedded_experts_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "crafted_router.json")))
    d = fs.TINY
    H, E, I, k = d.hidden, d.n_experts, d.inter, d.top_k
    wr = np.zeros((E, H), np.float32)
    wr[:, 0] = g["router_column0"]
    rng = np.random.default_rng(5)
    xv = rng.standard_normal((2, H)).astype(np.float32)
    xv[:, 0] = g["x0"]
    x = _bf16(xv)
    r = _bf16(rng.standard_normal((2, H)))
    w13, w2, ws13, ws2 = _embedded_layer(d, g["shared_up_scale"])
    out, idx, w = oracle.moe_bf16(d, x, r, _bf16(wr), None, w13, w2, ws13, ws2)
    expect_idx = np.array(g["expected_topk_idx"])
    np.testing.assert_array_equal(idx, np.tile(expect_idx, (2, 1)))
    L = g["x0"] * np.array(g["router_column0"])[expect_idx]
    s = 1.0 / (1.0 + np.exp(-L))
    np.testing.assert_allclose(w[0], s / s.sum(), rtol=1e-15)
    X = _f64(x)
    a = X[:, :I] / (1.0 + np.exp(-X[:, :I])) * X[:, :I]    # silu(g) * u with g = u = x[:I]
    ups = 1.0 + expect_idx / 8.0
    routed = (s / s.sum() * ups).sum()
    expect = _f64(r).copy()
    expect[:, :I] += g["shared_up_scale"] * a
    expect[:, :I] += routed * np.roll(a, -1, axis=1)       # (P a)[i] = a[(i+1) mod I]
    np.testing.assert_allclose(out, expect, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(out[:, I:], _f64(r)[:, I:])


def test_identical_experts_reduce_to_one_expert():
    """All routed experts equal: the routed part is (sum of weights) * f(x) = f(x)
    whatever the routing, so out = residual + f_shared(x) + f(x)."""
    d = fs.TINY
    W = fs.layer_weights(51, d)
    w13 = W["w13"][:1].expand(d.n_experts, -1, -1).contiguous()
    w2 = W["w2"][:1].expand(d.n_experts, -1, -1).contiguous()
    x, r = fs.tokens(52, 6, d.hidden)
    out, _, _ = oracle.moe_bf16(d, x, r, W["wr"], None, w13, w2, W["ws13"], W["ws2"])
    X = _f64(x)

    def ffn(w13e, w2e):
        W13, W2 = _f64(w13e), _f64(w2e)
        gg, uu = X @ W13[:d.inter].T, X @ W13[d.inter:].T
        return (gg / (1.0 + np.exp(-gg)) * uu) @ W2.T

    expect = _f64(r) + ffn(W["ws13"][0], W["ws2"][0]) + ffn(W["w13"][0], W["w2"][0])
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-12)


def test_silu_form_matches_page_expression():
    """The page writes SiLU-and-mul as g / (1 + exp(-g)) times the up value.
    With Wg = Wu = [I | 0] and Wd = [I; 0], out - residual - shared = silu(x) * x."""
    d = fs.TINY
    I = d.inter
    w13, w2, ws13, ws2 = _embedded_layer(d, shared_up=0.0)
    # Make every routed expert identical with s_e = 1 and no shift.
    eye = np.zeros((I, d.hidden), np.float32)
    eye[np.arange(I), np.arange(I)] = 1.0
    w13n = np.zeros((d.n_experts, 2 * I, d.hidden), np.float32)
    w13n[:, :I] = eye
    w13n[:, I:] = eye
    w2n = np.zeros((d.n_experts, d.hidden, I), np.float32)
    w2n[:, np.arange(I), np.arange(I)] = 1.0
    vals = np.array([0.0, 1.0, -1.0, 2.0, -3.0, 10.0, -10.0, 0.5], np.float32)
    xv = np.zeros((1, d.hidden), np.float32)
    xv[0, :len(vals)] = vals
    x = _bf16(xv)
    r = torch.zeros((1, d.hidden), dtype=torch.bfloat16)
    W = fs.layer_weights(61, d)
    out, _, _ = oracle.moe_bf16(d, x, r, W["wr"], None, _bf16(w13n), _bf16(w2n), ws13, ws2)
    v = vals.astype(np.float64)
    expect = v / (1.0 + np.exp(-v)) * v
    np.testing.assert_allclose(out[0, :len(vals)], expect, rtol=1e-15, atol=1e-300)
    assert out[0, 0] == 0.0
    assert abs(out[0, 1] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


# ---------------------------------------------------------------- NVFP4 codes

E2M1_SPEC = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # OCP MX v1.0, FP4 E2M1 magnitudes


def test_e2m1_all_codes_match_spec_table():
    for c in range(16):
        mag = E2M1_SPEC[c & 7]
        want = -mag if c & 8 else mag
        got = oracle.e2m1(c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want)


def test_e4m3_all_codes_match_library_decode_and_spec_points():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        got = oracle.e4m3(c)
        if np.isnan(lib[c]):
            assert math.isnan(got), c
        else:
            assert got == lib[c], (c, got, lib[c])
    assert oracle.e4m3(0x7E) == 448.0          # largest finite
    assert oracle.e4m3(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3(0x38) == 1.0
    assert math.isnan(oracle.e4m3(0x7F)) and math.isnan(oracle.e4m3(0xFF))


def _random_nvfp4(d, seed, E, S):
    """Random packed NVFP4 tensors with power-of-two tensor scales and block
    scales in [2^-3, 2^3], so every dequantised weight is exact in bf16."""
    rng = np.random.default_rng(seed)
    H, I = d.hidden, d.inter

    def proj(n, rows, K, parts):
        q = rng.integers(0, 256, size=(n, rows, K // 2), dtype=np.uint8)
        sf = rng.integers(0x20, 0x50, size=(n, rows, K // 16), dtype=np.uint8)  # 2^-3 .. 2^3
        ts = (2.0 ** rng.integers(-8, -4, size=(n, parts))).astype(np.float32)
        return q, sf, ts

    nv = {}
    nv["w13_q"], nv["w13_sf"], nv["w13_ts"] = proj(E, 2 * I, H, 2)
    nv["w2_q"], nv["w2_sf"], w2_ts = proj(E, H, I, 1)
    nv["w2_ts"] = w2_ts[:, 0].copy()
    nv["ws13_q"], nv["ws13_sf"], nv["ws13_ts"] = proj(S, 2 * I, H, 2)
    nv["ws2_q"], nv["ws2_sf"], ws2_ts = proj(S, H, I, 1)
    nv["ws2_ts"] = ws2_ts[:, 0].copy()
    return nv


def _dequant_independent(q, sf, ts, split):
    """Dequantise with torch's e4m3 decoder and the spec e2m1 table."""
    table = np.array(E2M1_SPEC + [-v for v in E2M1_SPEC])
    codes = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), np.uint8)
    codes[..., 0::2] = q & 15
    codes[..., 1::2] = q >> 4
    vals = table[codes]
    scale = torch.as_tensor(sf).view(torch.float8_e4m3fn).double().numpy()
    vals = vals * np.repeat(scale, 16, axis=-1)
    rows = q.shape[-2]
    tsv = np.ones(q.shape[:-2] + (rows,))
    if ts.ndim == 2 and ts.shape[-1] == 2:
        tsv[..., :split] = ts[..., 0:1]
        tsv[..., split:] = ts[..., 1:2]
    else:
        tsv[...] = ts.reshape(-1, 1)
    return vals * tsv[..., None]


def test_nvfp4_layer_equals_bf16_layer_on_dequantised_weights():
    d = fs.TINY
    E, S = d.n_experts, d.n_shared
    nv = _random_nvfp4(d, 71, E, S)
    W = fs.layer_weights(72, d)
    x, r = fs.tokens(73, 4, d.hidden)
    I = d.inter
    w13 = _dequant_independent(nv["w13_q"], nv["w13_sf"], nv["w13_ts"], I)
    w2 = _dequant_independent(nv["w2_q"], nv["w2_sf"], nv["w2_ts"], None)
    ws13 = _dequant_independent(nv["ws13_q"], nv["ws13_sf"], nv["ws13_ts"], I)
    ws2 = _dequant_independent(nv["ws2_q"], nv["ws2_sf"], nv["ws2_ts"], None)
    for a in (w13, w2, ws13, ws2):   # exactly representable in bf16
        assert np.array_equal(_f64(_bf16(a)), a)
    o_bf, i_bf, w_bf = oracle.moe_bf16(d, x, r, W["wr"], None, _bf16(w13), _bf16(w2),
                                       _bf16(ws13), _bf16(ws2))
    o_fp, i_fp, w_fp = oracle.moe_nvfp4(d, x, r, W["wr"], None, nv)
    np.testing.assert_array_equal(i_fp, i_bf)
    np.testing.assert_array_equal(w_fp, w_bf)
    np.testing.assert_allclose(o_fp, o_bf, rtol=1e-14, atol=1e-14)


def test_nvfp4_packer_roundtrip_within_format_error():
    """The packer (input preparation, not the method) keeps every weight within
    half an e2m1 step of its block scale."""
    d = fs.TINY
    W = fs.layer_weights(81, d)
    q, sf, ts = fs.pack_nvfp4(W["w13"], row_split=d.inter)
    back = _dequant_independent(q.numpy(), sf.numpy(), ts.numpy(), d.inter)
    ref = _f64(W["w13"])
    blk = np.abs(ref).reshape(*ref.shape[:-1], -1, 16).max(axis=-1)
    err = np.abs(back - ref).reshape(*ref.shape[:-1], -1, 16).max(axis=-1)
    assert np.all(err <= blk * 0.25 + 1e-12)


# ---------------------------------------------------------------- bucketing

def test_bucketing_matches_definition_and_invariants():
    d = fs.FULL
    W = fs.layer_weights(91, fs.Dims(hidden=64, n_experts=256, top_k=6, inter=32))
    x, _ = fs.tokens(92, 128, 64)
    bias = fs.logit_offsets(93, 256)
    idx, _, _ = oracle.route(fs.Dims(hidden=64, n_experts=256, top_k=6, inter=32), x, W["wr"], bias)
    uniq, offsets, pairs = oracle.bucket(idx, 256)
    B, k = idx.shape
    # Definition, written independently: sort (expert, token) keys.
    tok = np.repeat(np.arange(B), k)
    slot = np.tile(np.arange(k), B)
    ex = idx.reshape(-1)
    order = np.lexsort((tok, ex))
    np.testing.assert_array_equal(pairs, (tok * 8 + slot)[order])
    np.testing.assert_array_equal(uniq, np.unique(ex))
    counts = np.diff(offsets)
    assert counts.sum() == B * k and np.all(counts > 0)
    np.testing.assert_array_equal(counts, np.bincount(ex, minlength=256)[uniq])
    assert np.all(np.diff(uniq) > 0)
    seen = set((p >> 3, p & 7) for p in pairs.tolist())
    assert len(seen) == B * k
    for u, e in enumerate(uniq):
        for p in pairs[offsets[u]:offsets[u + 1]]:
            assert idx[p >> 3, p & 7] == e
    assert d.top_k == k


# ---------------------------------------------------------------- rmsnorm

def test_rmsnorm_closed_forms():
    H = 2048
    c = np.array([[2.0] * H, [-0.5] * H], np.float32)
    out = oracle.rmsnorm(_bf16(c), eps=1e-6)
    np.testing.assert_allclose(out[0], 2.0 / math.sqrt(4.0 + 1e-6), rtol=1e-15)
    np.testing.assert_allclose(out[1], -0.5 / math.sqrt(0.25 + 1e-6), rtol=1e-15)
    x, _ = fs.tokens(101, 4, H)
    y = oracle.rmsnorm(x, eps=0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-13)
    y2 = oracle.rmsnorm(_bf16(_f64(x) * 4.0), eps=0.0)   # scale invariance (exact x4 in bf16)
    np.testing.assert_allclose(y2, y, rtol=1e-14)


# ---------------------------------------------------------------- q/k norm + RoPE
# The attention side of a decode step: per-head Q/K RMSNorm with a learned gain,
# then RoPE (element i paired with i + D/2, angle pos * theta^(-2i/D); theta = 0
# on the layers without positional encoding), V unchanged.

def _qkv_rows(seed, B, nq, nkv, D):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((B, (nq + 2 * nkv) * D), generator=g).to(torch.bfloat16)


def test_qk_norm_rope_hand_computed_head():
    # D = 4, one query and one KV head, eps = 0.  q = [1, 0, 0, 0] has RMS 1/2,
    # so it normalises to [2, 0, 0, 0]; k = [0, 1, 0, 0] to [0, 2, 0, 0], times
    # its gain 2 at element 1.  theta = 100: frequencies 1 and 100^(-1/2) = 0.1;
    # at position 3 the pairs (0, 2) and (1, 3) turn by 3 and 0.3 radians.
    qkv = _bf16([[1, 0, 0, 0, 0, 1, 0, 0, 1.5, -2, 3, 0.25]])
    q, k, v = oracle.qk_norm_rope(qkv, _bf16([1, 1, 1, 1]), _bf16([0.5, 2, 1, 1]),
                                  np.array([3], np.int32), 1, 1, 100.0, eps=0.0)
    np.testing.assert_allclose(q[0, 0], [2 * math.cos(3), 0, 2 * math.sin(3), 0], atol=1e-15)
    np.testing.assert_allclose(k[0, 0], [0, 4 * math.cos(0.3), 0, 4 * math.sin(0.3)], atol=1e-15)
    assert v[0, 0].tolist() == [1.5, -2.0, 3.0, 0.25]


def test_qk_norm_eps_sits_under_the_root():
    # every element c = 2^-5 and eps = c^2 = 2^-10: n = c / sqrt(c^2 + eps) = 1/sqrt(2)
    D = 8
    qkv = _bf16([[2.0 ** -5] * (3 * D)])
    q, k, _ = oracle.qk_norm_rope(qkv, _bf16([1] * D), _bf16([1] * D), np.array([0], np.int32),
                                  1, 1, 0.0, eps=2.0 ** -10)
    np.testing.assert_allclose(q, 1 / math.sqrt(2), rtol=1e-15)
    np.testing.assert_allclose(k, 1 / math.sqrt(2), rtol=1e-15)


def test_qk_norm_rope_invariants():
    nq, nkv, D, theta = 32, 4, 128, 1.0e6
    qkv = _qkv_rows(7, 3, nq, nkv, D)
    ones = _bf16([1] * D)
    pos = np.array([0, 5, 200000], np.int32)
    q0, k0, v0 = oracle.qk_norm_rope(qkv, ones, ones, pos, nq, nkv, 0.0, eps=0.0)
    q1, k1, v1 = oracle.qk_norm_rope(qkv, ones, ones, pos, nq, nkv, theta, eps=0.0)
    # unit gain, no eps: every normalised head has RMS 1
    np.testing.assert_allclose(np.mean(q0 * q0, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(np.mean(k0 * k0, axis=-1), 1.0, rtol=1e-13)
    # position 0 turns nothing
    np.testing.assert_allclose(q1[0], q0[0], atol=1e-15)
    np.testing.assert_allclose(k1[0], k0[0], atol=1e-15)
    # a rotation keeps the length of every (i, i + D/2) pair
    h = D // 2
    for a, b in ((q0, q1), (k0, k1)):
        np.testing.assert_allclose(a[..., :h] ** 2 + a[..., h:] ** 2,
                                   b[..., :h] ** 2 + b[..., h:] ** 2, rtol=1e-12, atol=1e-14)
    # V passes unchanged, bit for bit
    raw = _f64(qkv).reshape(3, nq + 2 * nkv, D)
    assert np.array_equal(v0, raw[:, nq + nkv:]) and np.array_equal(v1, v0)
    # gains scale their own heads only
    g2 = _bf16([2] * D)
    q2, k2, _ = oracle.qk_norm_rope(qkv, g2, ones, pos, nq, nkv, theta, eps=0.0)
    np.testing.assert_allclose(q2, 2 * q1, rtol=1e-15)
    np.testing.assert_allclose(k2, k1, rtol=0)


def test_rope_scores_depend_on_relative_position_only():
    # a query at position m against a key at position n: q.k is the same for
    # (m, n) and (m + s, n + s), per query head and KV head
    nq, nkv, D, theta = 4, 2, 128, 1.0e6
    qkv = _qkv_rows(11, 1, nq, nkv, D).repeat(4, 1)
    ones = _bf16([1] * D)
    pos = np.array([10, 3, 1010, 1003], np.int32)
    q, k, _ = oracle.qk_norm_rope(qkv, ones, ones, pos, nq, nkv, theta, eps=1e-6)
    s_near = np.einsum("hd,gd->hg", q[0], k[1])
    s_far = np.einsum("hd,gd->hg", q[2], k[3])
    np.testing.assert_allclose(s_far, s_near, rtol=1e-9, atol=1e-9)
    # and it does change with the distance
    q5, k5, _ = oracle.qk_norm_rope(qkv, ones, ones, np.array([10, 4, 0, 0], np.int32), nq, nkv,
                                    theta, eps=1e-6)
    assert np.max(np.abs(np.einsum("hd,gd->hg", q5[0], k5[1]) - s_near)) > 1e-3


def test_margin_helper_on_planted_ties():
    L = np.array([[3.0, 1.0, 2.0, 2.0, 0.0]])
    assert topk_margin(L, 2)[0] == 0.0 and topk_margin(L, 1)[0] == 1.0
