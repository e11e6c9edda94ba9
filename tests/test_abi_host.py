"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments on the host
before any CUDA call."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import moe_decode_sigmoid_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from moe_decode_sigmoid_gb300 import build
    build.build()
    return m.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "flint_moe.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const char\*|size_t|flint_status)\s+(flint_\w+)\s*\(",
                                 src, re.M)))


def test_header_declarations_match_binding_list():
    assert sorted(m.EXPORTS) == _declared()


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code, name in [(0, "FLINT_OK"), (1, "FLINT_ERR_INVALID_ARG"), (2, "FLINT_ERR_UNSUPPORTED"),
                       (3, "FLINT_ERR_WORKSPACE"), (4, "FLINT_ERR_CUDA"),
                       (5, "FLINT_ERR_DEVICE_TIMEOUT")]:
        assert m.status_string(code) == name
    assert m.status_string(99) == "FLINT_ERR_UNKNOWN"


def test_workspace_bytes(L):
    a = m.flint_moe_workspace_bytes(1)
    b = m.flint_moe_workspace_bytes(128)
    c = m.flint_moe_workspace_bytes(256)
    assert 0 < a < b < c
    assert (b - a) == 127 * 7 * (512 + 2048) * 4   # only the h and y rows grow with the batch
    assert a % 256 == 0 and b % 256 == 0
    assert m.flint_moe_workspace_bytes(0) == 0
    assert m.flint_moe_workspace_bytes(257) == 0
    bad = m.Dims(2048, 256, 6, 256, 1)
    assert m.flint_moe_workspace_bytes(8, bad) == 0
    assert m.flint_moe_workspace_bytes(8, m.SELECT_DIMS) == m.flint_moe_workspace_bytes(8)
    assert m.flint_moe_workspace_bytes(8, m.Dims(2048, 256, 6, 512, 1, 2)) == 0  # no such mode


# Fake device addresses: validation fails before anything is dereferenced.
A = 0x100000
WS = 0x7000000


def _decode(L, dims=None, batch=1, x=A, res=A + 0x10000, wr=A, bias=None, w13=A, w2=A, ws13=A,
            ws2=A, out=A + 0x20000, idx=None, w=None, ws=WS, wsb=None):
    if wsb is None:
        wsb = m.flint_moe_workspace_bytes(max(1, min(batch, 256)))
    d = ctypes.byref(dims if dims is not None else m.FULL_DIMS)
    return L.flint_moe_decode_bf16(d, batch, x, res, wr, bias, w13, w2, ws13, ws2, out, idx, w,
                                   ws, wsb, None)


def test_decode_rejects_bad_arguments_before_launch(L):
    assert _decode(L, dims=m.Dims(2048, 128, 6, 512, 1)) == m.FLINT_ERR_UNSUPPORTED
    assert _decode(L, dims=m.Dims(4096, 256, 6, 512, 1)) == m.FLINT_ERR_UNSUPPORTED
    assert _decode(L, dims=m.Dims(2048, 256, 8, 512, 1)) == m.FLINT_ERR_UNSUPPORTED
    assert _decode(L, batch=0) == m.FLINT_ERR_INVALID_ARG
    assert _decode(L, batch=257, wsb=1 << 30) == m.FLINT_ERR_INVALID_ARG
    assert _decode(L, x=None) == m.FLINT_ERR_INVALID_ARG
    assert _decode(L, x=A + 2) == m.FLINT_ERR_INVALID_ARG            # misaligned
    assert _decode(L, w13=None) == m.FLINT_ERR_INVALID_ARG
    assert _decode(L, bias=A + 2) == m.FLINT_ERR_INVALID_ARG         # misaligned optional
    assert _decode(L, idx=A + 6) == m.FLINT_ERR_INVALID_ARG
    assert _decode(L, ws=None) == m.FLINT_ERR_WORKSPACE
    assert _decode(L, ws=WS + 8) == m.FLINT_ERR_WORKSPACE
    assert _decode(L, batch=8, wsb=m.flint_moe_workspace_bytes(4)) == m.FLINT_ERR_WORKSPACE
    # out overlapping x, or partially overlapping residual, or the workspace
    assert _decode(L, out=A + 0x100) == m.FLINT_ERR_INVALID_ARG
    assert _decode(L, res=A + 0x20000 + 0x10) == m.FLINT_ERR_INVALID_ARG
    assert _decode(L, out=WS + 0x100) == m.FLINT_ERR_INVALID_ARG
    d = ctypes.byref(m.FULL_DIMS)
    assert L.flint_moe_decode_bf16(None, 1, A, A, A, None, A, A, A, A, A, None, None, WS,
                                   1 << 30, None) == m.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_decode_nvfp4_w4a16(d, 1, A, A + 0x10000, A, None, *([A] * 11), None,
                                          A + 0x20000, None, None, WS, 1 << 30,
                                          None) == m.FLINT_ERR_INVALID_ARG


def test_decode_prenorm_rejects_bad_arguments_before_launch(L):
    f = L.flint_moe_decode_bf16_prenorm
    res, out = A + 0x10000, A + 0x20000

    def call(dims=m.FULL_DIMS, batch=1, res_=res, eps=1e-6, wr=A, w13=A, out_=out, ws=WS,
             wsb=None):
        if wsb is None:
            wsb = m.flint_moe_workspace_bytes(max(1, min(batch, 256)))
        return f(ctypes.byref(dims), batch, res_, eps, wr, None, w13, A, A, A, out_, None, None,
                 ws, wsb, None)

    assert call(dims=m.Dims(2048, 128, 6, 512, 1)) == m.FLINT_ERR_UNSUPPORTED
    assert call(batch=0) == m.FLINT_ERR_INVALID_ARG
    assert call(res_=None) == m.FLINT_ERR_INVALID_ARG
    assert call(res_=res + 2) == m.FLINT_ERR_INVALID_ARG             # misaligned
    assert call(wr=None) == m.FLINT_ERR_INVALID_ARG
    assert call(w13=None) == m.FLINT_ERR_INVALID_ARG
    assert call(eps=-1e-6) == m.FLINT_ERR_INVALID_ARG
    assert call(eps=float("nan")) == m.FLINT_ERR_INVALID_ARG
    assert call(ws=None) == m.FLINT_ERR_WORKSPACE
    assert call(batch=8, wsb=m.flint_moe_workspace_bytes(4)) == m.FLINT_ERR_WORKSPACE
    # out partially overlapping the residual, or the workspace; the residual
    # inside the workspace (the norm may be written there)
    assert call(out_=res + 0x100) == m.FLINT_ERR_INVALID_ARG
    assert call(out_=WS + 0x100) == m.FLINT_ERR_INVALID_ARG
    assert call(res_=WS + 0x1000) == m.FLINT_ERR_INVALID_ARG
    assert f(None, 1, res, 1e-6, A, None, A, A, A, A, out, None, None, WS, 1 << 30,
             None) == m.FLINT_ERR_INVALID_ARG


def test_route_bucket_rmsnorm_reject_bad_arguments(L):
    d = ctypes.byref(m.FULL_DIMS)
    wsb = m.flint_moe_workspace_bytes(4)
    assert L.flint_moe_route(d, 4, None, A, None, A, A, WS, wsb, None) == m.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_route(d, 4, A, A, None, A, A, WS, 16, None) == m.FLINT_ERR_WORKSPACE
    assert L.flint_moe_bucket(d, 4, A, A, A, None, A, WS, wsb, None) == m.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_rmsnorm_bf16(d, 4, A, A + 0x100, 1e-6, None) == m.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_rmsnorm_bf16(d, 4, A, A + 0x10000, -1.0, None) == m.FLINT_ERR_INVALID_ARG
    assert L.flint_moe_workspace_init(None, wsb, 0, None) == m.FLINT_ERR_WORKSPACE
    assert L.flint_moe_workspace_init(WS, 64, 0, None) == m.FLINT_ERR_WORKSPACE
    assert L.flint_moe_debug_arm_stall(None, wsb, None) == m.FLINT_ERR_WORKSPACE


def test_qk_norm_rope_kv_rejects_bad_arguments(L):
    f = L.flint_qk_norm_rope_kv_bf16
    d = ctypes.byref(m.ATTN_DIMS)
    row = (m.N_Q_HEADS + 2 * m.N_KV_HEADS) * m.HEAD_DIM
    B, slots = 4, 64
    qkv, qn, kn, pos, sl = A, A + 0x10000, A + 0x10100, A + 0x10200, A + 0x10300
    q, kc, vc = A + 0x20000, A + 0x40000, A + 0x60000

    def call(dims=d, batch=B, qkv_=qkv, theta=1.0e6, eps=1e-6, q_=q, kc_=kc, vc_=vc, n=slots,
             pos_=pos):
        return f(dims, batch, qkv_, qn, kn, pos_, sl, theta, eps, q_, kc_, vc_, n, None)

    assert call(dims=None) == m.FLINT_ERR_INVALID_ARG
    assert call(dims=ctypes.byref(m.AttnDims(32, 8, 128))) == m.FLINT_ERR_UNSUPPORTED
    assert call(dims=ctypes.byref(m.AttnDims(32, 4, 64))) == m.FLINT_ERR_UNSUPPORTED
    assert call(batch=0) == m.FLINT_ERR_INVALID_ARG
    assert call(batch=m.MAX_BATCH + 1) == m.FLINT_ERR_INVALID_ARG
    assert call(qkv_=qkv + 2) == m.FLINT_ERR_INVALID_ARG          # bf16 rows: 16-byte alignment
    assert call(pos_=pos + 2) == m.FLINT_ERR_INVALID_ARG          # int32 vectors: 4 bytes
    assert call(qkv_=None) == m.FLINT_ERR_INVALID_ARG
    assert call(theta=-1.0) == m.FLINT_ERR_INVALID_ARG
    assert call(theta=float("nan")) == m.FLINT_ERR_INVALID_ARG
    assert call(eps=float("inf")) == m.FLINT_ERR_INVALID_ARG
    assert call(n=0) == m.FLINT_ERR_INVALID_ARG
    assert call(q_=qkv + B * row * 2 - 16) == m.FLINT_ERR_INVALID_ARG       # q_out overlaps qkv
    assert call(vc_=kc + slots * 4 * 128 * 2 - 16) == m.FLINT_ERR_INVALID_ARG  # caches overlap


def test_binding_checks_what_the_c_call_cannot():
    """The C calls take bare pointers: the binding rejects a tensor whose dtype,
    shape, layout or device differs from the header's layout, naming it, before
    anything is launched (a plain int passes as a raw device pointer)."""
    import torch
    cpu = torch.device("cpu")
    f = "flint_moe_decode_bf16"
    x = torch.zeros((4, 2048), dtype=torch.bfloat16)
    assert m._arg(f, "x", x, torch.bfloat16, (4, 2048), cpu) == x.data_ptr()
    assert m._arg(f, "bias", None, torch.float32, (256,), cpu, optional=True) is None
    assert m._arg(f, "w", 0x1000, torch.bfloat16, (1,), cpu) == 0x1000
    bad = {
        "dtype": x.float(),
        "shape": torch.zeros((4, 1024), dtype=torch.bfloat16),
        "layout": torch.zeros((2048, 4), dtype=torch.bfloat16).t(),
        "device": x.to("meta"),
        "type": [0] * 8,
    }
    for why, t in bad.items():
        with pytest.raises(m.FlintError) as e:
            m._arg(f, "x", t, torch.bfloat16, (4, 2048), cpu)
        assert e.value.status == m.FLINT_ERR_INVALID_ARG and "x must be" in str(e.value), why
    with pytest.raises(m.FlintError):
        m._arg(f, "w13", None, torch.bfloat16, (256, 1024, 2048), cpu)
    with pytest.raises(m.FlintError) as e:
        m._arg(f, "pairs", torch.zeros(5, dtype=torch.int32), torch.int32, None, cpu, min_numel=6)
    assert "pairs" in str(e.value)
    # activations must live on a GPU: a host tensor is refused before the call
    with pytest.raises(m.FlintError) as e:
        m.flint_moe_decode_bf16(x, x, None, None, None, None, None, None, x, None)
    assert "CUDA" in str(e.value)
    with pytest.raises(m.FlintError):
        m.flint_moe_rmsnorm_bf16(torch.zeros((4, 100), dtype=torch.bfloat16), x)


def test_binding_refuses_a_host_workspace():
    import torch
    ws = torch.zeros(m.flint_moe_workspace_bytes(1), dtype=torch.uint8)
    for call in (m.flint_moe_workspace_init, m.flint_moe_get_device_status,
                 m.flint_moe_debug_arm_stall):
        with pytest.raises(m.FlintError) as e:
            call(ws)
        assert "workspace must be" in str(e.value) and "CUDA" in str(e.value)
