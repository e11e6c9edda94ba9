"""fp64 CPU oracle of the Flint decode MoE layer -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU legs (the
cpu_baseline record and the `--impl reference` arm) may import this package.  It wraps the plain C implementation in
oracle/flint_moe_ref.c (built by oracle/build.py) and takes host tensors
(torch CPU tensors or NumPy arrays).  It shares nothing with the CUDA path.

Parity pins for every function here are in tests/test_oracle_pins.py; the
separately written dense NumPy brute force is oracle/brute.py.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int


class _Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("offset_mode", ctypes.c_int32)]


def load(path: str) -> ctypes.CDLL:
    """Loads an oracle library build (the tests' mutation check loads builds of
    altered copies of the source this way)."""
    L = ctypes.CDLL(path)
    L.ref_e2m1.restype = ctypes.c_double
    L.ref_e2m1.argtypes = [ctypes.c_uint8]
    L.ref_e4m3.restype = ctypes.c_double
    L.ref_e4m3.argtypes = [ctypes.c_uint8]
    L.ref_route.restype = _I
    L.ref_route.argtypes = [_P, _I, _P, _P, _P, _P, _P, _P]
    L.ref_moe_bf16.restype = _I
    L.ref_moe_bf16.argtypes = [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P]
    L.ref_moe_bf16_given_routing.restype = _I
    L.ref_moe_bf16_given_routing.argtypes = [_P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]
    L.ref_moe_nvfp4.restype = _I
    L.ref_moe_nvfp4.argtypes = [_P, _I, _P, _P, _P, _P] + [_P] * 12 + [_I, _P, _P, _P]
    L.ref_moe_nvfp4_given_routing.restype = _I
    L.ref_moe_nvfp4_given_routing.argtypes = [_P, _I, _P, _P, _P, _P] + [_P] * 12 + [_I, _P]
    L.ref_bucket.restype = _I
    L.ref_bucket.argtypes = [_I, _I, _I, _P, _P, _P, _P]
    L.ref_rmsnorm.restype = None
    L.ref_rmsnorm.argtypes = [_I, _I, _P, ctypes.c_double, _P]
    L.ref_qk_norm_rope.restype = None
    L.ref_qk_norm_rope.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, ctypes.c_double,
                                   ctypes.c_double, _P, _P, _P]
    L.ref_max_threads.restype = _I
    L.ref_max_threads.argtypes = []
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(_build.build())
    return _lib


def _np(a, dtype=None):
    """Host array view: torch CPU tensors are viewed without copy (bf16 as uint16)."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.device.type == "cpu", "the oracle takes host tensors"
            a = a.contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16)
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype is not None:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _dims(d):
    return _Dims(d.hidden, d.n_experts, d.top_k, d.inter, d.n_shared,
                 getattr(d, "offset_mode", 0))


def e2m1(code: int) -> float:
    return lib().ref_e2m1(int(code) & 0xFF)


def e4m3(code: int) -> float:
    return lib().ref_e4m3(int(code) & 0xFF)


def route(dims, x, wr, bias=None):
    """Returns (idx int32 [B,k], w f64 [B,k], logits f64 [B,E])."""
    x = _np(x, np.uint16); wr = _np(wr, np.uint16)
    b = _np(bias, np.float32)
    B = x.shape[0]
    idx = np.zeros((B, dims.top_k), np.int32)
    w = np.zeros((B, dims.top_k), np.float64)
    logits = np.zeros((B, dims.n_experts), np.float64)
    d = _dims(dims)
    rc = lib().ref_route(ctypes.byref(d), B, _ptr(x), _ptr(wr), _ptr(b), _ptr(logits),
                         _ptr(idx), _ptr(w))
    assert rc == 0
    return idx, w, logits


def moe_bf16(dims, x, residual, wr, bias, w13, w2, ws13, ws2, nthreads=0):
    """Whole layer.  Returns (out f64 [B,H], idx int32 [B,k], w f64 [B,k])."""
    x = _np(x, np.uint16); residual = _np(residual, np.uint16); wr = _np(wr, np.uint16)
    b = _np(bias, np.float32)
    w13 = _np(w13, np.uint16); w2 = _np(w2, np.uint16)
    ws13 = _np(ws13, np.uint16); ws2 = _np(ws2, np.uint16)
    B = x.shape[0]
    out = np.zeros((B, dims.hidden), np.float64)
    idx = np.zeros((B, dims.top_k), np.int32)
    w = np.zeros((B, dims.top_k), np.float64)
    d = _dims(dims)
    rc = lib().ref_moe_bf16(ctypes.byref(d), B, _ptr(x), _ptr(residual), _ptr(wr), _ptr(b),
                            _ptr(w13), _ptr(w2), _ptr(ws13), _ptr(ws2), int(nthreads),
                            _ptr(out), _ptr(idx), _ptr(w))
    assert rc == 0
    return out, idx, w


def moe_bf16_given_routing(dims, x, residual, idx, w, w13, w2, ws13, ws2, nthreads=0):
    """Expert part for the given routing.  Returns out f64 [B,H]."""
    x = _np(x, np.uint16); residual = _np(residual, np.uint16)
    idx = _np(idx, np.int32); w = _np(w, np.float64)
    w13 = _np(w13, np.uint16); w2 = _np(w2, np.uint16)
    ws13 = _np(ws13, np.uint16); ws2 = _np(ws2, np.uint16)
    B = x.shape[0]
    out = np.zeros((B, dims.hidden), np.float64)
    d = _dims(dims)
    rc = lib().ref_moe_bf16_given_routing(ctypes.byref(d), B, _ptr(x), _ptr(residual),
                                          _ptr(idx), _ptr(w), _ptr(w13), _ptr(w2),
                                          _ptr(ws13), _ptr(ws2), int(nthreads), _ptr(out))
    assert rc == 0
    return out


def _fp4_args(nv):
    keys = ["w13_q", "w13_sf", "w13_ts", "w2_q", "w2_sf", "w2_ts",
            "ws13_q", "ws13_sf", "ws13_ts", "ws2_q", "ws2_sf", "ws2_ts"]
    arrs = [_np(nv[k], np.float32 if k.endswith("_ts") else np.uint8) for k in keys]
    return arrs, [_ptr(a) for a in arrs]


def moe_nvfp4(dims, x, residual, wr, bias, nv, nthreads=0):
    """NVFP4 layer; nv holds the twelve packed tensors.  Returns (out, idx, w)."""
    x = _np(x, np.uint16); residual = _np(residual, np.uint16); wr = _np(wr, np.uint16)
    b = _np(bias, np.float32)
    keep, ptrs = _fp4_args(nv)
    B = x.shape[0]
    out = np.zeros((B, dims.hidden), np.float64)
    idx = np.zeros((B, dims.top_k), np.int32)
    w = np.zeros((B, dims.top_k), np.float64)
    d = _dims(dims)
    rc = lib().ref_moe_nvfp4(ctypes.byref(d), B, _ptr(x), _ptr(residual), _ptr(wr), _ptr(b),
                             *ptrs, int(nthreads), _ptr(out), _ptr(idx), _ptr(w))
    assert rc == 0
    del keep
    return out, idx, w


def moe_nvfp4_given_routing(dims, x, residual, idx, w, nv, nthreads=0):
    x = _np(x, np.uint16); residual = _np(residual, np.uint16)
    idx = _np(idx, np.int32); w = _np(w, np.float64)
    keep, ptrs = _fp4_args(nv)
    B = x.shape[0]
    out = np.zeros((B, dims.hidden), np.float64)
    d = _dims(dims)
    rc = lib().ref_moe_nvfp4_given_routing(ctypes.byref(d), B, _ptr(x), _ptr(residual),
                                           _ptr(idx), _ptr(w), *ptrs, int(nthreads), _ptr(out))
    assert rc == 0
    del keep
    return out


def bucket(idx, n_experts):
    """Returns (uniq [U], offsets [U+1], pairs [B*k]) as int32 arrays."""
    idx = _np(idx, np.int32)
    B, k = idx.shape
    uniq = np.zeros((n_experts,), np.int32)
    offsets = np.zeros((n_experts + 1,), np.int32)
    pairs = np.zeros((B * k,), np.int32)
    U = lib().ref_bucket(B, k, n_experts, _ptr(idx), _ptr(uniq), _ptr(offsets), _ptr(pairs))
    return uniq[:U].copy(), offsets[:U + 1].copy(), pairs


def rmsnorm(x, eps=1e-6):
    x = _np(x, np.uint16)
    B, H = x.shape
    out = np.zeros((B, H), np.float64)
    lib().ref_rmsnorm(B, H, _ptr(x), float(eps), _ptr(out))
    return out


def qk_norm_rope(qkv, q_norm, k_norm, positions, n_q_heads, n_kv_heads, theta, eps=1e-6):
    """Per-head Q/K RMSNorm (learned gain) and RoPE (rotate-half, theta = 0:
    none) of a decode step's projection rows qkv [B, (nq + 2 nkv) * D] (bf16);
    returns (q [B, nq, D], k [B, nkv, D], v [B, nkv, D]) in fp64."""
    qkv = _np(qkv, np.uint16)
    qn, kn = _np(q_norm, np.uint16), _np(k_norm, np.uint16)
    pos = _np(positions, np.int32)
    B = qkv.shape[0]
    D = qn.shape[0]
    assert qkv.shape[1] == (n_q_heads + 2 * n_kv_heads) * D and kn.shape[0] == D and pos.shape == (B,)
    q = np.zeros((B, n_q_heads, D), np.float64)
    k = np.zeros((B, n_kv_heads, D), np.float64)
    v = np.zeros((B, n_kv_heads, D), np.float64)
    lib().ref_qk_norm_rope(B, n_q_heads, n_kv_heads, D, _ptr(qkv), _ptr(qn), _ptr(kn), _ptr(pos),
                           float(theta), float(eps), _ptr(q), _ptr(k), _ptr(v))
    return q, k, v


def max_threads() -> int:
    return lib().ref_max_threads()
