"""Python binding of the Flint decode-MoE C ABI (include/flint_moe.h).

Argument marshalling only: every function below forwards torch tensors' device
pointers and the current CUDA stream to the same-named C entry point in
lib/libflint_moe.so; every step of the layer runs in that library's CUDA
kernels.  There is no fallback: if the library is missing or fails to load,
importing the binding's functions raises.

Build the library with `python -m moe_decode_sigmoid_gb300.build` (or
`__graft_entry__.build()`).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libflint_moe.so")

FLINT_OK = 0
FLINT_ERR_INVALID_ARG = 1
FLINT_ERR_UNSUPPORTED = 2
FLINT_ERR_WORKSPACE = 3
FLINT_ERR_CUDA = 4
FLINT_ERR_DEVICE_TIMEOUT = 5
MAX_BATCH = 256

HIDDEN, N_EXPERTS, TOP_K, INTER, N_SHARED = 2048, 256, 6, 512, 1

# Every symbol include/flint_moe.h declares.
EXPORTS = (
    "flint_status_string", "flint_moe_workspace_bytes", "flint_moe_workspace_init",
    "flint_moe_get_device_status", "flint_moe_route", "flint_moe_bucket",
    "flint_moe_decode_bf16", "flint_moe_decode_nvfp4_w4a16", "flint_moe_rmsnorm_bf16",
    "flint_moe_debug_arm_stall", "flint_moe_gateup_bf16", "flint_moe_down_bf16",
    "flint_moe_decode_bf16_noalloc",
)
NOALLOC_MAX_BATCH = 8


class FlintError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_shared", ctypes.c_int32)]


FULL_DIMS = Dims(HIDDEN, N_EXPERTS, TOP_K, INTER, N_SHARED)

_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """Loads the CUDA library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libflint_moe.so not built (%s); run moe_decode_sigmoid_gb300/build.py"
                          % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    L.flint_status_string.restype = ctypes.c_char_p
    L.flint_status_string.argtypes = [ctypes.c_int]
    L.flint_moe_workspace_bytes.restype = _SZ
    L.flint_moe_workspace_bytes.argtypes = [_P, _I32]
    L.flint_moe_workspace_init.restype = ctypes.c_int
    L.flint_moe_workspace_init.argtypes = [_P, _SZ, ctypes.c_uint64, _P]
    L.flint_moe_get_device_status.restype = ctypes.c_int
    L.flint_moe_get_device_status.argtypes = [_P, _P]
    L.flint_moe_debug_arm_stall.restype = ctypes.c_int
    L.flint_moe_debug_arm_stall.argtypes = [_P, _SZ, _P]
    L.flint_moe_route.restype = ctypes.c_int
    L.flint_moe_route.argtypes = [_P, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.flint_moe_bucket.restype = ctypes.c_int
    L.flint_moe_bucket.argtypes = [_P, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]
    L.flint_moe_decode_bf16.restype = ctypes.c_int
    L.flint_moe_decode_bf16.argtypes = [_P, _I32] + [_P] * 12 + [_SZ, _P]
    L.flint_moe_decode_nvfp4_w4a16.restype = ctypes.c_int
    L.flint_moe_decode_nvfp4_w4a16.argtypes = [_P, _I32] + [_P] * 20 + [_SZ, _P]
    L.flint_moe_gateup_bf16.restype = ctypes.c_int
    L.flint_moe_gateup_bf16.argtypes = [_P, _I32, _P, _P, _P, _P, _SZ, _P]
    L.flint_moe_down_bf16.restype = ctypes.c_int
    L.flint_moe_down_bf16.argtypes = [_P, _I32, _P, _P, _P, _P, _P, _SZ, _P]
    L.flint_moe_rmsnorm_bf16.restype = ctypes.c_int
    L.flint_moe_rmsnorm_bf16.argtypes = [_P, _I32, _P, _P, ctypes.c_float, _P]
    L.flint_moe_decode_bf16_noalloc.restype = ctypes.c_int
    L.flint_moe_decode_bf16_noalloc.argtypes = [_P, _I32] + [_P] * 13
    _lib = L
    return L


def status_string(status: int) -> str:
    try:
        return lib().flint_status_string(int(status)).decode()
    except ImportError:
        return "status %d" % status


def _check(status: int, where: str) -> None:
    if status != FLINT_OK:
        raise FlintError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dims(dims):
    return ctypes.byref(FULL_DIMS if dims is None else dims)


# ---------------------------------------------------------------- entry points

def flint_moe_workspace_bytes(max_batch: int, dims: Dims | None = None) -> int:
    return int(lib().flint_moe_workspace_bytes(_dims(dims), int(max_batch)))


def flint_moe_workspace_init(workspace: torch.Tensor, wait_limit_ns: int = 0, stream=None):
    _check(lib().flint_moe_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                          int(wait_limit_ns), _stream(stream)),
           "flint_moe_workspace_init")


def flint_moe_get_device_status(workspace: torch.Tensor, stream=None) -> int:
    return int(lib().flint_moe_get_device_status(_ptr(workspace), _stream(stream)))


def flint_moe_debug_arm_stall(workspace: torch.Tensor, stream=None):
    _check(lib().flint_moe_debug_arm_stall(_ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _stream(stream)), "flint_moe_debug_arm_stall")


def _ws(workspace):
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def flint_moe_route(x, w_router, logit_bias, topk_idx, topk_w, workspace, stream=None,
                    dims: Dims | None = None):
    wp, wb = _ws(workspace)
    _check(lib().flint_moe_route(_dims(dims), x.shape[0], _ptr(x), _ptr(w_router), _ptr(logit_bias),
                                 _ptr(topk_idx), _ptr(topk_w), wp, wb, _stream(stream)),
           "flint_moe_route")


def flint_moe_bucket(topk_idx, uniq, offsets, pairs, n_uniq, workspace, stream=None,
                     dims: Dims | None = None):
    wp, wb = _ws(workspace)
    _check(lib().flint_moe_bucket(_dims(dims), topk_idx.shape[0], _ptr(topk_idx), _ptr(uniq),
                                  _ptr(offsets), _ptr(pairs), _ptr(n_uniq), wp, wb,
                                  _stream(stream)), "flint_moe_bucket")


def flint_moe_decode_bf16(x, residual, w_router, logit_bias, w13, w2, ws13, ws2, out, workspace,
                          topk_idx_out=None, topk_w_out=None, stream=None,
                          dims: Dims | None = None):
    wp, wb = _ws(workspace)
    _check(lib().flint_moe_decode_bf16(_dims(dims), x.shape[0], _ptr(x), _ptr(residual),
                                       _ptr(w_router), _ptr(logit_bias), _ptr(w13), _ptr(w2),
                                       _ptr(ws13), _ptr(ws2), _ptr(out), _ptr(topk_idx_out),
                                       _ptr(topk_w_out), wp, wb, _stream(stream)),
           "flint_moe_decode_bf16")


def flint_moe_decode_bf16_noalloc(x, residual, w_router, logit_bias, w13, w2, ws13, ws2, out,
                                  topk_idx_out=None, topk_w_out=None, device_status_out=None,
                                  stream=None, dims: Dims | None = None):
    """flint_moe_decode_bf16 without a workspace (the library's static device
    array instead; batch <= NOALLOC_MAX_BATCH).  For callers that cannot
    allocate device memory; calls whose GPU work overlaps race."""
    _check(lib().flint_moe_decode_bf16_noalloc(
        _dims(dims), x.shape[0], _ptr(x), _ptr(residual), _ptr(w_router), _ptr(logit_bias),
        _ptr(w13), _ptr(w2), _ptr(ws13), _ptr(ws2), _ptr(out), _ptr(topk_idx_out),
        _ptr(topk_w_out), _ptr(device_status_out), _stream(stream)),
        "flint_moe_decode_bf16_noalloc")


def flint_moe_gateup_bf16(x, w13, ws13, workspace, stream=None, dims: Dims | None = None):
    wp, wb = _ws(workspace)
    _check(lib().flint_moe_gateup_bf16(_dims(dims), x.shape[0], _ptr(x), _ptr(w13), _ptr(ws13),
                                       wp, wb, _stream(stream)), "flint_moe_gateup_bf16")


def flint_moe_down_bf16(residual, w2, ws2, out, workspace, stream=None, dims: Dims | None = None):
    wp, wb = _ws(workspace)
    _check(lib().flint_moe_down_bf16(_dims(dims), residual.shape[0], _ptr(residual), _ptr(w2),
                                     _ptr(ws2), _ptr(out), wp, wb, _stream(stream)),
           "flint_moe_down_bf16")


NVFP4_KEYS = ("w13_q", "w13_sf", "w13_ts", "w2_q", "w2_sf", "w2_ts",
              "ws13_q", "ws13_sf", "ws13_ts", "ws2_q", "ws2_sf", "ws2_ts")


def flint_moe_decode_nvfp4_w4a16(x, residual, w_router, logit_bias, nv: dict, out, workspace,
                                 topk_idx_out=None, topk_w_out=None, stream=None,
                                 dims: Dims | None = None):
    """nv holds the twelve packed tensors named in NVFP4_KEYS."""
    wp, wb = _ws(workspace)
    _check(lib().flint_moe_decode_nvfp4_w4a16(
        _dims(dims), x.shape[0], _ptr(x), _ptr(residual), _ptr(w_router), _ptr(logit_bias),
        *[_ptr(nv[k]) for k in NVFP4_KEYS], _ptr(out), _ptr(topk_idx_out), _ptr(topk_w_out),
        wp, wb, _stream(stream)), "flint_moe_decode_nvfp4_w4a16")


def flint_moe_rmsnorm_bf16(inp, out, eps: float = 1e-6, stream=None, dims: Dims | None = None):
    _check(lib().flint_moe_rmsnorm_bf16(_dims(dims), inp.shape[0], _ptr(inp), _ptr(out),
                                        float(eps), _stream(stream)), "flint_moe_rmsnorm_bf16")


# ---------------------------------------------------------------- conveniences

def new_workspace(max_batch: int, device="cuda", wait_limit_ns: int = 0) -> torch.Tensor:
    """Allocates (through torch) and initialises a workspace for max_batch tokens."""
    n = flint_moe_workspace_bytes(max_batch)
    if n == 0:
        raise FlintError(FLINT_ERR_INVALID_ARG, "new_workspace")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    flint_moe_workspace_init(ws, wait_limit_ns)
    return ws
