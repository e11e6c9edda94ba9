"""Python binding of the Flint decode-MoE C ABI (include/flint_moe.h).

Argument marshalling only: every function below forwards torch tensors' device
pointers and the current CUDA stream to the same-named C entry point in
lib/libflint_moe.so; every step of the layer runs in that library's CUDA
kernels.  There is no fallback: if the library is missing or fails to load,
importing the binding's functions raises.

The C entry points take bare pointers, so the binding checks what they cannot:
each tensor's dtype, shape (as include/flint_moe.h lays it out), contiguity and
device (all on the activations' CUDA device), raising FlintError with
FLINT_ERR_INVALID_ARG before anything is launched.  A plain int is taken as a
raw device pointer the caller vouches for.

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
    "flint_moe_decode_bf16_noalloc", "flint_qk_norm_rope_kv_bf16",
    "flint_moe_decode_bf16_prenorm",
)
NOALLOC_MAX_BATCH = 8
# Batches up to which flint_moe_decode_bf16_prenorm is one launch (the
# persistent kernel normalises its input itself); 5..8 tokens take the RMSNorm
# kernel + the persistent kernel, larger batches the RMSNorm + three kernels.
PRENORM_FUSED_MAX_BATCH = 4


class FlintError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


FLINT_OFFSET_LOGIT = 0    # offsets move ranking and weights (default)
FLINT_OFFSET_SELECT = 1   # offsets steer the ranking only


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("offset_mode", ctypes.c_int32)]


FULL_DIMS = Dims(HIDDEN, N_EXPERTS, TOP_K, INTER, N_SHARED, FLINT_OFFSET_LOGIT)
SELECT_DIMS = Dims(HIDDEN, N_EXPERTS, TOP_K, INTER, N_SHARED, FLINT_OFFSET_SELECT)

# The attention side of a decode step (flint_qk_norm_rope_kv_bf16).
N_Q_HEADS, N_KV_HEADS, HEAD_DIM = 32, 4, 128


class AttnDims(ctypes.Structure):
    _fields_ = [("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


ATTN_DIMS = AttnDims(N_Q_HEADS, N_KV_HEADS, HEAD_DIM)

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
    L.flint_moe_decode_bf16_prenorm.restype = ctypes.c_int
    L.flint_moe_decode_bf16_prenorm.argtypes = ([_P, _I32, _P, ctypes.c_float] + [_P] * 10 +
                                                [_SZ, _P])
    L.flint_moe_decode_bf16_noalloc.restype = ctypes.c_int
    L.flint_moe_decode_bf16_noalloc.argtypes = [_P, _I32] + [_P] * 13
    L.flint_qk_norm_rope_kv_bf16.restype = ctypes.c_int
    L.flint_qk_norm_rope_kv_bf16.argtypes = ([_P, _I32] + [_P] * 5 + [ctypes.c_float] * 2 +
                                             [_P] * 3 + [ctypes.c_int64, _P])
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


_BF16, _F32, _I32T, _U8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def _bad(where, name, what, t):
    got = ("%s %s%s on %s" % (t.dtype, tuple(t.shape), "" if t.is_contiguous() else
                              " (not contiguous)", t.device)
           if isinstance(t, torch.Tensor) else type(t).__name__)
    raise FlintError(FLINT_ERR_INVALID_ARG, "%s: %s must be %s, got %s" % (where, name, what, got))


def _arg(where, name, t, dtype, shape, dev, optional=False, min_numel=None):
    """Device pointer of t after checking it against the layout the C call
    assumes: dtype, exact shape (or at least min_numel elements), contiguous,
    on device dev."""
    if t is None:
        if optional:
            return None
        raise FlintError(FLINT_ERR_INVALID_ARG, "%s: %s is required" % (where, name))
    if isinstance(t, int):
        return t
    if not (isinstance(t, torch.Tensor) and t.dtype == dtype and t.device == dev and
            (t.shape == shape if shape is not None else t.numel() >= min_numel) and
            t.is_contiguous()):
        what = "a contiguous %s tensor %s on %s" % (
            dtype, shape if shape is not None else "of >= %d elements" % min_numel, dev)
        _bad(where, name, what, t)
    return t.data_ptr()


def _batch(where, name, t, hidden):
    """(batch, device) of a [batch, hidden] activation tensor on the current
    CUDA device (the library launches on, and sizes its grids for, the
    current device)."""
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dim() == 2 and t.shape[1] == hidden):
        _bad(where, name, "a [batch, %d] tensor on a CUDA device" % hidden, t)
    _on_current_device(where, name, t)
    return t.shape[0], t.device


def _on_current_device(where, name, t):
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise FlintError(FLINT_ERR_INVALID_ARG,
                         "%s: %s is on %s but the current device is cuda:%d (use "
                         "torch.cuda.device(...) around the call)" % (where, name, t.device, cur))


def _ws_arg(where, workspace, dev):
    """(pointer, bytes) of a workspace: a contiguous uint8 tensor on dev."""
    if isinstance(workspace, torch.Tensor):
        if not (workspace.dtype == _U8 and workspace.dim() == 1 and workspace.device == dev and
                workspace.is_contiguous()):
            _bad(where, "workspace", "a contiguous 1-D uint8 tensor on %s" % dev, workspace)
    return _ws(workspace)


def _d(dims):
    return FULL_DIMS if dims is None else dims


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


def _ws_only(where, workspace):
    """(pointer, bytes) of a workspace passed on its own: a contiguous uint8
    tensor on the current CUDA device."""
    if not (isinstance(workspace, torch.Tensor) and workspace.is_cuda):
        _bad(where, "workspace", "a contiguous 1-D uint8 tensor on a CUDA device", workspace)
    _on_current_device(where, "workspace", workspace)
    return _ws_arg(where, workspace, workspace.device)


def flint_moe_workspace_init(workspace: torch.Tensor, wait_limit_ns: int = 0, stream=None):
    wp, wb = _ws_only("flint_moe_workspace_init", workspace)
    _check(lib().flint_moe_workspace_init(wp, wb, int(wait_limit_ns), _stream(stream)),
           "flint_moe_workspace_init")


def flint_moe_get_device_status(workspace: torch.Tensor, stream=None) -> int:
    wp, _ = _ws_only("flint_moe_get_device_status", workspace)
    return int(lib().flint_moe_get_device_status(wp, _stream(stream)))


def flint_moe_debug_arm_stall(workspace: torch.Tensor, stream=None):
    wp, wb = _ws_only("flint_moe_debug_arm_stall", workspace)
    _check(lib().flint_moe_debug_arm_stall(wp, wb, _stream(stream)), "flint_moe_debug_arm_stall")


def _ws(workspace):
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def flint_moe_route(x, w_router, logit_bias, topk_idx, topk_w, workspace, stream=None,
                    dims: Dims | None = None):
    f, d = "flint_moe_route", _d(dims)
    B, dev = _batch(f, "x", x, d.hidden)
    args = (_arg(f, "x", x, _BF16, (B, d.hidden), dev),
            _arg(f, "w_router", w_router, _BF16, (d.n_experts, d.hidden), dev),
            _arg(f, "logit_bias", logit_bias, _F32, (d.n_experts,), dev, optional=True),
            _arg(f, "topk_idx", topk_idx, _I32T, (B, d.top_k), dev),
            _arg(f, "topk_w", topk_w, _F32, (B, d.top_k), dev))
    wp, wb = _ws_arg(f, workspace, dev)
    _check(lib().flint_moe_route(_dims(dims), B, *args, wp, wb, _stream(stream)), f)


def flint_moe_bucket(topk_idx, uniq, offsets, pairs, n_uniq, workspace, stream=None,
                     dims: Dims | None = None):
    f, d = "flint_moe_bucket", _d(dims)
    B, dev = _batch(f, "topk_idx", topk_idx, d.top_k)
    args = (_arg(f, "topk_idx", topk_idx, _I32T, (B, d.top_k), dev),
            _arg(f, "uniq", uniq, _I32T, None, dev, min_numel=d.n_experts),
            _arg(f, "offsets", offsets, _I32T, None, dev, min_numel=d.n_experts + 1),
            _arg(f, "pairs", pairs, _I32T, None, dev, min_numel=B * d.top_k),
            _arg(f, "n_uniq", n_uniq, _I32T, None, dev, min_numel=1))
    wp, wb = _ws_arg(f, workspace, dev)
    _check(lib().flint_moe_bucket(_dims(dims), B, *args, wp, wb, _stream(stream)), f)


def _layer_args(f, d, B, dev, x, residual, w_router, logit_bias, w13, w2, ws13, ws2, out,
                topk_idx_out, topk_w_out):
    """Checked pointers of the BF16 layer's arguments, in the C call's order."""
    H, E, K, I, S = d.hidden, d.n_experts, d.top_k, d.inter, d.n_shared
    return (_arg(f, "x", x, _BF16, (B, H), dev),
            _arg(f, "residual", residual, _BF16, (B, H), dev),
            _arg(f, "w_router", w_router, _BF16, (E, H), dev),
            _arg(f, "logit_bias", logit_bias, _F32, (E,), dev, optional=True),
            _arg(f, "w13", w13, _BF16, (E, 2 * I, H), dev),
            _arg(f, "w2", w2, _BF16, (E, H, I), dev),
            _arg(f, "ws13", ws13, _BF16, (S, 2 * I, H), dev),
            _arg(f, "ws2", ws2, _BF16, (S, H, I), dev),
            _arg(f, "out", out, _BF16, (B, H), dev),
            _arg(f, "topk_idx_out", topk_idx_out, _I32T, (B, K), dev, optional=True),
            _arg(f, "topk_w_out", topk_w_out, _F32, (B, K), dev, optional=True))


def flint_moe_decode_bf16(x, residual, w_router, logit_bias, w13, w2, ws13, ws2, out, workspace,
                          topk_idx_out=None, topk_w_out=None, stream=None,
                          dims: Dims | None = None):
    f, d = "flint_moe_decode_bf16", _d(dims)
    B, dev = _batch(f, "x", x, d.hidden)
    args = _layer_args(f, d, B, dev, x, residual, w_router, logit_bias, w13, w2, ws13, ws2, out,
                       topk_idx_out, topk_w_out)
    wp, wb = _ws_arg(f, workspace, dev)
    _check(lib().flint_moe_decode_bf16(_dims(dims), B, *args, wp, wb, _stream(stream)), f)


def flint_moe_decode_bf16_prenorm(residual, w_router, logit_bias, w13, w2, ws13, ws2, out,
                                  workspace, norm_eps: float = 1e-6, topk_idx_out=None,
                                  topk_w_out=None, stream=None, dims: Dims | None = None):
    """flint_moe_decode_bf16 whose input is RMSNorm(residual) (unit gain,
    norm_eps), computed inside the call: one launch per layer for batches of
    at most 8 tokens."""
    f, d = "flint_moe_decode_bf16_prenorm", _d(dims)
    B, dev = _batch(f, "residual", residual, d.hidden)
    args = _layer_args(f, d, B, dev, residual, residual, w_router, logit_bias, w13, w2, ws13, ws2,
                       out, topk_idx_out, topk_w_out)
    wp, wb = _ws_arg(f, workspace, dev)
    _check(lib().flint_moe_decode_bf16_prenorm(_dims(dims), B, args[1], float(norm_eps), *args[2:],
                                               wp, wb, _stream(stream)), f)


def flint_moe_decode_bf16_noalloc(x, residual, w_router, logit_bias, w13, w2, ws13, ws2, out,
                                  topk_idx_out=None, topk_w_out=None, device_status_out=None,
                                  stream=None, dims: Dims | None = None):
    """flint_moe_decode_bf16 without a workspace (the library's static device
    array instead; batch <= NOALLOC_MAX_BATCH).  For callers that cannot
    allocate device memory; calls whose GPU work overlaps race."""
    f, d = "flint_moe_decode_bf16_noalloc", _d(dims)
    B, dev = _batch(f, "x", x, d.hidden)
    args = _layer_args(f, d, B, dev, x, residual, w_router, logit_bias, w13, w2, ws13, ws2, out,
                       topk_idx_out, topk_w_out)
    st = _arg(f, "device_status_out", device_status_out, _I32T, None, dev, optional=True,
              min_numel=1)
    _check(lib().flint_moe_decode_bf16_noalloc(_dims(dims), B, *args, st, _stream(stream)), f)


def flint_moe_gateup_bf16(x, w13, ws13, workspace, stream=None, dims: Dims | None = None):
    f, d = "flint_moe_gateup_bf16", _d(dims)
    B, dev = _batch(f, "x", x, d.hidden)
    args = (_arg(f, "x", x, _BF16, (B, d.hidden), dev),
            _arg(f, "w13", w13, _BF16, (d.n_experts, 2 * d.inter, d.hidden), dev),
            _arg(f, "ws13", ws13, _BF16, (d.n_shared, 2 * d.inter, d.hidden), dev))
    wp, wb = _ws_arg(f, workspace, dev)
    _check(lib().flint_moe_gateup_bf16(_dims(dims), B, *args, wp, wb, _stream(stream)), f)


def flint_moe_down_bf16(residual, w2, ws2, out, workspace, stream=None, dims: Dims | None = None):
    f, d = "flint_moe_down_bf16", _d(dims)
    B, dev = _batch(f, "residual", residual, d.hidden)
    args = (_arg(f, "residual", residual, _BF16, (B, d.hidden), dev),
            _arg(f, "w2", w2, _BF16, (d.n_experts, d.hidden, d.inter), dev),
            _arg(f, "ws2", ws2, _BF16, (d.n_shared, d.hidden, d.inter), dev),
            _arg(f, "out", out, _BF16, (B, d.hidden), dev))
    wp, wb = _ws_arg(f, workspace, dev)
    _check(lib().flint_moe_down_bf16(_dims(dims), B, *args, wp, wb, _stream(stream)), f)


NVFP4_KEYS = ("w13_q", "w13_sf", "w13_ts", "w2_q", "w2_sf", "w2_ts",
              "ws13_q", "ws13_sf", "ws13_ts", "ws2_q", "ws2_sf", "ws2_ts")


def flint_moe_decode_nvfp4_w4a16(x, residual, w_router, logit_bias, nv: dict, out, workspace,
                                 topk_idx_out=None, topk_w_out=None, stream=None,
                                 dims: Dims | None = None):
    """nv holds the twelve packed tensors named in NVFP4_KEYS."""
    f, d = "flint_moe_decode_nvfp4_w4a16", _d(dims)
    H, E, K, I, S = d.hidden, d.n_experts, d.top_k, d.inter, d.n_shared
    B, dev = _batch(f, "x", x, H)
    shapes = {}
    for pre, n in (("w", E), ("ws", S)):
        shapes[pre + "13_q"] = (_U8, (n, 2 * I, H // 2))
        shapes[pre + "13_sf"] = (_U8, (n, 2 * I, H // 16))
        shapes[pre + "13_ts"] = (_F32, (n, 2))
        shapes[pre + "2_q"] = (_U8, (n, H, I // 2))
        shapes[pre + "2_sf"] = (_U8, (n, H, I // 16))
        shapes[pre + "2_ts"] = (_F32, (n,))
    packed = [_arg(f, k, nv.get(k), shapes[k][0], shapes[k][1], dev) for k in NVFP4_KEYS]
    args = (_arg(f, "x", x, _BF16, (B, H), dev),
            _arg(f, "residual", residual, _BF16, (B, H), dev),
            _arg(f, "w_router", w_router, _BF16, (E, H), dev),
            _arg(f, "logit_bias", logit_bias, _F32, (E,), dev, optional=True),
            *packed,
            _arg(f, "out", out, _BF16, (B, H), dev),
            _arg(f, "topk_idx_out", topk_idx_out, _I32T, (B, K), dev, optional=True),
            _arg(f, "topk_w_out", topk_w_out, _F32, (B, K), dev, optional=True))
    wp, wb = _ws_arg(f, workspace, dev)
    _check(lib().flint_moe_decode_nvfp4_w4a16(_dims(dims), B, *args, wp, wb, _stream(stream)), f)


def flint_moe_rmsnorm_bf16(inp, out, eps: float = 1e-6, stream=None, dims: Dims | None = None):
    f, d = "flint_moe_rmsnorm_bf16", _d(dims)
    B, dev = _batch(f, "inp", inp, d.hidden)
    args = (_arg(f, "inp", inp, _BF16, (B, d.hidden), dev),
            _arg(f, "out", out, _BF16, (B, d.hidden), dev))
    _check(lib().flint_moe_rmsnorm_bf16(_dims(dims), B, *args, float(eps), _stream(stream)), f)


def flint_qk_norm_rope_kv_bf16(qkv, q_norm, k_norm, positions, slot_mapping, q_out, k_cache,
                               v_cache, rope_theta: float, eps: float = 1e-6, stream=None):
    """Per-head Q/K RMSNorm + RoPE (rope_theta = 0: none) of a decode step's
    projection rows qkv [B, (32 + 2*4) * 128], writing the query heads to
    q_out [B, 32, 128] and the key / value heads to row slot_mapping[t] of
    k_cache / v_cache [slots, 4, 128]; positions and slot_mapping are int32 [B]."""
    f = "flint_qk_norm_rope_kv_bf16"
    row = (N_Q_HEADS + 2 * N_KV_HEADS) * HEAD_DIM
    B, dev = _batch(f, "qkv", qkv, row)
    if not (isinstance(k_cache, torch.Tensor) and k_cache.dim() == 3):
        _bad(f, "k_cache", "a [slots, %d, %d] tensor" % (N_KV_HEADS, HEAD_DIM), k_cache)
    slots = k_cache.shape[0]
    cache = (slots, N_KV_HEADS, HEAD_DIM)
    args = (_arg(f, "qkv", qkv, _BF16, (B, row), dev),
            _arg(f, "q_norm", q_norm, _BF16, (HEAD_DIM,), dev),
            _arg(f, "k_norm", k_norm, _BF16, (HEAD_DIM,), dev),
            _arg(f, "positions", positions, _I32T, (B,), dev),
            _arg(f, "slot_mapping", slot_mapping, _I32T, (B,), dev))
    outs = (_arg(f, "q_out", q_out, _BF16, (B, N_Q_HEADS, HEAD_DIM), dev),
            _arg(f, "k_cache", k_cache, _BF16, cache, dev),
            _arg(f, "v_cache", v_cache, _BF16, cache, dev))
    _check(lib().flint_qk_norm_rope_kv_bf16(ctypes.byref(ATTN_DIMS), B, *args, float(rope_theta),
                                            float(eps), *outs, slots, _stream(stream)), f)


# ---------------------------------------------------------------- conveniences

def new_workspace(max_batch: int, device="cuda", wait_limit_ns: int = 0) -> torch.Tensor:
    """Allocates (through torch) and initialises a workspace for max_batch tokens."""
    n = flint_moe_workspace_bytes(max_batch)
    if n == 0:
        raise FlintError(FLINT_ERR_INVALID_ARG, "new_workspace")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    flint_moe_workspace_init(ws, wait_limit_ns)
    return ws
