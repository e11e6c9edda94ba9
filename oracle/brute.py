"""Dense NumPy brute force of the Flint decode MoE layer -- TEST INFRASTRUCTURE.

Written separately from the C oracle to pin it: it evaluates EVERY expert for
every token (dense), ranks experts with one stable full sort of the negated
logits (a stable sort keeps the lower index first among equal logits), and
combines with a dense weight matrix that is zero outside the selected set.
Same definition as the C oracle (sigmoid top-k with renormalised weights,
SwiGLU experts, shared expert with weight 1, residual add), reached by a
different route.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(a) -> np.ndarray:
    """bf16 bit patterns (uint16/int16 array or torch bf16 tensor) -> float64."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.contiguous().view(torch.int16).numpy()
    except ImportError:  # pragma: no cover
        pass
    u = np.ascontiguousarray(a).view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def dense_routing(x, wr, bias, top_k, select_only=False):
    """Returns (logits [B,E], order [B,E] full ranking, dense weights [B,E]).
    logits are the ranking keys (router scores plus offsets); with
    select_only the sigmoid takes the router scores without the offsets."""
    X = bf16_to_f64(x)
    Wr = bf16_to_f64(wr)
    raw = X @ Wr.T
    logits = raw
    if bias is not None:
        logits = raw + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    order = np.argsort(-logits, axis=1, kind="stable")
    sel = order[:, :top_k]
    scores = 1.0 / (1.0 + np.exp(-(raw if select_only else logits)))
    dense_w = np.zeros_like(logits)
    rows = np.arange(logits.shape[0])[:, None]
    dense_w[rows, sel] = scores[rows, sel]
    dense_w /= dense_w.sum(axis=1, keepdims=True)
    return logits, order, dense_w


def _ffn_all_tokens(X, w13_e, w2_e, inter):
    W13 = bf16_to_f64(w13_e)
    W2 = bf16_to_f64(w2_e)
    G = X @ W13[:inter].T
    U = X @ W13[inter:].T
    A = G * (1.0 / (1.0 + np.exp(-G))) * U
    return A @ W2.T


def dense_moe_bf16(x, residual, wr, bias, w13, w2, ws13, ws2, top_k, select_only=False):
    """Returns (out [B,H], selected idx [B,k], their weights [B,k])."""
    X = bf16_to_f64(x)
    out = bf16_to_f64(residual).copy()
    inter = w13.shape[1] // 2
    logits, order, dense_w = dense_routing(x, wr, bias, top_k, select_only)
    for s in range(ws13.shape[0]):
        out += _ffn_all_tokens(X, ws13[s], ws2[s], inter)
    for e in range(w13.shape[0]):
        out += dense_w[:, e:e + 1] * _ffn_all_tokens(X, w13[e], w2[e], inter)
    sel = order[:, :top_k]
    rows = np.arange(X.shape[0])[:, None]
    return out, sel.astype(np.int32), dense_w[rows, sel]
