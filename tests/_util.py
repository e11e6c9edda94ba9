"""Shared test helpers: the output error rule and small numeric utilities."""
from __future__ import annotations

import numpy as np

# Output tolerance: max relative error 2e-2 on bf16 outputs with fp32
# accumulation, measured against max(|ref|, 0.1 * rms(ref)) so that elements
# near zero do not blow the ratio up.  Applied to `out` and to the MoE delta
# `out - residual`, so the residual cannot mask expert errors.
REL_TOL = 2e-2
# Router margin: tokens whose fp64 gap between the k-th and (k+1)-th logit is
# at least TAU must select exactly the oracle's experts (the fp32 accumulation
# error of a 2048-term dot of unit-scale terms is ~1e-6).
TAU = 1e-4


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    floor = 0.1 * np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    denom = np.maximum(np.abs(ref), floor)
    denom = np.where(denom > 0, denom, 1.0)
    return float(np.max(np.abs(got - ref) / denom)) if ref.size else 0.0


def half_ulp_bf16(v) -> np.ndarray:
    """Half a bf16 ulp at |v| (the largest error of rounding v to bf16, RNE)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def rel_err_delta(got_out, ref_out, resid) -> float:
    """Error rule for the MoE delta (out - residual) of a bf16 output: the final
    rounding of out to bf16 (half an ulp of out) is unavoidable and is not
    charged to the delta; the rest is measured like rel_err."""
    got_out = np.asarray(got_out, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64)
    ref_d = ref_out - np.asarray(resid, dtype=np.float64)
    floor = 0.1 * np.sqrt(np.mean(ref_d * ref_d)) if ref_d.size else 0.0
    denom = np.maximum(np.abs(ref_d), floor)
    denom = np.where(denom > 0, denom, 1.0)
    excess = np.maximum(np.abs(got_out - ref_out) - half_ulp_bf16(ref_out), 0.0)
    return float(np.max(excess / denom)) if ref_d.size else 0.0


def bf16_bits_to_f64(a) -> np.ndarray:
    import torch
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    u = np.ascontiguousarray(a).view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def topk_margin(logits: np.ndarray, k: int) -> np.ndarray:
    """Per-token fp64 gap between the k-th and (k+1)-th largest logit."""
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]
