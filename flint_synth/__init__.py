"""Seeded synthetic inputs for the Flint decode MoE layer.

This module only draws and packs inputs; it holds none of the layer's
arithmetic (no routing, no expert FFN, no combine).  Both the CUDA path and the
CPU oracle consume what it returns, so the two sides always see bit-identical
inputs.

Recipe (the pages fix only the shapes: hidden 2048, 256 routed experts, top-6
plus one shared expert -- [vLLM Day-0 Support for Recursive's Flint,
"Flint Model Architecture"]; the intermediate size 512 and the value
distributions are this library's choices):
  - every weight ~ N(0, 0.02), rounded to bf16 (round-to-nearest-even);
  - x_pre ~ N(0, 1) per token; residual = bf16(x_pre);
    x = bf16(x_pre / sqrt(mean(x_pre^2) + 1e-6))  (unit-RMS activations);
  - optional per-expert logit offsets ~ N(0, 0.5) in fp32 (skewed expert load);
  - NVFP4 weights are packed from the bf16 draws (see pack_nvfp4).
Draws use torch's seeded generators on the requested device; a given
(seed, device type) always yields the same tensors.
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = [
    "Dims", "FULL", "TINY", "layer_weights", "tokens", "logit_offsets",
    "pack_nvfp4", "nvfp4_layer", "E2M1_VALUES", "attn_inputs",
]


@dataclasses.dataclass(frozen=True)
class Dims:
    hidden: int = 2048
    n_experts: int = 256
    top_k: int = 6
    inter: int = 512
    n_shared: int = 1
    offset_mode: int = 0   # 0: logit offsets move ranking and weights; 1: ranking only


FULL = Dims()
TINY = Dims(hidden=64, n_experts=16, top_k=6, inter=32, n_shared=1)

WEIGHT_STD = 0.02
RMS_EPS = 1e-6
OFFSET_STD = 0.5


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _normal_bf16(shape, std, g, device) -> torch.Tensor:
    # Draw in chunks along dim 0 to bound the fp32 temporary.
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rows = shape[0]
    per_row = 1
    for s in shape[1:]:
        per_row *= s
    step = max(1, (1 << 26) // max(per_row, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        tmp = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device,
                          dtype=torch.float32)
        out[r0:r1] = (tmp * std).to(torch.bfloat16)
    return out


def layer_weights(seed: int, dims: Dims = FULL, device="cpu") -> dict:
    """Router, routed experts and shared expert(s) of one layer, all bf16.

    wr [E,H]; w13 [E,2I,H] (rows 0..I-1 gate, I..2I-1 up); w2 [E,H,I];
    ws13 [S,2I,H]; ws2 [S,H,I].
    """
    g = _gen(seed, device)
    H, E, I, S = dims.hidden, dims.n_experts, dims.inter, dims.n_shared
    return {
        "wr": _normal_bf16((E, H), WEIGHT_STD, g, device),
        "w13": _normal_bf16((E, 2 * I, H), WEIGHT_STD, g, device),
        "w2": _normal_bf16((E, H, I), WEIGHT_STD, g, device),
        "ws13": _normal_bf16((S, 2 * I, H), WEIGHT_STD, g, device),
        "ws2": _normal_bf16((S, H, I), WEIGHT_STD, g, device),
    }


def tokens(seed: int, batch: int, hidden: int = FULL.hidden, device="cpu"):
    """(x, residual) bf16 [batch, hidden]: unit-RMS activations and the raw draw."""
    g = _gen(seed, device)
    x_pre = torch.randn((batch, hidden), generator=g, device=device, dtype=torch.float32)
    residual = x_pre.to(torch.bfloat16)
    scale = torch.rsqrt(x_pre.double().pow(2).mean(dim=1, keepdim=True) + RMS_EPS)
    x = (x_pre.double() * scale).to(torch.bfloat16)
    return x, residual


def logit_offsets(seed: int, n_experts: int = FULL.n_experts, device="cpu") -> torch.Tensor:
    """Per-expert fp32 offsets ~ N(0, 0.5) that skew expert load."""
    g = _gen(seed, device)
    return torch.randn((n_experts,), generator=g, device=device,
                       dtype=torch.float32) * OFFSET_STD


def attn_inputs(seed: int, batch: int, cache_slots: int, n_q: int = 32, n_kv: int = 4,
                head_dim: int = 128, max_pos: int = 1 << 18, device="cpu") -> dict:
    """Inputs of a decode step's attention side (per-head Q/K norm + RoPE +
    KV-cache write; GQA 32 / 4 heads: [vLLM Day-0 Support for Recursive's
    Flint, "Flint Model Architecture"]):
      qkv [batch, (n_q + 2 n_kv) * head_dim] bf16 ~ N(0, 1) (projection rows);
      q_norm, k_norm [head_dim] bf16 ~ N(1, 0.1) (per-element gains);
      positions [batch] int32 uniform in [0, max_pos) (2^18: the 262k context);
      slot_mapping [batch] int32: distinct cache rows, every 7th token -1
      (padding);
      k_cache, v_cache [cache_slots, n_kv, head_dim] bf16 ~ N(0, 1) (rows the
      step must leave as they are).
    The value distributions are this library's choices; the pages give none."""
    assert cache_slots >= batch
    g = _gen(seed, device)
    row = (n_q + 2 * n_kv) * head_dim
    qkv = torch.randn((batch, row), generator=g, device=device).to(torch.bfloat16)
    q_norm = (1.0 + 0.1 * torch.randn((head_dim,), generator=g, device=device)).to(torch.bfloat16)
    k_norm = (1.0 + 0.1 * torch.randn((head_dim,), generator=g, device=device)).to(torch.bfloat16)
    positions = torch.randint(0, max_pos, (batch,), generator=g, device=device, dtype=torch.int32)
    slots = torch.randperm(cache_slots, generator=g, device=device)[:batch].to(torch.int32)
    slots[6::7] = -1
    cache = (cache_slots, n_kv, head_dim)
    k_cache = torch.randn(cache, generator=g, device=device).to(torch.bfloat16)
    v_cache = torch.randn(cache, generator=g, device=device).to(torch.bfloat16)
    return {"qkv": qkv, "q_norm": q_norm, "k_norm": k_norm, "positions": positions,
            "slot_mapping": slots, "k_cache": k_cache, "v_cache": v_cache}


# --- NVFP4 packing -----------------------------------------------------------
# e2m1 magnitudes by 3-bit code (OCP Microscaling Formats v1.0, FP4 E2M1).
E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
# Midpoints between neighbouring magnitudes; at an exact midpoint round-to-even
# keeps the even code, i.e. rounds up across the midpoints 0.75, 1.75 and 3.5.
_MID_DOWN = (0.25, 1.25, 2.5, 5.0)
_MID_UP = (0.75, 1.75, 3.5)
E2M1_MAX = 6.0
E4M3_MAX = 448.0


def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    a = v.abs().clamp(max=E2M1_MAX)
    code = torch.zeros(a.shape, dtype=torch.int32, device=a.device)
    for m in _MID_DOWN:
        code += (a > m).to(torch.int32)
    for m in _MID_UP:
        code += (a >= m).to(torch.int32)
    sign = ((v < 0) & (code > 0)).to(torch.int32) << 3
    return (code | sign).to(torch.uint8)


def pack_nvfp4(w: torch.Tensor, row_split: int | None = None):
    """Pack bf16 weights [..., rows, K] into (q, sf, ts).

    q  uint8 [..., rows, K/2]  e2m1 codes, low nibble = even k
    sf uint8 [..., rows, K/16] E4M3FN block scales (16 consecutive k)
    ts fp32  [..., n_parts]    one tensor scale per part; rows are split into
                               parts [0, row_split) and [row_split, rows) when
                               row_split is given (gate / up), else one part.
    ts = amax / (6 * 448); sf = e4m3(amax16 / (6 * ts)); q = e2m1(w / (sf * ts)).
    """
    *lead, rows, K = w.shape
    assert K % 16 == 0
    wf = w.float()
    parts = [(0, rows)] if row_split is None else [(0, row_split), (row_split, rows)]
    q_codes = torch.empty(wf.shape, dtype=torch.uint8, device=w.device)
    sf = torch.empty(tuple(lead) + (rows, K // 16), dtype=torch.uint8, device=w.device)
    ts = torch.empty(tuple(lead) + (len(parts),), dtype=torch.float32, device=w.device)
    for pi, (r0, r1) in enumerate(parts):
        blk = wf[..., r0:r1, :]
        amax = blk.abs().amax(dim=(-2, -1))
        t = torch.where(amax > 0, amax / (E2M1_MAX * E4M3_MAX), torch.ones_like(amax))
        ts[..., pi] = t
        tb = t[..., None, None]
        b16 = blk.reshape(*blk.shape[:-1], K // 16, 16)
        amax16 = b16.abs().amax(dim=-1)
        s_code = (amax16 / (E2M1_MAX * tb)).clamp(max=E4M3_MAX).to(torch.float8_e4m3fn)
        sf[..., r0:r1, :] = s_code.view(torch.uint8)
        s_val = s_code.float()
        denom = (s_val * tb)[..., None]
        scaled = torch.where(denom > 0, b16 / torch.where(denom > 0, denom, torch.ones_like(denom)),
                             torch.zeros_like(b16))
        q_codes[..., r0:r1, :] = _e2m1_codes(scaled).reshape(blk.shape)
    q = q_codes[..., 0::2] | (q_codes[..., 1::2] << 4)
    return q.contiguous(), sf.contiguous(), ts.contiguous()


def nvfp4_layer(W: dict, dims: Dims = FULL) -> dict:
    """The twelve packed NVFP4 tensors of a layer, from its bf16 weights:
    w13_q/w13_sf/w13_ts (gate and up scaled separately), w2_q/w2_sf/w2_ts, and
    the same for the shared expert(s) (ws13_*, ws2_*)."""
    nv = {}
    for pre, w13, w2 in (("w", W["w13"], W["w2"]), ("ws", W["ws13"], W["ws2"])):
        q, sf, ts = pack_nvfp4(w13, row_split=dims.inter)
        nv[pre + "13_q"], nv[pre + "13_sf"], nv[pre + "13_ts"] = q, sf, ts
        q, sf, ts = pack_nvfp4(w2)
        nv[pre + "2_q"], nv[pre + "2_sf"], nv[pre + "2_ts"] = q, sf, ts[..., 0].contiguous()
    return nv
