"""flint_moe_decode_bf16_noalloc: the decode layer for callers that cannot
allocate device memory (hosts that own every byte of the GPU themselves, such
as a serving engine with fixed memory pools or a runtime with a build-time
memory budget).  Instead of a caller-allocated workspace it runs on one static
device array inside the library.

The GPU test calls it twice in a row through the C ABI -- a batch of 8 tokens,
then a batch of 3 with logit offsets, so the second call starts from whatever
the first left in the shared array -- and checks each call's outputs, routing
and device status against flint_moe_decode_bf16 on a normal workspace: both
run the same kernels, so the outputs and routing must agree bit for bit.  The
file is named so that pytest collects it last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import flint_synth as fs
from tests._util import REL_TOL, bf16_bits_to_f64, rel_err, rel_err_delta

D = fs.FULL
K = D.top_k


def test_noalloc_rejects_batches_beyond_its_limit():
    """Checked on the host before any CUDA call (runs without a GPU)."""
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as m
    L = m.lib()
    A = 0x100000   # fake device addresses: nothing is dereferenced
    d = ctypes.byref(m.FULL_DIMS)
    for batch in (0, m.NOALLOC_MAX_BATCH + 1, 256):
        assert L.flint_moe_decode_bf16_noalloc(d, batch, A, A + 0x10000, A, None, A, A, A, A,
                                               A + 0x20000, None, None, None,
                                               None) == m.FLINT_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row():
    from moe_decode_sigmoid_gb300 import build
    build.build()
    import moe_decode_sigmoid_gb300 as m
    dev = torch.device("cuda:0")
    W = fs.layer_weights(1001, D, device=dev)
    cases = [(8, None, 31), (3, fs.logit_offsets(7, device=dev), 32)]

    results = []
    for B, bias, seed in cases:   # two no-alloc calls back to back, no sync between
        x, res = fs.tokens(seed, B, device=dev)
        out = torch.empty_like(res)
        idx = torch.full((B, K), -1, dtype=torch.int32, device=dev)
        w = torch.zeros((B, K), dtype=torch.float32, device=dev)
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        m.flint_moe_decode_bf16_noalloc(x, res, W["wr"], bias, W["w13"], W["w2"], W["ws13"],
                                        W["ws2"], out, idx, w, status)
        results.append((B, bias, x, res, out, idx, w, status))
    torch.cuda.synchronize()

    ws = m.new_workspace(8, device=dev)
    for B, bias, x, res, out, idx, w, status in results:
        assert int(status.item()) == m.FLINT_OK
        ref_out = torch.empty_like(res)
        ref_idx = torch.full((B, K), -1, dtype=torch.int32, device=dev)
        ref_w = torch.zeros((B, K), dtype=torch.float32, device=dev)
        m.flint_moe_decode_bf16(x, res, W["wr"], bias, W["w13"], W["w2"], W["ws13"], W["ws2"],
                                ref_out, ws, ref_idx, ref_w)
        torch.cuda.synchronize()
        assert m.flint_moe_get_device_status(ws) == m.FLINT_OK
        # Same kernels on the same inputs: the same bits.
        assert torch.equal(idx, ref_idx)
        assert torch.equal(w, ref_w)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        got, ref, r = bf16_bits_to_f64(out), bf16_bits_to_f64(ref_out), bf16_bits_to_f64(res)
        assert rel_err(got, ref) <= REL_TOL
        assert rel_err_delta(got, ref, r) <= REL_TOL
