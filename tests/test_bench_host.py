"""Host-side pieces of bench.py that need no GPU: the needed-bytes formulas
behind the metric, the nvidia-smi clock record, the ncu traffic lookup and the
latency statistics."""
from __future__ import annotations

import json
import os

import pytest

import bench
import flint_synth as fs

D = fs.FULL


def test_needed_bytes_follow_the_layer_shapes():
    """(U + 1) experts (the routed ones read plus the shared one) and the router:
    each expert is gate + up [2I, H] and down [H, I] in bf16; NVFP4 stores half a
    byte per weight, one e4m3 scale per 16 weights and three fp32 tensor scales."""
    H, E, I = D.hidden, D.n_experts, D.inter
    weights = 2 * I * H + H * I
    router = E * H * 2
    for U in (0, 6, 43, 182, 256):
        assert bench.needed_bytes_bf16(U) == (U + 1) * weights * 2 + router
        assert bench.needed_bytes_nvfp4(U) == (U + 1) * (weights // 2 + weights // 16 + 3 * 4) + router
    assert bench.needed_bytes_bf16(6) == 45_088_768            # batch 1: six routed experts
    assert bench.GATEUP_BYTES_BF16 + bench.DOWN_BYTES_BF16 == bench.EXPERT_BYTES_BF16


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def test_clock_record_median_max_and_throttle_reasons(tmp_path):
    csv = tmp_path / "clocks.csv"
    csv.write_text(
        "index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], "
        "clocks_event_reasons.active, clocks_event_reasons.hw_slowdown, "
        "clocks_event_reasons.hw_thermal_slowdown, clocks_event_reasons.sw_thermal_slowdown, "
        "clocks_event_reasons.sw_power_cap\n"
        "0, 2070 MHz, 2070 MHz, 700.10 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1965 MHz, 2070 MHz, 1390.00 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
        "0, 2070 MHz, 2070 MHz, 900.00 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, [N/A], 2070 MHz, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]\n")
    s = object.__new__(bench.ClockSampler)
    s.proc, s.path = _FakeProc(), str(csv)
    rec = s.stop()
    assert rec == {"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"], "samples": 3}
    assert not os.path.exists(csv)
    s = object.__new__(bench.ClockSampler)
    s.proc, s.path = None, None
    assert s.stop()["samples"] == 0


def test_recorded_traffic_counts_only_for_the_captured_sources(monkeypatch):
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    key = next(iter(recs))
    kernel, batch = key.rsplit("_b", 1)
    rec = recs[key]
    assert rec["traffic_bytes"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    assert "--clock-control none" in rec["command"]
    monkeypatch.setattr(bench, "sources_sha", lambda tu=None: rec["sources_sha"])
    assert bench.recorded_traffic(kernel, int(batch)) == rec["traffic_bytes"]
    assert bench.recorded_traffic(kernel, int(batch) + 1) is None
    monkeypatch.setattr(bench, "sources_sha", lambda tu=None: "0" * 16)
    assert bench.recorded_traffic(kernel, int(batch)) is None


def test_sources_hash_is_stable_and_short():
    a, b = bench.sources_sha(), bench.sources_sha()
    assert a == b and len(a) == 16 and int(a, 16) >= 0
    assert bench.sources_sha("fused.cu") == bench.sources_sha("fused.cu")


def test_sources_hash_covers_exactly_the_include_closure(tmp_path, monkeypatch):
    csrc = tmp_path / "moe_decode_sigmoid_gb300" / "csrc"
    inc = tmp_path / "include"
    csrc.mkdir(parents=True)
    inc.mkdir()
    (csrc / "a.cu").write_text('#include "b.cuh"\n#include <cuda.h>\n')
    (csrc / "b.cuh").write_text('  #  include "api.h"\n')
    (csrc / "c.cu").write_text("// another kernel\n")
    (inc / "api.h").write_text("// the API\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    names = [os.path.basename(p) for p in bench.source_closure("a.cu")]
    assert names == ["a.cu", "api.h", "b.cuh"]
    h0 = bench.sources_sha("a.cu")
    (csrc / "c.cu").write_text("// changed, outside the closure\n")
    assert bench.sources_sha("a.cu") == h0
    (inc / "api.h").write_text("// changed, inside the closure\n")
    assert bench.sources_sha("a.cu") != h0


def test_chained_replays_time_exactly_the_requested_steps():
    assert bench.chain_blocks(2000, 8) == [8] * 250
    assert bench.chain_blocks(20, 8) == [8, 8, 4]
    assert bench.chain_blocks(5, 1) == [1] * 5
    assert bench.chain_blocks(3, 8) == [3]
    for steps in range(1, 40):
        for n in (1, 3, 8):
            b = bench.chain_blocks(steps, n)
            assert sum(b) == steps and all(1 <= k <= n for k in b)


def test_latency_statistics():
    st = bench.stats_us([0.010, 0.030, 0.020, 0.040, 0.050])   # ms
    assert st["mean"] == pytest.approx(30.0)
    assert (st["p10"], st["p50"], st["p90"]) == pytest.approx((10.0, 30.0, 40.0))


def test_peak_is_measured_or_the_stated_fallback():
    peak, kind = bench.peaks()
    assert kind in ("measured", "fallback") and peak > 0
    if kind == "fallback":
        assert peak == bench.FALLBACK_HBM_GBS


def test_profile_summaries_name_safe_commands_over_committed_files():
    """Every ncu command a profile summary gives leaves the GPU clocks alone and
    runs a program of this repository (the bench or the tests)."""
    import glob
    import re
    cmds = []
    for path in glob.glob(os.path.join(bench.ROOT, "profiles", "*")):
        if path.endswith(".json"):
            cmds += [(path, r["command"]) for r in json.load(open(path)).values()]
            continue
        for line in open(path).read().replace("\\\n", " ").splitlines():
            if line.strip().startswith("ncu "):
                cmds.append((path, line.strip()))
    assert len(cmds) >= 5
    for path, cmd in cmds:
        assert "--clock-control none" in cmd, (path, cmd)
        prog = re.search(r"\bpython(?: -m pytest)? (\S+)", cmd)
        assert prog, (path, cmd)
        assert os.path.exists(os.path.join(bench.ROOT, prog.group(1))), (path, cmd)
