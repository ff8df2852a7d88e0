"""The benchmark's host-side arithmetic on CPU: the algorithmic work it
divides by, the roofline it picks, and when stored ncu traffic applies.

The per-configuration totals are the closed forms of the layer: router
2·T·E·d, gate/up 4·d·F per kept assignment (+ 4·d·F_s per token for the
shared expert), down half of that; weight bytes 3·F·d per touched expert at
2 bytes (bf16) or 1 byte plus a 4-byte scale per weight row (E4M3).
"""

import dataclasses
import json

import pytest

import bench
from workloads import SHAPES

PEAKS = {"hbm_gbs": 6503.1, "bf16_tflops": 1755.4, "bf16_tflops_sustained": 1353.7}


def _work(name, kept_per_expert=None, touched=None, **kw):
    s = dataclasses.replace(SHAPES[name], **kw) if kw else SHAPES[name]
    n = touched if touched is not None else s.E
    per = kept_per_expert if kept_per_expert is not None else s.T * s.k // s.E
    counts = [per] * n + [0] * (s.E - n)
    return s, bench.algorithmic_work(s, counts)


def test_mixtral_flops():
    s, w = _work("mixtral")
    assert w["kept"] == 8192 and w["touched"] == 8
    assert w["flops_router"] == pytest.approx(2 * 4096 * 8 * 4096)
    assert w["flops"] / 1e9 == pytest.approx(2886.5, abs=0.1)
    assert w["flops_down"] * 2 == pytest.approx(w["flops_gate_up"])


def test_dsv3_prefill_flops_and_bytes():
    s, w = _work("dsv3_prefill")
    assert w["kept"] == 65536 and w["touched"] == 256
    assert w["flops_router"] / 1e9 == pytest.approx(30.06, abs=0.01)
    assert w["flops"] / 1e9 == pytest.approx(6524.1, abs=0.1)
    per_expert = 3 * 2048 * 7168 * 2
    assert per_expert == 88_080_384
    assert w["weight_bytes"] == 257 * per_expert + 256 * 7168 * 2   # + shared + router


def test_decode_bytes_per_touched_expert():
    s, w = _work("dsv3_decode", kept_per_expert=2, touched=223)
    assert w["weight_bytes"] == 224 * 88_080_384 + 256 * 7168 * 2
    assert w["weight_bytes"] / 1e9 == pytest.approx(19.73, abs=0.01)


def test_e4m3_bytes_are_codes_plus_row_scales():
    s, w = _work("dsv3_decode_fp8", kept_per_expert=2, touched=223)
    per_expert = 3 * 2048 * 7168 + (2 * 2048 + 7168) * 4
    assert w["bytes_gate_up"] + w["bytes_down"] == 224 * per_expert
    assert w["weight_bytes"] == 224 * per_expert + 256 * 7168 * 2   # router stays bf16


@pytest.mark.parametrize("name,kw,stage,want", [
    ("mixtral", {}, "gate_up", True),
    ("mixtral", {}, "down", True),
    ("dsv3_prefill", {}, "gate_up", True),
    ("dsv3_decode", dict(kept_per_expert=2, touched=223), "gate_up", False),
    # the Switch layer: 2701 kept tokens over 40 touched experts
    ("switch", dict(kept_per_expert=2701 // 40, touched=40), "gate_up", False),
])
def test_roofline_bound(name, kw, stage, want):
    s, w = _work(name, **kw)
    assert bench.tensor_bound(w, stage, PEAKS, "bf16_tflops") is want
    assert bench.tensor_bound(w, "combine", PEAKS, "bf16_tflops") is False


def test_stored_traffic_only_for_matching_sources(monkeypatch, tmp_path):
    digest = bench.source_digest()
    rec = {"mixtral": {"gate_up": {"dram_bytes_per_launch": 123, "source_digest": digest}},
           "other": {"gate_up": {"dram_bytes_per_launch": 456, "source_digest": "0" * 16}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda names=bench.GEMM_SOURCES: digest)
    assert bench.stored_traffic("mixtral", "gate_up") == 123
    assert bench.stored_traffic("other", "gate_up") is None      # kernel changed since
    assert bench.stored_traffic("mixtral", "down") is None       # never captured


def test_committed_traffic_records_name_their_capture():
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    for wl, stages in t.items():
        if wl.startswith("_"):
            continue
        assert wl in bench.WORKLOAD_TEXT
        for rec in stages.values():
            assert rec["dram_bytes_per_launch"] > 0
            assert bench.os.path.exists(bench.os.path.join(
                bench.ROOT, "profiles", rec["capture"].split(" ")[0]))


def test_clock_sampler_counts_only_the_timed_window():
    # NVML poller lines "host_time sm_mhz max_mhz reason_mask": two before the
    # window, three inside (one under the software power cap, bit 0x4, and an
    # unreported reason bit 0x1), one after
    cs = bench.ClockSampler(0)
    cs.source = "nvml"
    cs.t0, cs.t1 = 100.0, 100.02
    cs.nvml_lines = ["99.990 2032 2032 0", "99.995 2032 2032 0",
                     "100.000 1980 2032 5", "100.010 1200 2032 0", "100.020 1300 2032 1",
                     "100.030 2032 2032 4", "garbled"]
    s = cs.summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1300.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]
    assert tuple(bench.ClockSampler.REASONS) == ("hw_slowdown", "hw_thermal_slowdown",
                                                 "sw_thermal_slowdown", "sw_power_cap")


def test_clock_sampler_without_a_gpu_reports_no_samples():
    # no NVML library and no nvidia-smi here: the sampler must neither raise
    # nor invent samples
    cs = bench.ClockSampler(0)
    cs.start()
    cs.mark_begin()
    cs.mark_end()
    cs.stop()
    s = cs.summary()
    if cs.source is None:
        assert s == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    else:   # a machine with a GPU: whatever it sampled lies inside the window
        assert s["samples"] >= 0
