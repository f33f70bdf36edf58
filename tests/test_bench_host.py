"""Host-side arithmetic of bench.py, on CPU: the algorithmic bytes and FLOPs
behind the roofline fractions, the recorded-traffic lookup, the peak
fallback and the clock-record parsing.

The byte counts are checked against an independent enumeration of the
block's tensors (each input read once, each output written once, at the
shapes the operator's "Schema summary" gives), and against the per-block
figures of the measurement plan: 13,260,816 B for the rows-1 bf16 decode
block, 432.77 MB and 391.04 MB for the two 8192-row prefill blocks.
"""
import json
import os

import bench


def tensor_bytes(rows, C, H, R, es, prologue=True):
    CH = C * H
    shapes = {
        "streams": (rows, CH), "norm_scale": (CH,), "down_weight": (CH, R), "up_weight": (R, CH),
        "inject_weight": (CH, C),
        "pre_output": (rows, H), "post_gate": (rows, C), "streams_out": (rows, CH),
    }
    if prologue:
        shapes.update(prev_block_output=(rows, H), prev_post_gate=(rows, C))
    n = 0
    for s in shapes.values():
        k = 1
        for d in s:
            k *= d
        n += k
    return n * es


def test_block_bytes_is_every_tensor_once():
    for rows, C, H, R, es, pro in [(1, 4, 2560, 320, 2, True), (8, 4, 2560, 320, 2, True), (2, 4, 64, 16, 4, False),
                                   (8192, 8, 1280, 320, 2, True), (3, 1, 16384, 64, 2, False)]:
        assert bench.block_bytes(rows, C, H, R, es, prologue=pro) == tensor_bytes(rows, C, H, R, es, pro)


def test_block_bytes_match_the_measurement_plan():
    assert bench.block_bytes(1, 4, 2560, 320, 2) == 13_260_816
    assert round(bench.block_bytes(8192, 4, 2560, 320, 2) / 1e6, 2) == 432.77
    assert round(bench.block_bytes(8192, 8, 1280, 320, 2) / 1e6, 2) == 391.04
    # per row with a prologue: 51,216 B; without: 46,088 B
    assert bench.block_bytes(2, 4, 2560, 320, 2) - bench.block_bytes(1, 4, 2560, 320, 2) == 51_216
    assert (bench.block_bytes(2, 4, 2560, 320, 2, prologue=False)
            - bench.block_bytes(1, 4, 2560, 320, 2, prologue=False)) == 46_088


def test_block_flops_counts_the_three_contractions():
    # down (CH x R), up (R x CH) and inject (CH x C): one multiply and one add
    # per weight element and row
    for rows, C, H, R in [(1, 4, 2560, 320), (8192, 4, 2560, 320), (8192, 8, 1280, 320)]:
        CH = C * H
        macs = rows * (CH * R + R * CH + CH * C)
        assert bench.block_flops(rows, C, H, R) == 2 * macs
    assert round(bench.block_flops(8192, 4, 2560, 320) / 1e9, 2) == 108.05
    assert round(bench.block_flops(8192, 8, 1280, 320) / 1e9, 2) == 108.72


def test_recorded_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"dram_bytes_per_unit": 123, "source_hash": "abc", "sources": ["x.cu"]}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=(): "abc")
    assert bench.recorded_traffic("k") == 123
    assert bench.recorded_traffic("missing") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=(): "changed")
    assert bench.recorded_traffic("k") is None


def test_committed_traffic_record_names_existing_sources():
    j = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    csrc = os.path.join(bench.ROOT, "hyper_connection_rank_gb300", "csrc")
    for name, e in j.items():
        assert e["dram_bytes_per_unit"] > 0 and len(e["source_hash"]) == 16
        for fn in e["sources"]:
            assert os.path.exists(os.path.join(csrc, fn)), f"{name}: {fn} is not a kernel source"


def test_peak_fallback_without_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.peaks()
    assert p["source"] == "fallback" and p["hbm"] == 6800.0 and p["bf16"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0}))
    p = bench.peaks()
    assert p["source"] == "measured" and p["hbm"] == 7000.0 and p["bf16_sustained"] == 2000.0


class _FakeProc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_record_parsing():
    lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ]
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.p = _FakeProc("\n".join(lines))
    r = s.stop()
    assert r == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    s.p = None
    assert s.stop() is None
