"""bench.py's host-side helpers on CPU: the clock-sample summary, the
comment-insensitive source hash that guards the committed ncu traffic, and
the traffic lookup itself."""

import os
import shutil

import bench


def test_clock_summary_takes_the_median_and_the_active_reasons():
    import datetime

    s = bench.ClockSampler(0, interval_ms=20)
    s.lines = [
        "2026/12/02 10:00:00.000, 0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.020, 0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.040, 0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
        "2026/12/02 10:00:00.060, 0, n/a, 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s.window = [datetime.datetime(2026, 12, 2, 10, 0, 0, 10000),
                datetime.datetime(2026, 12, 2, 10, 0, 0, 50000)]
    s.soak_steps = 16
    out = s.summary()
    assert out["sm_mhz"] == 2070.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 3
    assert out["samples_in_timed_window"] == 2  # the samples at .020 and .040
    assert out["soak_steps_before_window"] == 16


def test_clock_summary_without_samples():
    assert bench.ClockSampler(0).summary() == {"sm_mhz": None, "sm_max_mhz": None,
                                               "reasons": [], "samples": 0}


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = os.path.join(bench.ROOT, "paged_kv_decode_08_gb300", "csrc")
    dst = tmp_path / "paged_kv_decode_08_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    k = dst / "kernels.cuh"
    text = k.read_text()
    k.write_text("// a new comment line\n\n" + text.replace("\n", "  // trailing\n", 3))
    assert bench.kernel_source_hash() == h0
    k.write_text(text + "\nstatic const int pkv_extra_constant = 1;\n")
    assert bench.kernel_source_hash() != h0


def test_traffic_is_reported_only_for_the_captured_kernels(monkeypatch):
    entry = bench.NCU_TRAFFIC["llama8b"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=None: entry["kernel_hash"])
    assert bench.ncu_traffic("llama8b", entry["num_splits"]) == entry["bytes_per_launch"]
    assert bench.ncu_traffic("llama8b", entry["num_splits"] + 1) is None
    assert bench.ncu_traffic("no_such_workload", 1) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda files=None: "0" * 16)
    assert bench.ncu_traffic("llama8b", entry["num_splits"]) is None


def test_every_traffic_entry_is_a_plausible_capture():
    for name, e in bench.NCU_TRAFFIC.items():
        assert len(e["kernel_hash"]) == 16, name
        assert e["bytes_per_launch"] > 0, name
        assert e["kernel"], name


def test_a_tcgen05_source_edit_leaves_the_other_kernels_traffic(tmp_path, monkeypatch):
    """Only the tcgen05 varlen kernel is built from varlen_tc.cuh: editing it
    changes that kernel's hash and no other."""
    src = os.path.join(bench.ROOT, "paged_kv_decode_08_gb300", "csrc")
    dst = tmp_path / "paged_kv_decode_08_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base, tc = bench.kernel_source_hash(), bench.kernel_source_hash(bench.TC_SOURCES)
    f = dst / "varlen_tc.cuh"
    f.write_text(f.read_text() + "\nstatic const int pkv_extra_constant = 2;\n")
    assert bench.kernel_source_hash() == base
    assert bench.kernel_source_hash(bench.TC_SOURCES) != tc
