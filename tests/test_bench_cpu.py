"""Host logic of the benchmark, on fake nvidia-smi output (CPU only)."""
import datetime

import bench


def _line(t, idx, uuid, sm, mx, hw="Not Active", thermal="Not Active", swt="Not Active", cap="Not Active"):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, {idx}, {uuid}, {sm}, {mx}, 900.5, 0x0, {hw}, {thermal}, {swt}, {cap}\n"


def test_clock_summary_keeps_the_window_and_the_gpu():
    t = 1_800_000_000.0
    lines = [_line(t - 1.0, 0, "GPU-aaa", 1000, 2070, thermal="Active"),   # before the region
             _line(t + 0.02, 0, "GPU-aaa", 2070, 2070),
             _line(t + 0.04, 0, "GPU-aaa", 2050, 2070, cap="Active"),
             _line(t + 0.06, 0, "GPU-aaa", 2070, 2070),
             _line(t + 0.05, 1, "GPU-bbb", 900, 2070, hw="Active"),        # another GPU
             "garbage line\n",
             _line(t + 2.0, 0, "GPU-aaa", 800, 2070, hw="Active")]         # after the region
    s = bench.summarize_clocks(lines, "GPU-AAA", t, t + 0.1)
    assert s["samples_in_window"] == 3 and s["samples"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples_in_the_window():
    t = 1_800_000_000.0
    lines = [_line(t - 0.5, 0, "GPU-aaa", 1980, 2070), _line(t + 0.5, 0, "GPU-aaa", 2070, 2070)]
    s = bench.summarize_clocks(lines, "GPU-aaa", t, t + 0.01)
    assert s["samples_in_window"] == 0 and s["samples"] == 2
    assert s["sm_mhz"] == (1980 + 2070) / 2
    assert bench.summarize_clocks([], "GPU-aaa")["reasons"] == ["no samples"]


def test_profiled_traffic_needs_the_current_source(tmp_path, monkeypatch):
    """The traffic of a committed ncu summary counts only when its source
    hash is the kernel file's current one; a note after the number is
    allowed; any missing or stale summary makes the total null."""
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "sparse_attention_prolog_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.src_hash("k.cu")
    (tmp_path / "profiles" / "a.txt").write_text(f"source_sha256_16: {h}\ntraffic_bytes_per_launch: 1000 (a note)\n")
    (tmp_path / "profiles" / "b.txt").write_text(f"source_sha256_16: {h}\ntraffic_bytes_per_launch: 24\n")
    assert bench.profiled_traffic([("k.cu", "a.txt"), ("k.cu", "b.txt")]) == 1024.0
    assert bench.profiled_traffic([("k.cu", "a.txt"), ("k.cu", "missing.txt")]) is None
    (csrc / "k.cu").write_text("kernel v2")
    assert bench.profiled_traffic([("k.cu", "a.txt")]) is None
