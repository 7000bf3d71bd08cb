"""Host logic of the benchmark, on fake nvidia-smi output (CPU only)."""
import datetime
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


REF_KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _json_lines(text):
    import json
    return [json.loads(line) for line in text.splitlines() if line.startswith("{")]


def _check_reference_line(d, n_gpus):
    import bench
    assert REF_KEYS <= set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == n_gpus
    assert (d["metric"], d["unit"], d["higher_is_better"]) == (bench.METRIC, bench.UNIT, True)
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` times the oracle on the host cores and
    prints one line with the headline's metric, unit and workload."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--ref-tokens", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 1)


def test_reference_arm_under_two_ranks():
    """Launched as two ranks (gloo on the CPU): rank 0 alone runs and prints
    the line; the other rank exits 0 without work."""
    import socket
    import subprocess
    import sys
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--ref-tokens", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0], 2)


def test_every_profile_summary_names_its_sources_and_command():
    """Each committed ncu summary gives the command that made it and the
    kernel sources it was taken on, and those sources are the current ones
    (a kernel changed after its capture would make the benchmark report
    its traffic as null)."""
    import glob
    paths = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.txt")))
    assert paths
    for path in paths:
        text = open(path).read()
        vals = dict((k.strip(), v.strip()) for k, v in (line.split(":", 1) for line in text.splitlines()
                                                         if ":" in line))
        assert "ncu" in text and "--clock-control none" in text, path
        srcs = [s.strip() for s in vals["sources"].split(",")]
        assert vals["source_sha256_16"] == bench.src_hash(*srcs), f"{path}: taken on other sources"
