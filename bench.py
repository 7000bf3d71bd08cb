#!/usr/bin/env python
"""Benchmark of the DSA decode step: Indexer Prolog -> Lightning Indexer ->
top-k -> sparse MLA attention, B=4 sequences, MTP1 (2 query tokens each),
64K keys per sequence, on one GB300 per process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is whole-job query tokens per
second measured on the device (CUDA events on the launching stream, one CUDA
graph per step, max over ranks).  By default the steps rotate over 4
independent device copies of every input (caches, weights, queries; about
1.4 GB), so no step finds its inputs in the 126 MB L2 left by the steps
before it; `--l2 flush` instead writes 256 MiB before every step (which also
evicts the kernels' code from L2).  `e2e` repeats
the step through the C ABI with host buffers (pinned H2D of the step's new
inputs, D2H of the attention output) timed on the host, launched as one CUDA
graph per step (the copies and calls issued one by one are reported beside
it as `eager_value`); `roofline` is the
dominant kernel's algorithmic bytes / its event-timed duration against the
measured HBM copy bandwidth.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sparse_attention_prolog_gb300 import dist as D  # noqa: E402
from sparse_attention_prolog_gb300 import workloads as W  # noqa: E402

METRIC = "decode query-tok/s (prolog+indexer+topk+sparse attn), B=4 MTP1 64K; % roofline"
UNIT = "query-tok/s"
WORKLOAD = ("decode B=4 x MTP1 (T=8 query tokens), KV 65536 per sequence; indexer H_I=64 d_I=128 int8, "
            "top-2048; sparse MLA attention 128 heads d_qk=576 d_v=512 bf16; prolog T=8 K_q=1536 D_x=7168")
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ bytes
def prolog_bytes(p) -> int:
    """Algorithmic HBM bytes of one prolog launch: every weight and input
    read once, every output written once."""
    n = p.q_lora.nbytes + p.q_lora_scale.nbytes + p.w_qb.nbytes + p.w_qb_scale.nbytes + p.x.nbytes
    n += p.w_k.nbytes + (p.w_proj.nbytes if p.w_proj is not None else 0)
    n += p.T * p.H_I * (p.d_I + 2) + p.T * (p.d_I + 2) + (p.T * p.H_I * 4 if p.w_proj is not None else 0)
    return int(n)


def indexer_bytes(inp) -> int:
    """Keys visible to some token of their sequence (int8 d_I + fp16 scale
    each) plus the query rows, their scales and weights."""
    keys = sum(int(inp.pos[inp.seq_of_token == b].max()) + 1 for b in range(inp.B))
    return int(keys * (inp.d_I + 2) + inp.T * inp.H_I * (inp.d_I + 2 + 4))


def attention_bytes(inp, idx: np.ndarray) -> int:
    """q, the distinct selected latent rows of each sequence (1152 B each),
    the index rows and the bf16 output."""
    rows = 0
    for b in range(inp.B):
        sel = idx[inp.seq_of_token == b]
        rows += np.unique(sel[sel >= 0]).size
    return int(inp.T * inp.H * inp.d_qk * 2 + rows * inp.d_qk * 2 + idx.size * 4 + inp.T * inp.H * inp.d_v * 2)


def topk_bytes(inp) -> int:
    """The selected indices.  The fp32 score rows the top-k reads are written
    by the indexer just before and stay in L2 (2 MB at decode), so they are
    not HBM traffic of the step."""
    return int(inp.T * inp.topk * 4)


# ----------------------------------------------------------------- clocks
CLOCK_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def _sample_time(stamp: str):
    """nvidia-smi's timestamp field ('YYYY/MM/DD HH:MM:SS.mmm', local time)
    as seconds since the epoch, or None."""
    import datetime
    try:
        return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return None


def summarize_clocks(lines, uuid: str, t0: float = None, t1: float = None) -> dict:
    """Median SM clock, the maximum clock and the throttle reasons seen in the
    samples of one GPU (matched by uuid; index 0 if no uuid matches) taken
    within [t0, t1] (host wall-clock seconds).  If no sample fell inside the
    window (a region shorter than the polling period) every sample is used
    and "samples_in_window" says 0."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) >= 11:
            rows.append(parts)
    want = uuid.lower().replace("gpu-", "")
    mine = [r for r in rows if r[2].lower().replace("gpu-", "") == want]
    if mine:
        rows = mine
    elif len({r[2] for r in rows}) > 1:
        rows = [r for r in rows if r[1] == "0"]
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    inside = rows
    if t0 is not None and t1 is not None:
        inside = [r for r in rows if (_sample_time(r[0]) is not None and t0 <= _sample_time(r[0]) <= t1)]
    used = inside if inside else rows
    num = lambda v: v.replace(".", "", 1).isdigit()
    sm = [float(r[3]) for r in used if num(r[3])]
    mx = [float(r[4]) for r in used if num(r[4])]
    reasons = sorted({CLOCK_REASONS[i] for r in used for i in range(4) if r[7 + i].lower() == "active"})
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": reasons, "samples": len(used), "samples_in_window": len(inside)}


class ClockSampler:
    """nvidia-smi polling every PERIOD_MS around a timed region: entering
    waits for the first sample, so the poller is live when the region
    starts; the summary keeps the samples stamped inside the region."""
    QUERY = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.t0 = self.t1 = None
        self.path = os.path.join(tempfile.gettempdir(), f"dsa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.PERIOD_MS)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        if self.proc is not None:
            deadline = time.time() + 5.0
            while time.time() < deadline and self.proc.poll() is None and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        self.t1 = time.time()
        if self.proc is not None:
            time.sleep(2 * self.PERIOD_MS / 1000.0)  # the samples of the region's last moments
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        with open(self.path) as f:
            return summarize_clocks(f.readlines(), self.uuid, self.t0, self.t1)


def device_uuid(dev) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return ""


# ------------------------------------------------------------------- ours
def src_hash(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sparse_attention_prolog_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(parts):
    """Sum over (kernel source, summary) pairs of the dram read+write bytes
    per launch in each committed ncu summary; None unless every summary
    exists and was taken on the current source of its kernel."""
    total = 0.0
    for kernel_file, summary in parts:
        path = os.path.join(ROOT, "profiles", summary)
        if not os.path.exists(path):
            return None
        vals = {}
        for line in open(path):
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("source_sha256_16") != src_hash(kernel_file):
            return None
        try:
            total += float(vals["traffic_bytes_per_launch"].split()[0])
        except (KeyError, ValueError):
            return None
    return total


def stage_times_in_graph(stage_fns_per_set, stream, prep, reps):
    """Mean ms of each stage inside one graph of the whole step (one graph
    per input set, replayed in rotation), from event nodes recorded between
    the stages.  None if events cannot be captured."""
    try:
        names = [n for n, _ in stage_fns_per_set[0]]
        graphs = []
        for fns in stage_fns_per_set:
            evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(fns) + 1)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                evs[0].record(stream)
                for i, (_, fn) in enumerate(fns):
                    fn(stream)
                    evs[i + 1].record(stream)
            graphs.append((g, evs))
        acc = [[] for _ in names]
        for r in range(reps + 2 * len(graphs)):
            g, evs = graphs[r % len(graphs)]
            with torch.cuda.stream(stream):
                prep()
                g.replay()
            stream.synchronize()
            if r >= 2 * len(graphs):
                for i in range(len(names)):
                    acc[i].append(evs[i].elapsed_time(evs[i + 1]))
    except (TypeError, RuntimeError):
        return None, None
    return ({n: statistics.mean(a) for n, a in zip(names, acc)},
            "event nodes between the C calls inside one step graph (same L2 policy as the timed steps)")


def stage_times_separate(stage_fns_per_set, stream, prep, reps):
    """Fallback: each stage in its own graph, replayed alone."""
    out = {}
    for si, (name, _) in enumerate(stage_fns_per_set[0]):
        graphs = []
        for fns in stage_fns_per_set:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                fns[si][1](stream)
            graphs.append(g)
        t = []
        for r in range(reps + 2 * len(graphs)):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                prep()
                a.record(stream)
                graphs[r % len(graphs)].replay()
                b.record(stream)
            stream.synchronize()
            if r >= 2 * len(graphs):
                t.append(a.elapsed_time(b))
        out[name] = statistics.mean(t)
    return out, "one graph per stage, replayed alone (same L2 policy as the timed steps)"


def run_ours(args, rank, world, local):
    from sparse_attention_prolog_gb300 import binding as B
    from sparse_attention_prolog_gb300.pipeline import DecodeBuffers, PrologBuffers

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.load()
    inp = W.decode_64k(seed=D.replica_seed(1002, rank))
    p = W.decode_64k_prolog(seed=D.replica_seed(2002, rank))
    n_sets = max(1, args.rotate) if args.l2 == "rotate" else 1
    sets = []
    for _ in range(n_sets):  # independent device copies of every input
        kc = torch.from_numpy(inp.k_cache).to(dev)
        ks = torch.from_numpy(inp.k_scale).to(dev)
        pro = PrologBuffers(p, dev, kc, ks)
        buf = DecodeBuffers(inp, dev, q_idx=pro.q_out, q_idx_scale=pro.q_scale_out, w_idx=pro.w_out, k_cache=kc,
                            k_scale=ks, keep_scores=True)
        sets.append((pro, buf))
    pro, buf = sets[0]
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if args.l2 == "flush" else None

    def prep():  # before every timed step, outside the events
        if flush is not None:
            flush.zero_()

    def step_of(pr, bu):
        def step(s):
            pr.run(s)
            bu.run(s)
        return step

    steps = [step_of(pr, bu) for pr, bu in sets]
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            for st in steps:
                st(stream)
    stream.synchronize()
    if B.device_error() != 0:
        raise RuntimeError("device-side error during warm-up")

    graphs = []
    for st in steps:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            st(stream)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for w in range(max(args.warmup, 3) * len(graphs)):
            prep()
            graphs[w % len(graphs)].replay()
    stream.synchronize()

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    # The clock poll (every 20 ms) needs a loaded window longer than a short
    # timed region: untimed replays of the same step graphs run just before
    # and after the timed steps, inside the sampler's window.
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for w in range(2 * len(graphs)):
            graphs[w % len(graphs)].replay()
        b.record(stream)
    stream.synchronize()
    est_ms = max(a.elapsed_time(b) / (2 * len(graphs)), 1e-3)
    soak_pre, soak_post = int(150.0 / est_ms) + 1, int(60.0 / est_ms) + 1

    def soak(n):
        with torch.cuda.stream(stream):
            for w in range(n):
                prep()
                graphs[w % len(graphs)].replay()

    with ClockSampler(device_uuid(dev)) as clk:
        soak(soak_pre)
        D.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for k in range(K):
                prep()
                starts[k].record(stream)
                graphs[k % len(graphs)].replay()
                ends[k].record(stream)
        torch.cuda.synchronize()
        D.barrier()
        soak(soak_post)
        torch.cuda.synchronize()
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms_max = D.max_over_ranks(ms, dev)
    tokens_total = D.sum_over_ranks(inp.T, dev)
    value = tokens_total / (ms_max / 1e3)
    clocks = clk.summary()
    clocks["window"] = (f"the {K} timed steps with {soak_pre} untimed replays of the same step graphs before "
                        f"and {soak_post} after them (one loaded window, sampled every {ClockSampler.PERIOD_MS} ms)")

    # Per-stage times inside the step: a second copy of the step graph with
    # event nodes at the boundaries of the three C calls (event nodes split
    # the programmatic-launch overlap, so this copy is not the timed one).
    stage_fns = [[("prolog", lambda s, pr=pr: pr.run(s)), ("indexer+topk", lambda s, bu=bu: bu.run_topk(s)),
                  ("attention+combine", lambda s, bu=bu: bu.run_attn(s))] for pr, bu in sets]
    reps = min(max(K, 5), 50)
    st_ms, stage_timing = stage_times_in_graph(stage_fns, stream, prep, reps)
    if st_ms is None:
        st_ms, stage_timing = stage_times_separate(stage_fns, stream, prep, reps)
    idx = buf.topk_idx.cpu().numpy()
    peak, peak_kind = measured_peaks()
    alg = {"prolog": prolog_bytes(p), "indexer+topk": indexer_bytes(inp) + topk_bytes(inp),
           "attention+combine": attention_bytes(inp, idx)}
    dom = max(alg, key=lambda k: st_ms[k])
    kfile = {"prolog": [("prolog.cu", "prolog_decode64k.txt")],
             "indexer+topk": [("indexer.cu", "indexer_decode64k.txt"), ("topk.cu", "topk_decode64k.txt")],
             "attention+combine": [("attention.cu", "attention_decode64k.txt"), ("attention.cu", "combine_decode64k.txt")]}[dom]
    achieved = alg[dom] / (st_ms[dom] / 1e3) / 1e9
    step_bytes = sum(alg.values())

    # end to end through the C ABI with host buffers: every step copies its
    # new inputs (queries, positions, slots, hidden states) from pinned host
    # memory into the input set it runs on and reads the attention output back
    names = ["q_lora", "q_lora_scale", "x", "pos_prolog", "slot", "pos", "q_attn"]

    def dev_inputs(pr, bu):
        return {"q_lora": pr.q_lora, "q_lora_scale": pr.q_lora_scale, "x": pr.x, "pos_prolog": pr.pos,
                "slot": pr.slot, "pos": bu.pos, "q_attn": bu.q_attn}

    pinned = {k: v.detach().cpu().pin_memory() for k, v in dev_inputs(pro, buf).items()}
    out_host = torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory()
    h2d_bytes = sum(pinned[k].numel() * pinned[k].element_size() for k in names)
    d2h_bytes = out_host.numel() * out_host.element_size()
    def e2e_step(k):  # copies in, the three C calls, the output back
        pr, bu = sets[k % len(sets)]
        dst = dev_inputs(pr, bu)
        for name in names:
            dst[name].copy_(pinned[name], non_blocking=True)
        steps[k % len(sets)](stream)
        out_host.copy_(bu.out, non_blocking=True)

    # As a serving loop launches it: one CUDA graph per input set holding the
    # copies and the C calls (every replay copies from the pinned buffers and
    # back); the same work issued call by call is reported beside it.
    e2e_graphs = []
    try:
        for k in range(len(sets)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                e2e_step(k)
            e2e_graphs.append(g)
    except RuntimeError:
        e2e_graphs = []

    def time_e2e(use_graphs):
        ts = []
        n_e2e = min(K, 50) + 2 * len(sets)
        for k in range(n_e2e):
            with torch.cuda.stream(stream):
                prep()
            stream.synchronize()
            t0 = time.perf_counter()
            with torch.cuda.stream(stream):
                if use_graphs:
                    e2e_graphs[k % len(sets)].replay()
                else:
                    e2e_step(k)
            stream.synchronize()
            if k >= 2 * len(sets):
                ts.append(time.perf_counter() - t0)
        return D.max_over_ranks(statistics.mean(ts), dev)

    e2e_eager_s = time_e2e(False)
    e2e_serial_s = time_e2e(True) if e2e_graphs else e2e_eager_s

    # As a serving loop overlaps them: step k+1's inputs are copied from
    # pinned memory into its input set on a copy stream while step k runs,
    # and step k's output is read back on a third stream while step k+1
    # runs.  The set of step k+1 was last used by step k+1-S (S sets), so
    # its copy waits for that step's read-back.  Every copy of every step is
    # inside the timed region.
    S = len(sets)
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    outs_host = [torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory() for _ in range(S)]
    copy_graphs, step_graphs = [], []
    try:
        for k in range(S):
            pr, bu = sets[k]
            dst = dev_inputs(pr, bu)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs_in, capture_error_mode="relaxed"):
                for name in names:
                    dst[name].copy_(pinned[name], non_blocking=True)
            copy_graphs.append(g)
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, stream=stream, capture_error_mode="relaxed"):
                steps[k](stream)
            step_graphs.append(g2)
    except RuntimeError:
        copy_graphs, step_graphs = [], []

    def time_e2e_pipelined(n):
        copied = [torch.cuda.Event() for _ in range(n)]
        computed = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        with torch.cuda.stream(stream):
            prep()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(cs_in):
            copy_graphs[0].replay()
            copied[0].record(cs_in)
        for k in range(n):
            if k + 1 < n:
                with torch.cuda.stream(cs_in):
                    if k + 1 - S >= 0:
                        cs_in.wait_event(done[k + 1 - S])
                    copy_graphs[(k + 1) % S].replay()
                    copied[k + 1].record(cs_in)
            with torch.cuda.stream(stream):
                stream.wait_event(copied[k])
                step_graphs[k % S].replay()
                computed[k].record(stream)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(computed[k])
                outs_host[k % S].copy_(sets[k % S][1].out, non_blocking=True)
                done[k].record(cs_out)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n

    if step_graphs:
        n_pipe = max(min(K, 2000), 8 * S)
        time_e2e_pipelined(4 * S)  # warm-up
        e2e_s = D.max_over_ranks(time_e2e_pipelined(n_pipe), dev)
        e2e_launch = (f"pipelined over {n_pipe} consecutive steps: per step one CUDA graph of the 7 host-to-device "
                      "copies from pinned memory (copy stream, into the step's rotated input set), one graph of "
                      "the three C calls (compute stream) and the device-to-host read of the attention output "
                      "(read-back stream), ordered by events; host wall clock from the first copy to the last "
                      "read-back, divided by the steps")
    else:
        e2e_s = e2e_serial_s
        e2e_launch = "one CUDA graph per step of the copies and the C calls, a synchronize after each"
    e2e_value = tokens_total / e2e_s

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 indexer (exact f16 MMA), bf16 attention, fp32 accumulate",
        "data": "synthetic (seeded; replica r uses seed + 100 r)",
        "config": {"workload": WORKLOAD, "global_batch": inp.B * world, "query_tokens_per_step": int(tokens_total),
                   "l2": (f"inputs larger than L2: {len(sets)} rotating device copies of every input "
                          f"({len(sets) * 0.36:.1f} GB), no flush" if args.l2 == "rotate"
                          else "flushed before every timed step (256 MiB write, outside the events)"),
                   "timing": "one CUDA graph per step, CUDA events on its stream", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes": alg[dom],
                     "traffic": profiled_traffic(kfile)},
        "step_roofline": {"algorithmic_bytes": step_bytes,
                          "roofline_us": round(step_bytes / (peak * 1e9) * 1e6, 3),
                          "frac": round(step_bytes / (peak * 1e9) / (ms_max / 1e3), 4)},
        "stages_ms": {k: round(v, 5) for k, v in st_ms.items()},
        "stages_timing": stage_timing,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d_bytes),
                "d2h_bytes_per_step": int(d2h_bytes), "ms_per_step": round(e2e_s * 1e3, 4),
                "launch": e2e_launch,
                "serial_value": round(tokens_total / e2e_serial_s, 1),
                "serial_ms_per_step": round(e2e_serial_s * 1e3, 4),
                "serial_launch": ("one step at a time: one CUDA graph of the copies in, the three C calls and the "
                                  "copy out, then a synchronize" if e2e_graphs else
                                  "one step at a time, copies and C calls issued one by one"),
                "eager_value": round(tokens_total / e2e_eager_s, 1),
                "eager_ms_per_step": round(e2e_eager_s * 1e3, 4)},
        "gpu_launches": K * 5,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, p, budget_s=args.cpu_budget)
    return result


# ---------------------------------------------------------------- oracle
def oracle_step(inp, p, tokens):
    """The whole decode step on the CPU oracle for the given query tokens:
    prolog (all T tokens' q / k / w rows are one GEMM of the sample),
    indexer scores, full-sort top-k and attention for `tokens`."""
    import oracle as O
    kc = inp.k_cache
    ks = inp.k_scale
    pr = O.indexer_prolog(p)
    kc_rows = {int(s): (pr["k"][i], pr["k_scale"][i]) for i, s in enumerate(p.slot)}
    idx = np.full((inp.T, inp.topk), -1, np.int64)
    for t in tokens:
        b = int(inp.seq_of_token[t])
        n = int(inp.pos[t]) + 1
        rows = O.logical_rows(inp, b, n)
        keys, kscale = kc[rows].copy(), ks[rows].copy()
        for j, r in enumerate(rows[-2:]):
            if int(r) in kc_rows:
                keys[n - 2 + j], kscale[n - 2 + j] = kc_rows[int(r)]
        sc = O.indexer_scores_token(pr["q"][t], pr["q_scale"][t], pr["w"][t], keys, kscale, n - 1)
        idx[t] = O.topk_indices(sc, n, inp.topk)
    out, _ = O.sparse_attention(inp, idx, tokens)
    return out


def cpu_baseline(inp, p, budget_s=20.0):
    t0 = time.perf_counter()
    done = 0
    reps = 0
    while True:
        oracle_step(inp, p, list(range(inp.T)))
        done += inp.T
        reps += 1
        if time.perf_counter() - t0 >= budget_s or reps >= 200:
            break
    el = time.perf_counter() - t0
    return {"value": round(done / el, 4), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} full decode step(s) of the same workload ({inp.T} query tokens each), numpy float64 "
                      "(BLAS threads up to the core count)", "seconds": round(el, 2)}


def run_reference(args, rank, world):
    inp = W.decode_64k(seed=1002)
    p = W.decode_64k_prolog(seed=2002)
    per_step = list(range(args.ref_tokens))

    def one():
        oracle_step(inp, p, per_step)

    for _ in range(args.warmup):
        one()
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one()
        t.append(time.perf_counter() - t0)
    s = statistics.mean(t)
    value = len(per_step) / s
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "global_batch": inp.B, "query_tokens_per_step": len(per_step)},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"each step: the prolog of all {inp.T} tokens plus indexer, top-k and "
                                   f"attention of {len(per_step)} query token(s)"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_act_quant(args):
    """The standalone activation quantiser on a [16384, 7168] bf16 matrix
    (235 MB in, 118 MB out: larger than L2, so no flush is needed), timed
    launch by launch with CUDA events; its roofline is the copy bandwidth
    (2 bytes read + 1 written per element + 4 per row scale)."""
    from sparse_attention_prolog_gb300 import binding as B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M, N = 16384, 7168
    rng = np.random.default_rng(4242)
    from sparse_attention_prolog_gb300.workloads import f32_to_bf16_bits
    bits = f32_to_bf16_bits((rng.standard_normal((M, N)) * np.exp(rng.uniform(-4, 4, (M, 1)))).astype(np.float32))
    x = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.int8, device=dev)
    sc = torch.empty((M,), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            B.dsa_act_quant(x, y, sc, False, stream)
    stream.synchronize()
    K = min(args.steps, 3000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with ClockSampler(device_uuid(dev)) as clk:
        with torch.cuda.stream(stream):
            for a, b in evs:
                a.record(stream)
                B.dsa_act_quant(x, y, sc, False, stream)
                b.record(stream)
        stream.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    nbytes = M * N * 3 + M * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    res = {"metric": "act_quant GB/s (bf16 [16384,7168] -> int8 + fp32 row scales)", "value": round(gbs, 1),
           "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
           "higher_is_better": True, "dtype": "bf16 in, fp32 scale, int8 out", "data": "synthetic (seeded)",
           "config": {"workload": "act_quant M=16384 N=7168 round_scale=0",
                      "l2": "inputs larger than L2 (235 MB read per launch)"},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                        "traffic": profiled_traffic([("quant.cu", "act_quant_16384x7168.txt")])},
           "gpu_launches": K, "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        import oracle as O
        sample = bits[:512]
        t0 = time.perf_counter()
        O.act_quant(sample)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round((512 * N * 3 + 512 * 4) / dt / 1e9, 3), "unit": "GB/s",
                               "cores": 1, "kind": "oracle", "sample": "512 rows of the same matrix, numpy"}
    return res


def run_int8_gemm(args):
    """The standalone int8 GEMM for 8 decode rows against a [24576, 7168]
    int8 weight (176 MB, larger than L2), timed launch by launch with CUDA
    events; a weight stream, so its roofline is the copy bandwidth."""
    from sparse_attention_prolog_gb300 import binding as B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M, N, K = 8, 24576, 7168
    gen = torch.Generator(device=dev).manual_seed(77)
    a = torch.randint(-128, 128, (M, K), dtype=torch.int8, device=dev, generator=gen)
    b = torch.randint(-128, 128, (N, K), dtype=torch.int8, device=dev, generator=gen)
    sa = torch.full((M,), 1.0 / 128, dtype=torch.float32, device=dev)
    sb = torch.full((N,), 1.0 / (128 * K ** 0.5), dtype=torch.float32, device=dev)
    c = torch.empty((M, N), dtype=torch.float16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            B.dsa_int8_gemm(a, sa, b, sb, c, stream)
    stream.synchronize()
    K_steps = min(args.steps, 3000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
    with ClockSampler(device_uuid(dev)) as clk:
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                e0.record(stream)
                B.dsa_int8_gemm(a, sa, b, sb, c, stream)
                e1.record(stream)
        stream.synchronize()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    nbytes = N * K + M * K + M * N * 2 + (M + N) * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    res = {"metric": "int8_gemm GB/s (a int8 [8,7168] x b int8 [24576,7168] -> fp16)", "value": round(gbs, 1),
           "unit": "GB/s", "n_gpus": 1, "steps": K_steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
           "higher_is_better": True, "dtype": "int8 in, int32 accumulate, fp32 dequant, fp16 out",
           "data": "synthetic (seeded)", "config": {"workload": "int8_gemm M=8 N=24576 K=7168",
                                                   "l2": "weight larger than L2 (176 MB per launch)"},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                        "traffic": profiled_traffic([("quant.cu", "int8_gemm_8x24576x7168.txt")])},
           "gpu_launches": K_steps, "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        import oracle as O
        an, bn = a.cpu().numpy(), b[:512].cpu().numpy()
        t0 = time.perf_counter()
        O.int8_gemm(an, sa.cpu().numpy(), bn, sb[:512].cpu().numpy())
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(512 * K / dt / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                               "sample": "512 weight rows of the same problem, numpy float64"}
    return res


def run_mhc(args):
    """The mHC mappings for 2^20 tokens with 4 streams (96 bytes in and 96
    out per token, 201 MB: larger than L2), timed launch by launch."""
    from sparse_attention_prolog_gb300 import binding as B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n, hc, iters = 1 << 20, 4, 20
    w = hc * (2 + hc)
    gen = torch.Generator(device=dev).manual_seed(5)
    mixes = torch.randn((n, w), device=dev, generator=gen)
    scale = torch.tensor([0.8, 1.3, 1.7], device=dev)
    base = torch.randn((w,), device=dev, generator=gen) * 0.5
    pre, post = torch.empty((n, hc), device=dev), torch.empty((n, hc), device=dev)
    comb = torch.empty((n, hc, hc), device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            B.dsa_mhc(mixes, scale, base, hc, iters, 1e-6, pre, post, comb, stream)
    stream.synchronize()
    K_steps = min(args.steps, 3000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
    with ClockSampler(device_uuid(dev)) as clk:
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                e0.record(stream)
                B.dsa_mhc(mixes, scale, base, hc, iters, 1e-6, pre, post, comb, stream)
                e1.record(stream)
        stream.synchronize()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    nbytes = n * w * 4 * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    res = {"metric": "mhc GB/s (n=2^20 tokens, hc=4, 20 Sinkhorn rounds)", "value": round(gbs, 1), "unit": "GB/s",
           "n_gpus": 1, "steps": K_steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
           "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded)",
           "config": {"workload": "mhc n=1048576 hc=4 iters=20", "l2": "inputs larger than L2 (201 MB per launch)"},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                        "traffic": profiled_traffic([("quant.cu", "mhc_1048576x4.txt")])},
           "gpu_launches": K_steps, "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        import oracle as O
        mx = mixes[:65536].cpu().numpy()
        t0 = time.perf_counter()
        O.mhc(mx, scale.cpu().numpy(), base.cpu().numpy(), hc, iters, 1e-6)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(65536 * w * 8 / dt / 1e9, 3), "unit": "GB/s", "cores": 1,
                               "kind": "oracle", "sample": "65536 tokens of the same input, numpy float64"}
    return res


def run_mla(args):
    """The MLA Prolog of one decode step (B=4 x MTP1 = 8 tokens, 128 heads,
    K_q = 1536, D_x = 7168): 85 MB of weights per call, so three weight sets
    (255 MB, larger than L2) are rotated call by call."""
    from sparse_attention_prolog_gb300 import binding as B
    from sparse_attention_prolog_gb300 import workloads as W
    from sparse_attention_prolog_gb300.pipeline import MlaBuffers
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T, H, K_q, D_x = 8, 128, 1536, 7168
    pos = np.array([65534, 65535] * 4, dtype=np.int32)
    slot = np.arange(T, dtype=np.int64) + 65528
    p = W.make_mla_inputs(T, pos, slot, seed=9001, H=H, K_q=K_q, D_x=D_x, max_pos=65536)
    bufs = [MlaBuffers(p, dev, 65536) for _ in range(3)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            bufs[i % 3].run(stream)
    stream.synchronize()
    assert B.device_error(stream) == 0
    K_steps = min(args.steps, 3000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
    with ClockSampler(device_uuid(dev)) as clk:
        with torch.cuda.stream(stream):
            for i, (e0, e1) in enumerate(evs):
                e0.record(stream)
                bufs[i % 3].run(stream)
                e1.record(stream)
        stream.synchronize()
    assert B.device_error(stream) == 0
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    weights = K_q * D_x * 2 + 576 * D_x * 2 + H * 192 * K_q + H * 192 * 2 + H * 128 * 512 * 2 + (K_q + 512) * 4
    io = T * D_x * 2 + T * K_q + T * 2 + T * H * 576 * 2 + T * 576 * 2
    nbytes = weights + io
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    res = {"metric": "mla_prolog GB/s (T=8 tokens, H=128, K_q=1536, D_x=7168)", "value": round(gbs, 1),
           "unit": "GB/s", "n_gpus": 1, "steps": K_steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
           "higher_is_better": True, "dtype": "bf16/int8", "data": "synthetic (seeded)",
           "config": {"workload": "mla_prolog decode T=8 H=128 K_q=1536 D_x=7168",
                      "l2": f"3 weight sets rotated ({3 * weights / 1e6:.0f} MB, larger than L2)",
                      "bytes_per_call": nbytes},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
                        "traffic": profiled_traffic([("mla.cu", "mla_prolog_decode_T8.txt")])},
           "gpu_launches": 3 * K_steps, "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        import oracle as O
        reps = 3
        t0 = time.perf_counter()
        for _ in range(reps):
            O.mla_prolog(p)
        dt = (time.perf_counter() - t0) / reps
        res["cpu_baseline"] = {"value": round(nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": os.cpu_count(),
                               "kind": "oracle", "sample": f"the same call, {reps} times, numpy float64 (BLAS threads "
                                                           "up to the core count)"}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2", choices=["rotate", "flush"], default="rotate",
                    help="keep each step's inputs out of L2 by rotating input copies, or by flushing")
    ap.add_argument("--rotate", type=int, default=4, help="input copies rotated with --l2 rotate")
    ap.add_argument("--op", choices=["step", "act_quant", "int8_gemm", "mhc", "mla_prolog"], default="step",
                    help="the decode step (default), or a standalone export: the activation quantiser, the int8 "
                         "GEMM, the mHC mappings, the MLA Prolog")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.op != "step":
        run = {"act_quant": run_act_quant, "int8_gemm": run_int8_gemm, "mhc": run_mhc,
               "mla_prolog": run_mla}[args.op]
        print(json.dumps(run(args)), flush=True)
        return
    rank, world, local = D.init()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        D.shutdown()
        return
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    D.barrier()
    D.shutdown()


if __name__ == "__main__":
    main()
