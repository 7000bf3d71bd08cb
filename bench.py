#!/usr/bin/env python
"""Benchmark of the DSA decode step: Indexer Prolog -> Lightning Indexer ->
top-k -> sparse MLA attention, B=4 sequences, MTP1 (2 query tokens each),
64K keys per sequence, on one GB300 per process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is whole-job query tokens per
second measured on the device (one CUDA graph per step, K graphs replayed back
to back between one pair of CUDA events on the launching stream, max over
ranks).  By default the steps rotate over 4
independent device copies of every input (caches, weights, queries; about
1.4 GB), so no step finds its inputs in the 126 MB L2 left by the steps
before it; `--l2 flush` instead writes 256 MiB before every step (which also
evicts the kernels' code from L2).  `e2e` repeats
the step through the C ABI with host buffers (pinned H2D of the step's new
inputs, D2H of the attention output) timed on the host: step k+1's copies
in and step k's read-back overlap step k's calls on their own streams, as a
serving loop runs them; the serial loop (copies, calls and read-back, then a
synchronize) and the calls issued one by one are reported beside it as
`serial_value` and `eager_value`; `roofline` is the
dominant kernel's algorithmic bytes / its event-timed duration against the
measured HBM copy bandwidth.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
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
SOAK_MS = (150.0, 60.0)  # untimed replays before / after the timed steps (the clock window)


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
    """Sum over (kernel sources, summary) pairs of the dram read+write bytes
    per launch in each committed ncu summary; None unless every summary
    exists and was taken on the current sources of its kernel (a kernel's
    sources are its .cu file and the headers it takes device code from,
    joined by '+')."""
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
        if vals.get("source_sha256_16") != src_hash(*kernel_file.split("+")):
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


def time_replays(graphs, K, stream, prep, dev):
    """ms per step of K replays of graphs[k % len(graphs)], with a barrier and
    a synchronize on both sides of the timed region, and the clocks of a
    loaded window around it: untimed replays of the same graphs run just
    before and after the timed ones, so that the 20 ms clock poll sees the
    region however short it is.  Without `prep` the K replays run back to
    back between one pair of CUDA events on the launching stream (total / K);
    with it (an L2 flush before every step), events around each replay keep
    the flush outside the timed region and the mean is returned."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for w in range(2 * len(graphs)):
            graphs[w % len(graphs)].replay()
        b.record(stream)
    stream.synchronize()
    est_ms = max(a.elapsed_time(b) / (2 * len(graphs)), 1e-3)
    soak_pre = int(SOAK_MS[0] / est_ms) + 1 if SOAK_MS[0] > 0 else 0
    soak_post = int(SOAK_MS[1] / est_ms) + 1 if SOAK_MS[1] > 0 else 0

    def soak(n):
        with torch.cuda.stream(stream):
            for w in range(n):
                if prep is not None:
                    prep()
                graphs[w % len(graphs)].replay()

    with ClockSampler(device_uuid(dev)) as clk:
        soak(soak_pre)
        D.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            if prep is None:
                a.record(stream)
                for k in range(K):
                    graphs[k % len(graphs)].replay()
                b.record(stream)
            else:
                for k in range(K):
                    prep()
                    starts[k].record(stream)
                    graphs[k % len(graphs)].replay()
                    ends[k].record(stream)
        torch.cuda.synchronize()
        D.barrier()
        soak(soak_post)
        torch.cuda.synchronize()
    if prep is None:
        ms = a.elapsed_time(b) / K
    else:
        ms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in zip(starts, ends))
    clocks = clk.summary()
    clocks["window"] = (f"the {K} timed steps with {soak_pre} untimed replays of the same step graphs before "
                        f"and {soak_post} after them (one loaded window, sampled every {ClockSampler.PERIOD_MS} ms)")
    return ms, clocks


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        fn(stream)
    return g


def pipelined_e2e(dev, stream, io, n, prep=lambda: None):
    """End to end through the C ABI, as a serving loop overlaps it.  io[k] =
    (copy_in, step, read_out) of input set k: copy_in(s) copies a step's
    inputs from pinned host memory into set k, step(s) issues the C calls on
    set k, read_out(s) copies the result into pinned host memory.  Step j
    uses set j % S; its inputs are copied on a copy stream while step j-1
    runs, its result is read back on a third stream while step j+1 runs, and
    the copy into a set waits for the read-back of the step that used it
    last.  Returns seconds per step over n steps (host wall clock from the
    first copy to the last read-back), or None if the copies or calls cannot
    be captured as graphs."""
    S = len(io)
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    try:
        copy_graphs = [capture(c, cs_in) for c, _, _ in io]
        step_graphs = [capture(st, stream) for _, st, _ in io]
    except RuntimeError:
        return None

    def run(m):
        copied = [torch.cuda.Event() for _ in range(m)]
        computed = [torch.cuda.Event() for _ in range(m)]
        done = [torch.cuda.Event() for _ in range(m)]
        with torch.cuda.stream(stream):
            prep()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(cs_in):
            copy_graphs[0].replay()
            copied[0].record(cs_in)
        for k in range(m):
            if k + 1 < m:
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
                io[k % S][2](cs_out)
                done[k].record(cs_out)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / m

    run(2 * S)  # warm-up
    return run(n)


def nbytes(*tensors) -> int:
    return int(sum(t.numel() * t.element_size() for t in tensors))


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
    ms, clocks = time_replays(graphs, K, stream, prep if flush is not None else None, dev)
    ms_max = D.max_over_ranks(ms, dev)
    tokens_total = D.sum_over_ranks(inp.T, dev)
    value = tokens_total / (ms_max / 1e3)

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
    kfile = {"prolog": [("prolog.cu+dsa_ptx.cuh", "prolog_decode64k.txt")],
             "indexer+topk": [("indexer.cu+dsa_ptx.cuh", "indexer_decode64k.txt"), ("topk.cu+dsa_ptx.cuh", "topk_decode64k.txt")],
             "attention+combine": [("attention.cu+dsa_ptx.cuh", "attention_decode64k.txt"), ("attention.cu+dsa_ptx.cuh", "combine_decode64k.txt")]}[dom]
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

    # As a serving loop overlaps them (see pipelined_e2e): step k+1's inputs
    # are copied while step k runs, step k's output is read back while step
    # k+1 runs; every copy of every step is inside the timed region.
    S = len(sets)
    outs_host = [torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory() for _ in range(S)]

    def io_of(k):
        pr, bu = sets[k]
        dst = dev_inputs(pr, bu)

        def copy_in(s_):
            for name in names:
                dst[name].copy_(pinned[name], non_blocking=True)

        def read_out(s_):
            outs_host[k].copy_(bu.out, non_blocking=True)
        return copy_in, steps[k], read_out

    n_pipe = max(min(K, 2000), 8 * S)
    e2e_s = pipelined_e2e(dev, stream, [io_of(k) for k in range(S)], n_pipe, prep)
    if e2e_s is not None:
        e2e_s = D.max_over_ranks(e2e_s, dev)
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
                   "timing": ("one CUDA graph per step, K replays back to back between one pair of CUDA events on its "
                              "stream" if flush is None else "one CUDA graph per step, CUDA events around each "
                              "replay (the flush before it outside)"), "parallelism": f"replicas x{world}"},
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


# ------------------------------------------------- the other three workloads
def measured_tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s) and its kind: the sustained cuBLAS
    figure (the prefill kernels run for milliseconds inside a long step); f16
    operands run at the bf16 rate."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured sustained bf16 dense (cuBLAS)"
        return float(d["bf16_tflops"]), "measured burst bf16 dense (cuBLAS)"
    return 1700.0, "fallback sustained bf16 dense"


def prolog_config(args, dev, K):
    """The Indexer Prolog alone: T=8 tokens at positions 0..7, no weight
    stream (14.6 MB per call).  Twelve input sets (175 MB) rotate, so no call
    finds its weights in L2."""
    from sparse_attention_prolog_gb300 import binding as B
    from sparse_attention_prolog_gb300.pipeline import PrologBuffers
    p = W.prolog_alone()
    S = 12
    sets = [PrologBuffers(p, dev) for _ in range(S)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            for pr in sets:
                pr.run(stream)
    stream.synchronize()
    if B.device_error() != 0:
        raise RuntimeError("device-side error in the prolog warm-up")
    graphs = [capture(pr.run, stream) for pr in sets]
    ms, clocks = time_replays(graphs, K, stream, None, dev)
    peak, peak_kind = measured_peaks()
    alg = prolog_bytes(p)
    achieved = alg / (ms / 1e3) / 1e9
    names = ["q_lora", "q_lora_scale", "x", "pos", "slot"]
    pinned = {n: getattr(sets[0], n).detach().cpu().pin_memory() for n in names}
    rows = int(p.slot.max()) + 1
    outs = [(torch.empty(sets[0].q_out.shape, dtype=torch.int8).pin_memory(),
             torch.empty(sets[0].q_scale_out.shape, dtype=torch.float16).pin_memory(),
             torch.empty((rows, p.d_I), dtype=torch.int8).pin_memory(),
             torch.empty((rows,), dtype=torch.float16).pin_memory()) for _ in range(S)]

    def io_of(k):
        pr = sets[k]

        def copy_in(s_):
            for n in names:
                getattr(pr, n).copy_(pinned[n], non_blocking=True)

        def read_out(s_):
            o = outs[k]
            o[0].copy_(pr.q_out, non_blocking=True)
            o[1].copy_(pr.q_scale_out, non_blocking=True)
            o[2].copy_(pr.k_cache[:rows], non_blocking=True)
            o[3].copy_(pr.k_scale_cache[:rows], non_blocking=True)
        return copy_in, pr.run, read_out

    n_pipe = max(min(K, 2000), 8 * S)
    e2e_s = pipelined_e2e(dev, stream, [io_of(k) for k in range(S)], n_pipe)
    res = {
        "metric": "prolog query-tok/s (Indexer Prolog alone, T=8); % roofline", "value": round(p.T / (ms / 1e3), 1),
        "unit": "query-tok/s", "n_gpus": 1, "steps": K, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "dtype": "int8 q GEMM (dp4a), bf16 k GEMM (tcgen05), fp32 epilogue", "data": "synthetic (seeded)",
        "config": {"workload": "Indexer Prolog alone: T=8, positions 0..7, H_I=64 d_I=128, K_q=1536, D_x=7168, "
                               "no weight stream", "l2": f"{S} rotating input sets ({S * alg / 1e6:.0f} MB), no flush"},
        "roofline": {"bound": "hbm", "kernel": "prolog_kernel", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes": alg,
                     "traffic": profiled_traffic([("prolog.cu+dsa_ptx.cuh", "prolog_alone_T8.txt")])},
        "gpu_launches": K, "clocks": clocks,
    }
    if e2e_s is not None:
        res["e2e"] = {"value": round(p.T / e2e_s, 1), "unit": "query-tok/s",
                      "h2d_bytes_per_step": nbytes(*pinned.values()), "d2h_bytes_per_step": nbytes(*outs[0]),
                      "ms_per_step": round(e2e_s * 1e3, 4),
                      "launch": f"pipelined over {n_pipe} calls (copy stream, compute stream, read-back stream)"}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = prolog_cpu_baseline(p)
    return res


def prolog_cpu_baseline(p):
    """The oracle's Indexer Prolog on the same inputs, repeated for ~3 s."""
    import oracle as O
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < 3.0:
        O.indexer_prolog(p)
        reps += 1
    el = time.perf_counter() - t0
    return {"value": round(reps * p.T / el, 3), "unit": "query-tok/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} full calls of the same workload, numpy float64"}


def prefill_config(args, dev, K):
    """Causal prefill: B=1, S=8192 query tokens over 8192 keys, top-2048
    among s <= t, 128 attention heads; the indexer and the attention are
    tensor-core bound, so the roofline is the dense tensor peak.  Its
    queries (1.2 GB) and outputs (1.1 GB) exceed L2: one input set."""
    from sparse_attention_prolog_gb300 import binding as B
    from sparse_attention_prolog_gb300.pipeline import DecodeBuffers
    inp = W.causal_prefill()
    buf = DecodeBuffers(inp, dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(2):
            buf.run(stream)
    stream.synchronize()
    if B.device_error() != 0:
        raise RuntimeError("device-side error in the prefill warm-up")
    graphs = [capture(buf.run, stream)]
    ms, clocks = time_replays(graphs, K, stream, None, dev)
    st_ms, stage_timing = stage_times_in_graph([[("indexer+topk", buf.run_topk), ("attention", buf.run_attn)]],
                                               stream, lambda: None, max(K, 3))
    if st_ms is None:
        st_ms, stage_timing = stage_times_separate([[("indexer+topk", buf.run_topk), ("attention", buf.run_attn)]],
                                                   stream, lambda: None, max(K, 3))
    n_vis = np.minimum(inp.pos.astype(np.int64) + 1, inp.max_L)
    idx_ops = float(n_vis.sum()) * inp.H_I * inp.d_I * 2
    att_flop = float(np.minimum(n_vis, inp.topk).sum()) * inp.H * (inp.d_qk + inp.d_v) * 2
    peak, peak_kind = measured_tensor_peak()
    stage = {"indexer+topk": idx_ops / (st_ms["indexer+topk"] / 1e3) / 1e12,
             "attention": att_flop / (st_ms["attention"] / 1e3) / 1e12}
    dom = max(st_ms, key=lambda k: st_ms[k])
    step_tf = (idx_ops + att_flop) / (ms / 1e3) / 1e12
    names = ["q_idx", "q_idx_scale", "w_idx", "pos", "q_attn"]
    pinned = {n: getattr(buf, n).detach().cpu().pin_memory() for n in names}
    out_host = torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory()

    def copy_in(s_):
        for n in names:
            getattr(buf, n).copy_(pinned[n], non_blocking=True)

    def read_out(s_):
        out_host.copy_(buf.out, non_blocking=True)

    n_pipe = max(min(K, 10), 3)
    e2e_s = pipelined_e2e(dev, stream, [(copy_in, buf.run, read_out)], n_pipe)
    res = {
        "metric": "prefill query-tok/s (indexer+topk+sparse attn), B=1 S=8192 causal top-2048; % tensor roofline",
        "value": round(inp.T / (ms / 1e3), 1), "unit": "query-tok/s", "n_gpus": 1, "steps": K,
        "ms_per_step": round(ms, 4), "higher_is_better": True,
        "dtype": "int8 indexer (exact f16 MMA), bf16 attention, fp32 accumulate", "data": "synthetic (seeded)",
        "config": {"workload": "causal prefill B=1, S=8192 query tokens over KV 8192, H_I=64 d_I=128 int8, top-2048 "
                               "(rows t<2048 keep t+1), sparse MLA attention 128 heads d_qk=576 d_v=512 bf16",
                   "l2": "inputs larger than L2 (1.3 GB of queries per step), one set, no flush"},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": round(stage[dom], 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(stage[dom] / peak, 4), "peak_kind": peak_kind,
                     "algorithmic_flops": idx_ops if dom == "indexer+topk" else att_flop,
                     "traffic": profiled_traffic([("indexer.cu+dsa_ptx.cuh", "indexer_prefill8192.txt"),
                                                  ("topk.cu+dsa_ptx.cuh", "topk_prefill8192.txt")] if dom == "indexer+topk"
                                                 else [("attention.cu+dsa_ptx.cuh", "attention_prefill8192.txt")])},
        "stage_roofline": {k: {"achieved_tflops": round(v, 1), "frac": round(v / peak, 4)} for k, v in stage.items()},
        "step_roofline": {"algorithmic_flops": idx_ops + att_flop, "achieved_tflops": round(step_tf, 1),
                          "frac": round(step_tf / peak, 4)},
        "stages_ms": {k: round(v, 4) for k, v in st_ms.items()}, "stages_timing": stage_timing,
        "gpu_launches": 3 * K, "clocks": clocks,
    }
    if e2e_s is not None:
        res["e2e"] = {"value": round(inp.T / e2e_s, 1), "unit": "query-tok/s",
                      "h2d_bytes_per_step": nbytes(*pinned.values()), "d2h_bytes_per_step": nbytes(out_host),
                      "ms_per_step": round(e2e_s * 1e3, 4),
                      "launch": f"pipelined over {n_pipe} steps on one input set (the next step's copy waits for "
                                "the previous read-back)"}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = prefill_cpu_baseline(inp, n_vis)
    return res


def prefill_cpu_baseline(inp, n_vis):
    """The oracle on 256 random rows of the prefill (indexer, top-k and
    attention), extrapolated to all 8192 rows: the indexer part by the
    rows' visible keys, the attention part by their selected rows."""
    import oracle as O
    rng = np.random.default_rng(4)
    sample = np.sort(rng.choice(inp.T, size=256, replace=False))
    t0 = time.perf_counter()
    idx = np.full((inp.T, inp.topk), -1, np.int64)
    for t in sample:
        n = int(inp.pos[t]) + 1
        rows = O.logical_rows(inp, 0, n)
        sc = O.indexer_scores_token(inp.q_idx[t], inp.q_idx_scale[t], inp.w_idx[t], inp.k_cache[rows],
                                    inp.k_scale[rows], n - 1)
        idx[t] = O.topk_indices(sc, n, inp.topk)
    t_idx = time.perf_counter() - t0
    t0 = time.perf_counter()
    O.sparse_attention(inp, idx, list(sample))
    t_att = time.perf_counter() - t0
    est = t_idx * n_vis.sum() / n_vis[sample].sum() + \
        t_att * np.minimum(n_vis, inp.topk).sum() / np.minimum(n_vis[sample], inp.topk).sum()
    return {"value": round(inp.T / est, 4), "unit": "query-tok/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{len(sample)} random rows of the 8192 (indexer, top-k and attention), extrapolated to all "
                      "rows by their visible keys and selected rows",
            "extrapolated": True, "seconds": round(t_idx + t_att, 2)}


def ragged_config(args, dev, K):
    """Long-context ragged decode: B=32 sequences of L ~ U[4096, 131072]
    keys, one query token each, both caches paged in 64-token blocks through
    a shuffled block table; the step is the prolog of the 32 tokens (new keys
    at each sequence's last position) + indexer/top-k + attention.  Its
    caches (2.8 GB) exceed L2: one input set."""
    from sparse_attention_prolog_gb300 import binding as B
    from sparse_attention_prolog_gb300.pipeline import DecodeBuffers, PrologBuffers
    inp = W.ragged_paged_decode()
    last = inp.seq_len.astype(np.int64) - 1
    slot = inp.block_table[np.arange(inp.B), last // inp.block_size].astype(np.int64) * inp.block_size + \
        last % inp.block_size
    p = W.make_prolog_inputs(T=inp.T, pos=inp.pos, slot=slot, seed=2005, max_pos=inp.max_L)
    kc = torch.from_numpy(inp.k_cache).to(dev)
    ks = torch.from_numpy(inp.k_scale).to(dev)
    pro = PrologBuffers(p, dev, kc, ks)
    buf = DecodeBuffers(inp, dev, q_idx=pro.q_out, q_idx_scale=pro.q_scale_out, w_idx=pro.w_out, k_cache=kc,
                        k_scale=ks, keep_scores=True)

    def step(s_):
        pro.run(s_)
        buf.run(s_)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            step(stream)
    stream.synchronize()
    if B.device_error() != 0:
        raise RuntimeError("device-side error in the ragged warm-up")
    graphs = [capture(step, stream)]
    ms, clocks = time_replays(graphs, K, stream, None, dev)
    fns = [[("prolog", pro.run), ("indexer+topk", buf.run_topk), ("attention+combine", buf.run_attn)]]
    st_ms, stage_timing = stage_times_in_graph(fns, stream, lambda: None, min(max(K, 5), 50))
    if st_ms is None:
        st_ms, stage_timing = stage_times_separate(fns, stream, lambda: None, min(max(K, 5), 50))
    idx = buf.topk_idx.cpu().numpy()
    alg = {"prolog": prolog_bytes(p), "indexer+topk": indexer_bytes(inp) + topk_bytes(inp),
           "attention+combine": attention_bytes(inp, idx)}
    dom = max(alg, key=lambda k: st_ms[k])
    peak, peak_kind = measured_peaks()
    achieved = alg[dom] / (st_ms[dom] / 1e3) / 1e9
    step_bytes = sum(alg.values())
    names = ["q_lora", "q_lora_scale", "x", "pos", "slot"]
    pinned = {n: getattr(pro, n).detach().cpu().pin_memory() for n in names}
    pinned["pos_idx"] = buf.pos.detach().cpu().pin_memory()
    pinned["q_attn"] = buf.q_attn.detach().cpu().pin_memory()
    out_host = torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory()

    def copy_in(s_):
        for n in names:
            getattr(pro, n).copy_(pinned[n], non_blocking=True)
        buf.pos.copy_(pinned["pos_idx"], non_blocking=True)
        buf.q_attn.copy_(pinned["q_attn"], non_blocking=True)

    def read_out(s_):
        out_host.copy_(buf.out, non_blocking=True)

    n_pipe = max(min(K, 200), 8)
    e2e_s = pipelined_e2e(dev, stream, [(copy_in, step, read_out)], n_pipe)
    res = {
        "metric": "ragged decode query-tok/s (prolog+indexer+topk+sparse attn), B=32 paged L~U[4K,128K]; % roofline",
        "value": round(inp.T / (ms / 1e3), 1), "unit": "query-tok/s", "n_gpus": 1, "steps": K,
        "ms_per_step": round(ms, 5), "higher_is_better": True,
        "dtype": "int8 indexer (exact f16 MMA), bf16 attention, fp32 accumulate", "data": "synthetic (seeded)",
        "config": {"workload": "ragged paged decode B=32 x 1 token, KV lengths ~ U[4096, 131072] (seeded, "
                               f"sum {int(inp.seq_len.sum())}), 64-token blocks, shuffled block table; H_I=64 d_I=128 "
                               "int8, top-2048; sparse MLA attention 128 heads; prolog T=32",
                   "l2": f"inputs larger than L2 ({(inp.k_cache.nbytes + inp.kv_cache.nbytes) / 1e9:.1f} GB of caches), "
                         "one set, no flush"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes": alg[dom],
                     "traffic": profiled_traffic({
                         "prolog": [("prolog.cu+dsa_ptx.cuh", "prolog_ragged32.txt")],
                         "indexer+topk": [("indexer.cu+dsa_ptx.cuh", "indexer_ragged32.txt"), ("topk.cu+dsa_ptx.cuh", "topk_ragged32.txt")],
                         "attention+combine": [("attention.cu+dsa_ptx.cuh", "attention_ragged32.txt"),
                                               ("attention.cu+dsa_ptx.cuh", "combine_ragged32.txt")]}[dom])},
        "step_roofline": {"algorithmic_bytes": step_bytes, "roofline_us": round(step_bytes / (peak * 1e9) * 1e6, 3),
                          "frac": round(step_bytes / (peak * 1e9) / (ms / 1e3), 4)},
        "stages_ms": {k: round(v, 5) for k, v in st_ms.items()}, "stages_timing": stage_timing,
        "gpu_launches": 5 * K, "clocks": clocks,
    }
    if e2e_s is not None:
        res["e2e"] = {"value": round(inp.T / e2e_s, 1), "unit": "query-tok/s",
                      "h2d_bytes_per_step": nbytes(*pinned.values()), "d2h_bytes_per_step": nbytes(out_host),
                      "ms_per_step": round(e2e_s * 1e3, 4),
                      "launch": f"pipelined over {n_pipe} steps on one input set (the next step's copy waits for "
                                "the previous read-back)"}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = ragged_cpu_baseline(inp, p)
    return res


def ragged_cpu_baseline(inp, p):
    """The oracle's prolog of all 32 tokens, then indexer, top-k and
    attention of every other sequence, extrapolated by the key counts."""
    import oracle as O
    picks = list(range(0, inp.B, 2))
    t0 = time.perf_counter()
    pr = O.indexer_prolog(p)
    t_pro = time.perf_counter() - t0
    t0 = time.perf_counter()
    idx_h = np.full((inp.T, inp.topk), -1, np.int64)
    for t in picks:
        n = int(inp.pos[t]) + 1
        rows = O.logical_rows(inp, t, n)
        sc = O.indexer_scores_token(pr["q"][t], pr["q_scale"][t], pr["w"][t], inp.k_cache[rows],
                                    inp.k_scale[rows], n - 1)
        idx_h[t] = O.topk_indices(sc, n, inp.topk)
    O.sparse_attention(inp, idx_h, picks)
    t_rest = time.perf_counter() - t0
    lens = inp.seq_len.astype(np.float64)
    est = t_pro + t_rest * lens.sum() / lens[picks].sum()
    return {"value": round(inp.T / est, 4), "unit": "query-tok/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"the prolog of all 32 tokens, then indexer, top-k and attention of {len(picks)} of the 32 "
                      "sequences, extrapolated by their key counts",
            "extrapolated": True, "seconds": round(t_pro + t_rest, 2)}


def mla_bytes(mp) -> int:
    """Algorithmic HBM bytes of one MLA Prolog call: its weights (w_dq, w_dkv,
    w_uq + scales, w_uk, gammas) read once, x read, q_lora, q and the latent
    rows written."""
    T, H, K_q, D_x = mp.T, mp.H, mp.K_q, mp.D_x
    weights = K_q * D_x * 2 + 576 * D_x * 2 + H * 192 * K_q + H * 192 * 2 + H * 128 * 512 * 2 + (K_q + 512) * 4
    return int(weights + T * D_x * 2 + T * K_q + T * 2 + T * H * 576 * 2 + T * 576 * 2)


def dia_config(args, dev, K):
    """One decode step of DeepSeek Indexer Attention at B=4, MTP1, 64K:
    MLA Prolog -> Indexer Prolog -> Lightning Indexer + top-k -> sparse
    attention, the attention's query and latent rows coming from the MLA
    Prolog.  Four input sets (caches and weights, 1.8 GB) rotate."""
    from sparse_attention_prolog_gb300 import binding as B
    from sparse_attention_prolog_gb300.pipeline import DiaBuffers
    dia = W.dia_decode()
    S = 4
    sets = [DiaBuffers(dia, dev) for _ in range(S)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            for st in sets:
                st.run(stream)
    stream.synchronize()
    if B.device_error() != 0:
        raise RuntimeError("device-side error in the DIA warm-up")
    graphs = [capture(st.run, stream) for st in sets]
    ms, clocks = time_replays(graphs, K, stream, None, dev)
    fns = [[("mla_prolog", st.mla.run), ("indexer_prolog", st.pro.run), ("indexer+topk", st.buf.run_topk),
            ("attention+combine", st.buf.run_attn)] for st in sets]
    reps = min(max(K, 5), 50)
    st_ms, stage_timing = stage_times_in_graph(fns, stream, lambda: None, reps)
    if st_ms is None:
        st_ms, stage_timing = stage_times_separate(fns, stream, lambda: None, reps)
    inp = dia.decode
    idx = sets[0].buf.topk_idx.cpu().numpy()
    alg = {"mla_prolog": mla_bytes(dia.mla), "indexer_prolog": prolog_bytes(dia.prolog),
           "indexer+topk": indexer_bytes(inp) + topk_bytes(inp), "attention+combine": attention_bytes(inp, idx)}
    peak, peak_kind = measured_peaks()
    dom = max(alg, key=lambda k: st_ms[k])
    achieved = alg[dom] / (st_ms[dom] / 1e3) / 1e9
    step_bytes = sum(alg.values())

    def dev_inputs(st):
        return {"x": st.mla.x, "pos_mla": st.mla.pos, "slot_mla": st.mla.slot, "pos_prolog": st.pro.pos,
                "slot_prolog": st.pro.slot, "pos": st.buf.pos}

    pinned = {k: v.detach().cpu().pin_memory() for k, v in dev_inputs(sets[0]).items()}
    outs = [torch.empty(sets[0].buf.out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(S)]

    def io_of(k):
        st = sets[k]
        dst = dev_inputs(st)

        def copy_in(s_):
            for n, t in dst.items():
                t.copy_(pinned[n], non_blocking=True)

        def read_out(s_):
            outs[k].copy_(st.buf.out, non_blocking=True)
        return copy_in, st.run, read_out

    n_pipe = max(min(K, 2000), 8 * S)
    e2e_s = pipelined_e2e(dev, stream, [io_of(k) for k in range(S)], n_pipe)
    res = {
        "metric": "DIA decode query-tok/s (MLA prolog+indexer prolog+indexer+topk+sparse attn), B=4 MTP1 64K; "
                  "% roofline",
        "value": round(inp.T / (ms / 1e3), 1), "unit": "query-tok/s", "n_gpus": 1, "steps": K,
        "ms_per_step": round(ms, 5), "higher_is_better": True,
        "dtype": "bf16 / int8 prologs, int8 indexer (exact f16 MMA), bf16 attention, fp32 accumulate",
        "data": "synthetic (seeded)",
        "config": {"workload": "DIA decode B=4 x MTP1 (T=8), KV 65536 per sequence: MLA Prolog (H=128, K_q=1536, "
                               "D_x=7168) -> Indexer Prolog (its q_lora and x) -> indexer H_I=64 d_I=128 int8, "
                               "top-2048 -> sparse MLA attention over the latent cache with the new rows",
                   "l2": f"{S} rotating input sets ({S * 0.44:.1f} GB), no flush"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "algorithmic_bytes": alg[dom],
                     "traffic": profiled_traffic({
                         "mla_prolog": [("mla.cu+w8tc.cuh+dsa_ptx.cuh", "mla_down_decode_T8.txt"), ("mla.cu+w8tc.cuh+dsa_ptx.cuh", "mla_up_decode_T8.txt"),
                                        ("mla.cu+w8tc.cuh+dsa_ptx.cuh", "mla_absorb_decode_T8.txt")],
                         "indexer_prolog": [("prolog.cu+dsa_ptx.cuh", "prolog_decode64k.txt")],
                         "indexer+topk": [("indexer.cu+dsa_ptx.cuh", "indexer_decode64k.txt"), ("topk.cu+dsa_ptx.cuh", "topk_decode64k.txt")],
                         "attention+combine": [("attention.cu+dsa_ptx.cuh", "attention_decode64k.txt"),
                                               ("attention.cu+dsa_ptx.cuh", "combine_decode64k.txt")]}[dom])},
        "step_roofline": {"algorithmic_bytes": step_bytes, "roofline_us": round(step_bytes / (peak * 1e9) * 1e6, 3),
                          "frac": round(step_bytes / (peak * 1e9) / (ms / 1e3), 4)},
        "stages_ms": {k: round(v, 5) for k, v in st_ms.items()}, "stages_timing": stage_timing,
        "gpu_launches": 8 * K, "clocks": clocks,
    }
    if e2e_s is not None:
        res["e2e"] = {"value": round(inp.T / e2e_s, 1), "unit": "query-tok/s",
                      "h2d_bytes_per_step": nbytes(*pinned.values()), "d2h_bytes_per_step": nbytes(outs[0]),
                      "ms_per_step": round(e2e_s * 1e3, 4),
                      "launch": f"pipelined over {n_pipe} steps (copy stream, compute stream, read-back stream)"}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = dia_cpu_baseline(dia)
    return res


def dia_cpu_baseline(dia):
    """The oracle's whole DIA step (MLA Prolog, Indexer Prolog on its
    q_lora, indexer, top-k and attention of all 8 tokens with its query and
    latent rows), repeated for ~5 s."""
    import oracle as O
    inp, mp, pp = dia.decode, dia.mla, dia.prolog

    def one():
        m = O.mla_prolog(mp)
        p2 = dataclasses.replace(pp, q_lora=m["q_lora"], q_lora_scale=m["q_lora_scale"])
        pr = O.indexer_prolog(p2)
        kc_rows = {int(s): (pr["k"][i], pr["k_scale"][i]) for i, s in enumerate(pp.slot)}
        idx = np.full((inp.T, inp.topk), -1, np.int64)
        for t in range(inp.T):
            b, n = int(inp.seq_of_token[t]), int(inp.pos[t]) + 1
            rows = O.logical_rows(inp, b, n)
            keys, ks = inp.k_cache[rows].copy(), inp.k_scale[rows].copy()
            for j, r in enumerate(rows[-2:]):
                if int(r) in kc_rows:
                    keys[n - 2 + j], ks[n - 2 + j] = kc_rows[int(r)]
            sc = O.indexer_scores_token(pr["q"][t], pr["q_scale"][t], pr["w"][t], keys, ks, n - 1)
            idx[t] = O.topk_indices(sc, n, inp.topk)
        q_bits = W.f32_to_bf16_bits(m["q"].astype(np.float32))
        kv = inp.kv_cache.copy()
        kv[mp.slot] = W.f32_to_bf16_bits(m["kv"].astype(np.float32))
        O.sparse_attention(dataclasses.replace(inp, q_attn=q_bits, kv_cache=kv), idx)

    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < 5.0 and reps < 50:
        one()
        reps += 1
    el = time.perf_counter() - t0
    return {"value": round(reps * inp.T / el, 4), "unit": "query-tok/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} full DIA step(s) of the same workload (8 query tokens each), numpy float64",
            "seconds": round(el, 2)}


EXTRA_CONFIGS = {"prolog": prolog_config, "prefill": prefill_config, "ragged": ragged_config, "dia": dia_config}


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
                        "traffic": profiled_traffic([("quant.cu+w8tc.cuh+dsa_ptx.cuh", "act_quant_16384x7168.txt")])},
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
                        "traffic": profiled_traffic([("quant.cu+w8tc.cuh+dsa_ptx.cuh", "int8_gemm_8x24576x7168.txt")])},
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


def run_int8_gemm_tc(args):
    """The int8 GEMM on the tensor cores at M=4096 activation rows, N=8192,
    K=1536 (the Indexer Prolog's q GEMM over a prefill block): 103 GFLOP per
    call against the dense tensor peak (f16 operands run at the bf16 rate;
    the burst figure, the kernel being timed alone).  Three input sets
    (258 MB, larger than L2) rotate."""
    from sparse_attention_prolog_gb300 import binding as B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M, N, K = 4096, 8192, 1536
    gen = torch.Generator(device=dev).manual_seed(78)
    sets = []
    for _ in range(3):
        a = torch.randint(-128, 128, (M, K), dtype=torch.int8, device=dev, generator=gen)
        b = torch.randint(-128, 128, (N, K), dtype=torch.int8, device=dev, generator=gen)
        sa = torch.full((M,), 1.0 / 128, dtype=torch.float32, device=dev)
        sb = torch.full((N,), 1.0 / (128 * K ** 0.5), dtype=torch.float32, device=dev)
        c = torch.empty((M, N), dtype=torch.float16, device=dev)
        sets.append((a, sa, b, sb, c))
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            B.dsa_int8_gemm(*sets[i % 3], stream)
    stream.synchronize()
    assert B.device_error(stream) == 0
    K_steps = min(args.steps, 1000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_steps)]
    with ClockSampler(device_uuid(dev)) as clk:
        with torch.cuda.stream(stream):
            for i, (e0, e1) in enumerate(evs):
                e0.record(stream)
                B.dsa_int8_gemm(*sets[i % 3], stream)
                e1.record(stream)
        stream.synchronize()
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    flops = 2.0 * M * N * K
    tf = flops / (ms * 1e-3) / 1e12
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak, peak_kind = 1900.0, "fallback bf16 dense burst"
    if os.path.exists(path):
        with open(path) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured bf16 dense burst (cuBLAS)"
    res = {"metric": "int8_gemm TFLOP/s (a int8 [4096,1536] x b int8 [8192,1536] -> fp16, tensor cores)",
           "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": K_steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 5), "higher_is_better": True,
           "dtype": "int8 in (exact f16 MMA), fp32 / int32 accumulate, fp16 out", "data": "synthetic (seeded)",
           "config": {"workload": "int8_gemm M=4096 N=8192 K=1536", "l2": "3 rotating input sets (258 MB)"},
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(tf / peak, 4), "peak_kind": peak_kind, "algorithmic_flops": flops,
                        "traffic": profiled_traffic([("gemm.cu+dsa_ptx.cuh", "int8_gemm_tc_4096x8192x1536.txt")])},
           "gpu_launches": K_steps, "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = int8_gemm_tc_cpu_baseline(sets[0])
    return res


def int8_gemm_tc_cpu_baseline(s0):
    """The oracle on 256 rows of a against all of b, scaled to the call."""
    import oracle as O
    a, sa, b, sb, _ = s0
    an, bn = a[:256].cpu().numpy(), b.cpu().numpy()
    t0 = time.perf_counter()
    O.int8_gemm(an, sa[:256].cpu().numpy(), bn, sb.cpu().numpy())
    dt = time.perf_counter() - t0
    flops = 2.0 * 256 * bn.shape[0] * bn.shape[1]
    return {"value": round(flops / dt / 1e12, 5), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "256 rows of a against all of b, numpy float64 (BLAS threads up to the core count)"}


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
                        "traffic": profiled_traffic([("quant.cu+w8tc.cuh+dsa_ptx.cuh", "mhc_1048576x4.txt")])},
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
                        "traffic": profiled_traffic([("mla.cu+w8tc.cuh+dsa_ptx.cuh", "mla_down_decode_T8.txt"),
                                                     ("mla.cu+w8tc.cuh+dsa_ptx.cuh", "mla_up_decode_T8.txt"),
                                                     ("mla.cu+w8tc.cuh+dsa_ptx.cuh", "mla_absorb_decode_T8.txt")])},
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
    ap.add_argument("--config", choices=["decode", "prolog", "prefill", "ragged", "dia"], default="decode",
                    help="the workload of the step: the headline decode (default; its line also carries the other "
                         "three under 'configs'), the Indexer Prolog alone, the causal prefill, the ragged paged "
                         "decode")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="do not add the prolog, prefill and ragged lines to the decode line")
    ap.add_argument("--op", choices=["step", "act_quant", "int8_gemm", "int8_gemm_tc", "mhc", "mla_prolog"],
                    default="step",
                    help="the decode step (default), or a standalone export: the activation quantiser, the int8 "
                         "GEMM, the mHC mappings, the MLA Prolog")
    ap.add_argument("--soak-ms", type=float, default=150.0,
                    help="untimed replays of the step before the timed steps (and 40%% of it after), so that the "
                         "clock samples cover a loaded window; 0 for none (profiling runs)")
    args = ap.parse_args()
    global SOAK_MS
    SOAK_MS = (args.soak_ms, 0.4 * args.soak_ms)
    if args.warmup < 3:
        args.warmup = 3
    if args.op != "step":
        run = {"act_quant": run_act_quant, "int8_gemm": run_int8_gemm, "int8_gemm_tc": run_int8_gemm_tc,
               "mhc": run_mhc, "mla_prolog": run_mla}[args.op]
        print(json.dumps(run(args)), flush=True)
        return
    extra_steps = {"prolog": 500, "prefill": 10, "ragged": 100, "dia": 500}
    if args.config != "decode":
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        D.init()
        res = EXTRA_CONFIGS[args.config](args, dev, max(min(args.steps, extra_steps[args.config]), 3))
        res["warmup"] = args.warmup
        print(json.dumps(res), flush=True)
        D.shutdown()
        return
    rank, world, local = D.init()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        D.shutdown()
        return
    res = run_ours(args, rank, world, local)
    if world == 1 and not args.no_extra_configs:
        # the other three workloads, one line each inside the headline line
        dev = torch.device("cuda", local)
        res["configs"] = {}
        for name, fn in EXTRA_CONFIGS.items():
            torch.cuda.empty_cache()
            try:
                r = fn(args, dev, max(min(args.steps, extra_steps[name]), 3))
                r["warmup"] = args.warmup
                res["configs"][name] = r
            except Exception as e:  # a failed extra line must not hide the headline
                res["configs"][name] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0:
        print(json.dumps(res), flush=True)
    D.barrier()
    D.shutdown()


if __name__ == "__main__":
    main()
