"""Benchmark of the paged KV-cache hot path on GB300.

One step = one decode step of one layer of the Llama-3-8B-shaped workload
(batch 64, stored lengths U[512, 4096], Hq 32 / Hkv 8 / head_dim 128 /
block_size 16, pool 1.25x the blocks needed, random block tables): the paged
write of each sequence's new K/V row, then in-place paged decode attention over
len + 1 tokens.  Inputs are resident in HBM; the decode reads ~604 MB of K/V
pages per step, far more than the 129 MB L2, so no flush is needed between
steps.

  python bench.py [--gpus N --steps K --warmup W] [--config C] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
(independent sequences, no collective in the data path: weak scaling) and the
time is the max over ranks.  The K timed steps follow the warm-up directly;
each timed region starts after a GPU-side hold during which the host enqueues
the K steps, and short regions are repeated (median reported) so that the
timed work adds up to ~150 ms.  The default single-GPU run also nests short
runs of the other four scenarios and of the page writes in the line
(`other_configs`).  `--config C` picks the workload (workloads.WORKLOADS):
1 the Llama-3-8B-shaped decode above (the default), 2 the same shapes with int8
pages and 16 new tokens per sequence (the gather of 16 x 2048 tokens timed
beside it), 4 256 skewed sequences sharing prefixes with 512-token splits,
3 chunked prefill (8 sequences, 512-token chunks) on the tensor cores
(TFLOP/s), 0 the tiny L2-resident decode step (per-call medians, warm and
flushed).  Other modes (each prints its own JSON line):

  --layers L         an L-layer decode step, eager launches against one CUDA graph
  --stream N_SLOTS   the Llama-3-8B-shaped batch decoded from a pinned host tier
                     through N_SLOTS scratch blocks
  --writes           the page writes alone: int8 at 64 x 16 tokens, bf16 at 8 x 512-token chunks
  --blocks           the host-side block manager's serving loop (no GPU)
  --impl reference   the float64 oracle on the host cores, bounded samples
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention HBM GB/s (% of GB300 peak) and seq-steps/s per layer"
PREFILL_METRIC = "chunked paged prefill attention TFLOP/s (8 sequences, 512-token chunks)"
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant
# kernel per workload number (decode_split_kernel for the decode workloads 1, 2
# and 4; prefill_tc_kernel for the prefill, 3), from the ncu captures summarised
# under profiles/, valid while the kernel's sources (comments and blank space
# aside) hash to source_sha.
NCU_TRAFFIC = {
    "decode": {"sources": ("decode.cu", "common.cuh", "launch.h", "tcgen05.cuh"), "source_sha": "49d4ee397a96c233",
               "bytes_per_launch": {1: 544752640 + 3192320, 2: 310436096 + 3242496, 4: 1318916864 + 12018944}},
    "prefill": {"sources": ("prefill_tc.cu", "common.cuh", "launch.h", "tcgen05.cuh"), "source_sha": "6734f6fa468fbe1b",
                "bytes_per_launch": {3: 197949952 + 17204224}},
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=1, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--split", type=int, default=0, help="decode split_tokens (0 = library default)")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="default run: skip the short runs of the other scenarios nested in the line")
    ap.add_argument("--blocks", action="store_true",
                    help="time the host-side block manager's per-step calls instead (no GPU)")
    ap.add_argument("--stream", type=int, default=0, metavar="N_SLOTS",
                    help="decode the Llama-3-8B-shaped batch from a pinned host tier through an "
                         "N_SLOTS-block scratch pool")
    ap.add_argument("--writes", action="store_true",
                    help="time the page writes alone (int8 write at 64 x 16 tokens, bf16 write of 8 x 512-token chunks)")
    ap.add_argument("--layers", type=int, default=0, metavar="L",
                    help="time an L-layer decode step (write + decode per layer, each layer its own pools), "
                         "eager launches against one CUDA graph of the whole step")
    return ap.parse_args()


def measured_peaks(key="hbm_gbs"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0}[key], "fallback"


def kernel_source_sha(names=("decode.cu", "common.cuh", "launch.h")):
    """Hash of the kernels' sources with comments and blank space removed, so
    that a stamp survives an edit of the comments but not of the code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_212_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over all ranks (the slowest
    rank's times); identity when no process group is initialised."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def gpu_hold(ms):
    """Puts a GPU-side wait of about `ms` on the current stream, so that the
    host enqueues the timed steps while the GPU waits: the timed region that
    starts after it then measures the GPU, not the host's launch rate."""
    import torch
    torch.cuda._sleep(max(1, int(ms * 1e-3 * 2.0e9)))     # clock cycles at ~2 GHz


def device_timed(step, K, stream, world, device, host_ms_per_step, est_ms_per_step,
                 min_total_ms=150.0, max_repeats=50):
    """Times exactly K steps on the device, R times over.  Every repeat is
    bracketed by a barrier and a synchronize on both sides; a GPU-side hold
    that covers the host's enqueue of the K steps sits before the start event,
    so the GPU runs the K steps back to back.  R is chosen so that the timed
    regions add up to about min_total_ms (at most max_repeats).  Returns the
    per-repeat elapsed ms (max over ranks for each repeat)."""
    import torch
    import torch.distributed as dist
    R = max(1, min(max_repeats, math.ceil(min_total_ms / max(K * est_ms_per_step, 1e-6))))
    hold = min(50.0, 0.3 + 1.25 * K * host_ms_per_step)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(R)]
    per = []
    for t0, t1 in evs:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        gpu_hold(hold)
        t0.record(stream)
        for _ in range(K):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        per.append(t0.elapsed_time(t1))
    return max_over_ranks(per, device)


def warm_up(step, W):
    """W untimed steps; returns (host ms per step spent enqueueing, GPU ms per
    step of the last half, both measured here)."""
    import torch
    for _ in range(max(1, W // 2)):
        step()
    torch.cuda.synchronize()
    n = max(1, W - W // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    e0.record()
    for _ in range(n):
        step()
    e1.record()
    host = (time.perf_counter() - h0) * 1e3 / n
    torch.cuda.synchronize()
    return host, e0.elapsed_time(e1) / n


def timing_note(per_repeat_ms, K, hold_note=True):
    return {"repeats": len(per_repeat_ms), "steps_per_repeat": K,
            "ms_per_step_median": round(statistics.median(per_repeat_ms) / K, 5),
            "ms_per_step_min": round(min(per_repeat_ms) / K, 5),
            "ms_per_step_max": round(max(per_repeat_ms) / K, 5),
            "how": ("each repeat: barrier + synchronize, a GPU-side hold while the host enqueues the K steps, "
                    "CUDA events around the K steps on the launching stream, synchronize + barrier; "
                    "ms_per_step is the median repeat / K" if hold_note else "")}


def weak_scaling_value(bytes_per_step_per_rank, world, ms_per_step):
    """Whole-job throughput in GB/s: every rank moves its own step bytes in
    the slowest rank's step time."""
    return world * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9


def ncu_traffic(kind, cfg):
    """Per-launch DRAM traffic of the dominant kernel from the committed ncu
    capture, or None when its sources changed since (or no capture exists)."""
    t = NCU_TRAFFIC[kind]
    if t["source_sha"] != kernel_source_sha(t["sources"]):
        return None
    return t["bytes_per_launch"].get(cfg)


def make_workload(cfg, device):
    from paged_kv_cache_212_gb300 import workloads as W
    if cfg == 0:
        w = W.tiny_decode(device=device)
    elif cfg == 1:
        w = W.llama8b_decode(device=device)
    elif cfg == 3:
        w = W.chunked_prefill(device=device)
    elif cfg == 2:
        w = W.llama8b_decode_int8(device=device)
    else:
        w = W.skewed_prefix_decode(device=device)
    return w


def algorithmic_bytes(w):
    """Bytes the step must move at minimum: K/V of every attended token (int8:
    codes + fp32 scales), Q and O, the table entries and lengths read; plus the
    write's new rows in and out (int8: codes + scales out)."""
    ctx = w.ctx_lens.long()
    hkv, d, bs = w.n_kv_heads, w.head_dim, w.block_size
    tokens = int(ctx.sum())
    if w.kv_format == "int8":
        kv = tokens * 2 * hkv * (d + 4)
    else:
        kv = tokens * 2 * hkv * d * 2
    qo = 2 * w.n_seqs * w.n_q_heads * d * 2
    tab = int(((ctx + bs - 1) // bs).sum()) * 4 + w.n_seqs * 4
    decode = kv + qo + tab
    rows = w.n_seqs * w.n_new * hkv
    if w.kv_format == "int8":
        write = 2 * rows * d * 2 + 2 * rows * (d + 4) + w.n_seqs * 8
    else:
        write = 2 * 2 * rows * d * 2 + w.n_seqs * 8
    return decode, write


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None

    def __enter__(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def fill_pool(P, w, device):
    """Untimed set-up: allocate the pools and place the resident prefix with
    the library's own write (int8 pages through the quantised write)."""
    import torch
    nb1 = w.n_blocks + 1
    if w.kv_format == "int8":
        kp = torch.zeros(w.pool_shape, dtype=torch.int8, device=device)
        vp = torch.zeros(w.pool_shape, dtype=torch.int8, device=device)
        ks = torch.zeros(w.scale_shape, dtype=torch.float32, device=device)
        vs = torch.zeros(w.scale_shape, dtype=torch.float32, device=device)
    else:
        kp = torch.zeros(w.pool_shape, dtype=torch.bfloat16, device=device)
        vp = torch.zeros(w.pool_shape, dtype=torch.bfloat16, device=device)
        ks = vs = None
    tables = w.tables.to(device)
    for seg in w.prefix:
        t = tables[seg.seq:seg.seq + 1]
        sp = torch.tensor([seg.start], dtype=torch.int32, device=device)
        if ks is not None:
            P.paged_kv_write_int8(seg.k[None].contiguous(), seg.v[None].contiguous(), kp, vp, ks, vs, t, sp)
        else:
            P.paged_kv_write(seg.k[None].contiguous(), seg.v[None].contiguous(), kp, vp, t, sp)
    torch.cuda.synchronize()
    del nb1
    return kp, vp, ks, vs


def cpu_baseline(cfg, budget_s=8.0):
    """The float64 oracle, as it stands, on the host cores: write + decode of
    the same workload's sequences, repeated until ~budget_s of wall time, once
    with one thread per host core and once single-threaded."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from oracle_pools import dims_of, empty_pools, write_prefix
    w = make_workload(cfg, "cpu")
    kp, vp, ks, vs = empty_pools(w, poison=False)
    write_prefix(w, kp, vp, ks, vs)
    decode_b, write_b = algorithmic_bytes(w)
    d = dims_of(w)

    def run(threads, n):
        sl = slice(0, n)
        reps, t0 = 0, time.perf_counter()
        while True:
            if w.kv_format == "int8":
                oracle.write_int8(w.k_new[sl], w.v_new[sl], kp, vp, ks, vs, d, w.tables[sl], w.start_pos[sl])
            else:
                oracle.write_bf16(w.k_new[sl], w.v_new[sl], kp, vp, d, w.tables[sl], w.start_pos[sl])
            oracle.decode(w.q[sl], kp, vp, d, w.tables[sl], w.ctx_lens[sl], w.softmax_scale, ks, vs,
                          n_threads=threads)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                return reps, el

    threads = os.cpu_count() or 1
    reps, el = run(threads, w.n_seqs)
    gbs = reps * (decode_b + write_b) / el / 1e9
    # single-threaded: the first n sequences, n such that a pass takes about a
    # quarter of the budget (the bytes counted are those of the n sequences)
    n1 = max(1, min(w.n_seqs, int(w.n_seqs * (budget_s / 4) / max(el / reps * threads, 1e-9))))
    reps1, el1 = run(1, n1)
    sub = make_sub_bytes(w, n1)
    gbs1 = reps1 * sub / el1 / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} full steps (write + float64 decode of all {w.n_seqs} sequences) in {el:.1f} s",
            "seq_steps_per_s": round(reps * w.n_seqs / el, 2),
            "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{reps1} steps of the first {n1} sequences in {el1:.1f} s",
                              "seq_steps_per_s": round(reps1 * n1 / el1, 2)}}


def prefill_row_flops(w):
    """Flops of each query row of the chunk: 4 Hq D (P_s + i + 1) per (s, i)."""
    import numpy as np
    P = np.asarray(w.stored_lens, np.int64)[:, None]
    i = np.arange(w.n_new, dtype=np.int64)[None, :]
    return 4 * w.n_q_heads * w.head_dim * (P + i + 1)


def oracle_prefill_sample(w, budget_s, threads):
    """The float64 oracle's chunk write + prefill over an evenly strided sample
    of the chunk's query rows (every sequence, rows i = 0, k, 2k, ...), k chosen
    so that one pass takes about budget_s.  Returns (flops per pass, a pass
    callable, description)."""
    import numpy as np
    import oracle
    from oracle_pools import dims_of, empty_pools, write_prefix
    kp, vp, _, _ = empty_pools(w, poison=False)
    write_prefix(w, kp, vp)
    d = dims_of(w)
    rowf = prefill_row_flops(w)

    def select(stride):
        sel = np.zeros((w.n_seqs, w.n_new), bool)
        sel[:, ::stride] = True
        return sel

    def one(sel):
        oracle.write_bf16(w.k_new, w.v_new, kp, vp, d, w.tables, w.start_pos)
        code, _, _ = oracle.prefill(w.q, kp, vp, d, w.tables, w.stored_lens, w.softmax_scale, row_select=sel,
                                    n_threads=threads)
        assert code == oracle.OK

    probe = select(w.n_new)                     # row 0 of every sequence
    t0 = time.perf_counter()
    one(probe)
    t_probe = time.perf_counter() - t0
    rate = float(rowf[probe].sum()) / max(t_probe, 1e-9)
    if t_probe <= budget_s:
        stride = max(1, int(np.ceil(float(rowf.sum()) / (rate * budget_s))))
        sel = select(stride)
        what = f"one query row in {stride} ({int(sel.sum())} of {w.n_seqs * w.n_new} rows, all heads)"
    else:
        # below one row per sequence: the single row whose key count best fits the budget
        want = rate * budget_s
        flat = rowf.reshape(-1)
        fits = np.flatnonzero(flat <= want)
        k = int(fits[np.argmax(flat[fits])]) if fits.size else int(np.argmin(flat))
        sel = np.zeros(flat.shape, bool)
        sel[k] = True
        sel = sel.reshape(rowf.shape)
        what = f"query row {k % w.n_new} of sequence {k // w.n_new} (all heads)"
    return float(rowf[sel].sum()), (lambda: one(sel)), "the chunk write + float64 prefill of " + what


def cpu_baseline_prefill(budget_s=12.0):
    """The float64 oracle's chunk write + prefill over a row sample, with one
    thread per host core and single-threaded."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    w = make_workload(3, "cpu")
    res = {}
    for threads in (os.cpu_count() or 1, 1):
        flops, run, what = oracle_prefill_sample(w, budget_s / 4, threads)
        reps, t0 = 0, time.perf_counter()
        while True:
            run()
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s / 4:
                break
        res[threads] = {"value": round(reps * flops / el / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
                        "sample": f"{reps} passes of {what} in {el:.1f} s"}
    many = os.cpu_count() or 1
    line = dict(res[many], kind="oracle")
    if many != 1:
        line["single_thread"] = res[1]
    return line


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle on the host cores, same metric and
    workload; each step is a bounded sample (the first n sequences)."""
    if rank != 0:
        return
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    import torch
    from oracle_pools import dims_of, empty_pools, write_prefix
    w = make_workload(args.config, "cpu")
    threads = os.cpu_count() or 1
    if args.config == 3:
        flops, run, what = oracle_prefill_sample(w, 150.0 / max(1, args.steps + args.warmup), threads)
        for _ in range(args.warmup):
            run()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            run()
        el = time.perf_counter() - t0
        tf = args.steps * flops / el / 1e12
        print(json.dumps({
            "impl": "reference", "metric": PREFILL_METRIC, "value": round(tf, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "n_seqs": w.n_seqs, "chunk": w.n_new},
            "cpu_baseline": {"value": round(tf, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": "each step: " + what},
            "e2e": {"value": round(tf, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
            flush=True)
        return
    kp, vp, ks, vs = empty_pools(w, poison=False)
    write_prefix(w, kp, vp, ks, vs)
    d = dims_of(w)

    def step(n, ctx0=None):
        sl = slice(0, n)
        if w.kv_format == "int8":
            oracle.write_int8(w.k_new[sl], w.v_new[sl], kp, vp, ks, vs, d, w.tables[sl], w.start_pos[sl])
        else:
            oracle.write_bf16(w.k_new[sl], w.v_new[sl], kp, vp, d, w.tables[sl], w.start_pos[sl])
        ctx = w.ctx_lens[sl].clone()
        if ctx0 is not None:
            ctx[0] = ctx0
        oracle.decode(w.q[sl], kp, vp, d, w.tables[sl], ctx, w.softmax_scale, ks, vs, n_threads=threads)

    def timed(*a):
        t0 = time.perf_counter()
        step(*a)
        return time.perf_counter() - t0

    # each step's sample fits 150 s / (steps + warmup): the first n sequences,
    # or, below one sequence, sequence 0 attending only its first ctx0 tokens
    budget = 150.0 / max(1, args.steps + args.warmup)
    t_full = timed(w.n_seqs)
    n = max(1, min(w.n_seqs, int(w.n_seqs * budget / max(t_full, 1e-9))))
    ctx0 = None
    if n == 1:
        full0 = int(w.ctx_lens[0])
        t_one = timed(1)
        if t_one > budget:
            ctx0 = max(w.n_new, min(full0, int(full0 * budget / t_one)))
    for _ in range(args.warmup):
        step(n, ctx0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(n, ctx0)
    el = time.perf_counter() - t0
    sub = make_sub_bytes(w, n, ctx0)
    gbs = args.steps * sub / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(w, args),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": (f"each step: write + float64 decode of the first {n} of {w.n_seqs} "
                                        "sequences" if ctx0 is None else
                                        f"each step: write + float64 decode of sequence 0 over its first {ctx0} "
                                        f"of {int(w.ctx_lens[0])} tokens")},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def make_sub_bytes(w, n, ctx0=None):
    """Algorithmic bytes of the step restricted to the first n sequences (and,
    with ctx0, sequence 0 attending only its first ctx0 tokens)."""
    import copy
    sub = copy.copy(w)
    sub.n_seqs = n
    sub.stored_lens = w.stored_lens[:n].clone()
    if ctx0 is not None:
        sub.stored_lens[0] = ctx0 - w.n_new
    sub.tables = w.tables[:n]
    dec, wr = algorithmic_bytes(sub)
    return dec + wr


def bench_config(w, args):
    ctx = w.ctx_lens
    return {"workload": w.name, "n_seqs": w.n_seqs, "ctx_min": int(ctx.min()), "ctx_max": int(ctx.max()),
            "ctx_total": int(ctx.sum()), "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "kv_pages": w.kv_format,
            "n_blocks": w.n_blocks, "layers_timed": 1, "split_tokens": args.split or w.split_tokens or "library default",
            "l2": "inputs larger than L2 (K/V pages read per step far exceed the 129 MB L2); no flush"}


def bench_gather(P, device, peak, reps=200):
    """The bf16 gather timed beside the int8 decode: 16 sequences of 2048 tokens into a
    contiguous [16, 8, 2048, 128] view (K and V), CUDA events over `reps` calls.
    Algorithmic bytes: every gathered K/V row read once and written once."""
    import torch
    from paged_kv_cache_212_gb300 import workloads as W
    w = W.gather_16x2048(device=device)
    kp, vp, _, _ = fill_pool(P, w, device)
    tables, lens = w.tables.to(device), w.stored_lens.to(device)
    out_tokens = w.extra["out_tokens"]
    ko = torch.empty((w.n_seqs, w.n_kv_heads, out_tokens, w.head_dim), dtype=torch.bfloat16, device=device)
    vo = torch.empty_like(ko)
    for _ in range(5):
        P.paged_kv_gather(kp, vp, tables, lens, out_tokens, k_out=ko, v_out=vo)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        P.paged_kv_gather(kp, vp, tables, lens, out_tokens, k_out=ko, v_out=vo)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nbytes = 2 * 2 * int(w.stored_lens.sum()) * w.n_kv_heads * w.head_dim * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": w.name, "ms_per_call": round(ms, 5), "algorithmic_bytes": nbytes,
            "achieved": round(gbs, 2), "unit": "GB/s", "frac": round(gbs / peak, 4), "calls": reps,
            "l2": "268 MB moved per call, larger than the 129 MB L2"}


def prefill_flops(w):
    """4 * Hq * D * sum over queries of the keys each attends (Q K^T and P V)."""
    import torch
    P = w.stored_lens.long()
    keys = int((P[:, None] + torch.arange(w.n_new)[None, :] + 1).sum())
    return 4 * w.n_q_heads * w.head_dim * keys


def run_prefill_bench(args, P, w, device, rank, world, K, W, with_e2e=True):
    """Chunked prefill (8 sequences): paged write of each sequence's 512-token
    chunk, then chunked paged prefill attention over prefix + chunk
    (tensor-core bound).  The
    step (write + prefill) and the prefill call alone are each timed as K
    calls on the device (see device_timed).  Returns the JSON line."""
    import torch
    import torch.distributed as dist
    kp, vp, _, _ = fill_pool(P, w, device)
    tables, start = w.tables.to(device), w.start_pos.to(device)
    k_new, v_new, q = w.k_new.to(device), w.v_new.to(device), w.q.to(device)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()

    def prefill():
        P.paged_prefill_attention(q, kp, vp, tables, start, w.softmax_scale, out=out, dev_status=status)

    def step():
        P.paged_kv_write(k_new, v_new, kp, vp, tables, start, dev_status=status)
        prefill()

    uuid = gpu_uuid(device)
    with ClockSampler(uuid) as clk:
        time.sleep(0.25)
        host_ms, est_ms = warm_up(step, max(3, W))
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        per = device_timed(step, K, stream, world, device, host_ms, est_ms)
        host_p, est_p = warm_up(prefill, 3)
        per_p = device_timed(prefill, K, stream, world, device, host_p, est_p)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    ms = statistics.median(per) / K
    pre_ms = statistics.median(per_p) / K
    flops = prefill_flops(w)
    peak, kind = measured_peaks("bf16_tflops")
    ach = flops / (pre_ms * 1e-3) / 1e12
    line = {"metric": PREFILL_METRIC, "value": round(world * flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "n_seqs": w.n_seqs, "chunk": w.n_new,
                       "prefix": [int(x) for x in w.stored_lens]},
            "timing": timing_note(per, K),
            "roofline": {"bound": "tensor", "kernel": "paged_prefill_attention", "achieved": round(ach, 2),
                         "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                         "traffic": ncu_traffic("prefill", 3),
                         "flops_per_launch": flops, "avg_launch_ms": round(pre_ms, 5),
                         "peak_source": f"{kind} bf16_tflops (burst)"},
            "gpu_launches": 2 * K * len(per) + K * len(per_p), "clocks": clk.summary()}
    if not with_e2e:
        return line
    # end to end: the chunk's rows, queries, tables and prefix lengths from pinned
    # host memory every step, the output back to pinned host memory
    h_in = tuple(x.cpu().pin_memory() for x in (w.k_new, w.v_new, w.q, w.tables, w.start_pos))
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = q.numel() * q.element_size()

    def call(views, o):
        dk, dv, dq, dtab, dstart = views
        P.paged_kv_write(dk, dv, kp, vp, dtab, dstart, dev_status=status)
        P.paged_prefill_attention(dq, kp, vp, dtab, dstart, w.softmax_scale, out=o, dev_status=status)

    e2e_run, cs, osm = pipelined_e2e(h_in, q, call, device, stream)
    e2e_steps = args.e2e_steps or max(10, min(K, 200))
    e2e_run(3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs.wait_event(e0)
    osm.wait_event(e0)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], device)[0]
    line["e2e"] = {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                   "steps": e2e_steps}
    return line


def blocks_serving_loop(mgr, n_slots, steps, rng_seed=20265):
    """A continuous-batching loop on a block manager (library or oracle: same
    method names).  Every step: reserve_step (preemption), begin_step (growth,
    copy-on-write pairs), export of the tables, end_step -- these four are
    timed; then, untimed, sequences that ran out of tokens are released and
    empty slots refilled with new prompts, a quarter of them as forks of a live
    sequence (sharing its blocks).  Returns (seconds in the four calls,
    copies, victims)."""
    import random
    rng = random.Random(rng_seed)
    budget = [rng.randrange(64, 1024) for _ in range(n_slots)]   # tokens each sequence still generates
    for s in range(n_slots):
        mgr.admit(s, rng.randrange(16, 2048))
    copies = victims = 0
    busy = 0.0
    for _ in range(steps):
        t0 = time.perf_counter()
        v = mgr.reserve_step()
        c = mgr.begin_step()
        mgr.export()
        mgr.end_step()
        busy += time.perf_counter() - t0
        victims += len(v)
        copies += len(c)
        _, lens, active = mgr.export()
        act = [int(x) for x in active]
        ln = [int(x) for x in lens]
        for s in range(n_slots):
            if act[s]:
                budget[s] -= 1
                if budget[s] > 0:
                    continue
                mgr.release(s)
                act[s] = 0
            n = rng.randrange(16, 2048)
            live = [t for t in range(n_slots) if act[t] and ln[t] < 2048]
            if live and rng.random() < 0.25:
                src = rng.choice(live)
                mgr.fork(src, s)
                act[s], ln[s] = 1, ln[src]
            elif mgr.can_admit([n]):
                mgr.admit(s, n)
                act[s], ln[s] = 1, n
            budget[s] = rng.randrange(64, 1024)
    return busy, copies, victims


def run_blocks_bench(args):
    """Host-side block manager (pagedkv_blocks.h) per-step cost on a 256-slot
    serving loop, the plain-Python oracle of the same rules timed beside it."""
    import paged_kv_cache_212_gb300 as P
    from paged_kv_cache_212_gb300 import build as B
    B.build()
    P.load_library()
    n_slots, bs, max_blocks = 256, 16, 256
    n_blocks = int(1.25 * n_slots * 2048 / bs)
    steps = min(args.steps, 2000)
    mgr = P.BlockManager(n_blocks, bs, n_slots, max_blocks)
    busy, copies, victims = blocks_serving_loop(mgr, n_slots, steps)
    line = {"metric": "block manager steps/s (256 slots: reserve_step, begin_step, export, end_step)",
            "value": round(steps / busy, 1), "unit": "steps/s", "n_gpus": 0, "steps": steps, "warmup": 0,
            "ms_per_step": round(1e3 * busy / steps, 4), "higher_is_better": True, "scaling": "none",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": "block manager serving loop", "n_slots": n_slots, "block_size": bs,
                       "n_blocks": n_blocks, "max_blocks": max_blocks, "copies": copies, "victims": victims},
            "note": "host code through the Python binding (ctypes call overhead included)"}
    if not args.no_cpu_baseline:
        sys.path.insert(0, ROOT)
        from oracle.block_manager import BlockManagerOracle
        osteps = max(1, min(steps, 200))
        ref = BlockManagerOracle(n_blocks, bs, n_slots, max_blocks)
        obusy, _, _ = blocks_serving_loop(ref, n_slots, osteps)
        line["cpu_baseline"] = {"value": round(osteps / obusy, 1), "unit": "steps/s", "cores": 1, "kind": "oracle",
                                "sample": f"first {osteps} steps of the same loop"}
    print(json.dumps(line), flush=True)


def run_stream_bench(args, P, device):
    """The Llama-3-8B-shaped decode with every K/V block in a pinned host tier,
    streamed through a device scratch pool of args.stream blocks (pagedkv_stream.h).
    When the batch has more blocks than the pool, the cyclic order evicts every
    block before its reuse, so each call restages the whole context over the
    CPU-GPU link: the link bounds this path."""
    import torch
    w = make_workload(1, device)
    kp, vp, _, _ = fill_pool(P, w, device)
    tables, start, ctx = w.tables.to(device), w.start_pos.to(device), w.ctx_lens.to(device)
    q = w.q.to(device)
    P.paged_kv_write(w.k_new.to(device), w.v_new.to(device), kp, vp, tables, start)
    torch.cuda.synchronize()
    host_k, host_v = kp.cpu().pin_memory(), vp.cpu().pin_memory()   # the tier: ids as in the tables
    del kp, vp
    n_slots = args.stream
    pool_k = torch.zeros((n_slots + 1,) + tuple(host_k.shape[1:]), dtype=torch.bfloat16, device=device)
    pool_v = torch.zeros_like(pool_k)
    sp = P.ScratchPool(n_slots, w.n_seqs)
    t_tab, t_len = w.tables.to(torch.int32), w.ctx_lens.to(torch.int32)
    ws = torch.empty(P.streamed_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, n_slots, w.block_size),
                     dtype=torch.uint8, device=device)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()

    def call():
        P.paged_decode_streamed(q, host_k, host_v, pool_k, pool_v, sp, t_tab, t_len, w.softmax_scale, out=out,
                                workspace=ws, dev_status=status)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the link's copy rate on this machine, measured here: the copy engine moving the
    # whole K tier (pinned host -> device, one contiguous copy), after one warm-up
    link_dst = torch.empty_like(host_k, device=device)
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    link_dst.copy_(host_k, non_blocking=True)
    l0.record(stream)
    for _ in range(3):
        link_dst.copy_(host_k, non_blocking=True)
    l1.record(stream)
    torch.cuda.synchronize()
    link_gbs = 3 * host_k.numel() * 2 / (l0.elapsed_time(l1) * 1e-3) / 1e9
    del link_dst
    # blocks staged per call (the plan is host bookkeeping: replay it on a copy)
    blocks = sum(-(-int(L) // w.block_size) for L in w.ctx_lens)
    steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    with ClockSampler(uuid) as clk:
        time.sleep(0.25)
        for _ in range(3):          # busy again right before the timed calls
            call()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    decode_b, _ = algorithmic_bytes(w)
    block_bytes = 2 * w.block_size * w.n_kv_heads * w.head_dim * 2
    staged = blocks * block_bytes if blocks > n_slots else 0
    line = {"metric": "streamed paged decode GB/s (Llama-3-8B-shaped batch 64 from a pinned host tier)",
            "value": round(decode_b / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": 1, "steps": steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "none", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "n_slots": n_slots, "blocks_per_call": blocks,
                       # a batch larger than the pool goes in tiles of half the pool
                       "tiles_per_call": -(-blocks // (n_slots // 2)) if blocks > n_slots else 1,
                       "host_tier_bytes": 2 * host_k.numel() * 2},
            "staging": {"bytes_per_call": staged, "gbs": round(staged / (ms * 1e-3) / 1e9, 2)},
            "roofline": ({"bound": "host-link", "achieved": round(staged / (ms * 1e-3) / 1e9, 2),
                          "peak": round(link_gbs, 2), "unit": "GB/s",
                          "frac": round(staged / (ms * 1e-3) / 1e9 / link_gbs, 4), "traffic": None,
                          "peak_source": "pinned host -> device copy-engine rate measured in this run"}
                         if staged else None),
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_small_bench(args, P, w, device, reps=None):
    """The tiny decode (4 sequences, all data in L2): the decode step (write +
    decode) timed call by call with CUDA events, median of the reps, once with the
    data warm in L2 and once with a buffer of twice the L2 size rewritten
    between reps outside the timed pair (flushed)."""
    import torch
    kp, vp, ks, vs = fill_pool(P, w, device)
    tables, start, ctx = w.tables.to(device), w.start_pos.to(device), w.ctx_lens.to(device)
    k_new, v_new, q = w.k_new.to(device), w.v_new.to(device), w.q.to(device)
    out = torch.empty_like(q)
    ws = torch.empty(P.decode_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, int(w.ctx_lens.sum())),
                     dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=device)

    def step():
        P.paged_decode_step(k_new, v_new, start, q, kp, vp, tables, ctx, w.softmax_scale, out=out, workspace=ws,
                            dev_status=status)

    reps = reps or max(50, min(args.steps, 2000))
    warm_n = max(5, args.warmup)

    def median_us(flushed):
        for _ in range(warm_n):
            step()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in evs:
            if flushed:
                flush.fill_(1.0)
            # a short GPU wait before each timed pair lets the host enqueue the
            # step ahead of the GPU, so the pair times the GPU, not the launches
            torch.cuda._sleep(100_000)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        t = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
        return {"median_us": round(t[len(t) // 2], 3), "p10_us": round(t[len(t) // 10], 3),
                "p90_us": round(t[(9 * len(t)) // 10], 3)}

    uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    with ClockSampler(uuid) as clk:
        time.sleep(0.25)
        warm = median_us(False)
        cold = median_us(True)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    decode_b, write_b = algorithmic_bytes(w)
    us = cold["median_us"]
    return {
        "metric": METRIC, "value": round((decode_b + write_b) / (us * 1e-6) / 1e9, 3), "unit": "GB/s",
        "n_gpus": 1, "steps": reps, "warmup": warm_n, "ms_per_step": round(us * 1e-3, 5), "higher_is_better": True,
        "scaling": "none", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(bench_config(w, args), l2=f"data fits in L2: value from the flushed median ({2 * l2 >> 20} "
                                                  "MiB rewritten between reps)"),
        "seq_steps_per_s_per_layer": round(w.n_seqs / (us * 1e-6), 1),
        "warm_l2": warm, "flushed_l2": cold,
        # one launch per step: this shape takes the small-batch path unless PKV_DECODE_IMPL=split
        "gpu_launches": (3 if os.environ.get("PKV_DECODE_IMPL") == "split" else 1) * reps * 2,
        "clocks": clk.summary()}


def run_layers_bench(args, P, device):
    """An args.layers-layer decode step of workload 0, 1 or 2 (tiny, Llama-3-8B
    shaped, its int8 variant): per layer the page write of the step's new rows and the paged decode
    over that layer's own pools (the tables are shared, as every layer of a
    model stores the same token positions), timed as eager calls and as one
    captured CUDA graph of the whole step."""
    import torch
    assert args.config in (0, 1, 2), "the layered step covers workloads 0, 1 and 2"
    w = make_workload(args.config, device)
    L = args.layers
    kp, vp, ks, vs = fill_pool(P, w, device)
    layers = []
    gen = torch.Generator().manual_seed(4242)
    for l in range(L):
        layers.append(dict(kp=kp if l == 0 else kp.clone(), vp=vp if l == 0 else vp.clone(),
                           ks=None if ks is None else (ks if l == 0 else ks.clone()),
                           vs=None if vs is None else (vs if l == 0 else vs.clone()),
                           q=torch.randn(w.q.shape, generator=gen).to(torch.bfloat16).to(device),
                           k_new=torch.randn(w.k_new.shape, generator=gen).to(torch.bfloat16).to(device),
                           v_new=torch.randn(w.v_new.shape, generator=gen).to(torch.bfloat16).to(device),
                           out=torch.empty(w.q.shape, dtype=torch.bfloat16, device=device)))
    tables, start, ctx = w.tables.to(device), w.start_pos.to(device), w.ctx_lens.to(device)
    ws = torch.empty(P.decode_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, int(w.ctx_lens.sum()),
                                              w.split_tokens), dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)

    def step():
        for x in layers:
            P.paged_decode_step(x["k_new"], x["v_new"], start, x["q"], x["kp"], x["vp"], tables, ctx,
                                w.softmax_scale, k_scales=x["ks"], v_scales=x["vs"], split_tokens=w.split_tokens,
                                out=x["out"], workspace=ws, dev_status=status)

    # the same calls through one DecodePlan per layer (the fixed arguments checked once)
    plans = [P.DecodePlan(x["kp"], x["vp"], tables, ctx, w.softmax_scale, w.n_q_heads, k_scales=x["ks"],
                          v_scales=x["vs"], split_tokens=w.split_tokens, out=x["out"], workspace=ws,
                          dev_status=status) for x in layers]

    def step_planned():
        for x, plan in zip(layers, plans):
            plan.run(x["q"], x["k_new"], x["v_new"], start)

    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    steps = max(3, min(args.steps, 2000))
    warm = max(3, args.warmup)

    def timed(fn):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    with ClockSampler(uuid) as clk:
        time.sleep(0.25)
        ms_eager = timed(step)
        ms_planned = timed(step_planned)
        ms_graph = timed(graph.replay)
    assert int(status.item()) == 0
    decode_b, write_b = algorithmic_bytes(w)
    line = {"metric": f"{L}-layer decode step seq-steps/s", "value": round(w.n_seqs / (ms_graph * 1e-3), 1),
            "unit": "seq-steps/s", "n_gpus": 1, "steps": steps, "warmup": warm, "ms_per_step": round(ms_graph, 4),
            "higher_is_better": True, "scaling": "none", "vs_baseline": None,
            "dtype": "int8" if w.kv_format == "int8" else "bf16", "data": "synthetic",
            "config": {"workload": w.name, "layers": L, "launch": "one CUDA graph per step",
                       "gb_per_s": round(L * (decode_b + write_b) / (ms_graph * 1e-3) / 1e9, 2),
                       # the tiny decode takes the one-launch small-batch path unless PKV_DECODE_IMPL=split
                       "kernel_launches_per_step": L * (1 if args.config == 0 and
                                                        os.environ.get("PKV_DECODE_IMPL") != "split" else 3)},
            "eager": {"ms_per_step": round(ms_eager, 4), "value": round(w.n_seqs / (ms_eager * 1e-3), 1),
                      "gb_per_s": round(L * (decode_b + write_b) / (ms_eager * 1e-3) / 1e9, 2)},
            "eager_planned": {"ms_per_step": round(ms_planned, 4),
                              "value": round(w.n_seqs / (ms_planned * 1e-3), 1),
                              "gb_per_s": round(L * (decode_b + write_b) / (ms_planned * 1e-3) / 1e9, 2),
                              "how": "one DecodePlan per layer, run(q, k_new, v_new, start_pos) per call"},
            "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def pipelined_e2e(ins, out_like, call, device, stream):
    """End-to-end steps through the public API: the step's inputs sit in one
    pinned host arena and are copied with one H2D per step into one of two
    device arenas (views feed call(views, out)); the output goes back to one
    of two pinned host buffers.  Input copies and output copies each run on
    their own stream, so step i + 1's inputs land while step i computes and
    step i's output drains while step i + 1 runs; every step still moves its
    own inputs and output.  Returns (run(n), input stream, output stream);
    run(n) ends with the caller's stream waiting for the last output."""
    import torch
    offs, total = [], 0
    for t in ins:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_arena = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(ins, offs):
        h_arena[o:o + t.numel() * t.element_size()].copy_(t.contiguous().view(-1).view(torch.uint8))
    d_arena = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]

    def views(buf):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(ins, offs)]

    d_views = [views(b) for b in d_arena]
    d_out = [torch.empty_like(out_like) for _ in range(2)]
    h_outs = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory() for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=device)     # inputs, host -> device
    out_stream = torch.cuda.Stream(device=device)      # outputs, device -> host (not behind the next inputs)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_drained = [torch.cuda.Event() for _ in range(2)]
    ev_out = torch.cuda.Event()

    def run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(ev_done[b])     # compute i - 2 no longer reads buffer b
                d_arena[b].copy_(h_arena, non_blocking=True)
                ev_in[b].record(copy_stream)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_drained[b])           # output i - 2 has left d_out[b]
            call(d_views[b], d_out[b])
            ev_done[b].record(stream)
            with torch.cuda.stream(out_stream):
                out_stream.wait_event(ev_done[b])
                h_outs[b].copy_(d_out[b], non_blocking=True)
                ev_drained[b].record(out_stream)
        ev_out.record(out_stream)
        stream.wait_event(ev_out)                          # the last output has reached the host

    return run, copy_stream, out_stream


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.blocks:
        if rank == 0:
            run_blocks_bench(args)
        return

    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    from paged_kv_cache_212_gb300 import build as B
    B.build()
    import paged_kv_cache_212_gb300 as P
    P.load_library()

    if args.writes:
        if rank == 0:
            print(json.dumps({"metric": "page write GB/s", "unit": "GB/s", "n_gpus": 1, "data": "synthetic",
                              "writes": bench_writes(P, device, measured_peaks()[0])}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    if args.stream or args.layers:
        if rank == 0:
            (run_stream_bench if args.stream else run_layers_bench)(args, P, device)
        if world > 1:
            dist.destroy_process_group()
        return
    w = make_workload(args.config, device)  # every rank owns an independent replica batch
    if args.config == 0:
        if rank == 0:
            line = run_small_bench(args, P, w, device)
            if world == 1 and not args.no_cpu_baseline:
                line["cpu_baseline"] = cpu_baseline(0)
            print(json.dumps(line), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    if args.config == 3:
        line = run_prefill_bench(args, P, w, device, rank, world, args.steps, args.warmup)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline_prefill()
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    line = run_decode_bench(args, P, w, device, rank, world, args.steps, args.warmup)
    if args.config == 2:
        line["gather"] = bench_gather(P, device, measured_peaks()[0])
    del w
    torch.cuda.empty_cache()
    if world == 1 and args.config == 1 and not args.no_other_configs:
        line["other_configs"] = other_configs(args, P, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_decode_bench(args, P, w, device, rank, world, K, W, with_e2e=True):
    """One decode step (paged write of the step's new rows + paged decode
    attention, one paged_decode_step call) of workload w, timed as K steps
    on the device (see device_timed), then end to end through the Python API
    with per-step host copies.  Returns the JSON line (a dict)."""
    import torch
    kp, vp, ks, vs = fill_pool(P, w, device)
    tables = w.tables.to(device)
    start = w.start_pos.to(device)
    ctx = w.ctx_lens.to(device)
    k_new, v_new, q = w.k_new.to(device), w.v_new.to(device), w.q.to(device)
    out = torch.empty_like(q)
    split = args.split or w.split_tokens
    ws_bytes = P.decode_workspace_bytes(w.n_seqs, w.n_q_heads, w.head_dim, int(w.ctx_lens.sum()), split)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream()
    int8 = w.kv_format == "int8"

    def step():
        # one call: the page write of this step's rows, then paged decode attention
        P.paged_decode_step(k_new, v_new, start, q, kp, vp, tables, ctx, w.softmax_scale, k_scales=ks,
                            v_scales=vs, split_tokens=split, out=out, workspace=ws, dev_status=status)

    uuid = gpu_uuid(device)
    with ClockSampler(uuid) as clk:
        time.sleep(0.25)  # the sampler is running before the warm-up starts
        host_ms, est_ms = warm_up(step, max(3, W))
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        # the timed region follows the warm-up directly: no idle gap before it
        per = device_timed(step, K, stream, world, device, host_ms, est_ms)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    ms_per_step = statistics.median(per) / K
    decode_b, write_b = algorithmic_bytes(w)
    step_b = decode_b + write_b
    peak, peak_kind = measured_peaks()
    value = weak_scaling_value(step_b, world, ms_per_step)
    achieved = step_b / (ms_per_step * 1e-3) / 1e9
    traffic = ncu_traffic("decode", w_index(w))
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8" if int8 else "bf16", "data": "synthetic",
        "config": bench_config(w, args),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "seq_steps_per_s_per_layer": round(world * w.n_seqs / (ms_per_step * 1e-3), 1),
        "ms_per_32_layer_step": round(32 * ms_per_step, 4),
        "timing": timing_note(per, K),
        "roofline": {"bound": "hbm",
                     "kernel": "paged_decode_step (plan + write, split, merge launches; split kernel dominant)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": step_b, "avg_launch_ms": round(ms_per_step, 5),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "gpu_launches": 3 * K * len(per),
        "clocks": clk.summary(),
    }
    if with_e2e:
        line["e2e"] = decode_e2e(P, w, kp, vp, ks, vs, split, ws, status, q, K, world, device, stream, args)
    return line


def W_CONFIGS():
    from paged_kv_cache_212_gb300 import workloads as W
    return W.WORKLOADS


def w_index(w):
    """The scenario number of a workload (from its seed)."""
    from paged_kv_cache_212_gb300 import workloads as W
    return w.seed - W.SEED_BASE


def gpu_uuid(device):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        return None


def decode_e2e(P, w, kp, vp, ks, vs, split, ws, status, q, K, world, device, stream, args):
    """The decode step end to end through the public API with pinned host
    buffers: per step the new rows, queries, tables, positions and lengths go
    host -> device and the output device -> host, inside the timed region."""
    import torch
    import torch.distributed as dist
    e2e_steps = args.e2e_steps or max(10, min(K, 2000))
    h_k, h_v, h_q = (x.cpu().pin_memory() for x in (w.k_new, w.v_new, w.q))
    h_tab, h_start, h_ctx = (x.cpu().pin_memory() for x in (w.tables, w.start_pos, w.ctx_lens))
    h_out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (h_k, h_v, h_q, h_tab, h_start, h_ctx))
    d2h = h_out.numel() * h_out.element_size()

    # one DecodePlan per device arena (its tables, lengths and output bound once);
    # each step runs it on that arena's queries, new rows and positions
    plans = {}

    def call(views, out):
        dk, dv, dq, dtab, dstart, dctx = views
        plan = plans.get(out.data_ptr())
        if plan is None:
            plan = plans[out.data_ptr()] = P.DecodePlan(kp, vp, dtab, dctx, w.softmax_scale, w.n_q_heads,
                                                        k_scales=ks, v_scales=vs, split_tokens=split, out=out,
                                                        workspace=ws, dev_status=status)
        plan.run(dq, dk, dv, dstart)

    e2e_run, copy_stream, out_stream = pipelined_e2e((h_k, h_v, h_q, h_tab, h_start, h_ctx), q, call, device,
                                                     stream)
    e2e_run(3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    out_stream.wait_event(e0)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], device)[0]
    decode_b, write_b = algorithmic_bytes(w)
    return {"value": round(weak_scaling_value(decode_b + write_b, world, e2e_ms), 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
            "steps": e2e_steps, "api": "DecodePlan.run (write + decode per step) on the copied inputs"}


def bench_writes(P, device, peak):
    """The page writes on their own: paged_kv_write_int8 at the int8
    workload's 64 x 16-token shape and paged_kv_write of the prefill
    workload's 8 x 512-token chunk, per-call CUDA events (median of 200),
    warm and with twice the L2 rewritten before each call."""
    import torch
    res = {}
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    for cfg in (2, 3):
        w = make_workload(cfg, device)
        int8 = cfg == 2
        nb1 = w.n_blocks + 1
        shape = (nb1, w.block_size, w.n_kv_heads, w.head_dim)
        kp = torch.zeros(shape, dtype=torch.int8 if int8 else torch.bfloat16, device=device)
        vp = torch.zeros_like(kp)
        ks = torch.zeros(shape[:3], dtype=torch.float32, device=device) if int8 else None
        vs = torch.zeros_like(ks) if int8 else None
        tables, start = w.tables.to(device), w.start_pos.to(device)
        k_new, v_new = w.k_new.to(device), w.v_new.to(device)

        def call():
            if int8:
                P.paged_kv_write_int8(k_new, v_new, kp, vp, ks, vs, tables, start)
            else:
                P.paged_kv_write(k_new, v_new, kp, vp, tables, start)

        rows = w.n_seqs * w.n_new * w.n_kv_heads
        nbytes = (2 * rows * w.head_dim * 2 + 2 * rows * (w.head_dim + 4)) if int8 else 2 * 2 * rows * w.head_dim * 2
        nbytes += w.n_seqs * 4 + int(((w.start_pos + w.n_new + w.block_size - 1) // w.block_size).sum()) * 4
        out = {"workload": w.name, "call": "paged_kv_write_int8" if int8 else "paged_kv_write",
               "rows": rows, "algorithmic_bytes": nbytes}
        for name, flushed in (("warm", False), ("flushed", True)):
            for _ in range(5):
                call()
            reps = 200
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for a, b in evs:
                if flushed:
                    flush.fill_(1.0)
                gpu_hold(0.05)
                a.record(stream)
                call()
                b.record(stream)
            torch.cuda.synchronize()
            t = sorted(a.elapsed_time(b) for a, b in evs)
            ms = t[len(t) // 2]
            out[name] = {"median_us": round(ms * 1e3, 3), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                         "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4)}
        res[str(cfg)] = out
        del kp, vp, ks, vs, w
        torch.cuda.empty_cache()
    return res


def other_configs(args, P, device):
    """Short runs of the other four scenarios, reported beside the headline
    (the headline's metric, value and config stay those of the Llama-3-8B
    decode): the int8 decode step with its gather, the chunked prefill, the
    skewed shared-prefix decode and the tiny L2-resident step, plus the page
    writes on their own."""
    import torch
    res = {}
    peak = measured_peaks()[0]
    keep = ("value", "unit", "ms_per_step", "steps", "warmup", "dtype", "pct_of_peak",
            "seq_steps_per_s_per_layer", "timing", "roofline", "clocks", "config", "gpu_launches")
    for cfg in (2, 4):
        w = make_workload(cfg, device)
        line = run_decode_bench(args, P, w, device, 0, 1, 200, 5, with_e2e=False)
        sub = {k: line[k] for k in keep if k in line}
        sub["metric"] = METRIC
        if cfg == 2:
            sub["gather"] = bench_gather(P, device, peak)
            # the same step on the tensor-core (tcgen05) decode kernel, selected
            # per call with PKV_DECODE_IMPL=tc
            prev = os.environ.get("PKV_DECODE_IMPL")
            os.environ["PKV_DECODE_IMPL"] = "tc"
            try:
                tc = run_decode_bench(args, P, w, device, 0, 1, 50, 5, with_e2e=False)
            finally:
                if prev is None:
                    os.environ.pop("PKV_DECODE_IMPL", None)
                else:
                    os.environ["PKV_DECODE_IMPL"] = prev
            sub["tensor_core_decode"] = {k: tc[k] for k in ("value", "unit", "ms_per_step", "pct_of_peak", "timing",
                                                            "gpu_launches") if k in tc}
        if cfg == 4:
            # shared prefix blocks are read by every member: report the unique bytes too
            sub["unique_kv_bytes_per_step"] = unique_kv_bytes(w)
        res[str(cfg)] = sub
        del w, line
        torch.cuda.empty_cache()
    w = make_workload(3, device)
    line = run_prefill_bench(args, P, w, device, 0, 1, 20, 5, with_e2e=False)
    res["3"] = {k: line[k] for k in ("metric",) + keep if k in line}
    del w, line
    torch.cuda.empty_cache()
    w = make_workload(0, device)
    line = run_small_bench(args, P, w, device, reps=300)
    res["0"] = {k: line[k] for k in ("metric", "value", "unit", "ms_per_step", "warm_l2", "flushed_l2",
                                     "seq_steps_per_s_per_layer", "clocks", "config") if k in line}
    del w, line
    torch.cuda.empty_cache()
    res["writes"] = bench_writes(P, device, peak)
    return res


def unique_kv_bytes(w):
    """K/V bytes of the blocks the step reads, each physical block once
    (valid tokens of each distinct block)."""
    bs = w.block_size
    per_tok = 2 * w.n_kv_heads * w.head_dim * 2
    seen = {}
    for s in range(w.n_seqs):
        L = int(w.ctx_lens[s])
        for j in range(-(-L // bs)):
            b = int(w.tables[s, j])
            seen[b] = max(seen.get(b, 0), min(bs, L - j * bs))
    return sum(seen.values()) * per_tok


if __name__ == "__main__":
    main()
