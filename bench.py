#!/usr/bin/env python3
"""Decode-step benchmark: KV append + split-KV decode attention + merge.

One step = one pass of the whole hot path over one batch: append the new
token's K/V to the cache, then decode attention over every sequence's cache.
Default workload: the PaLM-540B-style multiquery decode step (batch 64, 48
query heads over 1 KV head of 256, context 2048), one layer.

Prints ONE JSON line (rank 0). `value` is KV GB/s (algorithmic bytes of the
attention step: valid K/V rows + q + output, over the device time of the
step). Throughput in tokens/s (batch / step time) is reported beside it.

  python bench.py [--config palm] [--steps 50] [--warmup 5] [--impl ours|reference]

Under torchrun (--gpus N > 1) every rank runs its own replica of the
workload on its own GPU (the (sequence, KV head) units are independent, so
no data-path collective exists); timing is bracketed by a barrier and the
maximum over ranks is taken.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402
from kv_cache_decode_gb300 import roofline  # noqa: E402

METRIC = "decode-attention KV GB/s and % of GB300 HBM peak; decode tokens/s per shape"
UNIT = "GB/s"
# Every source of the attention kernels: a profile taken on other sources is stale.
# The sources each chunk-kernel engine is compiled from (the tcgen05 kernel
# also takes shared helpers from the mma.sync kernel's header).
CHUNK_SOURCES = {
    "mma": ["split_kv_chunk.cuh", "split_kv_chunk_variants.cuh", "common.cuh", "schedule.cuh", "params.h"],
    "tc": ["split_kv_chunk_tc.cuh", "split_kv_chunk_tc_launch.cuh", "tc_common.cuh", "split_kv_chunk.cuh",
           "common.cuh", "schedule.cuh", "params.h"],
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="palm", help="tiny|palm|mha|gqa|long|long_trialN")
    ap.add_argument("--n-split", type=int, default=0, help="0 = heuristic")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first N sequences (smaller profiling captures); 0 = the workload's")
    ap.add_argument("--out-dtype", default="bf16", choices=["bf16", "f32"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--page-size", type=int, default=0,
                    help="paged KV cache with pages of this many tokens; 0 = contiguous")
    ap.add_argument("--tokens", type=int, default=1,
                    help="query tokens per sequence (T > 1: a speculative check step; up to 64)")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "int8", "fp8"],
                    help="int8 / fp8 (E4M3): the cache quantized per (token, KV head) row")
    ap.add_argument("--softmax", default="online", choices=["online", "unified"],
                    help="unified: every split's partial softmax against one maximum phi (plain-sum merge)")
    ap.add_argument("--phi", type=float, default=0.0, help="the unified maximum, in logit units")
    ap.add_argument("--page-order", default="shuffled", choices=["shuffled", "sequential"],
                    help="paged: pages in random order over the pool, or each sequence's pages in a row")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other workloads (tiny, mha, gqa, long, the 16 long trials)")
    ap.add_argument("--probe", choices=["read"], default=None,
                    help="read: only run the read-only streaming probe over a range of sizes")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def max_over_ranks(values, device=None):
    """Each value's maximum over all ranks (one all_reduce of a float64 vector);
    the values unchanged when no process group is running. Every rank gets the
    result, so the slowest rank's time sets the job's rate."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_rate_gbs(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Whole-job rate: every rank processes bytes_per_rank_step per step (weak
    scaling, independent replicas), and a step lasts the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def chunk_source_hash(engine: str) -> str:
    h = hashlib.sha256()
    for name in CHUNK_SOURCES[engine]:
        with open(os.path.join(ROOT, "kv_cache_decode_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(config: str):
    """DRAM bytes per chunk-kernel launch from the committed ncu summary, or
    None when that summary was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(x.split("=", 1) for x in line.split())
        engine = "tc" if kv.get("kernel", "").startswith("split_kv_chunk_tc") else "mma"
        if kv.get("config") == config and kv.get("src_sha") == chunk_source_hash(engine):
            return int(float(kv["dram_bytes_per_launch"]))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        # nvidia-smi needs at least one sample period
        while time.time() - self.t0 < 0.5:
            time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.file.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_rate(w, inp, budget_s: float, repeats: int = 1, min_total_s: float = 0.0):
    """Time the oracle on a bounded sample of sequences: the first sequences
    that fit in about budget_s per pass, timed over `repeats` passes or, if
    longer, over as many passes as fill min_total_s. Returns (GB/s of
    algorithmic bytes, median seconds per pass, rows, cores, passes)."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    B = inp.q.shape[0]
    kc, vc, _ = oracle.kv_append(inp.k_cache[:1], inp.v_cache[:1], inp.k_new[:1], inp.v_new[:1], inp.pos[:1])
    t = time.perf_counter()
    oracle.decode_attention(inp.q[:1], kc, vc, inp.seq_lens[:1], w.scale)
    t1 = max(time.perf_counter() - t, 1e-4)
    n = int(max(1, min(B, budget_s / t1)))
    rows = np.arange(n)
    kc, vc, _ = oracle.kv_append(inp.k_cache[rows], inp.v_cache[rows], inp.k_new[rows],
                                 inp.v_new[rows], inp.pos[rows])
    times = []
    while len(times) < repeats or (sum(times) < min_total_s and len(times) < 1000):
        t = time.perf_counter()
        oracle.decode_attention(inp.q[rows], kc, vc, inp.seq_lens[rows], w.scale)
        times.append(time.perf_counter() - t)
    sec = statistics.median(times)
    nbytes = roofline.attention_step_bytes(inp.seq_lens[rows], w.Hq, w.Hkv, w.D)
    return nbytes / sec / 1e9, sec, n, cores, len(times)


def bench_config(w, B, Hq, Hkv, D, lens_np, args) -> dict:
    """The workload and run options, identical in both arms' lines."""
    return {"workload": w.name, "description": w.description, "batch": B, "n_heads_q": Hq,
            "n_heads_kv": Hkv, "head_dim": D, "context": [int(lens_np.min()), int(lens_np.max())],
            "out_dtype": args.out_dtype, "parallelism": f"replicas x{args.gpus}",
            "l2_flush": "K/V rows read from HBM every step: rotating cache copies totalling >= 3x L2",
            "kv_layout": (f"paged: {args.page_size}-token pages in {args.page_order} order" if args.page_size
                          else "contiguous"),
            "kv_dtype": args.kv_dtype, "query_tokens": args.tokens,
            "softmax": f"unified max, phi {args.phi}" if args.softmax == "unified" else "online max"}


def run_reference(args):
    """The reference arm: the float64 CPU oracle, as it stands, on the host's
    cores, over the whole batch of the workload every step."""
    rank, _, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    w = workloads.get(args.config)
    if args.batch:
        w = w.with_batch(min(args.batch, w.B))
    inp = workloads.step_inputs(w, pad_bits=0)
    kc, vc, _ = oracle.kv_append(inp.k_cache, inp.v_cache, inp.k_new, inp.v_new, inp.pos)
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        oracle.decode_attention(inp.q, kc, vc, inp.seq_lens, w.scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    sec = sum(times) / len(times)
    step_bytes = roofline.attention_step_bytes(inp.seq_lens, w.Hq, w.Hkv, w.D)
    value = step_bytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, w.B, w.Hq, w.Hkv, w.D, inp.seq_lens, args),
        "tokens_per_s": round(w.B / sec, 2),
        "timing": "wall clock (perf_counter) around each oracle pass over the whole batch",
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"all {w.B} sequences (all heads) per step, float64 C oracle, "
                                   f"mean of {len(times)} passes"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def rotation_count(kv_bytes: int, cache_bytes: int, l2: int) -> int:
    """Cache copies to rotate through so that a step's K/V rows are not
    L2-resident: together at least 3x L2, at most 16 copies or 40 GB."""
    R = max(1, math.ceil(3 * l2 / max(kv_bytes, 1)))
    return max(1, min(R, int(40e9 // max(cache_bytes, 1)), 16))


def time_replays(graphs, steps: int, warmup: int, round_graph=None) -> float:
    """Milliseconds per step of `steps` steps run as graph replays, queued
    behind a spin kernel so the GPU never waits for the host, between CUDA
    events on the replay stream. `graphs` hold one step each (round-robin over
    the cache copies); `round_graph`, if given, holds round_steps(R) steps, one
    on each copy in turn (as a model's graph holds many layers' steps), and is
    replayed for whole rounds, the single-step graphs for the rest."""
    import torch
    R = len(graphs)
    def run(n):
        for g in replay_plan(n, R, round_graph is not None):
            (round_graph if g == "round" else graphs[g]).replay()
    run(warmup)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2e6 + 2e5 * steps))
    e0.record()
    run(steps)
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


def isolated_replay_us(graph, reps: int) -> float:
    """Median device time of one graph replay with the GPU otherwise idle
    (the step's latency rather than its throughput), in microseconds."""
    import torch
    times = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        graph.replay()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    return statistics.median(times)


def round_steps(R: int) -> int:
    """Steps in a round graph: whole passes over the R cache copies, about 16."""
    return R * max(1, 16 // R)


def replay_plan(n: int, R: int, use_round: bool = True):
    """The graphs replayed for n steps, in order: "round" for a round graph
    (round_steps(R) steps, copies 0, 1, ..., R - 1, 0, ...), an int r for the
    single-step graph on copy r. The steps add up to exactly n, and the cache
    copies follow each other round-robin from copy 0."""
    RS = round_steps(R) if use_round else 1
    if not use_round:
        return [i % R for i in range(n)]
    return ["round"] * (n // RS) + [i % R for i in range(n % RS)]


def capture_round(step, R: int, dev):
    """One CUDA graph holding round_steps(R) steps, on copies 0, 1, ..., R - 1, 0, ..."""
    def all_steps():
        for i in range(round_steps(R)):
            step(i % R)
    return capture(all_steps, dev)


def capture(fn, dev):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream(device=dev)):
        fn()
    return g


def read_probe(kvd, dev, nbytes: int, l2: int, reps: int = 20) -> dict:
    """One read-only streaming pass over nbytes (kvd_probe_read), buffers
    rotated so the bytes come from HBM: median device time and GB/s."""
    import torch
    R = rotation_count(nbytes, nbytes, l2)
    bufs = [torch.ones(nbytes // 2, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    sink = torch.zeros(1024, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for i in range(3 * R):
        kvd.probe_read(bufs[i % R], sink=sink, status=status)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda._sleep(int(2e6 + 2e5 * reps))
    for i, (a, b) in enumerate(ev):
        a.record()
        kvd.probe_read(bufs[i % R], sink=sink, status=status)
        b.record()
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in ev)
    if int(status.item()) != 0:
        raise RuntimeError("read probe: a copy wait timed out")
    del bufs
    torch.cuda.empty_cache()
    return {"bytes": int(nbytes), "us": round(us, 3), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "copies_rotated": R}


def measure_shape(kvd, dev, w, steps: int, warmup: int, l2: int, peak: float, latency: bool = False) -> dict:
    """One workload's bf16 decode step (kvd_decode_step: append + attention),
    measured as the headline workload is: CUDA graphs over rotating cache
    copies, step time and the chunk kernel's time from CUDA events."""
    import torch
    inp = workloads.step_inputs(w, pad_bits=0)
    B, Hq, D = inp.q.shape
    S, Hkv = inp.k_cache.shape[1], inp.k_cache.shape[2]
    lens_np = inp.seq_lens.copy()
    step_bytes = roofline.attention_step_bytes(lens_np, Hq, Hkv, D)
    kv_bytes = roofline.attention_kv_bytes(lens_np, Hkv, D)
    R = rotation_count(kv_bytes, 2 * inp.k_cache.nbytes, l2)

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    kcs, vcs = [up(inp.k_cache)], [up(inp.v_cache)]
    for _ in range(R - 1):
        kcs.append(kcs[0].clone())
        vcs.append(vcs[0].clone())
    q, kn, vn = up(inp.q), up(inp.k_new), up(inp.v_new)
    pos, lens = torch.from_numpy(inp.pos).to(dev), torch.from_numpy(lens_np).to(dev)
    del inp
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    n_split, ws_bytes = kvd.decode_plan(B, Hq, Hkv, D, S)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    step = lambda r: kvd.decode_step(q, kcs[r], vcs[r], kn, vn, pos, lens, S, w.scale, out, workspace=ws)
    for i in range(3 * R):
        step(i % R)
    torch.cuda.synchronize()
    graphs = [capture(lambda r=r: step(r), dev) for r in range(R)]
    round_graph = capture_round(step, R, dev)
    res = {"batch": B, "n_heads_q": Hq, "n_heads_kv": Hkv, "head_dim": D,
           "context": [int(lens_np.min()), int(lens_np.max())], "n_split": n_split, "step_bytes": int(step_bytes)}
    if latency:
        res["latency_us"] = round(isolated_replay_us(graphs[0], 50), 3)
    ms = time_replays(graphs, steps, warmup, round_graph)
    ms_one = time_replays(graphs, steps, warmup)
    chunk_ms = time_chunk(kvd, lambda r: (kcs[r], vcs[r]), R, steps, q, kn, vn, pos, lens, S, w.scale, out, ws)
    gbs = step_bytes / (ms * 1e-3) / 1e9
    achieved = step_bytes / (chunk_ms * 1e-3) / 1e9
    res.update({"ms_per_step": round(ms, 5), "gbs": round(gbs, 1), "hbm_frac_of_step": round(gbs / peak, 4),
                "tokens_per_s": round(B / (ms * 1e-3), 1), "kernel_ms": round(chunk_ms, 5),
                "roofline_frac": round(achieved / peak, 4), "copies_rotated": R,
                "ms_per_step_one_step_graphs": round(ms_one, 5)})
    del kcs, vcs, graphs, round_graph
    torch.cuda.empty_cache()
    return res


def time_chunk(kvd, cache, R, steps, q, kn, vn, pos, lens, max_len, scale, out, ws, n_split=0) -> float:
    """Mean duration of the split-KV chunk kernel's launches (CUDA events on
    its stream, around each launch, after each step's append)."""
    import torch
    stream = torch.cuda.current_stream()
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda._sleep(int(2e6 + 2e5 * steps))
    for i in range(steps):
        kc, vc = cache(i % R)
        kvd.kv_append(kc, vc, kn, vn, pos)
        ea[i].record(stream)
        kvd.split_kv_chunk(q, kc, vc, lens, max_len, scale, out, workspace=ws, n_split=n_split)
        eb[i].record(stream)
        kvd.split_kv_merge(q, kc, vc, lens, max_len, scale, out, workspace=ws, n_split=n_split)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in zip(ea, eb))


def measure_long_trials(kvd, dev, steps: int, warmup: int, l2: int, peak: float) -> dict:
    """The 16 ragged long-context trials (lengths U[1, 131072] per trial): one
    step graph per cache copy, replayed with each trial's lengths. The K/V
    values do not change the work, so one seeded N(0, 1) cache drawn on the
    GPU serves every trial."""
    import torch
    w0 = workloads.long_trial(0)
    B, Hq, Hkv, D, S = w0.B, w0.Hq, w0.Hkv, w0.D, w0.S_max
    g = torch.Generator(device=dev)
    g.manual_seed(w0.seed)
    rnd = lambda *shape: torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    kc0, vc0 = rnd(B, S, Hkv, D), rnd(B, S, Hkv, D)
    R = rotation_count(B * S * Hkv * D * 4 // 2, 2 * kc0.numel() * 2, l2)
    kcs, vcs = [kc0] + [kc0.clone() for _ in range(R - 1)], [vc0] + [vc0.clone() for _ in range(R - 1)]
    q, kn, vn = rnd(B, Hq, D), rnd(B, Hkv, D), rnd(B, Hkv, D)
    lens = torch.zeros(B, dtype=torch.int32, device=dev)
    pos = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    n_split, ws_bytes = kvd.decode_plan(B, Hq, Hkv, D, S)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    step = lambda r: kvd.decode_step(q, kcs[r], vcs[r], kn, vn, pos, lens, S, w0.scale, out, workspace=ws)
    trials = []
    graphs = None
    for i in range(16):
        L = workloads.seq_lens(workloads.long_trial(i))
        lens.copy_(torch.from_numpy(L))
        pos.copy_(torch.from_numpy(np.maximum(L - 1, 0).astype(np.int32)))
        torch.cuda.synchronize()
        if graphs is None:
            for j in range(3 * R):
                step(j % R)
            torch.cuda.synchronize()
            graphs = [capture(lambda r=r: step(r), dev) for r in range(R)]
            round_graph = capture_round(step, R, dev)
        ms = time_replays(graphs, steps, warmup, round_graph)
        nbytes = roofline.attention_step_bytes(L, Hq, Hkv, D)
        gbs = nbytes / (ms * 1e-3) / 1e9
        trials.append({"trial": i, "tokens": int(L.sum()), "ms_per_step": round(ms, 5), "gbs": round(gbs, 1),
                       "hbm_frac_of_step": round(gbs / peak, 4)})
    del kcs, vcs, graphs, round_graph
    torch.cuda.empty_cache()
    fr = [t["hbm_frac_of_step"] for t in trials]
    return {"n_split": n_split, "trials": trials, "hbm_frac_of_step_median": round(statistics.median(fr), 4),
            "hbm_frac_of_step_min": min(fr), "hbm_frac_of_step_max": max(fr),
            "values": "one N(0,1) cache drawn on the GPU (torch generator, seed 500); each trial's own lengths"}


def run_ours(args):
    import torch

    import kv_cache_decode_gb300 as kvd

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peak_est, _ = measured_peaks()
    from kv_cache_decode_gb300 import _build
    _build.build()
    kvd.load()

    w = workloads.get(args.config)
    if args.batch:
        w = w.with_batch(min(args.batch, w.B))
    T = args.tokens
    multi = T > 1
    if multi and (args.page_size or args.kv_dtype != "bf16"):
        raise SystemExit("--tokens > 1 takes a contiguous bf16 cache")
    umax = args.softmax == "unified"
    if umax and (multi or args.page_size or args.kv_dtype != "bf16"):
        raise SystemExit("--softmax unified takes one query token and a contiguous bf16 cache")
    # T > 1: the same lengths, the last T tokens of each sequence new this step
    inp = (workloads.multi_step_inputs(w, T, pad_bits=0) if multi else workloads.step_inputs(w, pad_bits=0))
    B, Hq, D = inp.q.shape[0], inp.q.shape[-2], inp.q.shape[-1]
    S, Hkv = inp.k_cache.shape[1], inp.k_cache.shape[2]
    lens_np = inp.seq_lens
    max_len = int(w.S_max)
    int8 = args.kv_dtype in ("int8", "fp8")  # an 8-bit cache: codes and row scales
    fp8 = args.kv_dtype == "fp8"
    if int8 and args.page_size:
        raise SystemExit("--kv-dtype int8/fp8 takes a contiguous cache")
    step_bytes = (roofline.attention_step_bytes_q8(lens_np, Hq, Hkv, D) if int8
                  else roofline.attention_step_bytes(lens_np, Hq, Hkv, D))
    kv_bytes = roofline.attention_kv_bytes(lens_np, Hkv, D) // (2 if int8 else 1)
    if multi:
        step_bytes += 2 * B * (T - 1) * Hq * D * 2  # T queries in and T output rows out; the cache once
    append_bytes = roofline.append_bytes(B, Hkv, D)
    flops = roofline.attention_step_flops(lens_np, Hq, D)

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    paged = args.page_size > 0
    if paged:
        # The same rows spread over a shuffled pool of pages; the calls take the
        # pool and its block table instead of the contiguous cache.
        pinp = workloads.paged_step_inputs(inp, args.page_size, seed=w.seed, pad_bits=0,
                                           shuffle=args.page_order == "shuffled")
        k_src, v_src = pinp.k_pages, pinp.v_pages
        bt = torch.from_numpy(pinp.block_table).to(dev)
    else:
        k_src, v_src = inp.k_cache, inp.v_cache
    cache_bytes = 2 * k_src.nbytes
    # Rotate cache copies so that each step's K/V rows are not L2-resident.
    R = max(1, math.ceil(3 * l2 / max(kv_bytes, 1)))
    R = max(1, min(R, int(40e9 // max(cache_bytes, 1)), 16))
    kc0, vc0 = up(k_src), up(v_src)
    kcs, vcs = [kc0], [vc0]
    for _ in range(R - 1):
        kcs.append(kc0.clone())
        vcs.append(vc0.clone())
    if int8:
        # 8-bit copies quantized on the GPU from the bf16 cache (its cached rows)
        cached = torch.from_numpy(np.maximum(lens_np - 1, 0).astype(np.int32)).to(dev)
        q8 = []
        quantize = kvd.kv_quantize_fp8 if fp8 else kvd.kv_quantize_q8
        for kc_, vc_ in zip(kcs, vcs):
            codes = [torch.zeros(kc_.shape, dtype=torch.uint8 if fp8 else torch.int8, device=dev) for _ in range(2)]
            scales = [torch.zeros(kc_.shape[:3], dtype=torch.float32, device=dev) for _ in range(2)]
            quantize(kc_, codes[0], scales[0], cached, S)
            quantize(vc_, codes[1], scales[1], cached, S)
            q8.append((codes[0], codes[1], scales[0], scales[1]))
        del kcs[1:], vcs[1:]
        torch.cuda.synchronize()
    q, kn, vn = up(inp.q), up(inp.k_new), up(inp.v_new)
    pos = torch.from_numpy(inp.pos).to(dev)
    lens = torch.from_numpy(lens_np).to(dev)
    out_t = torch.bfloat16 if args.out_dtype == "bf16" else torch.float32
    out = torch.empty(inp.q.shape, dtype=out_t, device=dev)
    if multi:
        n_split, ws_bytes = kvd.decode_plan_multi(B, T, Hq, Hkv, D, max_len, 0, args.n_split, args.out_dtype)
    else:
        n_split, ws_bytes = kvd.decode_plan(B, Hq, Hkv, D, max_len, 0, args.n_split, args.out_dtype)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    launches_per_step = 2 + (1 if n_split > 1 else 0)

    def step(r, stream=None):
        # append the new token's K/V rows, then attend (one call, three launches)
        if multi:
            kvd.decode_step_multi(q, kcs[r], vcs[r], kn, vn, pos, lens, max_len, w.scale, out, workspace=ws,
                                  n_split=args.n_split, stream=stream)
        elif fp8:
            kq, vq, ks, vs = q8[r]
            kvd.decode_ex(q, kq, vq, lens, max_len, w.scale, out, k_scales=ks, v_scales=vs, k_new=kn, v_new=vn,
                          pos=pos, workspace=ws, n_split=args.n_split, stream=stream)
        elif int8:
            kq, vq, ks, vs = q8[r]
            kvd.decode_step_q8(q, kq, vq, ks, vs, kn, vn, pos, lens, max_len, w.scale, out, workspace=ws,
                               n_split=args.n_split, stream=stream)
        elif paged:
            kvd.decode_step_paged(q, kcs[r], vcs[r], kn, vn, pos, bt, lens, max_len, w.scale, out,
                                  workspace=ws, n_split=args.n_split, stream=stream)
        elif umax:
            kvd.decode_step_umax(q, kcs[r], vcs[r], kn, vn, pos, lens, max_len, w.scale, args.phi, out,
                                 workspace=ws, n_split=args.n_split, stream=stream)
        else:
            kvd.decode_step(q, kcs[r], vcs[r], kn, vn, pos, lens, max_len, w.scale, out, workspace=ws,
                            n_split=args.n_split, stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i % R)
    torch.cuda.synchronize()

    # CUDA graphs: one per cache copy, and one round graph holding a step on
    # every copy in turn (as a model's graph holds many layers' steps), replayed
    # back to back in the timed region (single-step graphs for a partial round).
    graphs = []
    cap_stream = torch.cuda.Stream(device=dev)
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            step(r)
        graphs.append(g)
    RS = round_steps(R)
    round_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(round_graph, stream=cap_stream):
        for i in range(RS):
            step(i % R)
    for g in graphs:
        g.replay()
    round_graph.replay()
    torch.cuda.synchronize()

    def run_steps(n):
        for g in replay_plan(n, R):
            (round_graph if g == "round" else graphs[g]).replay()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- timed region: K whole steps ----
    sampler = ClockSampler(local_rank)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    run_steps(args.warmup)
    barrier()
    torch.cuda.synchronize()
    # Queue the timed replays behind a spin kernel, so that the GPU never waits
    # for the host to launch the next step inside the timed region.
    torch.cuda._sleep(int(2e6 + 2e5 * args.steps))
    ev0.record()
    run_steps(args.steps)
    ev1.record()
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    total_ms = ev0.elapsed_time(ev1)
    # For comparison: the same steps as one graph launch each (adds the gap
    # between graph launches to every step).
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2e6 + 2e5 * args.steps))
    e_a.record()
    for i in range(args.steps):
        graphs[i % R].replay()
    e_b.record()
    e_b.synchronize()
    one_step_graphs_ms = e_a.elapsed_time(e_b) / args.steps

    # ---- chunk-kernel durations: events around each launch on its stream ----
    stream = torch.cuda.current_stream()
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda._sleep(int(2e6 + 2e5 * args.steps))  # let the host queue ahead of the GPU
    for i in range(args.steps):
        r = i % R
        if multi:
            # no separate multi-token chunk entry point: the whole attention call is timed
            kvd.kv_append_multi(kcs[r], vcs[r], kn, vn, pos)
            ea[i].record(stream)
            kvd.decode_attention_multi(q, kcs[r], vcs[r], lens, max_len, w.scale, out, workspace=ws,
                                       n_split=args.n_split)
            eb[i].record(stream)
            continue
        if int8:
            # no separate int8 chunk entry point: the whole attention call is timed
            kq, vq, ks, vs = q8[r]
            (kvd.kv_append_fp8 if fp8 else kvd.kv_append_q8)(kq, vq, ks, vs, kn, vn, pos)
            ea[i].record(stream)
            kvd.decode_ex(q, kq, vq, lens, max_len, w.scale, out, k_scales=ks, v_scales=vs, workspace=ws,
                          n_split=args.n_split)
            eb[i].record(stream)
            continue
        if paged:
            # no separate paged chunk entry point: the whole attention call is timed
            kvd.kv_append_paged(kcs[r], vcs[r], kn, vn, bt, pos)
            ea[i].record(stream)
            kvd.decode_attention_paged(q, kcs[r], vcs[r], bt, lens, max_len, w.scale, out, workspace=ws,
                                       n_split=args.n_split)
            eb[i].record(stream)
            continue
        kvd.kv_append(kcs[r], vcs[r], kn, vn, pos)
        ea[i].record(stream)
        kvd.split_kv_chunk(q, kcs[r], vcs[r], lens, max_len, w.scale, out, workspace=ws,
                           n_split=args.n_split)
        eb[i].record(stream)
        kvd.split_kv_merge(q, kcs[r], vcs[r], lens, max_len, w.scale, out, workspace=ws,
                           n_split=args.n_split)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    chunk_ms = [a.elapsed_time(b) for a, b in zip(ea, eb)]
    chunk_avg_ms = statistics.mean(chunk_ms)

    total_ms, chunk_avg_ms = max_over_ranks([total_ms, chunk_avg_ms], device=dev)

    ms_per_step = total_ms / args.steps
    value = job_rate_gbs(world, step_bytes, ms_per_step)
    tokens_per_s = world * B * T / (ms_per_step * 1e-3)  # query tokens scored per second

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        q_h = pin(inp.q.view(np.int16))
        kn_h, vn_h = pin(inp.k_new.view(np.int16)), pin(inp.v_new.view(np.int16))
        pos_h, lens_h = pin(inp.pos), pin(lens_np)
        bt_h = pin(pinp.block_table if paged else np.zeros(0, np.int32))
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = q_h.nbytes + kn_h.nbytes + vn_h.nbytes + pos_h.nbytes + lens_h.nbytes + bt_h.nbytes
        d2h = out_h.nbytes

        host_steps = None
        if not (paged or int8 or umax):
            # the library's host-input step: five input copies, the step, the output copy, in one call
            bf = lambda t: t.view(torch.bfloat16)
            # the step's inputs in one pinned packet laid out like the device staging buffer: one copy in
            staging = torch.empty(kvd.step_staging_bytes(B, T, Hq, Hkv, D), dtype=torch.uint8, device=dev)
            packet, pq, pkn, pvn, ppos, plens = kvd.alloc_host_packet(B, T, Hq, Hkv, D)
            for dst, src in ((pq, bf(q_h)), (pkn, bf(kn_h)), (pvn, bf(vn_h)), (ppos, pos_h), (plens, lens_h)):
                dst.copy_(src)
            # out=None: the kernels write the result straight into the pinned out_h
            host_steps = [kvd.HostStep(pq, pkn, pvn, ppos, plens, kcs[r], vcs[r], staging, max_len,
                                       w.scale, None, out_h, workspace=ws, n_split=args.n_split) for r in range(R)]

        def e2e_step(r):
            if host_steps is not None:
                host_steps[r]()
                return
            q.view(torch.int16).copy_(q_h, non_blocking=True)
            kn.view(torch.int16).copy_(kn_h, non_blocking=True)
            vn.view(torch.int16).copy_(vn_h, non_blocking=True)
            pos.copy_(pos_h, non_blocking=True)
            lens.copy_(lens_h, non_blocking=True)
            if paged:
                bt.copy_(bt_h, non_blocking=True)  # the table changes between steps in serving
            step(r)
            out_h.copy_(out, non_blocking=True)

        for i in range(args.warmup):
            e2e_step(i % R)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(args.steps):
            e2e_step(i % R)
        e1.record()
        e1.synchronize()
        wall_ms = (time.perf_counter() - t0) * 1e3
        e2e_ms = max(e0.elapsed_time(e1), wall_ms) / args.steps
        e2e_ms, = max_over_ranks([e2e_ms], device=dev)
        e2e = {"value": round(job_rate_gbs(world, step_bytes, e2e_ms), 2), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_ms, 4), "tokens_per_s": round(world * B * T / (e2e_ms * 1e-3), 1),
               "api": ("kvd_decode_step_host per step (inputs in one pinned packet, one copy in; the kernels "
                       "write the result into pinned host memory)" if host_steps is not None else
                       "torch copies in, the step call, a copy back, per step")}
        if host_steps is not None:
            # Where the time goes: the packet's copy in alone, the result's copy
            # out alone, the device step alone (ms_per_step above), and the same host step captured once
            # per cache copy in a CUDA graph (copy-in node, kernels writing the
            # result to host memory) and replayed: no per-step launch cost.
            hs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * 20)]
            for i in range(20):
                torch.cuda.synchronize()
                hs[2 * i].record()
                staging.copy_(packet, non_blocking=True)
                hs[2 * i + 1].record()
            torch.cuda.synchronize()
            h2d_us = statistics.median(hs[2 * i].elapsed_time(hs[2 * i + 1]) * 1e3 for i in range(20))
            # and the result's copy out alone (the kernels write it to host
            # memory themselves in the step; this is what a separate copy costs)
            od = torch.empty(out_h.shape, dtype=out_h.dtype, device=dev)
            for i in range(20):
                torch.cuda.synchronize()
                hs[2 * i].record()
                out_h.copy_(od, non_blocking=True)
                hs[2 * i + 1].record()
            torch.cuda.synchronize()
            d2h_us = statistics.median(hs[2 * i].elapsed_time(hs[2 * i + 1]) * 1e3 for i in range(20))
            del od
            # the steps bound to a capture stream (HostStep takes its stream when built)
            cs = torch.cuda.Stream(device=dev)
            host_steps_g = [kvd.HostStep(pq, pkn, pvn, ppos, plens, kcs[r], vcs[r], staging, max_len, w.scale,
                                         None, out_h, workspace=ws, n_split=args.n_split, stream=cs)
                            for r in range(R)]
            host_graphs = []
            for r in range(R):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cs):
                    host_steps_g[r]()
                host_graphs.append(g)
            g_ms = time_replays(host_graphs, args.steps, args.warmup)
            g_ms, = max_over_ranks([g_ms], device=dev)
            e2e["breakdown"] = {"h2d_copy_us": round(h2d_us, 2), "d2h_copy_us": round(d2h_us, 2),
                                "device_step_us": round(ms_per_step * 1e3, 2),
                                "api_call_us": round(e2e_ms * 1e3, 2),
                                "graph_replay_us": round(g_ms * 1e3, 2),
                                "graph_replay_gbs": round(job_rate_gbs(world, step_bytes, g_ms), 2)}
            del host_graphs

    if rank != 0:
        return

    peak, peak_kind = measured_peaks()
    achieved = step_bytes / (chunk_avg_ms * 1e-3) / 1e9
    traffic = None if (paged or int8 or multi or umax) else ncu_traffic(w.name)
    cpu = None
    if not args.no_cpu_baseline and not int8 and not multi:
        gbs, sec, n_rows, cores, passes = oracle_rate(w, inp, budget_s=10.0, repeats=1,
                                                      min_total_s=10.0)
        cpu = {"value": round(gbs, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{n_rows} of {B} sequences (all heads), float64 C oracle, "
                         f"median of {passes} passes of {sec:.3f} s"}

    # ---- the other workloads, the same way (default run only) ----
    per_config = None
    default_run = (w.name == "palm" and not (paged or int8 or multi or umax or args.batch or args.n_split)
                   and args.out_dtype == "bf16" and world == 1)
    probes = None
    if default_run and not args.no_per_config:
        per_config = {}
        for name in ("tiny", "mha", "gqa", "long"):
            per_config[name] = measure_shape(kvd, dev, workloads.get(name), min(args.steps, 20),
                                             max(args.warmup, 3), l2, peak_est, latency=(name == "tiny"))
        per_config["long_trials"] = measure_long_trials(kvd, dev, 10, 3, l2, peak_est)
        probes = [read_probe(kvd, dev, kv_bytes, l2), read_probe(kvd, dev, 2 << 30, l2)]

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(w, B, Hq, Hkv, D, lens_np, args),
        "n_split": n_split,
        "l2_detail": f"{R} rotating KV-cache copies ({R * kv_bytes / 1e6:.0f} MB of K/V rows vs {l2 / 1e6:.0f} MB L2)",
        "timing": (f"CUDA graphs of {round_steps(R)} steps, one on each rotating cache copy in turn "
                   "(as a model's graph holds many layers' steps), replayed back to back; single-step "
                   "graphs for a partial round; CUDA events on the replay stream"),
        "ms_per_step_one_step_graphs": round(one_step_graphs_ms, 5),
        "tokens_per_s": round(tokens_per_s, 1),
        "hbm_frac_of_step": round(value / world / peak, 4),
        "step_bytes": int(step_bytes), "append_bytes": int(append_bytes), "flops": int(flops),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("split_kv_chunk + split_kv_merge (multi-token)" if multi else
                                f"split_kv_chunk + split_kv_merge ({args.kv_dtype})" if int8 else
                                "split_kv_chunk + split_kv_merge (paged)" if paged else "split_kv_chunk"),
                     "peak_source": f"{peak_kind} copy bandwidth",
                     "kernel_ms": round(chunk_avg_ms, 5)},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "per_config": per_config,
        "read_probe": probes,
        "impl": "ours",
    }
    print(json.dumps(line), flush=True)


def run_probe(args):
    """--probe read: the read-only streaming probe alone, over the workloads'
    K/V byte counts and a few larger buffers; one JSON line."""
    import torch

    import kv_cache_decode_gb300 as kvd
    from kv_cache_decode_gb300 import _build
    _build.build()
    kvd.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20))
    sizes = {name: roofline.attention_kv_bytes(workloads.seq_lens(workloads.get(name)), workloads.get(name).Hkv,
                                               workloads.get(name).D) for name in ("palm", "long", "mha", "gqa")}
    sizes.update({"512MiB": 512 << 20, "2GiB": 2 << 30, "8GiB": 8 << 30})
    peak, kind = measured_peaks()
    res = {}
    for name, n in sizes.items():
        r = read_probe(kvd, dev, int(n) // 16 * 16, l2)
        r["frac_of_copy_peak"] = round(r["gbs"] / peak, 4)
        res[name] = r
    print(json.dumps({"probe": "read", "unit": "GB/s", "copy_peak": peak, "peak_source": kind, "results": res}),
          flush=True)


def main():
    args = parse_args()
    if args.probe:
        run_probe(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    rank, _, world = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
