#!/usr/bin/env python3
"""Benchmark of the sparse MLA decode hot path on GB300.

One step = one whole decode call, sparse_mla_decode (the split kernel with the splits
of each query merged on chip; split + combine kernels when the plan has more than 8
splits), for the batch-32 / 64-head / top-2048 workload (65536 cached rows per
sequence, half the picks from the last 4096 positions), inputs resident in HBM.

Steps run back to back, as the attention of consecutive layers does: step i decodes
layer i mod NL, and every layer has its own KV cache, q and index set.  NL is chosen
so that at least three L2 capacities of other layers' rows are read between two
reads of one layer, so the rows of every step come from HBM (inputs larger than L2;
no flush).  The steps are captured in CUDA graphs of up to 128 calls, replayed with
one pair of CUDA events around exactly K steps on the launching stream; the kernels
use programmatic dependent launch, so a step's launch overlaps the end of the one
before.  Workloads whose data cannot exceed L2 (the batch-1 and batch-4 shapes) are
timed one isolated step at a time instead: L2 flushed (a 256 MiB write) before each
step, events around each single-step graph replay.  The isolated time is reported
for every workload as context.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  With N > 1 (torchrun) every rank runs an independent replica
of the workload on its own GPU (no data exchange); `value` is the total over ranks.
`--impl reference` times the CPU float64 oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mla_decode_03_gb300 import workloads as W  # noqa: E402

METRIC = "decode queries/s and gathered-KV GB/s (% of HBM and tensor-pipe roofline)"
UNIT = "queries/s"
WORKLOAD = "c3"   # the headline workload; --workload selects another shape
N_INDEX_SETS = 8          # index sets of the isolated-step timing
FLUSH_BYTES = 256 << 20
MAX_LAYERS = 16
GRAPH_STEPS = 128         # decode calls per captured graph (back-to-back timing)
L2_TURNOVER = 3           # L2 capacities read between two reads of one layer
# DRAM bytes (read + write) per launch of the dominant kernel on this workload, from
# one ncu capture of the decode kernel on the batch-32 workload.  They describe the
# kernel source they were taken on: with any other source the field is null.
TRAFFIC_KERNEL_SRC = "sparse_mla_decode_03_gb300/csrc/smla_decode.cu"
TRAFFIC_SRC_SHA256_16 = "d623f299c93b8b75"
TRAFFIC_BYTES = 47548160 + 100352
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_traffic():
    """ncu DRAM bytes per launch, or None once the kernel source has changed."""
    import hashlib
    try:
        with open(os.path.join(ROOT, TRAFFIC_KERNEL_SRC), "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    return TRAFFIC_BYTES if sha == TRAFFIC_SRC_SHA256_16 else None


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def oracle_inputs(w, device):
    """Host copies of q bits and of the rows the queries reference (compact)."""
    L = W.seq_lengths(w)
    kv = W.make_cache(w, L, device=device)
    q = W.make_q(w, device=device)
    idx = W.make_indices(w, L)
    rows, remap = W.compact_rows(kv, idx)
    qbits = W.bf16_bits(q)
    del kv
    return qbits, rows, remap


def time_oracle(qbits, rows, remap, scale, budget_s: float, max_queries: int = 1 << 30):
    """Runs the oracle query by query (cycling over the batch) for about budget_s."""
    import oracle.mla_oracle as O
    B = qbits.shape[0]
    done, t0 = 0, time.perf_counter()
    while True:
        b = done % B
        O.sparse_mla_decode(qbits[b:b + 1], rows, remap[b:b + 1], scale)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= max_queries:
            return done, el


def cores_used() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """CPU model name of the host (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


SINGLE_THREAD_ENV = {k: "1" for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                       "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS")}


def oracle_child(path: str, seconds: float) -> None:
    """Child process of the single-core baseline: pinned to one core, one BLAS thread
    (set in its environment before numpy loads), times the oracle on the saved inputs
    and prints {"queries": n, "seconds": t}."""
    try:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    except Exception:
        pass
    d = np.load(path)
    n, el = time_oracle(d["q"], d["rows"], d["remap"], float(d["scale"]), seconds)
    print(json.dumps({"queries": n, "seconds": el, "cores": cores_used()}), flush=True)


def time_oracle_single_core(qbits, rows, remap, scale, seconds):
    """The oracle on one pinned core with one BLAS thread, in a child process."""
    import tempfile
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "oracle_inputs.npz")
        np.savez(path, q=qbits, rows=rows, remap=remap, scale=np.float64(scale))
        env = dict(os.environ, **SINGLE_THREAD_ENV)
        p = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", path,
                            "--cpu-seconds", str(seconds)], capture_output=True, text=True,
                           env=env, timeout=600)
        if p.returncode != 0:
            return None
        return json.loads(p.stdout.strip().splitlines()[-1])


def run_reference(args):
    ws, rank, _ = dist_env()
    if ws > 1 and rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    qbits, rows, remap = oracle_inputs(w, dev)
    per_step_s = min(2.0, 60.0 / max(1, args.steps))   # whole run about a minute or less
    time_oracle(qbits, rows, remap, w.softmax_scale, 0.0, max_queries=max(1, args.warmup))
    total_q, total_t, step_ms = 0, 0.0, []
    for _ in range(args.steps):
        n, el = time_oracle(qbits, rows, remap, w.softmax_scale, per_step_s)
        total_q += n
        total_t += el
        step_ms.append(1e3 * el / n * w.batch)
    value = total_q / total_t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(step_ms), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{total_q} queries of the workload, about {per_step_s:.0f} s "
                                   f"of oracle work per step, one query per call"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def aggregate_over_ranks(ms_values, device, world_size):
    """Max over ranks of each per-rank time (ms); identity when world_size == 1."""
    if world_size == 1:
        return list(ms_values)
    import torch.distributed as dist
    t = torch.tensor(list(ms_values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world_size, batch, ms_per_step):
    """Whole-job queries/s: every rank decodes its own batch in ms_per_step (the max)."""
    return world_size * batch / (ms_per_step * 1e-3)


def config_dict(w, S, fused=None, timing=None):
    d = {"workload": w.name, "batch": w.batch, "heads": w.heads, "topk": w.topk,
         "rows_per_seq": w.rows_per_seq, "index_law": w.index_law,
         "row_bytes": W.ROW_BYTES, "num_splits": S, "splits_merged_on_chip": fused}
    if timing:
        d.update(timing)
    return d


def plan_layers(step_bytes: int, cache_bytes: int, l2_bytes: int, free_bytes: int) -> int:
    """Number of layer caches for back-to-back timing, 0 when the data cannot exceed L2.

    Between two reads of one layer, (NL - 1) other steps read at least L2_TURNOVER
    L2 capacities; the caches together use at most 60 % of the free device memory.
    """
    need = -(-L2_TURNOVER * l2_bytes // max(step_bytes, 1)) + 1
    nl = max(2, need)
    if nl > MAX_LAYERS or nl * cache_bytes > 0.6 * free_bytes:
        return 0
    return nl


def run_gpu(args):
    import sparse_mla_decode_03_gb300 as smla
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    w = W.WORKLOADS[args.workload]
    L = W.seq_lengths(w)
    seed = w.seed + 7919 * rank
    kv = W.make_cache(w, L, device=dev, gen_seed=seed)
    q = W.make_q(w, device=dev, gen_seed=seed)
    idx_np = [W.make_indices(w, L, variant=v + 100 * rank) for v in range(N_INDEX_SETS)]
    idx_sets = [torch.as_tensor(i, device=dev) for i in idx_np]
    B, H = w.batch, w.heads
    params = smla.make_params(B, H, w.topk, kv.shape[0], kv.stride(0), w.softmax_scale)
    S, fused = smla.smla_decode_plan(params, 0)
    ws_bytes = smla.smla_workspace_size(params, S)
    wspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    o_part = torch.empty((B, H, S, 448), dtype=torch.float32, device=dev)
    lse_part = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    out = torch.empty((B, H, 448), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # ---- layers for back-to-back timing: each its own cache, q and index set ----
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or (129 << 20))
    step_bytes = statistics.mean(W.gathered_kv_bytes(i) for i in idx_np)
    cache_bytes = kv.numel() * kv.element_size()
    NL = plan_layers(int(step_bytes), cache_bytes, l2_bytes, torch.cuda.mem_get_info(dev)[0])
    if args.layers == 1:
        NL = 0                      # one cache: isolated steps (small device footprint)
    elif args.layers > 1:
        NL = args.layers
    layers = []   # (q, kv, idx, idx_np)
    for l in range(NL):
        if l == 0:
            layers.append((q, kv, idx_sets[0], idx_np[0]))
            continue
        lseed = seed + 104729 * l
        li = W.make_indices(w, L, variant=1000 + l + 100 * rank)
        layers.append((W.make_q(w, device=dev, gen_seed=lseed),
                       W.make_cache(w, L, device=dev, gen_seed=lseed),
                       torch.as_tensor(li, device=dev), li))
    back_to_back = NL > 0

    def decode(qq, kk, ii, **kw):
        smla.sparse_mla_decode(qq, kk, ii, w.softmax_scale, out=out, lse=lse, num_splits=S,
                               workspace=wspace, **kw)

    def split_only(qq, kk, ii, **kw):
        smla.sparse_mla_decode_split(qq, kk, ii, S, w.softmax_scale, o_part=o_part,
                                     lse_part=lse_part, **kw)

    for i in range(args.warmup):
        if back_to_back:
            decode(*layers[i % NL][:3], stream=stream)
        else:
            flush.zero_()
            decode(q, kv, idx_sets[i % N_INDEX_SETS], stream=stream)
    torch.cuda.synchronize(dev)
    if smla.smla_device_status() != 0:
        raise RuntimeError("device status set during warm-up")

    def capture(fn, first, n):
        """A CUDA graph of n consecutive steps starting at layer `first`."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(n):
                fn(*layers[(first + j) % NL][:3])
        return g

    class BackToBack:
        """Exactly K back-to-back steps as graph replays of G steps (+ a remainder)."""

        def __init__(self, fn, K):
            self.G = min(K, max(NL, (GRAPH_STEPS // NL) * NL))
            self.K = K
            self.full = capture(fn, 0, self.G)
            rem = K % self.G
            self.rem = capture(fn, 0, rem) if rem else None
            self.full.replay()                 # untimed: first replay of the graphs
            if self.rem is not None:
                self.rem.replay()
            torch.cuda.synchronize(dev)

        def load(self, seconds):
            """Untimed replays for about `seconds` (the clock sampler sees the load)."""
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < seconds:
                for _ in range(8):
                    self.full.replay()
                torch.cuda.synchronize(dev)

        def run(self):
            """ms per step over exactly K steps, one event pair on the launching stream."""
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(self.K // self.G):
                self.full.replay()
            if self.rem is not None:
                self.rem.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) / self.K

    def time_isolated(fn, K):
        """Mean ms of K single-step graph replays, L2 flushed before each."""
        gs = []
        for i in range(N_INDEX_SETS):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn(q, kv, idx_sets[i])
            gs.append(g)
        for i in range(3):
            flush.zero_()
            gs[i % N_INDEX_SETS].replay()
        torch.cuda.synchronize(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            gs[i % N_INDEX_SETS].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    K = args.steps
    if back_to_back:
        b2b = BackToBack(decode, K)
        # the dominant kernel: the fused step itself, or the split kernel of a
        # two-kernel step timed on its own the same way
        b2b_split = None if fused else BackToBack(split_only, K)
    sampler = ClockSampler(dev.index)
    sampler.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if back_to_back:
        b2b.load(0.6)
        ms = b2b.run()
        split_mean = ms if fused else b2b_split.run()
    else:
        ms = time_isolated(decode, K)
        split_mean = ms if fused else time_isolated(split_only, K)
    torch.cuda.synchronize(dev)
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    if smla.smla_device_status() != 0:
        raise RuntimeError("device status set during the timed region")
    iso_ms = time_isolated(decode, 20) if back_to_back else ms
    if back_to_back:
        timing = {"timing": f"back to back: CUDA-graph replays of {b2b.G} steps, one event "
                            f"pair around all {K} steps; programmatic dependent launch "
                            f"between steps; clocks sampled over 0.6 s of the same replays "
                            f"just before and during the timed steps",
                  "l2": f"inputs larger than L2: {NL} layers, each its own {cache_bytes / 1e9:.2f} GB "
                        f"cache, q and index set; step i reads layer i mod {NL}, so "
                        f"{(NL - 1) * step_bytes / 1e6:.0f} MB of other rows are read between two "
                        f"reads of a layer (L2 {l2_bytes / 1e6:.0f} MB)",
                  "layers": NL}
    else:
        timing = {"timing": "isolated steps: one single-step CUDA-graph replay per step, "
                            "events around each",
                  "l2": f"flushed before each step ({FLUSH_BYTES >> 20} MiB write); "
                        f"{N_INDEX_SETS} rotating index sets (the workload's data cannot "
                        f"exceed L2)",
                  "layers": 1}

    # ---- context: the per-head fp32 SIMT form of the same step (the pages' pre-MMA
    # kernel style), on the same inputs, outside the timed region above ----
    simt_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(5)]
    for i in range(6):
        flush.zero_()
        if i >= 1:
            simt_ev[i - 1][0].record(stream)
        smla.sparse_mla_decode_simt(q, kv, idx_sets[i % N_INDEX_SETS], w.softmax_scale,
                                    out=out, lse=lse, stream=stream)
        if i >= 1:
            simt_ev[i - 1][1].record(stream)
    torch.cuda.synchronize(dev)
    simt_ms = statistics.mean(a.elapsed_time(b) for a, b in simt_ev)

    # ---- end to end through the C ABI: inputs from pinned host memory and results
    # back to it, every step's copies inside the timed region.  Steps are pipelined
    # over three streams, as a serving loop would run them: the inputs of step i+1
    # and the results of step i-1 move while step i decodes, with NB rotating device
    # buffer sets.  The steps cycle over the same layers as the main timing (or the
    # index sets of the one cache). ----
    e2e_src = ([(l[0], l[1], l[2]) for l in layers] if back_to_back
               else [(q, kv, i) for i in idx_sets])
    n_src = len(e2e_src)
    q_h = [x[0].cpu().pin_memory() for x in e2e_src]
    idx_h = [x[2].cpu().pin_memory() for x in e2e_src]
    NB = 3
    q_d = [torch.empty_like(q) for _ in range(NB)]
    idx_d = [torch.empty_like(idx_sets[0]) for _ in range(NB)]
    out_d = [torch.empty_like(out) for _ in range(NB)]
    lse_d = [torch.empty_like(lse) for _ in range(NB)]
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(NB)]
    lse_h = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(NB)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(NB)]
    ev_dec = [torch.cuda.Event() for _ in range(NB)]
    ev_res = [torch.cuda.Event() for _ in range(NB)]

    def e2e_steps(n, cs, chained=True):
        """n pipelined steps; cs is the decode stream.  chained=False leaves out the
        slot-reuse waits of the first NB steps (inside a captured graph, which runs
        after the previous replay has completed)."""
        for i in range(n):
            k = i % NB
            src = e2e_src[i % n_src]
            reuse = chained or i >= NB
            if reuse:
                s_in.wait_event(ev_dec[k])    # slot k's inputs consumed by step i - NB
            with torch.cuda.stream(s_in):
                q_d[k].copy_(q_h[i % n_src], non_blocking=True)
                idx_d[k].copy_(idx_h[i % n_src], non_blocking=True)
            ev_in[k].record(s_in)
            cs.wait_event(ev_in[k])
            if reuse:
                cs.wait_event(ev_res[k])      # slot k's results of step i - NB read back
            smla.sparse_mla_decode(q_d[k], src[1], idx_d[k], w.softmax_scale, out=out_d[k],
                                   lse=lse_d[k], num_splits=S, workspace=wspace, stream=cs)
            ev_dec[k].record(cs)
            s_out.wait_event(ev_dec[k])
            with torch.cuda.stream(s_out):
                out_h[k].copy_(out_d[k], non_blocking=True)
                lse_h[k].copy_(lse_d[k], non_blocking=True)
            ev_res[k].record(s_out)

    if back_to_back:
        # G pipelined steps per CUDA graph (copies as memcpy nodes, the three streams as
        # graph branches), replayed back to back; eager issue if capture fails
        G = NB * n_src * max(1, 120 // (NB * n_src))
        g_e2e = None
        try:
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e):
                cs = torch.cuda.current_stream()
                s_in.wait_stream(cs)
                s_out.wait_stream(cs)
                e2e_steps(G, cs, chained=False)
                cs.wait_stream(s_in)
                cs.wait_stream(s_out)
        except Exception:
            g_e2e = None
            torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        if g_e2e is not None:
            g_e2e.replay()
            torch.cuda.synchronize(dev)
            reps = max(1, -(-min(K, 2000) // G))
            Ke = reps * G
            e_t0 = torch.cuda.Event(enable_timing=True)
            e_t1 = torch.cuda.Event(enable_timing=True)
            e_t0.record(stream)
            for _ in range(reps):
                g_e2e.replay()
            e_t1.record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = e_t0.elapsed_time(e_t1) / Ke
            e2e_how = (f"sparse_mla_decode on device copies of pinned host q and indices, results "
                       f"copied back to pinned host buffers; copies and decode pipelined over "
                       f"three streams (3 rotating buffer sets), captured as CUDA graphs of {G} "
                       f"steps and replayed back to back, one event pair around all {Ke} steps")
        else:
            e2e_steps(2 * NB, stream)
            torch.cuda.synchronize(dev)
            Ke = max(10, min(K, 2000))
            e_t0 = torch.cuda.Event(enable_timing=True)
            e_t1 = torch.cuda.Event(enable_timing=True)
            e_t0.record(s_in)
            e2e_steps(Ke, stream)
            e_t1.record(s_out)
            torch.cuda.synchronize(dev)
            e2e_ms = e_t0.elapsed_time(e_t1) / Ke
            e2e_how = ("sparse_mla_decode on device copies of pinned host q and indices, results "
                       "copied back to pinned host buffers; copies and decode pipelined over "
                       "three streams (3 rotating buffer sets), issued eagerly, one event pair "
                       "around all steps")
    else:
        # data that cannot exceed L2: one step at a time, L2 flushed before each
        Ke = max(10, min(K // 4, 500))
        ee = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
        for i in range(3 + Ke):
            flush.zero_()
            if i >= 3:
                ee[i - 3][0].record(stream)
            q_d[0].copy_(q_h[0], non_blocking=True)
            idx_d[0].copy_(idx_h[i % n_src], non_blocking=True)
            smla.sparse_mla_decode(q_d[0], kv, idx_d[0], w.softmax_scale, out=out_d[0],
                                   lse=lse_d[0], num_splits=S, workspace=wspace, stream=stream)
            out_h[0].copy_(out_d[0], non_blocking=True)
            lse_h[0].copy_(lse_d[0], non_blocking=True)
            if i >= 3:
                ee[i - 3][1].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in ee)
        e2e_how = ("one step at a time on one stream: L2 flushed, copy of pinned host q and "
                   "indices, sparse_mla_decode, copy of the results to pinned host buffers; "
                   "events around each step")
    h2d = q.numel() * q.element_size() + idx_sets[0].numel() * 4
    d2h = out.numel() * out.element_size() + lse.numel() * 4

    # ---- aggregate over ranks ----
    ms, split_mean, e2e_ms = aggregate_over_ranks([ms, split_mean, e2e_ms], dev, ws)
    value = job_throughput(ws, B, ms)
    e2e_value = job_throughput(ws, B, e2e_ms)

    hbm_peak, tc_peak, peak_kind = read_peaks()
    timed_idx = [l[3] for l in layers] if back_to_back else idx_np
    mean_valid_bytes = statistics.mean(W.gathered_kv_bytes(i) for i in timed_idx)
    split_bytes = mean_valid_bytes + q.numel() * 2 + B * w.topk * 4
    if fused:   # the fused kernel also writes the final out and lse
        split_bytes += out.numel() * out.element_size() + lse.numel() * 4
    achieved = split_bytes / (split_mean * 1e-3) / 1e9
    flops = statistics.mean(W.algorithmic_flops(w, i) for i in timed_idx)
    tc_achieved = flops / (split_mean * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "dtype_detail": "tensor-core operands f16 (FP8 e4m3 nope dequantised exactly, bf16 "
                        "q and rope converted), fp32 accumulation and softmax; inputs FP8/bf16, "
                        "output bf16 + fp32 lse",
        "config": config_dict(w, S, fused, timing),
        "gathered_kv_gbs": ws * mean_valid_bytes / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm",
                     "kernel": "split_kernel (splits merged on chip)" if fused else "split_kernel",
                     "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "peak_source": f"hbm_gbs ({peak_kind})",
                     # measured on the headline workload only
                     "traffic": measured_traffic()
                     if (fused and args.workload == WORKLOAD) else None,
                     "algorithmic_bytes_per_launch": split_bytes,
                     "launch_ms": split_mean,
                     "tensor_frac": tc_achieved / tc_peak,
                     "tensor_tflops": tc_achieved},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": Ke,
                "how": e2e_how},
        "gpu_launches": K * (1 if fused else 2),   # per step: fused, or split + combine
        "context": {"isolated_ms_per_step": iso_ms,
                    "isolated": "one step alone: L2 flushed before it, events around a "
                                "single-step graph replay (includes the whole launch latency)",
                    "simt_ms_per_step": simt_ms, "tensor_core_speedup": simt_ms / iso_ms,
                    "simt": "sparse_mla_decode_simt: one CTA per (query, head), fp32, rows "
                            "re-read per head; 5 plain launches, L2 flushed"},
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:   # the oracle baseline: N = 1 only
        qb = W.bf16_bits(q)
        rows, remap = W.compact_rows(kv, idx_np[0])
        del kv, layers
        n, el = time_oracle(qb, rows, remap, w.softmax_scale, args.cpu_seconds)
        one = time_oracle_single_core(qb, rows, remap, w.softmax_scale, args.cpu_seconds / 2)
        line["cpu_baseline"] = {"value": n / el, "unit": UNIT, "cores": cores_used(),
                                "kind": "oracle", "cpu_model": cpu_model(),
                                "sample": f"{n} queries of the same workload (cycling over the "
                                          f"batch of {B}), {el:.1f} s, numpy float64, all "
                                          f"host cores",
                                "single_core": None if one is None else {
                                    "value": one["queries"] / one["seconds"], "unit": UNIT,
                                    "cores": one["cores"],
                                    "sample": f"{one['queries']} queries, {one['seconds']:.1f} s, "
                                              f"pinned to one core, one BLAS thread"}}
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="layer caches for back-to-back timing (0: enough to exceed L2 three "
                         "times over; 1: one cache, isolated flushed steps)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(W.WORKLOADS),
                    help="workload shape (default: the batch-32 headline workload)")
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        oracle_child(args.oracle_child, args.cpu_seconds)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
