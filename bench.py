"""Benchmark of the MoE expert LoRA fold on GB300 (prints ONE JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
    python bench.py --workload NAME --profile-launches 2     (short untimed case for ncu)

A step is one pass of the hot path over one batch of synthetic input: one
fold launch for the decode workloads, one launch that folds every row window
for the prefill workloads, one router-fold launch for the router.  The
headline workload is the largest configuration, the 163840-row prefill
(16384 tokens, top-10, 512 experts at rank 32, k_in 512, n_out 2048); every
other workload is measured in the same run under "workloads", each with the
same set of figures.

value      rows folded-or-skipped per second: the K steps are captured in one
           CUDA graph, the graph is replayed R times, each replay timed with
           CUDA events on its stream; the median replay sets the value, the
           fastest and slowest are reported beside it.  The steps rotate over
           input sets whose total exceeds L2 (each step's inputs are cold in
           L2), inputs resident in HBM.
e2e        the same metric through the C ABI with host buffers: per step the
           host route + row map and table packing, pinned host->device copies
           of x, routing, row map, tables and base_out, the fold, and the
           device->host copy of base_out, wall-clock timed with a device sync.
roofline   algorithmic bytes of one launch / its median duration vs the
           measured HBM copy bandwidth of this GPU model (MEASURED_PEAKS.json).
decode     besides the chained steps (one fold after another, where a fold's
           early start overlaps its predecessor), each decode workload also
           reports an isolated fold (the GPU idle before it, nothing to
           overlap; isolated_floor_us is the same measurement around a trivial
           kernel, the event and launch latency included in it) and a contended one (each fold right after an HBM-bound
           copy kernel moving the expert GEMM's bytes; the fold's incremental
           time over the copies alone).
cpu_baseline / --impl reference
           the fp64 CPU oracle as it stands, on a bounded sample of the same
           workload, single-threaded and on all host cores (OpenMP over rows).
Multi-GPU (torchrun): replicas -- every rank folds its own copy of the
workload, no collective on the data path; barrier + max-over-ranks timing.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE LoRA fold rows/s and achieved HBM GB/s (% of GB300 roofline), 1 GPU"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
SOAK_S = 0.6  # seconds of untimed replays under the clock sampler before the timed region
REF_TOTAL_S = 120.0  # wall-clock bound of the reference arm's timed steps
REPLAYS = 10  # timed replays of the K-step graph (median reported, min / max beside it)
DEFAULT_WORKLOAD = "prefill_large"
DECODE = ("decode_down", "decode_gate_up", "decode_down_multi")

# workload name -> (generator, description)
WORKLOADS = {
    "decode_down": "decode gather BGMV, down-proj: 64 tokens x top-8 (512 rows), 128 experts "
                   "all adapted, rank 16, k_in 768, n_out 2048, bf16",
    "decode_gate_up": "decode gather BGMV, gate/up: 256 tokens x top-8 (2048 rows), 64 of 128 "
                      "experts adapted, rank 64, k_in 2048, n_out 768; 154 active / 64 base / 38 pad",
    "decode_down_multi": "multi-adapter decode gather BGMV, down-proj: decode_down's shape with 4 "
                         "adapters installed at once (4 x 128 cells, all adapted), request slots "
                         "uniform over the 4",
    "prefill_down": "prefill grouped fold, down-proj: 8 streams U[256,768] tokens x top-8, 128 "
                    "experts, rank 16, k_in 768, n_out 2048, skewed routing, windows of 8192 rows",
    "prefill_down_xrows": "prefill grouped fold, down-proj, per-row input (x_rows [rows, 768], one "
                          "row per sorted row): prefill_down's routing, experts and windows",
    "prefill_large": "large prefill grouped fold: 16384 tokens x top-10 (163840 rows), 512 experts, "
                     "rank 32, k_in 512, n_out 2048, skewed routing, windows of 32768 rows",
    "router": "router fold (one-entry route): 16384 tokens, k_in 2048, n_out 512, rank 32",
    "tiny_decode": "tiny decode gather fold: 4 tokens x top-2, 8 experts (2 unadapted), rank 8",
    "prefill_down_fused": "expert GEMM with the fold in its epilogue, down-proj: prefill_down_xrows "
                          "plus every expert's weight W_e [2048, 768]; out = x_rows W_e^T + fold",
    "prefill_large_fused": "expert GEMM with the fold in its epilogue at the large prefill's scale: "
                           "163840 sorted rows, x_rows [163840, 512], 512 experts' W_e [2048, 512], "
                           "rank 32",
}


# ------------------------------------------------------------------ helpers
def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor TFLOP/s of this GPU model: the measured burst figure
    (a kernel timed on its own), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


KERNEL_HEADERS = ("lora_moe_expert_gb300/csrc/mlg_ptx.cuh", "lora_moe_expert_gb300/csrc/mlg_internal.h",
                  "lora_moe_expert_gb300/csrc/mlg_tiles.cuh")


def source_hash(path):
    """Hash of a kernel source together with the headers it includes."""
    h = hashlib.sha256()
    for p in (path,) + tuple(os.path.join(ROOT, k) for k in KERNEL_HEADERS):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_src, workload):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since it was captured; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        ent = rec[workload]
        if ent["source_sha"] != source_hash(os.path.join(ROOT, kernel_src)):
            return None
        return ent["dram_bytes_per_launch"]
    except Exception:
        return None


def algorithmic(w, row_map, tables):
    """(rows, folded_rows, bytes, flops) of one step: the bytes the method must
    move -- x rows of tokens with a folding row (of folding rows, for per-row
    x), A_e + B_e of each expert hit,
    the base_out read + write of each folding row, and the index arrays."""
    a, b, _ = tables
    E = a.size
    if w.kind == "gather":
        rows = w.indices.size
        tok = np.arange(rows) // w.top_k
        e = w.indices.astype(np.int64)
        if w.n_adapters:  # the row's cell in the slot-major multi-adapter tables
            s = row_map[tok].astype(np.int64)
            ok_id = (s >= 0) & (s < w.n_adapters) & (e >= 0) & (e < w.n_experts_model)
            e = np.where(ok_id, s * w.n_experts_model + e, -1)
    elif w.kind == "grouped":
        rows = w.rows
        e = np.repeat(np.arange(w.n_experts_model), np.diff(w.expert_offsets))
        e = np.concatenate([e, np.full(rows - e.size, -1)])
        tok = w.src // w.top_k
    else:
        rows = w.rows
        e = np.zeros(rows, np.int64)
        tok = np.arange(rows)
    ok = (e >= 0) & (e < E)
    ec = np.clip(e, 0, max(E - 1, 0))
    ok &= (a[ec] != 0) & (b[ec] != 0)
    if row_map is not None:
        ok &= row_map[tok] >= 0
    folded = int(ok.sum())
    experts = np.unique(e[ok]).size
    tokens = np.unique(tok[ok]).size
    r, k, n = w.max_rank, w.k_in, w.n_out
    idx_bytes = rows * 4 + (row_map.size * 4 if row_map is not None else 0) + E * 20
    if w.kind == "grouped":
        idx_bytes += (w.n_experts_model + 1) * 4
    if w.weights is not None:
        # expert GEMM with the fold: every row of a span with a weight is read
        # (x_rows) and written once (out), each such expert's W_e is read once
        e_span = np.repeat(np.arange(w.n_experts_model), np.diff(w.expert_offsets))
        e_span = np.concatenate([e_span, np.full(rows - e_span.size, -1)])
        has_w = e_span >= 0
        written = int(has_w.sum())
        w_experts = np.unique(e_span[has_w]).size
        ok &= has_w
        folded = int(ok.sum())
        experts = np.unique(e[ok]).size
        nbytes = (written * k * 2 + w_experts * n * k * 2 + experts * r * (k + n) * 2
                  + written * n * 2 + idx_bytes)
        flops = 2 * written * k * n + 2 * folded * r * (k + n)
        return rows, folded, int(nbytes), int(flops)
    n_x = folded if w.x_rows is not None else tokens  # per-row x: one x row per folding row
    nbytes = n_x * k * 2 + experts * r * (k + n) * 2 + folded * n * 4 + idx_bytes
    flops = 2 * folded * r * (k + n)
    return rows, folded, int(nbytes), int(flops)


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, settle_s=0.3):
        self.gpu = gpu_index
        self.settle_s = settle_s
        self.proc = None
        # raw samples: a temporary file unless BENCH_CLOCKS_DIR names a folder to keep them in
        folder = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(folder, f"bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            time.sleep(self.settle_s)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[4:8]):
                    if v.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ oracle timing
def time_oracle(w, budget_s=10.0, threads=1):
    """The fp64 oracle as it stands on host cores, on a bounded sample of the
    workload: whole-workload passes for small workloads, else a row sample
    (sampled rows / elapsed).  threads: OpenMP threads of the oracle's row
    loops (0 = every core).  Returns (rows_per_s, sample description, threads)."""
    import oracle

    o = oracle.get()
    used = o.set_threads(threads)
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    length = (w.n_adapters * w.n_experts_model) if w.n_adapters else None
    if w.weights is not None:  # one table cell per expert of the stacked weights
        length = w.n_experts_model
    at, bt, st = he.tables(o, length=length)
    flops_row = 2 * w.max_rank * (w.k_in + w.n_out)
    if w.weights is not None:  # the expert GEMM as well
        flops_row += 2 * w.k_in * w.n_out
        keep = np.ascontiguousarray(w.weights, np.uint16)
        wt = np.zeros(at.size, np.uint64)
        step = keep.shape[1] * keep.shape[2] * 2
        for e in range(min(at.size, keep.shape[0])):
            wt[e] = keep.ctypes.data + e * step
    full_cost = w.rows * flops_row
    rng = np.random.default_rng(0)
    t0 = time.perf_counter()
    done = 0
    passes = 0
    if full_cost <= 2e9 * used:
        while time.perf_counter() - t0 < budget_s or passes == 0:
            if w.kind == "gather" and w.n_adapters:
                _, ra = o.build_moe_row_adapter_decode_multi(w.adapter_slots, w.padded_n,
                                                             w.n_adapters, w.has_moe_lora)
                o.gather_fold_multi(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank,
                                    w.n_out, w.top_k, w.n_experts_model, w.n_adapters)
            elif w.kind == "gather":
                ra = o.build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, w.active,
                                                    w.has_moe_lora)
                o.gather_fold(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank,
                              w.n_out, w.top_k)
            elif w.kind == "grouped" and w.weights is not None:
                ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
                o.grouped_gemm_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra, wt, at, bt, st,
                                          w.base, w.k_in, w.max_rank, w.n_out, w.top_k, 0, w.rows)
            elif w.kind == "grouped" and w.x_rows is not None:
                ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
                o.grouped_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra, at, bt, st, w.base,
                                     w.k_in, w.max_rank, w.n_out, w.top_k, 0, w.rows)
            elif w.kind == "grouped":
                ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
                for s, e in o.grouped_down_windows(w.rows, w.cap):
                    o.grouped_fold(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base, w.k_in,
                                   w.max_rank, w.n_out, w.top_k, s, e)
            else:
                o.router_fold(w.x, None, at, bt, st, w.base, w.k_in, w.max_rank, w.n_out)
            done += w.rows
            passes += 1
        dt = time.perf_counter() - t0
        o.set_threads(0)
        return (done / dt, f"{passes} whole-workload pass(es) of {w.rows} rows in {dt:.1f} s "
                           f"on {used} thread(s)", used)
    chunk = 64 * used
    while time.perf_counter() - t0 < budget_s or done == 0:
        rows = np.sort(rng.choice(w.rows, size=min(chunk, w.rows), replace=False)).astype(np.int32)
        if w.kind == "grouped" and w.weights is not None:
            ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
            o.grouped_gemm_fold_xrows_rows(w.x_rows, w.expert_offsets, w.src, ra, wt, at, bt, st,
                                           w.base[rows], rows, w.k_in, w.max_rank, w.n_out,
                                           w.top_k, 0, w.rows)
        elif w.kind == "grouped" and w.x_rows is not None:
            ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
            o.grouped_fold_xrows_rows(w.x_rows, w.expert_offsets, w.src, ra, at, bt, st,
                                      w.base[rows], rows, w.k_in, w.max_rank, w.n_out, w.top_k,
                                      0, w.rows)
        elif w.kind == "grouped":
            ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
            o.grouped_fold_rows(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base[rows], rows,
                                w.k_in, w.max_rank, w.n_out, w.top_k, 0, w.rows)
        elif w.kind == "gather":
            ra = o.build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, w.active,
                                                w.has_moe_lora)
            o.gather_fold_rows(w.x, w.indices, ra, at, bt, st, w.base[rows], rows, w.k_in,
                               w.max_rank, w.n_out, w.top_k)
        else:
            o.gather_fold_rows(w.x, np.zeros(w.rows, np.int32), None, at, bt, st, w.base[rows],
                               rows, w.k_in, w.max_rank, w.n_out, 1)
        done += rows.size
    dt = time.perf_counter() - t0
    o.set_threads(0)
    return (done / dt, f"{done} sampled rows of {w.rows} in {dt:.1f} s (row-by-row oracle) on "
                       f"{used} thread(s)", used)


def cpu_baseline(w, budget_s):
    """The oracle on one host core and on all of them (same bits either way)."""
    one, d1, _ = time_oracle(w, budget_s, threads=1)
    alln, dn, used = time_oracle(w, budget_s, threads=0)
    return {"value": alln, "unit": "rows/s", "cores": used, "kind": "oracle", "sample": dn,
            "single_thread_value": one, "single_thread_sample": d1,
            "host_cpu_count": os.cpu_count()}


# ------------------------------------------------------------------ GPU arm
def n_sets_for(w_bytes):
    """Input sets the timed steps rotate over: at least two, and enough that
    their total is twice the L2."""
    return max(2, min(32, int(np.ceil(2.0 * L2_BYTES / max(w_bytes, 1)))))


# The kernel that folds each named workload (the decode fold takes expert
# pairs of rank 16 or 32 that fit half an SM; other decode shapes go to the
# cluster kernel).
KERNEL_OF = {"decode_down": "mlg_decode.cu", "decode_gate_up": "mlg_gather.cu",
             "tiny_decode": "mlg_gather.cu", "prefill_down": "mlg_grouped.cu",
             "prefill_large": "mlg_grouped.cu", "router": "mlg_grouped.cu",
             "prefill_down_xrows": "mlg_grouped.cu", "decode_down_multi": "mlg_decode.cu",
             "prefill_down_fused": "mlg_gemm_fold.cu", "prefill_large_fused": "mlg_gemm_fold.cu"}


def kernel_source(workload):
    return "lora_moe_expert_gb300/csrc/" + KERNEL_OF[workload]


def make_sets(name, device, seed_base):
    """Device-resident input sets of a workload.  Sets past the first draw
    fresh inputs when the workload is small; a workload larger than half the
    L2 reuses the first set's host arrays in new device allocations (the
    timing only needs distinct memory, and drawing them would take longer
    than the measurement)."""
    from lora_moe_expert_gb300 import synth
    from lora_moe_expert_gb300.device import FoldProblem

    gen = synth.NAMED[name]
    w0 = gen()
    p0 = FoldProblem(w0, device=device)
    ws_bytes = (w0.x.nbytes + w0.base.nbytes + sum(e.A.nbytes + e.B.nbytes for e in w0.experts)
                + (w0.x_rows.nbytes if w0.x_rows is not None else 0)
                + (w0.weights.nbytes if w0.weights is not None else 0))
    nsets = n_sets_for(ws_bytes)
    big = ws_bytes > L2_BYTES // 2
    probs = [p0] + [FoldProblem(w0 if big else gen(seed=seed_base + i), device=device)
                    for i in range(1, nsets)]
    return probs, ws_bytes


def _events(n):
    import torch

    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def time_graph(graph, stream, replays, barrier=False, sampler=None):
    """Milliseconds of each of `replays` timed replays of `graph` (CUDA events
    on `stream`), after a soak of untimed replays (under the clock sampler
    when one is given)."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(3):
            graph.replay()
        stream.synchronize()
        if sampler is not None:
            t_soak = time.perf_counter()
            while time.perf_counter() - t_soak < SOAK_S:
                graph.replay()
                stream.synchronize()
    if barrier and torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = _events(replays)
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            e0.record(stream)
            graph.replay()
            e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def capture(fn, stream):
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def time_isolated(probs, n, stream, body=None):
    """Each fold alone: the GPU spins in a sleep kernel while the host enqueues
    an event, the fold and an event, so the fold starts on an idle stream with
    nothing to overlap.  Milliseconds per fold, n samples over the sets.  With
    `body`, the same measurement of body(i) instead of a fold."""
    import torch

    ev = _events(n)
    with torch.cuda.stream(stream):
        for i, (e0, e1) in enumerate(ev):
            torch.cuda._sleep(1000000)  # ~0.5 ms: the host enqueues the fold meanwhile
            e0.record(stream)
            if body is None:
                probs[i % len(probs)].run(stream=stream)
            else:
                body(i)
            e1.record(stream)
    stream.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in ev]


def isolated_floor(stream, n=40):
    """The same isolated measurement around a trivial kernel (an add on 16
    floats): the event and launch latency any kernel timed this way pays."""
    import torch

    t = torch.zeros(16, device=stream.device)
    return statistics.median(time_isolated(None, n, stream, body=lambda i: t.add_(1)))


def expert_gemm_bytes(w):
    """Bytes of the expert GEMM a decode fold follows in a model: the weight
    W_e [n_out, k_in] of every expert the routing hits (whether or not it is
    adapted), x and the output rows."""
    idx = w.indices.astype(np.int64)
    hit = np.unique(idx[(idx >= 0) & (idx < w.n_experts_model)]).size
    return hit * w.n_out * w.k_in * 2 + w.x.nbytes + w.base.nbytes


def time_contended(probs, steps, stream, copy_bytes, replays):
    """Each fold right after an HBM-bound copy kernel (an elementwise bf16
    multiply by one, reading and writing copy_bytes / 2 each): the fold's
    incremental milliseconds over the copies alone, per step."""
    import torch

    n = max(1, copy_bytes // 4)
    src = torch.ones(n, dtype=torch.bfloat16, device=stream.device)
    dst = torch.empty_like(src)

    def copies_and_folds():
        for i in range(steps):
            torch.mul(src, 1.0, out=dst)
            probs[i % len(probs)].run(stream=stream)

    def copies():
        for _ in range(steps):
            torch.mul(src, 1.0, out=dst)

    g_both, g_copy = capture(copies_and_folds, stream), capture(copies, stream)
    t_both = statistics.median(time_graph(g_both, stream, replays))
    t_copy = statistics.median(time_graph(g_copy, stream, replays))
    del g_both, g_copy
    return (t_both - t_copy) / steps, t_copy / steps


def gpu_measure(name, steps, warmup, device, seed_base=1000, replays=REPLAYS, e2e=True,
                decode_extra=True, barrier=False):
    import torch

    import lora_moe_expert_gb300 as mlg

    probs, ws_bytes = make_sets(name, device, seed_base)
    nsets = len(probs)
    # The input sets may differ in size (prefill lengths are drawn per seed):
    # the per-step figures are the mean over the steps the timed graph runs.
    alg = np.array([algorithmic(probs[i % nsets].w, probs[i % nsets].row_map_host,
                                probs[i % nsets].tables_host) for i in range(steps)], np.float64)
    rows, folded, nbytes, flops = alg.mean(axis=0)
    launches_per_step = 1  # the grouped form folds all windows in one launch
    w0 = probs[0].w

    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):  # eager warm-up steps
            probs[i % nsets].run(stream=stream)
    stream.synchronize()
    errors_before = mlg.mlg_read_device_errors(clear=True)

    def chain():
        for i in range(steps):
            probs[i % nsets].run(stream=stream)

    graph = capture(chain, stream)
    with ClockSampler(torch.cuda.current_device(), settle_s=0.0) as clocks:
        ms = time_graph(graph, stream, replays, barrier=barrier, sampler=clocks)
    del graph
    out = {"rows": rows, "folded_rows": folded, "alg_bytes": nbytes, "alg_flops": flops,
           "rows_set0": w0.rows, "ms_replays": ms, "ms_total": statistics.median(ms),
           "launches_per_step": launches_per_step, "replays": replays, "sets": nsets,
           "set_bytes": ws_bytes, "clocks": clocks.summary(), "kind": w0.kind}
    if decode_extra and name in DECODE:
        iso = time_isolated(probs, 40, stream)
        out["isolated_ms"] = statistics.median(iso)
        out["isolated_ms_min"] = min(iso)
        out["isolated_floor_ms"] = isolated_floor(stream)
        cb = expert_gemm_bytes(w0)
        inc, copy_ms = time_contended(probs, min(steps, 20), stream, cb, max(3, replays // 2))
        out["contended_ms"] = inc
        out["contended_copy_bytes"] = cb
        out["contended_copy_ms"] = copy_ms
    if w0.weights is not None:
        # the same step unfused: the plain expert GEMM (LoRA cells zero), then
        # the per-row x fold reading its output back
        def gemm_only():
            for i in range(steps):
                probs[i % nsets].run(stream=stream, lora=False)

        def fold_only():
            for i in range(steps):
                q = probs[i % nsets]
                mlg.mlg_grouped_down_xrows(q.x_rows, q.expert_offsets, q.src, q.row_adapter,
                                           q.a_table, q.b_table, q.scale_table, q.base,
                                           q.w.k_in, q.w.max_rank, q.w.n_out, q.w.top_k,
                                           q.n_experts, 0, q.w.rows, q.w.cap, stream=stream)

        for nm_, fn in (("gemm_only_ms", gemm_only), ("fold_only_ms", fold_only)):
            g = capture(fn, stream)
            out[nm_] = statistics.median(time_graph(g, stream, replays))
            del g
    if mlg.mlg_read_device_errors(clear=True) or errors_before:
        raise RuntimeError("device error bits were set during the benchmark")
    if e2e:
        out["e2e"] = e2e_measure(probs[0], max(3, min(steps, 20 if w0.rows > 50000 else 50)),
                                 device)
    return out


def e2e_measure(prob, steps, device):
    """Through the public API with host buffers: route + map and table packing on
    the host, pinned H2D copies of the step's inputs, the fold, D2H of base_out.
    A prefill workload with more than one row window runs the range calls on
    pieces of at most 8192 rows (inside windows), so piece i's rows go up while
    piece i-1 folds and piece i-2's come back, on three streams; the
    GEMM + fold form writes every row of its spans, so its base_out is not
    uploaded.  Timed twice: with a synchronize after every step, and as a
    stream of steps where each upload waits only for the previous step's last
    use of the same device buffer (a piece's rows for its download, the
    tables / row map / token x for the step's last fold) and one synchronize
    ends the timed region -- the rate at which a caller feeding batches back
    to back folds them."""
    import torch

    import lora_moe_expert_gb300 as mlg
    from lora_moe_expert_gb300.device import pad_tables

    w = prob.w
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    xrows = w.x_rows is not None
    h_x = pin((w.x_rows if xrows else w.x).view(np.int16))
    d_x = prob.x_rows if xrows else prob.x
    h_base = pin(w.base.view(np.int16))
    h_out = torch.empty_like(h_base).pin_memory()
    h_idx = pin(w.indices) if w.kind == "gather" else None
    h_off = pin(w.expert_offsets) if w.kind == "grouped" else None
    h_src = pin(w.src) if w.kind == "grouped" else None
    s = torch.cuda.Stream(device=device)
    h2d = d2h = 0
    prev_fold = None  # the previous step's last fold (its tables, row map and x are then free)
    d2h_done = {}  # piece -> the previous step's download of that piece's rows

    def step(sync):
        nonlocal h2d, d2h, prev_fold
        h2d = d2h = 0
        if prev_fold is not None:
            s.wait_event(prev_fold)
        with torch.cuda.stream(s):
            if w.kind == "gather" and w.n_adapters:
                m = mlg.mlg_build_moe_row_adapter_decode_multi(w.adapter_slots, w.padded_n,
                                                               w.n_adapters, w.has_moe_lora)
            elif w.kind == "gather":
                m = mlg.mlg_build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, w.active,
                                                         w.has_moe_lora)
            elif w.kind == "grouped":
                m = mlg.mlg_build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
            else:
                m = None
            a, b, sc = mlg.mlg_pack_expert_tables(prob.pool.ids, prob.pool.a_addr,
                                                  prob.pool.b_addr, prob.pool.scale)
            if w.n_adapters:
                a, b, sc = pad_tables(a, b, sc, w.n_adapters * w.n_experts_model)
            mlg.mlg_upload_expert_tables(a, b, sc, prob.a_table, prob.b_table, prob.scale_table,
                                         stream=s)
            h2d += a.nbytes + b.nbytes + sc.nbytes
            if m is not None:
                mlg.mlg_upload_row_adapter(m, prob.row_adapter, stream=s)
                h2d += m.nbytes
            if windows is None or not xrows:  # token x: the whole of it, before any window
                d_x.view(torch.int16).copy_(h_x, non_blocking=True)
                h2d += h_x.numel() * 2
            if windows is None:
                prob.base.view(torch.int16).copy_(h_base, non_blocking=True)
                h2d += h_base.numel() * 2
            if h_idx is not None:
                prob.indices.copy_(h_idx, non_blocking=True)
                h2d += h_idx.numel() * 4
            if h_off is not None:
                prob.expert_offsets.copy_(h_off, non_blocking=True)
                prob.src.copy_(h_src, non_blocking=True)
                h2d += h_off.numel() * 4 + h_src.numel() * 4
            if windows is None:
                prob.run(stream=s)
                h_out.copy_(prob.base.view(torch.int16), non_blocking=True)
                d2h += h_out.numel() * 2
        if windows is not None:
            prev_fold = windowed(s)
        if sync:
            sync_all()

    def sync_all():
        s.synchronize()
        if windows is not None:
            s_cmp.synchronize()
            s_d2h.synchronize()

    # Windowed prefill forms: the window calls of the public API let window
    # i's base_out rows (and per-row x) go up while window i-1 folds and
    # window i-2's rows come back, on three streams (a caller's own pipeline).
    # The fused form writes every row, so its base_out is never uploaded.
    windows = None
    if w.kind == "grouped" and len(prob.windows) > 1:
        # pieces of at most 8192 rows inside each window (a call may take any
        # sub-range of a window: every row's result is independent of it)
        windows = []
        for (a0, a1) in prob.windows:
            n_p = -(-(a1 - a0) // 8192)
            windows += [(a0 + (a1 - a0) * i // n_p, a0 + (a1 - a0) * (i + 1) // n_p)
                        for i in range(n_p)]
        s_cmp = torch.cuda.Stream(device=device)
        s_d2h = torch.cuda.Stream(device=device)
    fused = prob.w_experts is not None

    def windowed(s_up):
        nonlocal h2d, d2h
        ra = prob.row_adapter
        done = None
        for k, (r0, r1) in enumerate(windows):
            if k in d2h_done:  # the previous step's download of these rows
                s_up.wait_event(d2h_done[k])
            with torch.cuda.stream(s_up):
                if xrows:
                    prob.x_rows[r0:r1].view(torch.int16).copy_(h_x[r0:r1], non_blocking=True)
                    h2d += (r1 - r0) * h_x.shape[1] * 2
                if not fused:
                    prob.base[r0:r1].view(torch.int16).copy_(h_base[r0:r1], non_blocking=True)
                    h2d += (r1 - r0) * h_base.shape[1] * 2
                up = torch.cuda.Event()
                up.record(s_up)
            s_cmp.wait_event(up)
            with torch.cuda.stream(s_cmp):
                if fused:
                    mlg.mlg_grouped_gemm_fold_xrows(prob.x_rows, prob.expert_offsets, prob.src, ra,
                                                    prob.w_experts, prob.a_table, prob.b_table,
                                                    prob.scale_table, prob.base, w.k_in,
                                                    w.max_rank, w.n_out, w.top_k, prob.n_experts,
                                                    r0, r1, w.cap, stream=s_cmp)
                elif xrows:
                    mlg.mlg_grouped_down_xrows(prob.x_rows, prob.expert_offsets, prob.src, ra,
                                               prob.a_table, prob.b_table, prob.scale_table,
                                               prob.base, w.k_in, w.max_rank, w.n_out, w.top_k,
                                               prob.n_experts, r0, r1, w.cap, stream=s_cmp)
                else:
                    mlg.mlg_grouped_down(prob.x, prob.expert_offsets, prob.src, ra, prob.a_table,
                                         prob.b_table, prob.scale_table, prob.base, w.k_in,
                                         w.max_rank, w.n_out, w.top_k, prob.n_experts, r0, r1,
                                         stream=s_cmp)
                done = torch.cuda.Event()
                done.record(s_cmp)
            s_d2h.wait_event(done)
            with torch.cuda.stream(s_d2h):
                h_out[r0:r1].copy_(prob.base[r0:r1].view(torch.int16), non_blocking=True)
                d2h += (r1 - r0) * h_out.shape[1] * 2
                ev = torch.cuda.Event()
                ev.record(s_d2h)
                d2h_done[k] = ev
        return done

    for _ in range(3):
        step(True)
    t0 = time.perf_counter()
    for _ in range(steps):
        step(True)
    dt_sync = (time.perf_counter() - t0) / steps
    t0 = time.perf_counter()
    for _ in range(steps):
        step(False)
    sync_all()
    dt = (time.perf_counter() - t0) / steps
    return {"s_per_step": dt, "s_per_step_synced": dt_sync, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps}


# ------------------------------------------------------------------ replicas
def replica_seed_base(rank: int) -> int:
    """Seed offset of a replica's rotating input sets (distinct per rank)."""
    return 1000 + 97 * rank


def max_over_ranks(value: float, device) -> float:
    """The step time of the job: the maximum over ranks (timing only -- the
    fold itself exchanges nothing between replicas)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_step: int, world: int, ms_step: float) -> float:
    """Whole-job throughput: every replica folds its own batch per step."""
    return world * rows_per_step / (ms_step * 1e-3)


# ------------------------------------------------------------------ main
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from lora_moe_expert_gb300 import synth

    w = synth.NAMED[args.workload]()
    steps_rows = []
    for _ in range(args.warmup):
        time_oracle(w, budget_s=0.0, threads=0)
    # Each step is a bounded sample: the whole timed run stays within about
    # REF_TOTAL_S whatever --steps is (at most --ref-budget seconds a step).
    budget = min(args.ref_budget, REF_TOTAL_S / max(args.steps, 1))
    t0 = time.perf_counter()
    samples = []
    used = 1
    for _ in range(args.steps):
        rps, desc, used = time_oracle(w, budget_s=budget, threads=0)
        steps_rows.append(rps)
        samples.append(desc)
    total = time.perf_counter() - t0
    value = statistics.mean(steps_rows)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "description": WORKLOADS[args.workload],
                       "parallelism": "none (host oracle, OpenMP over rows)"},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": used, "kind": "oracle",
                             "sample": samples[0], "host_cpu_count": os.cpu_count()},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profile_case(name, launches, device):
    """A short, untimed run for profilers: one input set, the step `launches`
    times (the first launch of a fresh process pays module loading)."""
    import torch

    import lora_moe_expert_gb300 as mlg
    from lora_moe_expert_gb300 import synth
    from lora_moe_expert_gb300.device import FoldProblem

    prob = FoldProblem(synth.NAMED[name](), device=device)
    for _ in range(launches):
        prob.run()
    torch.cuda.synchronize(device)
    if mlg.mlg_read_device_errors(clear=True):
        raise RuntimeError("device error bits were set")
    print(f"profile case {name}: {launches} launch(es) done", flush=True)
    return 0


def summarize(name, r, peak, steps, cpu=None):
    """Per-workload figures from one gpu_measure result."""
    ms = r["ms_total"] / steps
    per_launch = ms / r["launches_per_step"]
    gbs = r["alg_bytes"] / r["launches_per_step"] / (per_launch * 1e-3) / 1e9
    out = {"rows_per_s": r["rows"] / (ms * 1e-3), "us_per_step": ms * 1e3,
           "us_per_step_min": min(r["ms_replays"]) / steps * 1e3,
           "us_per_step_max": max(r["ms_replays"]) / steps * 1e3,
           "replays": r["replays"], "launches_per_step": r["launches_per_step"],
           "rows_per_step": r["rows"], "folded_rows_per_step": r["folded_rows"],
           "alg_bytes_per_step": r["alg_bytes"], "achieved_gbs": gbs, "frac_of_peak": gbs / peak,
           "tflops": r["alg_flops"] / (ms * 1e-3) / 1e12,
           "traffic": recorded_traffic(kernel_source(name), name),
           "l2": f"{r['sets']} rotating input sets of {r['set_bytes'] / 2**20:.0f} MiB",
           "clocks": r["clocks"]}
    if "isolated_ms" in r:
        iso, con = r["isolated_ms"], r["contended_ms"]
        out["isolated_us"] = iso * 1e3
        out["isolated_us_min"] = r["isolated_ms_min"] * 1e3
        out["isolated_floor_us"] = r["isolated_floor_ms"] * 1e3
        out["isolated_frac_of_peak"] = r["alg_bytes"] / (iso * 1e-3) / 1e9 / peak
        out["contended_us"] = con * 1e3
        out["contended_frac_of_peak"] = (r["alg_bytes"] / (con * 1e-3) / 1e9 / peak
                                         if con > 0 else None)
        out["contended_copy_bytes"] = r["contended_copy_bytes"]
        out["contended_copy_us"] = r["contended_copy_ms"] * 1e3
    if "gemm_only_ms" in r:
        out["gemm_only_us"] = r["gemm_only_ms"] / steps * 1e3
        out["fold_only_us"] = r["fold_only_ms"] / steps * 1e3
        out["unfused_us"] = out["gemm_only_us"] + out["fold_only_us"]
        out["fused_speedup"] = out["unfused_us"] / out["us_per_step"]
        out["tensor_tflops_peak"] = tensor_peak()[0]
        t_hbm = r["alg_bytes"] / (peak * 1e9)
        t_tc = r["alg_flops"] / (tensor_peak()[0] * 1e12)
        out["bound"] = "hbm" if t_hbm >= t_tc else "tensor"
        out["roofline_frac"] = max(t_hbm, t_tc) / (ms * 1e-3)
    if "e2e" in r:
        e = r["e2e"]
        out["e2e"] = {"value": r["rows_set0"] / e["s_per_step"], "unit": "rows/s",
                      "h2d_bytes_per_step": e["h2d_bytes_per_step"],
                      "d2h_bytes_per_step": e["d2h_bytes_per_step"],
                      "value_synchronized_steps": r["rows_set0"] / e["s_per_step_synced"]}
    if cpu is not None:
        out["cpu_baseline"] = cpu
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--extra", default="decode_down,decode_gate_up,decode_down_multi,prefill_down,"
                                       "prefill_down_xrows,router,prefill_down_fused,"
                                       "prefill_large_fused",
                    help="other workloads measured in the same run (comma list, or 'none')")
    ap.add_argument("--replays", type=int, default=REPLAYS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=3.0,
                    help="seconds of oracle work per (workload, thread count) sample")
    ap.add_argument("--ref-budget", type=float, default=10.0)
    ap.add_argument("--profile-launches", type=int, default=0,
                    help="profiler case: run the workload's step this many times on cuda:0, "
                         "untimed, and exit (no JSON line)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    import __graft_entry__

    __graft_entry__.build()
    if args.profile_launches > 0:
        return profile_case(args.workload, args.profile_launches, device)

    main_res = gpu_measure(args.workload, args.steps, args.warmup, device,
                           seed_base=replica_seed_base(rank), replays=args.replays,
                           barrier=True)
    ms_step = max_over_ranks(main_res["ms_total"] / args.steps, device)
    main_res["e2e"]["s_per_step"] = max_over_ranks(main_res["e2e"]["s_per_step"], device)
    main_res["e2e"]["s_per_step_synced"] = max_over_ranks(main_res["e2e"]["s_per_step_synced"],
                                                          device)
    peak, peak_kind = measured_peaks()
    per_launch_ms = ms_step / main_res["launches_per_step"]
    achieved = main_res["alg_bytes"] / main_res["launches_per_step"] / (per_launch_ms * 1e-3) / 1e9
    extras = {}
    if args.extra != "none" and rank == 0:
        from lora_moe_expert_gb300 import synth

        for nm in [s for s in args.extra.split(",") if s and s != args.workload]:
            try:
                r = gpu_measure(nm, args.steps, 3, device, replays=args.replays)
                cpu = None if args.no_cpu_baseline else cpu_baseline(synth.NAMED[nm](),
                                                                      args.cpu_budget)
                extras[nm] = summarize(nm, r, peak, args.steps, cpu)
            except Exception as ex:  # report, do not hide
                extras[nm] = {"error": repr(ex)[:300]}
    if rank != 0:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
        return 0

    cpu = None
    if not args.no_cpu_baseline:
        from lora_moe_expert_gb300 import synth

        cpu = cpu_baseline(synth.NAMED[args.workload](), args.cpu_budget)
    e2e = main_res["e2e"]
    spread = [m / args.steps for m in main_res["ms_replays"]]
    line = {
        "metric": METRIC,
        "value": job_rows_per_s(main_res["rows"], ws, ms_step),
        "unit": "rows/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "ms_per_step_min": min(spread),
        "ms_per_step_max": max(spread),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "description": WORKLOADS[args.workload],
                   "rows_per_step": main_res["rows"], "folded_rows_per_step": main_res["folded_rows"],
                   "rows_note": "mean over the timed steps' input sets",
                   "l2": f"inputs rotate over {main_res['sets']} sets of "
                         f"{main_res['set_bytes'] / 2**20:.1f} MiB (> L2 in total)",
                   "timing": f"CUDA events around each of {args.replays} replays of one "
                             f"CUDA graph of the {args.steps} steps; median replay "
                             f"(min / max beside it)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "alg_bytes_per_launch": int(main_res["alg_bytes"] / main_res["launches_per_step"]),
                     "traffic": recorded_traffic(kernel_source(args.workload), args.workload)},
        "tflops": main_res["alg_flops"] / (ms_step * 1e-3) / 1e12,
        "cpu_baseline": cpu,
        "e2e": {"value": job_rows_per_s(main_res["rows_set0"], ws, e2e["s_per_step"] * 1e3),
                "unit": "rows/s",
                "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
                "value_synchronized_steps": job_rows_per_s(main_res["rows_set0"], ws,
                                                           e2e["s_per_step_synced"] * 1e3)},
        "gpu_launches": args.replays * args.steps * main_res["launches_per_step"],
        "clocks": main_res["clocks"],
        "workloads": extras,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
