"""Seeded synthetic workloads for the MoE expert LoRA fold.

This module only draws inputs: activations, expert pairs, routing, row
order and adapter slots.  It contains none of the fold's arithmetic, no
routing rule, no row-map rule and no table packing, so the CUDA path and the
CPU oracle can both consume what it returns without sharing any of the
method.  Everything is numpy, seeded with ``numpy.random.default_rng``.

Recipe (stand-in for Qwen3-MoE / Qwen3-Next serving traffic; no dataset,
no trained weights):

* bf16 values are fp32 draws rounded to nearest-even;
* x ~ N(0, 1); A_e ~ N(0, 1/k_in); B_e ~ N(0, 1/rank); scale_e ~ U(0.5, 2);
  base_out ~ N(0, 1) (the second N argument is the variance);
* decode routing: top_k of per-token N(0, 1) logits (descending, no repeats);
* prefill routing: the same with a per-expert bias ~ N(0, 1.5) added to the
  logits (skewed expert counts), then a stable counting sort of the flat
  (token, slot) rows by expert gives ``expert_offsets`` and ``src``.

Shapes of the named workloads:

* ``tiny_decode``      4 tokens, top-2, 8 experts (ids 1, 3 unadapted), one
                       routed id 9, k_in 64, n_out 96, rank 8,
                       adapter slots [0, -1, 0, 2], active 0, padded_n 4
* ``decode_down``      64 tokens, top-8, 128 experts all adapted, rank 16,
                       k_in 768, n_out 2048, every token active
* ``prefill_down``     8 streams of U[256, 768] tokens, top-8, 128 experts,
                       rank 16, k_in 768, n_out 2048, windows of 8192 rows
* ``decode_gate_up``   256 tokens, top-8, 64 of 128 experts adapted, rank 64,
                       k_in 2048, n_out 768; 154 active, 64 base, 38 padding
* ``prefill_down_xrows`` ``prefill_down`` with a per-row input: x_rows
                       [rows, 768] ~ N(0, 1), one row per sorted row (the
                       expert's intermediate activation in a down projection)
* ``decode_down_multi`` ``decode_down``'s shape with 4 adapters installed at
                       once (every expert adapted in each), each request's
                       slot uniform over the 4; tables of 4 x 128 cells
* ``prefill_large``    16384 tokens, top-10, 512 experts, rank 32, k_in 512,
                       n_out 2048, windows of 32768 rows
* ``router``           one-entry route over 16384 tokens, k_in 2048,
                       n_out 512, rank 32
* ``prefill_down_fused`` ``prefill_down_xrows`` plus every expert's GEMM
                       weight W_e [2048, 768] ~ N(0, 1/768): the expert GEMM
                       with the fold in its epilogue
* ``prefill_large_fused`` ``prefill_large`` with a per-row input x_rows
                       [163840, 512] and the 512 experts' weights
                       W_e [2048, 512] ~ N(0, 1/512), the same fused form
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np


def bf16_bits(f32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng, shape, variance: float = 1.0) -> np.ndarray:
    v = rng.standard_normal(shape, dtype=np.float32)
    if variance != 1.0:
        v *= np.float32(np.sqrt(variance))
    return bf16_bits(v)


@dataclasses.dataclass
class Expert:
    expert_id: int
    A: np.ndarray  # bf16 bits [max_rank, k_in]
    B: np.ndarray  # bf16 bits [n_out, max_rank]
    scale: float


@dataclasses.dataclass
class Workload:
    name: str
    kind: str  # "gather" | "grouped" | "router"
    k_in: int
    max_rank: int
    n_out: int
    top_k: int
    n_tokens: int
    x: np.ndarray  # bf16 bits [n_tokens, k_in]
    base: np.ndarray  # bf16 bits [rows, n_out]
    experts: List[Expert]
    n_experts_model: int
    # gather form
    indices: Optional[np.ndarray] = None  # int32 [n_slots]
    adapter_slots: Optional[np.ndarray] = None  # int32, decode request slots
    padded_n: int = 0
    active: int = 0
    has_moe_lora: bool = True
    # grouped form
    expert_offsets: Optional[np.ndarray] = None  # int32 [n_experts_model + 1]
    src: Optional[np.ndarray] = None  # int32 [rows], sorted row -> flat row
    cu_seqlens: Optional[np.ndarray] = None  # int32 [batch + 1]
    stream_slots: Optional[np.ndarray] = None  # int32 [batch]
    cap: int = 0
    x_rows: Optional[np.ndarray] = None  # bf16 bits [rows, k_in]: per-row input, sorted order
    # multi-adapter form: tables of n_adapters * n_experts_model cells, slot-major
    # (expert_id of an Expert is its cell, slot * n_experts_model + expert)
    n_adapters: int = 0
    # expert GEMM weights for the fused GEMM + fold form: bf16 bits
    # [n_experts_model, n_out, k_in], the experts' W_e stacked; base then holds
    # the output buffer's prior contents (rows outside the range keep them)
    weights: Optional[np.ndarray] = None

    @property
    def rows(self) -> int:
        return int(self.base.shape[0])


def _experts(rng, ids, k_in, max_rank, n_out, rank: Optional[int] = None) -> List[Expert]:
    """Pairs for the given ids; rows/cols at or past `rank` are zero padding."""
    rank = max_rank if rank is None else rank
    out = []
    for eid in ids:
        A = np.zeros((max_rank, k_in), np.uint16)
        B = np.zeros((n_out, max_rank), np.uint16)
        A[:rank] = _normal_bf16(rng, (rank, k_in), 1.0 / k_in)
        B[:, :rank] = _normal_bf16(rng, (n_out, rank), 1.0 / rank)
        s = float(rng.uniform(0.5, 2.0))
        out.append(Expert(int(eid), A, B, float(np.float32(s))))
    return out


def top_k_routing(rng, n_tokens: int, n_experts: int, top_k: int,
                  bias_variance: float = 0.0) -> np.ndarray:
    """[n_tokens, top_k] expert ids: the top_k of N(0,1) logits (+ per-expert bias)."""
    if top_k > n_experts:
        raise ValueError(f"top_k={top_k} exceeds n_experts={n_experts}")
    logits = rng.standard_normal((n_tokens, n_experts), dtype=np.float32)
    if bias_variance > 0:
        bias = rng.standard_normal(n_experts, dtype=np.float32) * np.float32(np.sqrt(bias_variance))
        logits += bias[None, :]
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :top_k].astype(np.int32)


def sort_rows_by_expert(flat_experts: np.ndarray, n_experts: int) -> Tuple[np.ndarray, np.ndarray]:
    """Stable counting sort of flat rows by expert: (expert_offsets [E+1], src [rows])."""
    counts = np.bincount(flat_experts, minlength=n_experts).astype(np.int64)
    offsets = np.zeros(n_experts + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    src = np.argsort(flat_experts, kind="stable").astype(np.int32)
    return offsets.astype(np.int32), src


def tiny_decode(seed: int = 0) -> Workload:
    rng = np.random.default_rng(seed)
    T, K, E, k_in, n_out, r = 4, 2, 8, 64, 96, 8
    idx = top_k_routing(rng, T, E, K).reshape(-1)
    idx[int(rng.integers(0, T * K))] = 9  # one routed id past the table
    x = _normal_bf16(rng, (T, k_in))
    base = _normal_bf16(rng, (T * K, n_out))
    experts = _experts(rng, [0, 2, 4, 5, 6, 7], k_in, r, n_out)
    return Workload("tiny_decode", "gather", k_in, r, n_out, K, T, x, base, experts, E,
                    indices=idx, adapter_slots=np.array([0, -1, 0, 2], np.int32), padded_n=4,
                    active=0, has_moe_lora=True)


def decode_down(seed: int = 1) -> Workload:
    rng = np.random.default_rng(seed)
    T, K, E, k_in, n_out, r = 64, 8, 128, 768, 2048, 16
    idx = top_k_routing(rng, T, E, K).reshape(-1)
    x = _normal_bf16(rng, (T, k_in))
    base = _normal_bf16(rng, (T * K, n_out))
    experts = _experts(rng, range(E), k_in, r, n_out)
    return Workload("decode_down", "gather", k_in, r, n_out, K, T, x, base, experts, E,
                    indices=idx, adapter_slots=np.zeros(T, np.int32), padded_n=T, active=0)


def decode_gate_up(seed: int = 3) -> Workload:
    rng = np.random.default_rng(seed)
    T, K, E, k_in, n_out, r = 256, 8, 128, 2048, 768, 64
    idx = top_k_routing(rng, T, E, K).reshape(-1)
    adapted = np.sort(rng.choice(E, size=E // 2, replace=False))
    slots = np.array([0] * 154 + [-1] * 64, np.int32)
    rng.shuffle(slots)  # 218 real requests; entries 218..255 are padding
    x = _normal_bf16(rng, (T, k_in))
    base = _normal_bf16(rng, (T * K, n_out))
    experts = _experts(rng, adapted, k_in, r, n_out)
    return Workload("decode_gate_up", "gather", k_in, r, n_out, K, T, x, base, experts, E,
                    indices=idx, adapter_slots=slots, padded_n=T, active=0)


def _prefill(name, rng, lengths, K, E, k_in, n_out, r, cap, adapted=None) -> Workload:
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    flat = top_k_routing(rng, T, E, K, bias_variance=1.5).reshape(-1)
    offsets, src = sort_rows_by_expert(flat, E)
    x = _normal_bf16(rng, (T, k_in))
    base = _normal_bf16(rng, (T * K, n_out))
    experts = _experts(rng, range(E) if adapted is None else adapted, k_in, r, n_out)
    return Workload(name, "grouped", k_in, r, n_out, K, T, x, base, experts, E,
                    expert_offsets=offsets, src=src, cu_seqlens=cu,
                    stream_slots=np.zeros(len(lengths), np.int32), cap=cap, active=0)


def prefill_down(seed: int = 2) -> Workload:
    rng = np.random.default_rng(seed)
    lengths = rng.integers(256, 769, size=8)
    return _prefill("prefill_down", rng, lengths, 8, 128, 768, 2048, 16, 8192)


def prefill_down_xrows(seed: int = 2) -> Workload:
    w = prefill_down(seed)
    rng = np.random.default_rng(seed + 5000)
    w.name = "prefill_down_xrows"
    w.x_rows = _normal_bf16(rng, (w.rows, w.k_in))
    return w


def add_expert_weights(w: Workload, seed: int) -> Workload:
    """Give a per-row x prefill workload the stacked expert GEMM weights,
    W_e ~ N(0, 1/k_in), [n_experts_model, n_out, k_in]."""
    rng = np.random.default_rng(seed)
    w.weights = _normal_bf16(rng, (w.n_experts_model, w.n_out, w.k_in), 1.0 / w.k_in)
    return w


def prefill_down_fused(seed: int = 2) -> Workload:
    """prefill_down_xrows with every expert's down-projection weight: the
    expert GEMM and the fold in one pass."""
    w = prefill_down_xrows(seed)
    w.name = "prefill_down_fused"
    return add_expert_weights(w, seed + 7000)


def prefill_large(seed: int = 4) -> Workload:
    rng = np.random.default_rng(seed)
    return _prefill("prefill_large", rng, np.array([16384]), 10, 512, 512, 2048, 32, 32768)


def prefill_large_fused(seed: int = 4) -> Workload:
    """The large prefill as the expert GEMM with the fold in its epilogue: a
    per-row input x_rows [163840, 512] and the 512 experts' stacked weights
    W [512, 2048, 512]."""
    w = prefill_large(seed)
    rng = np.random.default_rng(seed + 5000)
    w.name = "prefill_large_fused"
    w.x_rows = _normal_bf16(rng, (w.rows, w.k_in))
    return add_expert_weights(w, seed + 7000)


def router(seed: int = 4) -> Workload:
    rng = np.random.default_rng(seed + 1000)
    T, k_in, n_out, r = 16384, 2048, 512, 32
    x = _normal_bf16(rng, (T, k_in))
    base = _normal_bf16(rng, (T, n_out))
    experts = _experts(rng, [0], k_in, r, n_out)
    return Workload("router", "router", k_in, r, n_out, 1, T, x, base, experts, 1)


def custom_gather(seed: int, n_tokens: int, top_k: int, n_experts: int, k_in: int, n_out: int,
                  max_rank: int, adapted_frac: float = 1.0, base_frac: float = 0.0,
                  pad: int = 0, rank: Optional[int] = None, bad_ids: int = 0) -> Workload:
    """A decode batch of arbitrary shape (for parity sweeps and edge cases)."""
    rng = np.random.default_rng(seed)
    idx = top_k_routing(rng, n_tokens, n_experts, top_k).reshape(-1)
    for _ in range(bad_ids):  # ids past the table, or negative
        idx[int(rng.integers(0, idx.size))] = int(rng.choice([n_experts + 3, -1, 1 << 30]))
    n_adapt = max(1, int(round(adapted_frac * n_experts)))
    adapted = np.sort(rng.choice(n_experts, size=n_adapt, replace=False))
    real = max(0, n_tokens - pad)
    slots = np.where(rng.random(real) < base_frac, -1, 0).astype(np.int32)
    x = _normal_bf16(rng, (n_tokens, k_in))
    base = _normal_bf16(rng, (n_tokens * top_k, n_out))
    experts = _experts(rng, adapted, k_in, max_rank, n_out, rank)
    return Workload(f"gather_{n_tokens}x{top_k}_{k_in}_{n_out}_r{max_rank}", "gather", k_in,
                    max_rank, n_out, top_k, n_tokens, x, base, experts, n_experts,
                    indices=idx, adapter_slots=slots, padded_n=n_tokens, active=0)


def custom_gather_multi(seed: int, n_tokens: int, top_k: int, n_experts: int, k_in: int,
                        n_out: int, max_rank: int, n_adapters: int, adapted_frac: float = 1.0,
                        base_frac: float = 0.0, pad: int = 0, bad_ids: int = 0) -> Workload:
    """A decode batch over several adapters at once: request slots are drawn
    over [0, n_adapters) (base requests -1), each adapter adapts its own
    subset of experts, and the expert pairs are keyed by cell
    slot * n_experts + expert."""
    rng = np.random.default_rng(seed)
    idx = top_k_routing(rng, n_tokens, n_experts, top_k).reshape(-1)
    for _ in range(bad_ids):
        idx[int(rng.integers(0, idx.size))] = int(rng.choice([n_experts + 3, -1, 1 << 30]))
    n_adapt = max(1, int(round(adapted_frac * n_experts)))
    cells = []
    for s in range(n_adapters):
        adapted = np.sort(rng.choice(n_experts, size=n_adapt, replace=False))
        cells += [s * n_experts + int(e) for e in adapted]
    real = max(0, n_tokens - pad)
    slots = rng.integers(0, n_adapters, real).astype(np.int32)
    slots[rng.random(real) < base_frac] = -1
    x = _normal_bf16(rng, (n_tokens, k_in))
    base = _normal_bf16(rng, (n_tokens * top_k, n_out))
    experts = _experts(rng, cells, k_in, max_rank, n_out)
    return Workload(f"gather_multi{n_adapters}_{n_tokens}x{top_k}_{k_in}_{n_out}_r{max_rank}",
                    "gather", k_in, max_rank, n_out, top_k, n_tokens, x, base, experts, n_experts,
                    indices=idx, adapter_slots=slots, padded_n=n_tokens, active=0,
                    n_adapters=n_adapters)


def decode_down_multi(seed: int = 6) -> Workload:
    w = custom_gather_multi(seed, 64, 8, 128, 768, 2048, 16, 4)
    w.name = "decode_down_multi"
    return w


def custom_grouped(seed: int, lengths, top_k: int, n_experts: int, k_in: int, n_out: int,
                   max_rank: int, cap: int, adapted_frac: float = 1.0,
                   stream_base: Optional[List[int]] = None,
                   rank: Optional[int] = None, per_row_x: bool = False,
                   gemm_weights: bool = False) -> Workload:
    """A packed prefill batch of arbitrary shape (for parity sweeps and edge cases)."""
    rng = np.random.default_rng(seed)
    n_adapt = max(1, int(round(adapted_frac * n_experts)))
    adapted = np.sort(rng.choice(n_experts, size=n_adapt, replace=False))
    lengths = np.asarray(lengths, np.int64)
    w = _prefill(f"grouped_{int(lengths.sum())}x{top_k}_{k_in}_{n_out}_r{max_rank}", rng,
                 lengths, top_k, n_experts, k_in, n_out, max_rank, cap, adapted)
    if rank is not None and rank < max_rank:
        for e in w.experts:
            e.A[rank:] = 0
            e.B[:, rank:] = 0
    if stream_base is not None:
        w.stream_slots = np.array([-1 if b else 0 for b in stream_base], np.int32)
    if per_row_x:
        w.x_rows = _normal_bf16(rng, (w.rows, k_in))
    if gemm_weights:
        add_expert_weights(w, seed + 7000)
    return w


def custom_router(seed: int, n_tokens: int, k_in: int, n_out: int, max_rank: int) -> Workload:
    rng = np.random.default_rng(seed)
    x = _normal_bf16(rng, (n_tokens, k_in))
    base = _normal_bf16(rng, (n_tokens, n_out))
    experts = _experts(rng, [0], k_in, max_rank, n_out)
    return Workload(f"router_{n_tokens}_{k_in}_{n_out}_r{max_rank}", "router", k_in, max_rank,
                    n_out, 1, n_tokens, x, base, experts, 1)


NAMED = {
    "tiny_decode": tiny_decode,
    "decode_down": decode_down,
    "prefill_down": prefill_down,
    "prefill_down_xrows": prefill_down_xrows,
    "decode_gate_up": decode_gate_up,
    "decode_down_multi": decode_down_multi,
    "prefill_large": prefill_large,
    "router": router,
    "prefill_down_fused": prefill_down_fused,
    "prefill_large_fused": prefill_large_fused,
}
