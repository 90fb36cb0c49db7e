"""Oracle side of the parity tests and the comparison rules.

Comparison rules (the fold's contract):
  * a folded bf16 element passes when |out - ref| <= 4e-3 * max(1, |ref|),
    ref being the unrounded fp64 oracle value;
  * an element that must not fold keeps its input bits exactly (-0.0 too);
  * guard rows around base_out keep their sentinel bits.
The 4e-3 bound: the output is one round-to-nearest-even to bf16 (half an ulp,
2^-9 relative = 1.95e-3 of |ref| at most, 3.9e-3 absolute just below 2), so
the fp32 arithmetic before the rounding may add up to ~9e-5 at |ref| ~ 1.

That bound alone cannot tell a good pre-rounding value from a poor one: the
final rounding's half ulp dominates it.  So every check also compares each
folded element with RNE_bf16(ref), the correctly rounded exact value.  An
element may differ from it only when ref lies within RNE_BAND * max(1, |ref|)
of a rounding boundary (the midpoint between two adjacent bf16 values): an
fp32 result a little off the exact value can fall on the other side of such
a midpoint, nothing else can.  With h carried in fp32 (or as bf16 hi + lo,
~2^-18 relative) the pre-rounding error of these workloads is ~1e-5 or less;
h rounded to bf16 would err by ~2^-9 * |delta| (~1e-3), far outside the band.
"""
from __future__ import annotations

import numpy as np

import oracle
from lora_moe_expert_gb300 import synth

TOL = 4e-3
RNE_BAND = 2.0 ** -14


def rne_bf16_f64(ref: np.ndarray) -> np.ndarray:
    """bf16 bits of fp64 values rounded to nearest-even, and each value's
    distance to the nearest bf16 rounding boundary (midpoint).  The fp64 ->
    fp32 step can only move a value onto a midpoint from within one fp32 ulp
    of it, and such values lie inside any band the checks use."""
    ref = np.asarray(ref, np.float64)
    f32 = ref.astype(np.float32)
    bits = synth.bf16_bits(f32)
    u = f32.view(np.uint32)
    lo = (u & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    hi = ((u & np.uint32(0xFFFF0000)) + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    mid = 0.5 * (lo + hi)
    return bits, np.abs(ref - mid)


def weight_table(w, n_table):
    """Host table of the host addresses of each expert's slice of the stacked
    w.weights (0 past them), and the array it points into (keep it alive
    while the oracle runs)."""
    keep = np.ascontiguousarray(w.weights, np.uint16)
    table = np.zeros(n_table, np.uint64)
    step = keep.shape[1] * keep.shape[2] * 2
    for e in range(min(n_table, keep.shape[0])):
        table[e] = keep.ctypes.data + e * step
    return table, keep


def oracle_reference(w, o=None, row_offset=None, row_end=None):
    """(ref fp64, folded bool, keepalive) for the whole workload.  For the
    expert GEMM with the fold (w.weights set) the mask marks the rows the
    call writes (the GEMM rows, folded or not); every other row keeps its
    bits."""
    o = o or oracle.get()
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    if w.n_adapters:
        at, bt, st = he.tables(o, length=w.n_adapters * w.n_experts_model)
        status, ra = o.build_moe_row_adapter_decode_multi(w.adapter_slots, w.padded_n,
                                                          w.n_adapters, w.has_moe_lora)
        assert status == 0, status
        ref, folded = o.gather_fold_multi(w.x, w.indices, ra, at, bt, st, w.base, w.k_in,
                                          w.max_rank, w.n_out, w.top_k, w.n_experts_model,
                                          w.n_adapters)
        return ref, folded, (he, at.size)
    if w.weights is not None:  # the expert GEMM with the fold in its epilogue
        n_table = w.n_experts_model
        at, bt, st = he.tables(o, length=n_table)
        wt, keep_w = weight_table(w, n_table)
        ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
        lo = 0 if row_offset is None else row_offset
        hi = w.rows if row_end is None else row_end
        ref, written, _ = o.grouped_gemm_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra, wt,
                                                    at, bt, st, w.base, w.k_in, w.max_rank,
                                                    w.n_out, w.top_k, lo, hi)
        return ref, written, (he, at.size, keep_w)
    at, bt, st = he.tables(o)
    if w.kind == "gather":
        ra = o.build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, w.active,
                                            w.has_moe_lora)
        ref, folded = o.gather_fold(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank,
                                    w.n_out, w.top_k)
    elif w.kind == "grouped":
        ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
        lo = 0 if row_offset is None else row_offset
        hi = w.rows if row_end is None else row_end
        if w.x_rows is not None:
            ref, folded = o.grouped_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra, at, bt, st,
                                               w.base, w.k_in, w.max_rank, w.n_out, w.top_k, lo,
                                               hi)
        else:
            ref, folded = o.grouped_fold(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base,
                                         w.k_in, w.max_rank, w.n_out, w.top_k, lo, hi)
    else:
        ref, folded = o.router_fold(w.x, None, at, bt, st, w.base, w.k_in, w.max_rank, w.n_out)
    return ref, folded, (he, at.size)


def check_fold(out_bits: np.ndarray, base_bits: np.ndarray, ref: np.ndarray,
               folded: np.ndarray, tol: float = TOL, band: float = RNE_BAND) -> dict:
    """Assert the comparison rules; returns error statistics (rne_mismatch: folded
    elements whose bits differ from RNE_bf16(ref), each within the band of a
    rounding boundary)."""
    out_bits = np.asarray(out_bits, np.uint16)
    base_bits = np.asarray(base_bits, np.uint16)
    assert out_bits.shape == ref.shape == base_bits.shape
    keep = ~folded
    if keep.any():
        diff = out_bits[keep] != base_bits[keep]
        assert not diff.any(), f"{int(diff.sum())} elements of unfolded rows changed"
    stats = {"rows": int(folded.size), "folded_rows": int(folded.sum()), "max_err": 0.0,
             "max_rel": 0.0}
    if folded.any():
        out = synth.bf16_to_f32(out_bits[folded]).astype(np.float64)
        r = ref[folded]
        err = np.abs(out - r)
        bound = tol * np.maximum(1.0, np.abs(r))
        worst = np.argmax(err - bound)
        assert np.all(err <= bound), (
            f"{int((err > bound).sum())} folded elements out of tolerance; worst "
            f"out={out.flat[worst]!r} ref={r.flat[worst]!r}")
        stats["max_err"] = float(err.max())
        stats["max_rel"] = float((err / bound).max())
        rne, mid_dist = rne_bf16_f64(r)
        miss = out_bits[folded] != rne
        near = mid_dist <= band * np.maximum(1.0, np.abs(r))
        far = miss & ~near
        assert not far.any(), (
            f"{int(far.sum())} folded elements differ from RNE_bf16(ref) away from a rounding "
            f"boundary; first ref={r[far][0]!r} out={out[far][0]!r}")
        stats["rne_mismatch"] = int(miss.sum())
        stats["rne_mismatch_max_dist"] = float(
            (mid_dist[miss] / np.maximum(1.0, np.abs(r[miss]))).max()) if miss.any() else 0.0
    return stats
