"""fp64 CPU oracle for the MoE expert LoRA fold -- TEST INFRASTRUCTURE ONLY.

This package is the checker the CUDA path is compared against.  Only the
test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import it; the product package ``lora_moe_expert_gb300``
never imports, links or calls it, and the two share no source.

The arithmetic lives in ``mlg_oracle.c`` (plain C, fp64, compiled with gcc);
this module only marshals numpy arrays through ctypes.  Each wrapper names the
documentation item it follows:

* moe_row_adapter.rs -- ``resolve_moe_lora_route``,
  ``ensure_decode_route_servable``, ``build_moe_row_adapter_host``,
  ``build_moe_row_adapter_decode``;
* moe_lora_grouped module index -- the zero-cell / out-of-range invariant,
  ``pack_expert_tables``, ``grouped_down_windows``, ``grouped_down_wc``,
  ``gather_row_token``, ``moe_lora_gather_bgmv``, ``moe_lora_grouped_down``,
  and ``MoeExpertRoute`` (the router fold as a one-entry route).

Parity status: the host rules are pinned by page-derived fixtures and
invariants; the fold is pinned by closed forms (rank-1 unit vectors, exact
small-integer cases), a library-matmul special case, and invariants
(skips, linearity, cross-form and window equivalence).  The pages print no
worked numeric example of the fold.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mlg_oracle.c")
LIBRARY = os.path.join(_HERE, "libmlg_oracle.so")

ROUTE_FOLD, ROUTE_SKIP, ROUTE_REFUSE = 0, 1, 2
OK, NONE, EMPTY, CAP_ZERO, REFUSE, TOO_SMALL = 0, -1, -2, -3, -4, -6


def build(source: str = SOURCE, library: str = LIBRARY, extra_flags: Sequence[str] = ()) -> str:
    """Compile the oracle with gcc (plain -O2: no fast-math, so no reassociation).

    -fopenmp lets the row loops run on several threads (oracle_set_threads);
    each row is still computed by one thread in the serial order, so the
    results do not depend on the thread count."""
    if (
        os.path.exists(library)
        and source == SOURCE
        and not extra_flags
        and os.path.getmtime(library) >= os.path.getmtime(source)
    ):
        return library
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fopenmp", *extra_flags, "-o", library,
           source]
    subprocess.run(cmd, check=True)
    return library


_p = ctypes.c_void_p
_i32, _i64, _u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a test build)."""

    def __init__(self, library: Optional[str] = None):
        self.lib = ctypes.CDLL(library or build())
        L = self.lib
        L.oracle_set_threads.argtypes = [_i32]
        L.oracle_set_threads.restype = _i32
        L.oracle_resolve_moe_lora_route.argtypes = [_i32, _i32, _i32]
        L.oracle_resolve_moe_lora_route.restype = _i32
        L.oracle_ensure_decode_route_servable.argtypes = [_i32]
        L.oracle_ensure_decode_route_servable.restype = _i32
        L.oracle_build_moe_row_adapter_decode.argtypes = [_p, _i64, _i64, _i32, _i32, _p]
        L.oracle_build_moe_row_adapter_decode.restype = None
        L.oracle_build_moe_row_adapter_decode_multi.argtypes = [_p, _i64, _i64, _i32, _i32, _p]
        L.oracle_build_moe_row_adapter_decode_multi.restype = _i32
        L.oracle_gather_fold_multi.argtypes = [_p] * 9 + [_i32] * 7
        L.oracle_gather_fold_multi.restype = _i32
        L.oracle_build_moe_row_adapter_host.argtypes = [_p, _i64, _p, _i64, _p, _i64, _p]
        L.oracle_build_moe_row_adapter_host.restype = _i32
        L.oracle_pack_expert_tables.argtypes = [_p, _p, _p, _p, _i64, _p, _p, _p, _i64, _p]
        L.oracle_pack_expert_tables.restype = _i32
        L.oracle_grouped_down_windows.argtypes = [_u32, _u32, _p, _p, _i64]
        L.oracle_grouped_down_windows.restype = _i64
        L.oracle_grouped_down_wc.argtypes = [_u32, _u32, _u32]
        L.oracle_grouped_down_wc.restype = _u32
        L.oracle_gather_row_token.argtypes = [_u32, _u32]
        L.oracle_gather_row_token.restype = _u32
        L.oracle_gather_fold.argtypes = [_p] * 9 + [_i32] * 6
        L.oracle_gather_fold.restype = _i32
        L.oracle_grouped_fold.argtypes = [_p] * 10 + [_i64] + [_i32] * 7
        L.oracle_grouped_fold.restype = _i32
        L.oracle_grouped_fold_xrows.argtypes = [_p] * 10 + [_i64] + [_i32] * 7
        L.oracle_grouped_fold_xrows.restype = _i32
        L.oracle_grouped_fold_xrows_rows.argtypes = [_p] * 9 + [_i32, _p, _p] + [_i32] * 7
        L.oracle_grouped_fold_xrows_rows.restype = _i32
        L.oracle_router_fold.argtypes = [_p] * 8 + [_i32] * 4
        L.oracle_router_fold.restype = _i32
        L.oracle_gather_fold_rows.argtypes = [_p] * 8 + [_i32, _p, _p] + [_i32] * 5
        L.oracle_gather_fold_rows.restype = _i32
        L.oracle_grouped_fold_rows.argtypes = [_p] * 9 + [_i32, _p, _p] + [_i32] * 7
        L.oracle_grouped_fold_rows.restype = _i32
        L.oracle_grouped_gemm_fold_xrows.argtypes = [_p] * 12 + [_i64] + [_i32] * 7
        L.oracle_grouped_gemm_fold_xrows.restype = _i32
        L.oracle_grouped_gemm_fold_xrows_rows.argtypes = [_p] * 10 + [_i32, _p, _p, _p] + [_i32] * 7
        L.oracle_grouped_gemm_fold_xrows_rows.restype = _i32

    def set_threads(self, n: int) -> int:
        """Threads of the row loops (n < 1: every core); returns the count in force
        (1 for a build without OpenMP).  Results are the same bits for any count."""
        return int(self.lib.oracle_set_threads(n))

    # ---- host rules -------------------------------------------------------
    def resolve_moe_lora_route(self, adapter_slot: int, active: int, has_moe_lora: bool) -> int:
        return self.lib.oracle_resolve_moe_lora_route(adapter_slot, active, int(bool(has_moe_lora)))

    def ensure_decode_route_servable(self, route: int) -> int:
        return self.lib.oracle_ensure_decode_route_servable(route)

    def build_moe_row_adapter_decode(self, adapter_slots, padded_n: int, active: int,
                                     has_moe_lora: bool) -> np.ndarray:
        slots = np.ascontiguousarray(adapter_slots, dtype=np.int32)
        out = np.empty(padded_n, dtype=np.int32)
        self.lib.oracle_build_moe_row_adapter_decode(
            _ptr(slots), slots.size, padded_n, active, int(bool(has_moe_lora)), _ptr(out))
        return out

    def build_moe_row_adapter_decode_multi(self, adapter_slots, padded_n: int, n_adapters: int,
                                           has_moe_lora: bool):
        """(status, map): the multi-adapter decode map, or REFUSE with nothing written."""
        slots = np.ascontiguousarray(adapter_slots, dtype=np.int32)
        out = np.full(padded_n, 0x5A5A5A5A, dtype=np.int32)
        st = self.lib.oracle_build_moe_row_adapter_decode_multi(
            _ptr(slots), slots.size, padded_n, n_adapters, int(bool(has_moe_lora)), _ptr(out))
        return st, out

    def build_moe_row_adapter_host(self, cu_seqlens, adapter_slots) -> Optional[np.ndarray]:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        slots = np.ascontiguousarray(adapter_slots, dtype=np.int32)
        total = ctypes.c_int64(0)
        st = self.lib.oracle_build_moe_row_adapter_host(
            _ptr(cu), cu.size, _ptr(slots), slots.size, None, 0, ctypes.byref(total))
        if st == NONE:
            return None
        out = np.empty(max(total.value, 0), dtype=np.int32)
        st = self.lib.oracle_build_moe_row_adapter_host(
            _ptr(cu), cu.size, _ptr(slots), slots.size, _ptr(out), out.size, ctypes.byref(total))
        assert st == OK, st
        return out

    def pack_expert_tables(self, ids, a_addr, b_addr, scale):
        """Returns (a_table u64, b_table u64, scale_table f32) or None for empty input."""
        ids = np.ascontiguousarray(ids, dtype=np.uint32)
        a = np.ascontiguousarray(a_addr, dtype=np.uint64)
        b = np.ascontiguousarray(b_addr, dtype=np.uint64)
        s = np.ascontiguousarray(scale, dtype=np.float32)
        n_exp = ctypes.c_int64(0)
        st = self.lib.oracle_pack_expert_tables(_ptr(ids), _ptr(a), _ptr(b), _ptr(s), ids.size,
                                                None, None, None, 0, ctypes.byref(n_exp))
        if st == EMPTY:
            return None
        E = n_exp.value
        at, bt, stab = np.empty(E, np.uint64), np.empty(E, np.uint64), np.empty(E, np.float32)
        st = self.lib.oracle_pack_expert_tables(_ptr(ids), _ptr(a), _ptr(b), _ptr(s), ids.size,
                                                _ptr(at), _ptr(bt), _ptr(stab), E,
                                                ctypes.byref(n_exp))
        assert st == OK, st
        return at, bt, stab

    def grouped_down_windows(self, total_rows: int, cap: int):
        """List of (start, end); raises ValueError on cap == 0 (the pages' panic)."""
        n = self.lib.oracle_grouped_down_windows(total_rows, cap, None, None, 0)
        if n == CAP_ZERO:
            raise ValueError("grouped_down_windows: cap == 0")
        starts, ends = np.empty(n, np.uint32), np.empty(n, np.uint32)
        n2 = self.lib.oracle_grouped_down_windows(total_rows, cap, _ptr(starts), _ptr(ends), n)
        assert n2 == n
        return [(int(s), int(e)) for s, e in zip(starts, ends)]

    def grouped_down_wc(self, row_offset: int, row_end: int, m_tile: int) -> int:
        return self.lib.oracle_grouped_down_wc(row_offset, row_end, m_tile)

    def gather_row_token(self, row: int, top_k: int) -> int:
        return self.lib.oracle_gather_row_token(row, top_k)

    # ---- folds -------------------------------------------------------------
    @staticmethod
    def _u16(a):
        a = np.ascontiguousarray(a)
        assert a.dtype == np.uint16, a.dtype
        return a

    def gather_fold(self, x, indices, row_adapter, a_table, b_table, scale_table, base,
                    k_in, max_rank, n_out, top_k):
        """Returns (ref fp64 [n_slots, n_out], folded bool [n_slots])."""
        x, base = self._u16(x), self._u16(base)
        idx = np.ascontiguousarray(indices, np.int32)
        ra = np.ascontiguousarray(row_adapter, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        n_slots = idx.size
        ref = np.empty((n_slots, n_out), np.float64)
        folded = np.empty(n_slots, np.uint8)
        st = self.lib.oracle_gather_fold(_ptr(x), _ptr(idx), _ptr(ra), _ptr(at), _ptr(bt),
                                         _ptr(st_), _ptr(base), _ptr(ref), _ptr(folded), n_slots,
                                         k_in, max_rank, n_out, top_k, at.size)
        assert st == OK, st
        return ref, folded.astype(bool)

    def grouped_fold(self, x, expert_offsets, src, row_adapter, a_table, b_table, scale_table,
                     base, k_in, max_rank, n_out, top_k, row_offset, row_end):
        """Returns (ref fp64 [total_rows, n_out], folded bool [total_rows])."""
        x, base = self._u16(x), self._u16(base)
        off = np.ascontiguousarray(expert_offsets, np.int32)
        src = np.ascontiguousarray(src, np.int32)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        total = base.shape[0]
        ref = np.empty((total, n_out), np.float64)
        folded = np.empty(total, np.uint8)
        st = self.lib.oracle_grouped_fold(_ptr(x), _ptr(off), _ptr(src), _ptr(ra), _ptr(at),
                                          _ptr(bt), _ptr(st_), _ptr(base), _ptr(ref),
                                          _ptr(folded), total, k_in, max_rank, n_out, top_k,
                                          at.size, row_offset, row_end)
        assert st == OK, st
        return ref, folded.astype(bool)

    def gather_fold_multi(self, x, indices, row_adapter, a_table, b_table, scale_table, base,
                          k_in, max_rank, n_out, top_k, n_experts, n_adapters):
        """Multi-adapter gather fold over slot-major tables of n_adapters * n_experts cells."""
        x, base = self._u16(x), self._u16(base)
        idx = np.ascontiguousarray(indices, np.int32)
        ra = np.ascontiguousarray(row_adapter, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        assert at.size == bt.size == st_.size == n_experts * n_adapters
        n = idx.size
        ref = np.empty((n, n_out), np.float64)
        folded = np.empty(n, np.uint8)
        st = self.lib.oracle_gather_fold_multi(_ptr(x), _ptr(idx), _ptr(ra), _ptr(at), _ptr(bt),
                                               _ptr(st_), _ptr(base), _ptr(ref), _ptr(folded), n,
                                               k_in, max_rank, n_out, top_k, n_experts, n_adapters)
        assert st == OK, st
        return ref, folded.astype(bool)

    def grouped_fold_xrows(self, x_rows, expert_offsets, src, row_adapter, a_table, b_table,
                           scale_table, base, k_in, max_rank, n_out, top_k, row_offset, row_end):
        """Per-row x variant: sorted row r takes x_rows[r]."""
        x, base = self._u16(x_rows), self._u16(base)
        off = np.ascontiguousarray(expert_offsets, np.int32)
        src = np.ascontiguousarray(src, np.int32)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        total = base.shape[0]
        ref = np.empty((total, n_out), np.float64)
        folded = np.empty(total, np.uint8)
        st = self.lib.oracle_grouped_fold_xrows(_ptr(x), _ptr(off), _ptr(src), _ptr(ra), _ptr(at),
                                                _ptr(bt), _ptr(st_), _ptr(base), _ptr(ref),
                                                _ptr(folded), total, k_in, max_rank, n_out, top_k,
                                                at.size, row_offset, row_end)
        assert st == OK, st
        return ref, folded.astype(bool)

    def grouped_gemm_fold_xrows(self, x_rows, expert_offsets, src, row_adapter, w_table,
                                a_table, b_table, scale_table, out_in, k_in, max_rank, n_out,
                                top_k, row_offset, row_end):
        """Expert GEMM with the per-row x fold in its epilogue.  Returns
        (ref fp64 [total_rows, n_out], written bool, folded bool); rows not
        written keep out_in."""
        x, out_in = self._u16(x_rows), self._u16(out_in)
        off = np.ascontiguousarray(expert_offsets, np.int32)
        src = np.ascontiguousarray(src, np.int32)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        wt = np.ascontiguousarray(w_table, np.uint64)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        assert wt.size == at.size == bt.size == st_.size
        total = out_in.shape[0]
        ref = np.empty((total, n_out), np.float64)
        written = np.empty(total, np.uint8)
        folded = np.empty(total, np.uint8)
        st = self.lib.oracle_grouped_gemm_fold_xrows(
            _ptr(x), _ptr(off), _ptr(src), _ptr(ra), _ptr(wt), _ptr(at), _ptr(bt), _ptr(st_),
            _ptr(out_in), _ptr(ref), _ptr(written), _ptr(folded), total, k_in, max_rank, n_out,
            top_k, at.size, row_offset, row_end)
        assert st == OK, st
        return ref, written.astype(bool), folded.astype(bool)

    def grouped_gemm_fold_xrows_rows(self, x_rows, expert_offsets, src, row_adapter, w_table,
                                     a_table, b_table, scale_table, prior_rows, rows, k_in,
                                     max_rank, n_out, top_k, row_offset, row_end):
        """The listed sorted rows of the expert GEMM with the fold; prior_rows
        [len(rows), n_out] are their values before the call.  Returns (ref,
        written, folded) for those rows."""
        x, prior = self._u16(x_rows), self._u16(prior_rows)
        off = np.ascontiguousarray(expert_offsets, np.int32)
        src = np.ascontiguousarray(src, np.int32)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        wt = np.ascontiguousarray(w_table, np.uint64)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        rows = np.ascontiguousarray(rows, np.int32)
        ref = np.empty((rows.size, n_out), np.float64)
        written = np.empty(rows.size, np.uint8)
        folded = np.empty(rows.size, np.uint8)
        st = self.lib.oracle_grouped_gemm_fold_xrows_rows(
            _ptr(x), _ptr(off), _ptr(src), _ptr(ra), _ptr(wt), _ptr(at), _ptr(bt), _ptr(st_),
            _ptr(prior), _ptr(rows), rows.size, _ptr(ref), _ptr(written), _ptr(folded), k_in,
            max_rank, n_out, top_k, at.size, row_offset, row_end)
        assert st == OK, st
        return ref, written.astype(bool), folded.astype(bool)

    def router_fold(self, x, row_adapter, a_table, b_table, scale_table, base, k_in, max_rank,
                    n_out):
        x, base = self._u16(x), self._u16(base)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        T = base.shape[0]
        ref = np.empty((T, n_out), np.float64)
        folded = np.empty(T, np.uint8)
        st = self.lib.oracle_router_fold(_ptr(x), _ptr(ra), _ptr(at), _ptr(bt), _ptr(st_),
                                         _ptr(base), _ptr(ref), _ptr(folded), T, k_in, max_rank,
                                         n_out)
        assert st == OK, st
        return ref, folded.astype(bool)

    def gather_fold_rows(self, x, indices, row_adapter, a_table, b_table, scale_table,
                         base_rows, rows, k_in, max_rank, n_out, top_k):
        """Fold only `rows` (flat rows); base_rows [len(rows), n_out] are their inputs."""
        x, base_rows = self._u16(x), self._u16(base_rows)
        idx = np.ascontiguousarray(indices, np.int32)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        rows = np.ascontiguousarray(rows, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        ref = np.empty((rows.size, n_out), np.float64)
        folded = np.empty(rows.size, np.uint8)
        st = self.lib.oracle_gather_fold_rows(_ptr(x), _ptr(idx), _ptr(ra), _ptr(at), _ptr(bt),
                                              _ptr(st_), _ptr(base_rows), _ptr(rows), rows.size,
                                              _ptr(ref), _ptr(folded), k_in, max_rank, n_out,
                                              top_k, at.size)
        assert st == OK, st
        return ref, folded.astype(bool)

    def grouped_fold_rows(self, x, expert_offsets, src, row_adapter, a_table, b_table,
                          scale_table, base_rows, rows, k_in, max_rank, n_out, top_k,
                          row_offset, row_end):
        x, base_rows = self._u16(x), self._u16(base_rows)
        off = np.ascontiguousarray(expert_offsets, np.int32)
        src = np.ascontiguousarray(src, np.int32)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        rows = np.ascontiguousarray(rows, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        ref = np.empty((rows.size, n_out), np.float64)
        folded = np.empty(rows.size, np.uint8)
        st = self.lib.oracle_grouped_fold_rows(_ptr(x), _ptr(off), _ptr(src), _ptr(ra), _ptr(at),
                                               _ptr(bt), _ptr(st_), _ptr(base_rows), _ptr(rows),
                                               rows.size, _ptr(ref), _ptr(folded), k_in,
                                               max_rank, n_out, top_k, at.size, row_offset,
                                               row_end)
        assert st == OK, st
        return ref, folded.astype(bool)

    def grouped_fold_xrows_rows(self, x_rows, expert_offsets, src, row_adapter, a_table,
                                b_table, scale_table, base_rows, rows, k_in, max_rank, n_out,
                                top_k, row_offset, row_end):
        """Fold only the sorted `rows` of the per-row x form."""
        x, base_rows = self._u16(x_rows), self._u16(base_rows)
        off = np.ascontiguousarray(expert_offsets, np.int32)
        src = np.ascontiguousarray(src, np.int32)
        ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, np.int32)
        rows = np.ascontiguousarray(rows, np.int32)
        at, bt = np.ascontiguousarray(a_table, np.uint64), np.ascontiguousarray(b_table, np.uint64)
        st_ = np.ascontiguousarray(scale_table, np.float32)
        ref = np.empty((rows.size, n_out), np.float64)
        folded = np.empty(rows.size, np.uint8)
        st = self.lib.oracle_grouped_fold_xrows_rows(_ptr(x), _ptr(off), _ptr(src), _ptr(ra),
                                                     _ptr(at), _ptr(bt), _ptr(st_),
                                                     _ptr(base_rows), _ptr(rows), rows.size,
                                                     _ptr(ref), _ptr(folded), k_in, max_rank,
                                                     n_out, top_k, at.size, row_offset, row_end)
        assert st == OK, st
        return ref, folded.astype(bool)


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


class HostExperts:
    """Keeps host copies of expert pairs alive and hands out their addresses.

    The oracle's tables hold host addresses (0 = no adapter), mirroring the
    device tables that hold device addresses.
    """

    def __init__(self, experts):
        # experts: iterable of (expert_id, A bits [r, k_in] u16, B bits [n_out, r] u16, scale)
        self._keep = []
        self.ids, self.a_addr, self.b_addr, self.scale = [], [], [], []
        for eid, A, B, s in experts:
            A = np.ascontiguousarray(A, np.uint16)
            B = np.ascontiguousarray(B, np.uint16)
            self._keep += [A, B]
            self.ids.append(int(eid))
            self.a_addr.append(A.ctypes.data)
            self.b_addr.append(B.ctypes.data)
            self.scale.append(float(s))

    def tables(self, oracle: Optional[Oracle] = None, length: Optional[int] = None):
        """Packed tables; with `length`, padded with empty cells to that many."""
        o = oracle or get()
        at, bt, st = o.pack_expert_tables(self.ids, self.a_addr, self.b_addr, self.scale)
        if length is not None and length > at.size:
            pad = length - at.size
            at = np.concatenate([at, np.zeros(pad, at.dtype)])
            bt = np.concatenate([bt, np.zeros(pad, bt.dtype)])
            st = np.concatenate([st, np.zeros(pad, st.dtype)])
        return at, bt, st
