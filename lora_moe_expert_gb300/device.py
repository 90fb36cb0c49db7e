"""Device-resident fold problems: allocation and upload plumbing around libmlg.

``FoldProblem`` takes a host workload (``synth.Workload``: bf16 bit arrays,
routing, expert pairs) and builds what a caller of the library holds on the
GPU: x, base_out, the routing arrays, one 256-byte-aligned pool for the
expert pairs, the expert tables (packed and uploaded by libmlg) and the row
map (built and uploaded by libmlg).  ``run()`` is the hot path: one call of
the fold entry point (per window for the grouped form).  torch provides
device memory and streams only; no arithmetic of the fold happens here.
"""
from __future__ import annotations

from typing import List, Optional, Tuple

import numpy as np
import torch

import lora_moe_expert_gb300 as mlg

_ALIGN = 256


def _dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def _bits_tensor(a: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bits -> a torch bf16 tensor holding the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).to(device).view(
        torch.bfloat16)


def pad_tables(a, b, s, length: int):
    """Extend packed tables with zero cells to `length` entries."""
    pad = length - a.size
    if pad < 0:
        raise ValueError(f"tables of {a.size} cells exceed {length}")
    return (np.concatenate([a, np.zeros(pad, a.dtype)]), np.concatenate([b, np.zeros(pad, b.dtype)]),
            np.concatenate([s, np.zeros(pad, s.dtype)]))


class ExpertPool:
    """All expert pairs of a workload in one allocation, each 256-byte aligned."""

    def __init__(self, experts, device):
        offs: List[Tuple[int, int, int, int, float]] = []
        pos = 0
        for e in experts:
            a_off = pos
            pos += (e.A.nbytes + _ALIGN - 1) // _ALIGN * _ALIGN
            b_off = pos
            pos += (e.B.nbytes + _ALIGN - 1) // _ALIGN * _ALIGN
            offs.append((e.expert_id, a_off, b_off, e.A.nbytes, e.scale))
        host = np.zeros(max(pos, _ALIGN), np.uint8)
        for e, (_, a_off, b_off, _, _) in zip(experts, offs):
            host[a_off:a_off + e.A.nbytes] = e.A.view(np.uint8).reshape(-1)
            host[b_off:b_off + e.B.nbytes] = e.B.view(np.uint8).reshape(-1)
        self.buffer = _dev(host, device)
        base = self.buffer.data_ptr()
        self.ids = [o[0] for o in offs]
        self.a_addr = [base + o[1] for o in offs]
        self.b_addr = [base + o[2] for o in offs]
        self.scale = [o[4] for o in offs]
        self.nbytes = pos


class FoldProblem:
    def __init__(self, w, device="cuda", stream=None, guard_rows: int = 0,
                 pool: Optional[ExpertPool] = None):
        self.w = w
        self.device = torch.device(device)
        self.stream = stream
        self.pool = pool or ExpertPool(w.experts, self.device)
        a, b, s = mlg.mlg_pack_expert_tables(self.pool.ids, self.pool.a_addr, self.pool.b_addr,
                                             self.pool.scale)
        if w.n_adapters:  # slot-major sets of n_experts_model cells; trailing holes are zero
            a, b, s = pad_tables(a, b, s, w.n_adapters * w.n_experts_model)
        if w.weights is not None:  # one table cell per expert of the stacked weights
            a, b, s = pad_tables(a, b, s, w.n_experts_model)
        self.n_experts = int(a.size)
        self.a_table = torch.empty(self.n_experts, dtype=torch.int64, device=self.device)
        self.b_table = torch.empty(self.n_experts, dtype=torch.int64, device=self.device)
        self.scale_table = torch.empty(self.n_experts, dtype=torch.float32, device=self.device)
        self.tables_host = (a, b, s)
        mlg.mlg_upload_expert_tables(a, b, s, self.a_table, self.b_table, self.scale_table,
                                     stream=self._stream())
        self.x = _bits_tensor(w.x, self.device)
        self.x_rows = None if w.x_rows is None else _bits_tensor(w.x_rows, self.device)
        self.guard_rows = guard_rows
        self.base_full = _bits_tensor(
            np.concatenate([np.full((guard_rows, w.n_out), 0x7FC1, np.uint16), w.base,
                            np.full((guard_rows, w.n_out), 0x7FC1, np.uint16)]), self.device)
        self.base = self.base_full[guard_rows:guard_rows + w.rows]
        self.row_map_host = None
        self.row_adapter = None
        if w.kind == "gather":
            self.indices = _dev(w.indices.astype(np.int32), self.device)
            if w.n_adapters:
                self.row_map_host = mlg.mlg_build_moe_row_adapter_decode_multi(
                    w.adapter_slots, w.padded_n, w.n_adapters, w.has_moe_lora)
            else:
                self.row_map_host = mlg.mlg_build_moe_row_adapter_decode(
                    w.adapter_slots, w.padded_n, w.active, w.has_moe_lora)
        elif w.kind == "grouped":
            self.expert_offsets = _dev(w.expert_offsets.astype(np.int32), self.device)
            self.src = _dev(w.src.astype(np.int32), self.device)
            self.row_map_host = mlg.mlg_build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
            self.windows = mlg.mlg_grouped_down_windows(w.rows, w.cap)
        if self.row_map_host is not None:
            self.row_adapter = torch.empty(self.row_map_host.size, dtype=torch.int32,
                                           device=self.device)
            mlg.mlg_upload_row_adapter(self.row_map_host, self.row_adapter, stream=self._stream())
        self.w_experts = None
        self.zero_table = None
        if w.weights is not None:  # the stacked expert GEMM weights
            if w.weights.shape[0] != self.n_experts:
                raise ValueError("stacked weights must cover every table cell")
            self.w_experts = _bits_tensor(w.weights, self.device)
            self.zero_table = torch.zeros(self.n_experts, dtype=torch.int64, device=self.device)

    def _stream(self):
        return self.stream if self.stream is not None else torch.cuda.current_stream(self.device)

    def run(self, stream=None, use_row_map: bool = True, per_window: bool = False,
            lora: bool = True) -> None:
        """Enqueue the fold (the whole hot path for this problem) on `stream`.

        The grouped form folds all windows of grouped_down_windows(rows, cap)
        in one launch; per_window=True launches mlg_grouped_down once per
        window instead (same bits).  A workload with per-row inputs (x_rows)
        runs the per-row x form over all rows; one with expert GEMM weights runs
        the GEMM with the fold in its epilogue (lora=False: zero LoRA tables,
        the plain grouped expert GEMM)."""
        w = self.w
        s = stream if stream is not None else self._stream()
        if w.kind == "gather" and w.n_adapters:
            mlg.mlg_gather_bgmv_multi(self.x, self.indices, self.row_adapter, self.a_table,
                                      self.b_table, self.scale_table, self.base, w.rows, w.k_in,
                                      w.max_rank, w.n_out, w.top_k, w.n_experts_model,
                                      w.n_adapters, stream=s)
        elif w.kind == "gather":
            mlg.mlg_gather_bgmv(self.x, self.indices, self.row_adapter, self.a_table,
                                self.b_table, self.scale_table, self.base, w.rows, w.k_in,
                                w.max_rank, w.n_out, w.top_k, self.n_experts, stream=s)
        elif w.kind == "grouped" and self.w_experts is not None:
            ra = self.row_adapter if use_row_map else None
            a, b = (self.a_table, self.b_table) if lora else (self.zero_table, self.zero_table)
            mlg.mlg_grouped_gemm_fold_xrows(self.x_rows, self.expert_offsets, self.src, ra,
                                            self.w_experts, a, b, self.scale_table, self.base,
                                            w.k_in, w.max_rank, w.n_out, w.top_k, self.n_experts,
                                            0, w.rows, w.cap, stream=s)
        elif w.kind == "grouped":
            ra = self.row_adapter if use_row_map else None
            if self.x_rows is not None:
                mlg.mlg_grouped_down_xrows(self.x_rows, self.expert_offsets, self.src, ra,
                                           self.a_table, self.b_table, self.scale_table,
                                           self.base, w.k_in, w.max_rank, w.n_out, w.top_k,
                                           self.n_experts, 0, w.rows, w.cap, stream=s)
            elif per_window:
                for start, end in self.windows:
                    mlg.mlg_grouped_down(self.x, self.expert_offsets, self.src, ra,
                                         self.a_table, self.b_table, self.scale_table, self.base,
                                         w.k_in, w.max_rank, w.n_out, w.top_k, self.n_experts,
                                         start, end, stream=s)
            else:
                mlg.mlg_grouped_down_all_windows(self.x, self.expert_offsets, self.src, ra,
                                                 self.a_table, self.b_table, self.scale_table,
                                                 self.base, w.k_in, w.max_rank, w.n_out,
                                                 w.top_k, self.n_experts, w.rows, w.cap,
                                                 stream=s)
        else:
            mlg.mlg_router_fold(self.x, None, self.a_table, self.b_table, self.scale_table,
                                self.base, w.rows, w.k_in, w.max_rank, w.n_out, stream=s)

    def reset(self) -> None:
        """Restore base_out to the workload's input values."""
        self.base.copy_(_bits_tensor(self.w.base, self.device))

    def base_bits(self) -> np.ndarray:
        return self.base.view(torch.int16).cpu().numpy().view(np.uint16)

    def guard_bits(self) -> np.ndarray:
        g = self.guard_rows
        full = self.base_full.view(torch.int16).cpu().numpy().view(np.uint16)
        return np.concatenate([full[:g], full[g + self.w.rows:]])
