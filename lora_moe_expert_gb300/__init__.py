"""Python binding of libmlg, the GB300 (sm_103a) MoE expert LoRA fold.

Argument marshalling only: every call goes straight to the C ABI declared in
``include/mlg.h`` under the same name.  Device arguments may be torch CUDA
tensors (their ``data_ptr()`` is passed) or raw integer addresses; host
arguments are numpy arrays.  A non-OK status raises :class:`MlgError`.

There is no CPU fallback: if ``libmlg.so`` has not been built, :func:`lib`
raises.  Build it with ``python -m lora_moe_expert_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libmlg.so")

MLG_OK = 0
MLG_ERR_INVALID_ARG = -1
MLG_ERR_EMPTY = -2
MLG_ERR_CAP_ZERO = -3
MLG_ERR_REFUSE = -4
MLG_ERR_UNSUPPORTED = -5
MLG_ERR_BUFFER_TOO_SMALL = -6
MLG_ERR_CUDA = -7
MLG_ROUTE_FOLD, MLG_ROUTE_SKIP, MLG_ROUTE_REFUSE = 0, 1, 2
MLG_MAX_RANK = 64
MLG_FOLD_AFTER_PRECEDING = 1
# test and benchmark hooks (include/mlg_test.h; not part of the public interface)
MLG_TEST_GATHER_CLUSTER = 1
MLG_TEST_GROUPED_CTAS = 2
MLG_TEST_GATHER_NSPLIT = 3
MLG_TEST_GATHER_PATH = 4
MLG_TEST_GATHER_SPECULATION = 5


class MlgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = f" (cudaError {mlg_last_cuda_error()})" if status == MLG_ERR_CUDA else ""
        super().__init__(f"{what}: {status_string(status)} ({status}){detail}")


class ExpertEntry(ctypes.Structure):
    _fields_ = [("expert_id", ctypes.c_uint32), ("reserved0", ctypes.c_uint32),
                ("a_addr", ctypes.c_uint64), ("b_addr", ctypes.c_uint64),
                ("scale", ctypes.c_float), ("reserved1", ctypes.c_uint32)]


class Window(ctypes.Structure):
    _fields_ = [("start", ctypes.c_uint32), ("end", ctypes.c_uint32)]


_p, _i32, _u32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
_SIGNATURES = {
    "mlg_gather_bgmv": ([_p] * 7 + [_i32] * 6 + [_p], _i32),
    "mlg_gather_bgmv_ex": ([_p] * 7 + [_i32] * 6 + [_u32, _p], _i32),
    "mlg_gather_bgmv_multi_ex": ([_p] * 7 + [_i32] * 7 + [_u32, _p], _i32),
    "mlg_grouped_down": ([_p] * 8 + [_i32] * 7 + [_p], _i32),
    "mlg_router_fold": ([_p] * 6 + [_i32] * 4 + [_p], _i32),
    "mlg_grouped_down_all_windows": ([_p] * 8 + [_i32] * 6 + [_u32, _p], _i32),
    "mlg_grouped_down_xrows": ([_p] * 8 + [_i32] * 7 + [_u32, _p], _i32),
    "mlg_grouped_gemm_fold_xrows": ([_p] * 9 + [_i32] * 7 + [_u32, _p], _i32),
    "mlg_resolve_moe_lora_route": ([_i32, _i32, _i32], _i32),
    "mlg_ensure_decode_route_servable": ([_i32], _i32),
    "mlg_build_moe_row_adapter_decode": ([_p, _sz, _sz, _i32, _i32, _p], _i32),
    "mlg_build_moe_row_adapter_host": ([_p, _sz, _p, _sz, _p, _sz, _p], _i32),
    "mlg_build_moe_row_adapter_decode_multi": ([_p, _sz, _sz, _i32, _i32, _p], _i32),
    "mlg_gather_bgmv_multi": ([_p] * 7 + [_i32] * 7 + [_p], _i32),
    "mlg_pack_expert_tables": ([_p, _sz, _p, _p, _p, _sz, _p], _i32),
    "mlg_upload_expert_tables": ([_p, _p, _p, _u32, _p, _p, _p, _p], _i32),
    "mlg_upload_row_adapter": ([_p, _sz, _p, _p], _i32),
    "mlg_grouped_down_windows": ([_u32, _u32, _p, _sz, _p], _i32),
    "mlg_grouped_down_wc": ([_u32, _u32], _u32),
    "mlg_gather_row_token": ([_u32, _u32], _u32),
    "mlg_m_tile": ([], _u32),
    "mlg_status_string": ([_i32], ctypes.c_char_p),
    "mlg_last_cuda_error": ([], _i32),
    "mlg_version": ([], _i32),
    "mlg_read_device_errors": ([_p, _i32], _i32),
    "mlg_test_set_knob": ([_i32, _i32], _i32),
}

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded libmlg (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(f"libmlg is not built ({LIBRARY} missing); run "
                               "`python -m lora_moe_expert_gb300.build` -- there is no fallback")
        L = ctypes.CDLL(LIBRARY)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _addr(t) -> Optional[int]:
    """Device address of a torch tensor / raw int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != MLG_OK:
        raise MlgError(status, what)


def _host(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _hp(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- folds
def mlg_gather_bgmv(x, indices, row_adapter, a_table, b_table, scale_table, base_out,
                    n_slots, k_in, max_rank, n_out, top_k, n_experts, stream=None) -> None:
    _check(lib().mlg_gather_bgmv(_addr(x), _addr(indices), _addr(row_adapter), _addr(a_table),
                                 _addr(b_table), _addr(scale_table), _addr(base_out), n_slots,
                                 k_in, max_rank, n_out, top_k, n_experts, _stream(stream)),
           "mlg_gather_bgmv")


def mlg_gather_bgmv_ex(x, indices, row_adapter, a_table, b_table, scale_table, base_out,
                       n_slots, k_in, max_rank, n_out, top_k, n_experts, flags,
                       stream=None) -> None:
    _check(lib().mlg_gather_bgmv_ex(_addr(x), _addr(indices), _addr(row_adapter),
                                    _addr(a_table), _addr(b_table), _addr(scale_table),
                                    _addr(base_out), n_slots, k_in, max_rank, n_out, top_k,
                                    n_experts, flags, _stream(stream)),
           "mlg_gather_bgmv_ex")


def mlg_gather_bgmv_multi_ex(x, indices, row_adapter, a_table, b_table, scale_table, base_out,
                             n_slots, k_in, max_rank, n_out, top_k, n_experts, n_adapters,
                             flags, stream=None) -> None:
    _check(lib().mlg_gather_bgmv_multi_ex(_addr(x), _addr(indices), _addr(row_adapter),
                                          _addr(a_table), _addr(b_table), _addr(scale_table),
                                          _addr(base_out), n_slots, k_in, max_rank, n_out,
                                          top_k, n_experts, n_adapters, flags, _stream(stream)),
           "mlg_gather_bgmv_multi_ex")


def mlg_gather_bgmv_multi(x, indices, row_adapter, a_table, b_table, scale_table, base_out,
                          n_slots, k_in, max_rank, n_out, top_k, n_experts, n_adapters,
                          stream=None) -> None:
    _check(lib().mlg_gather_bgmv_multi(_addr(x), _addr(indices), _addr(row_adapter),
                                       _addr(a_table), _addr(b_table), _addr(scale_table),
                                       _addr(base_out), n_slots, k_in, max_rank, n_out, top_k,
                                       n_experts, n_adapters, _stream(stream)),
           "mlg_gather_bgmv_multi")


def mlg_grouped_down(x, expert_offsets, src, row_adapter, a_table, b_table, scale_table,
                     base_out, k_in, max_rank, n_out, top_k, n_experts, row_offset, row_end,
                     stream=None) -> None:
    _check(lib().mlg_grouped_down(_addr(x), _addr(expert_offsets), _addr(src),
                                  _addr(row_adapter), _addr(a_table), _addr(b_table),
                                  _addr(scale_table), _addr(base_out), k_in, max_rank, n_out,
                                  top_k, n_experts, row_offset, row_end, _stream(stream)),
           "mlg_grouped_down")


def mlg_grouped_down_all_windows(x, expert_offsets, src, row_adapter, a_table, b_table,
                                 scale_table, base_out, k_in, max_rank, n_out, top_k, n_experts,
                                 total_rows, cap, stream=None) -> None:
    _check(lib().mlg_grouped_down_all_windows(
        _addr(x), _addr(expert_offsets), _addr(src), _addr(row_adapter), _addr(a_table),
        _addr(b_table), _addr(scale_table), _addr(base_out), k_in, max_rank, n_out, top_k,
        n_experts, total_rows, cap, _stream(stream)), "mlg_grouped_down_all_windows")


def mlg_grouped_down_xrows(x_rows, expert_offsets, src, row_adapter, a_table, b_table,
                           scale_table, base_out, k_in, max_rank, n_out, top_k, n_experts,
                           row_offset, row_end, cap, stream=None) -> None:
    _check(lib().mlg_grouped_down_xrows(
        _addr(x_rows), _addr(expert_offsets), _addr(src), _addr(row_adapter), _addr(a_table),
        _addr(b_table), _addr(scale_table), _addr(base_out), k_in, max_rank, n_out, top_k,
        n_experts, row_offset, row_end, cap, _stream(stream)), "mlg_grouped_down_xrows")


def mlg_grouped_gemm_fold_xrows(x_rows, expert_offsets, src, row_adapter, w_experts, a_table,
                                b_table, scale_table, out, k_in, max_rank, n_out, top_k,
                                n_experts, row_offset, row_end, cap, stream=None) -> None:
    _check(lib().mlg_grouped_gemm_fold_xrows(
        _addr(x_rows), _addr(expert_offsets), _addr(src), _addr(row_adapter), _addr(w_experts),
        _addr(a_table), _addr(b_table), _addr(scale_table), _addr(out), k_in, max_rank, n_out,
        top_k, n_experts, row_offset, row_end, cap, _stream(stream)),
        "mlg_grouped_gemm_fold_xrows")


def mlg_router_fold(x, row_adapter, a_table, b_table, scale_table, base_out, n_tokens, k_in,
                    max_rank, n_out, stream=None) -> None:
    _check(lib().mlg_router_fold(_addr(x), _addr(row_adapter), _addr(a_table), _addr(b_table),
                                 _addr(scale_table), _addr(base_out), n_tokens, k_in, max_rank,
                                 n_out, _stream(stream)),
           "mlg_router_fold")


# ---------------------------------------------------------------- host helpers
def mlg_resolve_moe_lora_route(adapter_slot: int, active: int, has_moe_lora: bool) -> int:
    return lib().mlg_resolve_moe_lora_route(adapter_slot, active, int(bool(has_moe_lora)))


def mlg_ensure_decode_route_servable(route: int) -> None:
    _check(lib().mlg_ensure_decode_route_servable(route), "mlg_ensure_decode_route_servable")


def mlg_build_moe_row_adapter_decode(adapter_slots, padded_n: int, active: int,
                                     has_moe_lora: bool) -> np.ndarray:
    slots = _host(adapter_slots, np.int32)
    out = np.empty(padded_n, np.int32)
    _check(lib().mlg_build_moe_row_adapter_decode(_hp(slots), slots.size, padded_n, active,
                                                  int(bool(has_moe_lora)), _hp(out)),
           "mlg_build_moe_row_adapter_decode")
    return out


def mlg_build_moe_row_adapter_decode_multi(adapter_slots, padded_n: int, n_adapters: int,
                                           has_moe_lora: bool) -> np.ndarray:
    slots = _host(adapter_slots, np.int32)
    out = np.empty(padded_n, np.int32)
    _check(lib().mlg_build_moe_row_adapter_decode_multi(_hp(slots), slots.size, padded_n,
                                                        n_adapters, int(bool(has_moe_lora)),
                                                        _hp(out)),
           "mlg_build_moe_row_adapter_decode_multi")
    return out


def mlg_build_moe_row_adapter_host(cu_seqlens, adapter_slots) -> np.ndarray:
    cu = _host(cu_seqlens, np.int32)
    slots = _host(adapter_slots, np.int32)
    total = ctypes.c_size_t(0)
    st = lib().mlg_build_moe_row_adapter_host(_hp(cu), cu.size, _hp(slots), slots.size, None, 0,
                                              ctypes.byref(total))
    if st not in (MLG_OK, MLG_ERR_BUFFER_TOO_SMALL):
        _check(st, "mlg_build_moe_row_adapter_host")
    out = np.empty(total.value, np.int32)
    _check(lib().mlg_build_moe_row_adapter_host(_hp(cu), cu.size, _hp(slots), slots.size,
                                                _hp(out), out.size, ctypes.byref(total)),
           "mlg_build_moe_row_adapter_host")
    return out


# mlg_expert_entry as a numpy record (same 32-byte layout as ExpertEntry), so a
# table of entries is filled by array assignment rather than field by field.
_ENTRY_DT = np.dtype([("expert_id", "<u4"), ("reserved0", "<u4"), ("a_addr", "<u8"),
                      ("b_addr", "<u8"), ("scale", "<f4"), ("reserved1", "<u4")])
assert _ENTRY_DT.itemsize == ctypes.sizeof(ExpertEntry)


def mlg_pack_expert_tables(ids, a_addr, b_addr, scale):
    """Returns host tables (a u64, b u64, scale f32); n_experts = len(a)."""
    n = len(ids)
    rec = np.zeros(max(n, 1), _ENTRY_DT)
    if n:
        rec["expert_id"][:n] = np.asarray(ids, np.int64).astype(np.uint32)
        rec["a_addr"][:n] = np.asarray(a_addr).astype(np.uint64)
        rec["b_addr"][:n] = np.asarray(b_addr).astype(np.uint64)
        rec["scale"][:n] = np.asarray(scale, np.float32)
    entries = rec.ctypes.data_as(ctypes.c_void_p)
    n_exp = ctypes.c_uint32(0)
    st = lib().mlg_pack_expert_tables(entries, n, None, None, None, 0, ctypes.byref(n_exp))
    if st != MLG_ERR_BUFFER_TOO_SMALL:
        _check(st, "mlg_pack_expert_tables")
    E = n_exp.value
    a, b, s = np.empty(E, np.uint64), np.empty(E, np.uint64), np.empty(E, np.float32)
    _check(lib().mlg_pack_expert_tables(entries, n, _hp(a), _hp(b), _hp(s), E,
                                        ctypes.byref(n_exp)), "mlg_pack_expert_tables")
    return a, b, s


def mlg_upload_expert_tables(a_host, b_host, scale_host, a_dev, b_dev, scale_dev,
                             stream=None) -> None:
    a, b, s = _host(a_host, np.uint64), _host(b_host, np.uint64), _host(scale_host, np.float32)
    _check(lib().mlg_upload_expert_tables(_hp(a), _hp(b), _hp(s), a.size, _addr(a_dev),
                                          _addr(b_dev), _addr(scale_dev), _stream(stream)),
           "mlg_upload_expert_tables")


def mlg_upload_row_adapter(map_host, map_dev, stream=None) -> None:
    m = _host(map_host, np.int32)
    _check(lib().mlg_upload_row_adapter(_hp(m), m.size, _addr(map_dev), _stream(stream)),
           "mlg_upload_row_adapter")


def mlg_grouped_down_windows(total_rows: int, cap: int):
    n = ctypes.c_size_t(0)
    st = lib().mlg_grouped_down_windows(total_rows, cap, None, 0, ctypes.byref(n))
    if st != MLG_ERR_BUFFER_TOO_SMALL or n.value == 0:
        _check(st, "mlg_grouped_down_windows")
        if n.value == 0:
            return []
    out = (Window * n.value)()
    _check(lib().mlg_grouped_down_windows(total_rows, cap, out, n.value, ctypes.byref(n)),
           "mlg_grouped_down_windows")
    return [(w.start, w.end) for w in out]


def mlg_grouped_down_wc(row_offset: int, row_end: int) -> int:
    return lib().mlg_grouped_down_wc(row_offset, row_end)


def mlg_gather_row_token(row: int, top_k: int) -> int:
    return lib().mlg_gather_row_token(row, top_k)


def mlg_m_tile() -> int:
    return lib().mlg_m_tile()


def status_string(status: int) -> str:
    return lib().mlg_status_string(status).decode()


def mlg_last_cuda_error() -> int:
    return lib().mlg_last_cuda_error()


def mlg_version() -> int:
    return lib().mlg_version()


def mlg_read_device_errors(clear: bool = True) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().mlg_read_device_errors(ctypes.byref(v), int(clear)), "mlg_read_device_errors")
    return v.value


def mlg_test_set_knob(knob: int, value: int) -> None:
    """Test / benchmark hook (include/mlg_test.h): process-wide, not thread-safe;
    results never depend on it."""
    _check(lib().mlg_test_set_knob(knob, value), "mlg_test_set_knob")
