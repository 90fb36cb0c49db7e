"""libmlg host half: exported symbols, host helpers against the oracle and the
page-derived fixtures (bit-exact), and host-side validation of the fold entry
points.  CPU only: no call here reaches the GPU."""
import itertools
import os
import re
import subprocess

import numpy as np
import pytest

import golden_io
import oracle
import lora_moe_expert_gb300 as mlg
from lora_moe_expert_gb300 import build as mlg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mlg_build.build()
    return mlg.lib()


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^MLG_API\s+[\w\s\*]*?\b(mlg_\w+)\(", text, re.M))
    return names


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert len(declared) >= 19
    out = subprocess.run(["nm", "-D", "--defined-only", mlg.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = declared - exported
    assert not missing, missing
    for name in declared:
        getattr(L, name)


def test_product_does_not_touch_oracle():
    """The product package never imports, loads or names the oracle."""
    pkg = os.path.join(ROOT, "lora_moe_expert_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "mlg_oracle" not in text and "oracle_" not in text, f
    out = subprocess.run(["nm", "-D", mlg.LIBRARY], capture_output=True, text=True).stdout
    assert "oracle" not in out


def test_route_truth_table(L, o):
    for slot, active, has, exp in golden_io.route_cases():
        assert mlg.mlg_resolve_moe_lora_route(slot, active, bool(has)) == exp
    for slot, active, has in itertools.product(range(-3, 5), range(-1, 4), (0, 1)):
        assert mlg.mlg_resolve_moe_lora_route(slot, active, bool(has)) == \
            o.resolve_moe_lora_route(slot, active, bool(has))


def test_ensure_decode_route_servable(L):
    mlg.mlg_ensure_decode_route_servable(mlg.MLG_ROUTE_FOLD)
    mlg.mlg_ensure_decode_route_servable(mlg.MLG_ROUTE_SKIP)
    with pytest.raises(mlg.MlgError) as ei:
        mlg.mlg_ensure_decode_route_servable(mlg.MLG_ROUTE_REFUSE)
    assert ei.value.status == mlg.MLG_ERR_REFUSE
    assert "non-active adapter" in str(ei.value)
    with pytest.raises(mlg.MlgError):
        mlg.mlg_ensure_decode_route_servable(7)
    # the tiny decode batch holds a Refuse request (slot 2 under active 0)
    routes = [mlg.mlg_resolve_moe_lora_route(s, 0, True) for s in [0, -1, 0, 2]]
    assert routes == [0, 1, 0, 2]


def test_decode_map_fixtures(L):
    for slots, padded, active, has, exp in golden_io.decode_map_cases():
        assert mlg.mlg_build_moe_row_adapter_decode(slots, padded, active, bool(has)).tolist() \
            == exp


def test_decode_map_brute_force(L, o):
    vals = [-2, -1, 0, 1, 2]
    for n in range(0, 4):
        for slots in itertools.product(vals, repeat=n):
            for padded in range(0, 6):
                for active in (-1, 0, 1, 2):
                    for has in (False, True):
                        got = mlg.mlg_build_moe_row_adapter_decode(list(slots), padded, active,
                                                                   has)
                        exp = o.build_moe_row_adapter_decode(list(slots), padded, active, has)
                        assert np.array_equal(got, exp), (slots, padded, active, has)


def test_decode_map_multi_brute_force(L, o):
    vals = [-2, -1, 0, 1, 2, 3]
    for n in range(0, 4):
        for slots in itertools.product(vals, repeat=n):
            for padded in range(0, 5):
                for n_adapters in (1, 2, 3):
                    for has in (False, True):
                        st, exp = o.build_moe_row_adapter_decode_multi(list(slots), padded,
                                                                       n_adapters, has)
                        if st == 0:
                            got = mlg.mlg_build_moe_row_adapter_decode_multi(
                                list(slots), padded, n_adapters, has)
                            assert np.array_equal(got, exp), (slots, padded, n_adapters, has)
                        else:
                            with pytest.raises(mlg.MlgError) as ei:
                                mlg.mlg_build_moe_row_adapter_decode_multi(list(slots), padded,
                                                                           n_adapters, has)
                            assert ei.value.status == st == mlg.MLG_ERR_REFUSE
    with pytest.raises(mlg.MlgError) as ei:
        mlg.mlg_build_moe_row_adapter_decode_multi([0], 1, 0, True)
    assert ei.value.status == mlg.MLG_ERR_INVALID_ARG


def test_decode_map_multi_refusal_writes_nothing(L):
    import ctypes
    slots = np.array([0, 5, 1], np.int32)
    out = np.full(4, 77, np.int32)
    st = L.mlg_build_moe_row_adapter_decode_multi(slots.ctypes.data_as(ctypes.c_void_p), 3, 4, 2,
                                                  1, out.ctypes.data_as(ctypes.c_void_p))
    assert st == mlg.MLG_ERR_REFUSE and np.all(out == 77)


def test_host_map_fixtures(L):
    for cu, slots, exp in golden_io.host_map_cases():
        if exp is None:
            with pytest.raises(mlg.MlgError) as ei:
                mlg.mlg_build_moe_row_adapter_host(cu, slots)
            assert ei.value.status == mlg.MLG_ERR_INVALID_ARG
        else:
            assert mlg.mlg_build_moe_row_adapter_host(cu, slots).tolist() == exp


def test_host_map_brute_force(L, o):
    rng = np.random.default_rng(0)
    for _ in range(3000):
        n = int(rng.integers(0, 5))
        cu = rng.integers(-2, 7, size=n).astype(np.int32)
        if rng.random() < 0.6 and n:
            cu = np.sort(np.abs(cu)).astype(np.int32)
            cu[0] = 0 if rng.random() < 0.9 else cu[0]
        slots = rng.integers(-2, 4, size=max(0, n - 1 + int(rng.integers(-1, 2)))).astype(np.int32)
        exp = o.build_moe_row_adapter_host(cu, slots)
        if exp is None:
            with pytest.raises(mlg.MlgError):
                mlg.mlg_build_moe_row_adapter_host(cu, slots)
        else:
            assert np.array_equal(mlg.mlg_build_moe_row_adapter_host(cu, slots), exp)


def test_host_map_too_small_writes_nothing(L):
    import ctypes
    cu = np.array([0, 3, 5], np.int32)
    slots = np.array([1, 2], np.int32)
    out = np.full(4, 77, np.int32)
    total = ctypes.c_size_t(0)
    st = L.mlg_build_moe_row_adapter_host(cu.ctypes.data, 3, slots.ctypes.data, 2,
                                          out.ctypes.data, 4, ctypes.byref(total))
    assert st == mlg.MLG_ERR_BUFFER_TOO_SMALL and total.value == 5
    assert out.tolist() == [77] * 4
    # the page's [0, 4, 2]: None before any row is written
    cu = np.array([0, 4, 2], np.int32)
    st = L.mlg_build_moe_row_adapter_host(cu.ctypes.data, 3, slots.ctypes.data, 2,
                                          out.ctypes.data, 4, ctypes.byref(total))
    assert st == mlg.MLG_ERR_INVALID_ARG and out.tolist() == [77] * 4


def test_pack_fixtures(L):
    for entries, exp in golden_io.pack_cases():
        args = ([e[0] for e in entries], [e[1] for e in entries], [e[2] for e in entries],
                [e[3] for e in entries])
        if exp is None:
            with pytest.raises(mlg.MlgError) as ei:
                mlg.mlg_pack_expert_tables(*args)
            assert ei.value.status == mlg.MLG_ERR_EMPTY
            continue
        n, a, b, s = exp
        at, bt, st = mlg.mlg_pack_expert_tables(*args)
        assert at.tolist() == a and bt.tolist() == b and st.tolist() == s


def test_pack_brute_force(L, o):
    rng = np.random.default_rng(1)
    for _ in range(500):
        n = int(rng.integers(1, 9))
        ids = rng.integers(0, 12, size=n)
        a = rng.integers(0, 1 << 40, size=n) * 16 * (rng.random(n) < 0.8)
        b = rng.integers(0, 1 << 40, size=n) * 16
        s = rng.uniform(-2, 2, size=n).astype(np.float32)
        got = mlg.mlg_pack_expert_tables(ids, a, b, s)
        exp = o.pack_expert_tables(ids, a, b, s)
        for g, e in zip(got, exp):
            assert np.array_equal(g, e)


def test_pack_rejects_misaligned_and_small_buffer(L):
    import ctypes
    with pytest.raises(mlg.MlgError) as ei:
        mlg.mlg_pack_expert_tables([0, 1], [16, 24], [32, 48], [1.0, 1.0])
    assert ei.value.status == mlg.MLG_ERR_UNSUPPORTED
    ent = (mlg.ExpertEntry * 1)()
    ent[0].expert_id, ent[0].a_addr, ent[0].b_addr, ent[0].scale = 5, 16, 32, 1.0
    a = np.full(3, 9, np.uint64)
    n = ctypes.c_uint32(0)
    st = L.mlg_pack_expert_tables(ent, 1, a.ctypes.data, a.ctypes.data, a.ctypes.data, 3,
                                  ctypes.byref(n))
    assert st == mlg.MLG_ERR_BUFFER_TOO_SMALL and n.value == 6 and a.tolist() == [9, 9, 9]


def test_windows_and_wc(L, o):
    for total, cap, exp in golden_io.window_cases():
        if exp == "PANIC":
            with pytest.raises(mlg.MlgError) as ei:
                mlg.mlg_grouped_down_windows(total, cap)
            assert ei.value.status == mlg.MLG_ERR_CAP_ZERO
        else:
            assert mlg.mlg_grouped_down_windows(total, cap) == exp
    for total in range(0, 300, 11):
        for cap in range(1, 70, 7):
            assert mlg.mlg_grouped_down_windows(total, cap) == o.grouped_down_windows(total, cap)
    m = mlg.mlg_m_tile()
    assert m == 128
    for a, b, mt, exp in golden_io.wc_cases():
        if mt == m:
            assert mlg.mlg_grouped_down_wc(a, b) == exp
    for off in (0, 7, 1000):
        for length in range(0, 700, 9):
            assert mlg.mlg_grouped_down_wc(off, off + length) == o.grouped_down_wc(off, off +
                                                                                length, m)
    assert mlg.mlg_grouped_down_wc(10, 5) == 1


def test_row_token(L, o):
    for top_k in (1, 2, 3, 8, 10):
        for row in range(0, 100):
            assert mlg.mlg_gather_row_token(row, top_k) == o.gather_row_token(row, top_k)
    assert mlg.mlg_gather_row_token(5, 0) == 0


def test_fold_validation_on_host(L):
    """Invalid arguments are rejected before any device work (runs without a GPU)."""
    p = 1 << 20  # a 16-byte-aligned stand-in address; never dereferenced on error paths
    ok = dict(x=p, indices=p, row_adapter=p, a_table=p, b_table=p, scale_table=p, base_out=p,
              n_slots=8, k_in=64, max_rank=16, n_out=64, top_k=2, n_experts=4)

    def gather(**kw):
        args = {**ok, **kw}
        return L.mlg_gather_bgmv(args["x"], args["indices"], args["row_adapter"],
                                 args["a_table"], args["b_table"], args["scale_table"],
                                 args["base_out"], args["n_slots"], args["k_in"],
                                 args["max_rank"], args["n_out"], args["top_k"],
                                 args["n_experts"], 0)

    assert gather(top_k=0) == mlg.MLG_ERR_INVALID_ARG
    assert gather(n_slots=-1) == mlg.MLG_ERR_INVALID_ARG
    assert gather(k_in=12) == mlg.MLG_ERR_UNSUPPORTED
    assert gather(n_out=20) == mlg.MLG_ERR_UNSUPPORTED
    assert gather(max_rank=12) == mlg.MLG_ERR_UNSUPPORTED
    assert gather(max_rank=72) == mlg.MLG_ERR_UNSUPPORTED
    assert gather(max_rank=0) == mlg.MLG_ERR_INVALID_ARG
    assert gather(x=None) == mlg.MLG_ERR_INVALID_ARG
    assert gather(row_adapter=None) == mlg.MLG_ERR_INVALID_ARG
    assert gather(x=p + 8) == mlg.MLG_ERR_UNSUPPORTED
    assert gather(base_out=p + 2) == mlg.MLG_ERR_UNSUPPORTED
    assert gather(n_slots=0) == mlg.MLG_OK  # no-op, nothing launched
    assert gather(n_experts=0) == mlg.MLG_OK

    def multi(**kw):
        args = {**ok, "n_adapters": 3, **kw}
        return L.mlg_gather_bgmv_multi(args["x"], args["indices"], args["row_adapter"],
                                       args["a_table"], args["b_table"], args["scale_table"],
                                       args["base_out"], args["n_slots"], args["k_in"],
                                       args["max_rank"], args["n_out"], args["top_k"],
                                       args["n_experts"], args["n_adapters"], 0)

    assert multi(n_adapters=0) == mlg.MLG_ERR_INVALID_ARG
    assert multi(n_adapters=-1) == mlg.MLG_ERR_INVALID_ARG
    assert multi(n_experts=1 << 20, n_adapters=1 << 11) == mlg.MLG_ERR_UNSUPPORTED
    assert multi(top_k=0) == mlg.MLG_ERR_INVALID_ARG
    assert multi(row_adapter=None) == mlg.MLG_ERR_INVALID_ARG
    assert multi(k_in=12) == mlg.MLG_ERR_UNSUPPORTED
    assert multi(x=p + 8) == mlg.MLG_ERR_UNSUPPORTED
    assert multi(n_slots=0) == mlg.MLG_OK
    assert multi(n_experts=0) == mlg.MLG_OK

    def grouped(**kw):
        args = {**ok, "expert_offsets": p, "src": p, "row_offset": 0, "row_end": 100, **kw}
        return L.mlg_grouped_down(args["x"], args["expert_offsets"], args["src"],
                                  args["row_adapter"], args["a_table"], args["b_table"],
                                  args["scale_table"], args["base_out"], args["k_in"],
                                  args["max_rank"], args["n_out"], args["top_k"],
                                  args["n_experts"], args["row_offset"], args["row_end"], 0)

    assert grouped(row_end=5, row_offset=6) == mlg.MLG_ERR_INVALID_ARG
    assert grouped(row_offset=-1) == mlg.MLG_ERR_INVALID_ARG
    assert grouped(top_k=0) == mlg.MLG_ERR_INVALID_ARG
    assert grouped(src=None) == mlg.MLG_ERR_INVALID_ARG
    assert grouped(expert_offsets=None) == mlg.MLG_ERR_INVALID_ARG
    assert grouped(k_in=4) == mlg.MLG_ERR_UNSUPPORTED
    assert grouped(row_offset=50, row_end=50) == mlg.MLG_OK

    def all_windows(**kw):
        args = {**ok, "expert_offsets": p, "src": p, "total_rows": 100, "cap": 32, **kw}
        return L.mlg_grouped_down_all_windows(
            args["x"], args["expert_offsets"], args["src"], args["row_adapter"], args["a_table"],
            args["b_table"], args["scale_table"], args["base_out"], args["k_in"],
            args["max_rank"], args["n_out"], args["top_k"], args["n_experts"],
            args["total_rows"], args["cap"], 0)

    assert all_windows(cap=0) == mlg.MLG_ERR_CAP_ZERO
    assert all_windows(total_rows=-1) == mlg.MLG_ERR_INVALID_ARG
    assert all_windows(src=None) == mlg.MLG_ERR_INVALID_ARG
    assert all_windows(max_rank=20) == mlg.MLG_ERR_UNSUPPORTED
    assert all_windows(total_rows=0) == mlg.MLG_OK

    def xrows(**kw):
        args = {**ok, "expert_offsets": p, "src": p, "row_offset": 0, "row_end": 100, "cap": 32,
                **kw}
        return L.mlg_grouped_down_xrows(
            args["x"], args["expert_offsets"], args["src"], args["row_adapter"], args["a_table"],
            args["b_table"], args["scale_table"], args["base_out"], args["k_in"],
            args["max_rank"], args["n_out"], args["top_k"], args["n_experts"],
            args["row_offset"], args["row_end"], args["cap"], 0)

    assert xrows(cap=0) == mlg.MLG_ERR_CAP_ZERO
    assert xrows(row_offset=7, row_end=6) == mlg.MLG_ERR_INVALID_ARG
    assert xrows(row_offset=-2) == mlg.MLG_ERR_INVALID_ARG
    assert xrows(src=None) == mlg.MLG_ERR_INVALID_ARG
    assert xrows(x=None) == mlg.MLG_ERR_INVALID_ARG
    assert xrows(x=p + 4) == mlg.MLG_ERR_UNSUPPORTED
    assert xrows(top_k=0) == mlg.MLG_ERR_INVALID_ARG
    assert xrows(n_out=12) == mlg.MLG_ERR_UNSUPPORTED
    assert xrows(row_offset=40, row_end=40) == mlg.MLG_OK
    assert xrows(n_experts=0) == mlg.MLG_OK

    def router(**kw):
        args = {**ok, "n_tokens": 16, **kw}
        return L.mlg_router_fold(args["x"], args["row_adapter"], args["a_table"],
                                 args["b_table"], args["scale_table"], args["base_out"],
                                 args["n_tokens"], args["k_in"], args["max_rank"],
                                 args["n_out"], 0)

    assert router(n_tokens=-1) == mlg.MLG_ERR_INVALID_ARG
    assert router(a_table=None) == mlg.MLG_ERR_INVALID_ARG
    assert router(n_out=4) == mlg.MLG_ERR_UNSUPPORTED
    assert router(n_tokens=0) == mlg.MLG_OK

    def gemm_fold(**kw):
        args = {**ok, "expert_offsets": p, "src": p, "w": p, "row_offset": 0, "row_end": 100,
                "cap": 32, **kw}
        return L.mlg_grouped_gemm_fold_xrows(
            args["x"], args["expert_offsets"], args["src"], args["row_adapter"], args["w"],
            args["a_table"], args["b_table"], args["scale_table"], args["base_out"],
            args["k_in"], args["max_rank"], args["n_out"], args["top_k"], args["n_experts"],
            args["row_offset"], args["row_end"], args["cap"], 0)

    assert gemm_fold(cap=0) == mlg.MLG_ERR_CAP_ZERO
    assert gemm_fold(row_offset=7, row_end=6) == mlg.MLG_ERR_INVALID_ARG
    assert gemm_fold(row_offset=-2) == mlg.MLG_ERR_INVALID_ARG
    assert gemm_fold(top_k=0) == mlg.MLG_ERR_INVALID_ARG
    assert gemm_fold(n_experts=-1) == mlg.MLG_ERR_INVALID_ARG
    for name in ("x", "expert_offsets", "src", "w", "a_table", "b_table", "scale_table",
                 "base_out"):
        assert gemm_fold(**{name: None}) == mlg.MLG_ERR_INVALID_ARG, name
    assert gemm_fold(x=p + 4) == mlg.MLG_ERR_UNSUPPORTED
    assert gemm_fold(w=p + 8) == mlg.MLG_ERR_UNSUPPORTED
    assert gemm_fold(base_out=p + 2) == mlg.MLG_ERR_UNSUPPORTED
    assert gemm_fold(k_in=12) == mlg.MLG_ERR_UNSUPPORTED
    assert gemm_fold(n_out=12) == mlg.MLG_ERR_UNSUPPORTED
    assert gemm_fold(max_rank=72) == mlg.MLG_ERR_UNSUPPORTED
    assert gemm_fold(row_offset=40, row_end=40) == mlg.MLG_OK  # empty range: nothing launched
    assert gemm_fold(n_experts=0) == mlg.MLG_OK
    assert gemm_fold(row_adapter=None, row_offset=3, row_end=3) == mlg.MLG_OK  # the map is optional

    def gather_ex(flags, multi_form=False, **kw):
        args = {**ok, **kw}
        if multi_form:
            return L.mlg_gather_bgmv_multi_ex(
                args["x"], args["indices"], args["row_adapter"], args["a_table"], args["b_table"],
                args["scale_table"], args["base_out"], args["n_slots"], args["k_in"],
                args["max_rank"], args["n_out"], args["top_k"], args["n_experts"], 2, flags, 0)
        return L.mlg_gather_bgmv_ex(args["x"], args["indices"], args["row_adapter"],
                                    args["a_table"], args["b_table"], args["scale_table"],
                                    args["base_out"], args["n_slots"], args["k_in"],
                                    args["max_rank"], args["n_out"], args["top_k"],
                                    args["n_experts"], flags, 0)

    for multi_form in (False, True):
        # unknown flags are rejected before anything else; known ones pass validation
        assert gather_ex(2, multi_form) == mlg.MLG_ERR_INVALID_ARG
        assert gather_ex(0x80000000, multi_form) == mlg.MLG_ERR_INVALID_ARG
        assert gather_ex(2, multi_form, n_slots=0) == mlg.MLG_ERR_INVALID_ARG
        assert gather_ex(mlg.MLG_FOLD_AFTER_PRECEDING, multi_form, n_slots=0) == mlg.MLG_OK
        assert gather_ex(0, multi_form, top_k=0) == mlg.MLG_ERR_INVALID_ARG
        assert gather_ex(mlg.MLG_FOLD_AFTER_PRECEDING, multi_form, x=p + 8) == \
            mlg.MLG_ERR_UNSUPPORTED


def test_status_strings_and_tuning(L):
    for st in range(-7, 1):
        assert mlg.status_string(st)
    assert mlg.status_string(-99) == "unknown status"
    assert mlg.mlg_version() >= 10000
    with pytest.raises(mlg.MlgError):
        mlg.mlg_test_set_knob(99, 0)
    with pytest.raises(mlg.MlgError):
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_CLUSTER, 3)
    mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_CLUSTER, 0)
    for knob in (mlg.MLG_TEST_GATHER_PATH, mlg.MLG_TEST_GATHER_SPECULATION):
        with pytest.raises(mlg.MlgError):
            mlg.mlg_test_set_knob(knob, 3)
        mlg.mlg_test_set_knob(knob, 0)
