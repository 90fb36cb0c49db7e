"""Pins that tie the fp64 oracle to something other than itself.

Each pin is a function of an ``oracle.Oracle`` that raises AssertionError on a
mismatch, so the same pins run against the real oracle (test_oracle_pins.py)
and against deliberately broken copies of it (test_oracle_mutants.py, which
checks that every planted mistake trips at least one pin).

What pins what:

* host rules -- the hand-written fixtures in tests/golden/ (route truth table,
  decode and prefill row maps, table packing, windows, wc), plus invariants
  of the window split over a range of sizes;
* the fold -- closed forms (rank-1 unit-vector pairs give base + scale * x[t,i]
  in column j exactly), exact small-integer cases compared with an integer
  matrix product, a dense one-expert special case compared with numpy's
  float64 matmul, and invariants: rows that must not fold keep their input
  bit for bit, the delta is linear in the scale, the grouped form on sorted
  rows equals the gather form on flat rows, any window split equals one
  window, and the router fold equals a one-expert gather with top_k = 1.
"""
from __future__ import annotations

import numpy as np

import golden_io
from lora_moe_expert_gb300 import synth

from oracle import HostExperts


def _bits(values) -> np.ndarray:
    return synth.bf16_bits(np.asarray(values, np.float32))


def _f(bits) -> np.ndarray:
    return synth.bf16_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- host rules
def pin_route_truth_table(o):
    for slot, active, has, exp in golden_io.route_cases():
        got = o.resolve_moe_lora_route(slot, active, bool(has))
        assert got == exp, (slot, active, has, got, exp)
        err = o.ensure_decode_route_servable(got)
        assert (err != 0) == (exp == 2), (slot, active, has, err)


def pin_decode_maps(o):
    for slots, padded, active, has, exp in golden_io.decode_map_cases():
        got = o.build_moe_row_adapter_decode(slots, padded, active, bool(has))
        assert got.tolist() == exp, (slots, padded, active, has, got.tolist(), exp)


def pin_host_maps(o):
    for cu, slots, exp in golden_io.host_map_cases():
        got = o.build_moe_row_adapter_host(cu, slots)
        if exp is None:
            assert got is None, (cu, slots, got)
        else:
            assert got is not None and got.tolist() == exp, (cu, slots, got, exp)


def pin_pack(o):
    for entries, exp in golden_io.pack_cases():
        got = o.pack_expert_tables([e[0] for e in entries], [e[1] for e in entries],
                                   [e[2] for e in entries], [e[3] for e in entries])
        if exp is None:
            assert got is None
            continue
        n, a, b, s = exp
        at, bt, st = got
        assert at.size == n and at.tolist() == a and bt.tolist() == b, (entries, got)
        assert np.array_equal(st, np.asarray(s, np.float32)), (entries, st, s)


def pin_windows(o):
    for total, cap, exp in golden_io.window_cases():
        if exp == "PANIC":
            try:
                o.grouped_down_windows(total, cap)
            except ValueError:
                continue
            raise AssertionError("cap == 0 accepted")
        assert o.grouped_down_windows(total, cap) == exp, (total, cap)
    # invariants over a range: cover 0..total, contiguous, each <= cap, none empty,
    # and as few windows as the cap allows
    for total in range(0, 121, 7):
        for cap in range(1, 40, 3):
            w = o.grouped_down_windows(total, cap)
            assert sum(e - s for s, e in w) == total
            pos = 0
            for s, e in w:
                assert s == pos and 0 < e - s <= cap
                pos = e
            assert len(w) * cap >= total and (len(w) - 1) * cap < max(total, 1)


def pin_wc(o):
    for a, b, m, exp in golden_io.wc_cases():
        assert o.grouped_down_wc(a, b, m) == exp, (a, b, m)
    for m in (1, 32, 128):
        for length in range(0, 400, 13):
            wc = o.grouped_down_wc(10, 10 + length, m)
            assert wc >= 1 and wc * m >= length
            assert length == 0 or (wc - 1) * m < length


def pin_row_token(o):
    for top_k in (1, 2, 8, 10):
        for t in range(6):
            for k in range(top_k):
                assert o.gather_row_token(t * top_k + k, top_k) == t


# ---------------------------------------------------------------- the fold
def _unit_case():
    """Rank-1 unit pairs: expert e has A_e[0, i_e] = 1 and B_e[j_e, 0] = 1 only.
    Then the fold adds scale_e * x[t, i_e] to column j_e of the row, and nothing else."""
    k_in, n_out, r, T, K, E = 24, 40, 16, 5, 3, 6
    rng = np.random.default_rng(11)
    x = _bits(rng.integers(-8, 9, size=(T, k_in)) / 4.0)
    base = _bits(rng.integers(-8, 9, size=(T * K, n_out)) / 8.0)
    pick = [(3, 17), (0, 39), (23, 5), (11, 0), (7, 22), (19, 31)]
    scales = [0.5, 2.0, 1.0, 0.25, 1.5, 4.0]
    experts = []
    for e, (i, j) in enumerate(pick):
        A = np.zeros((r, k_in), np.uint16)
        B = np.zeros((n_out, r), np.uint16)
        A[0, i] = _bits([1.0])[0]
        B[j, 0] = _bits([1.0])[0]
        experts.append((e, A, B, scales[e]))
    idx = np.array([(t * 5 + k * 2) % E for t in range(T) for k in range(K)], np.int32)
    return k_in, n_out, r, T, K, x, base, experts, pick, scales, idx


def pin_fold_unit_vectors(o):
    k_in, n_out, r, T, K, x, base, experts, pick, scales, idx = _unit_case()
    he = HostExperts(experts)
    at, bt, st = he.tables(o)
    ra = np.zeros(T, np.int32)
    ref, folded = o.gather_fold(x, idx, ra, at, bt, st, base, k_in, r, n_out, K)
    assert folded.all()
    expect = _f(base).reshape(T * K, n_out).copy()
    xf = _f(x)
    for row in range(T * K):
        e = idx[row]
        i, j = pick[e]
        expect[row, j] += scales[e] * xf[row // K, i]
    assert np.array_equal(ref, expect), np.argwhere(ref != expect)[:5]


def pin_fold_exact_integers(o):
    """Small integers everywhere: every sum is exact in double, so the oracle must
    equal an integer matrix product (scale a power of two) exactly."""
    rng = np.random.default_rng(5)
    k_in, n_out, r, T, K, E = 40, 24, 8, 6, 2, 5
    xi = rng.integers(-3, 4, size=(T, k_in))
    Ai = rng.integers(-2, 3, size=(E, r, k_in))
    Bi = rng.integers(-2, 3, size=(E, n_out, r))
    basei = rng.integers(-16, 17, size=(T * K, n_out))
    scales = [0.5, 0.25, 2.0, 1.0, 0.125]
    experts = [(e, _bits(Ai[e]), _bits(Bi[e]), scales[e]) for e in range(E)]
    idx = rng.integers(0, E, size=T * K).astype(np.int32)
    ra = np.zeros(T, np.int32)
    at, bt, st = HostExperts(experts).tables(o)
    ref, _ = o.gather_fold(_bits(xi), idx, ra, at, bt, st, _bits(basei), k_in, r, n_out, K)
    for row in range(T * K):
        e, t = idx[row], row // K
        h = Ai[e] @ xi[t]  # integer, [r]
        d = Bi[e] @ h  # integer, [n_out]
        exp = basei[row] + scales[e] * d
        assert np.array_equal(ref[row], exp.astype(np.float64)), row


def pin_fold_dense_matmul(o):
    """All rows on one expert with every token active: the fold reduces to
    base + scale * (X A^T) B^T, a plain float64 matrix product."""
    rng = np.random.default_rng(7)
    k_in, n_out, r, T, K = 48, 72, 12, 7, 3
    x = _bits(rng.standard_normal((T, k_in)))
    base = _bits(rng.standard_normal((T * K, n_out)))
    A = _bits(rng.standard_normal((r, k_in)) / np.sqrt(k_in))
    B = _bits(rng.standard_normal((n_out, r)) / np.sqrt(r))
    at, bt, st = HostExperts([(2, A, B, 1.375)]).tables(o)
    idx = np.full(T * K, 2, np.int32)
    ref, folded = o.gather_fold(x, idx, np.zeros(T, np.int32), at, bt, st, base, k_in, r, n_out, K)
    X = np.repeat(_f(x), K, axis=0)
    exp = _f(base) + 1.375 * ((X @ _f(A).T) @ _f(B).T)
    assert folded.all()
    np.testing.assert_allclose(ref, exp, rtol=1e-12, atol=1e-12)


def pin_fold_skips_keep_input(o):
    """Rows that must not fold keep their input bit for bit: a negative row-map
    entry, an expert id at or past the table, a negative id, a zero table cell."""
    w = synth.custom_gather(21, n_tokens=9, top_k=3, n_experts=10, k_in=32, n_out=40,
                            max_rank=8, adapted_frac=0.6, base_frac=0.3, bad_ids=4)
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    E = at.size
    ra = o.build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, 0, True)
    ref, folded = o.gather_fold(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank,
                                w.n_out, w.top_k)
    for row in range(w.indices.size):
        e, t = int(w.indices[row]), row // w.top_k
        should = ra[t] >= 0 and 0 <= e < E and at[e] != 0 and bt[e] != 0
        assert folded[row] == should, (row, e, t)
        if not should:
            assert np.array_equal(ref[row], _f(w.base[row])), row
    assert folded.any() and (~folded).any()


def pin_fold_linear_in_scale(o):
    w = synth.custom_gather(3, n_tokens=5, top_k=2, n_experts=4, k_in=32, n_out=24, max_rank=8)
    ra = np.zeros(w.n_tokens, np.int32)
    he1 = HostExperts([(e.expert_id, e.A, e.B, 1.0) for e in w.experts])
    he2 = HostExperts([(e.expert_id, e.A, e.B, -2.0) for e in w.experts])
    ref1, _ = o.gather_fold(w.x, w.indices, ra, *he1.tables(o), w.base, w.k_in, w.max_rank,
                            w.n_out, w.top_k)
    ref2, _ = o.gather_fold(w.x, w.indices, ra, *he2.tables(o), w.base, w.k_in, w.max_rank,
                            w.n_out, w.top_k)
    b = _f(w.base)
    np.testing.assert_allclose(ref2 - b, -2.0 * (ref1 - b), rtol=1e-12, atol=1e-12)
    assert np.abs(ref1 - b).max() > 0.1


def _grouped_from_gather(w):
    """Sorted-row view of a decode batch: rows sorted by expert, ids past the
    model's expert count are put at the end (no span holds them)."""
    idx = w.indices.astype(np.int64)
    E = w.n_experts_model
    key = np.where((idx < 0) | (idx >= E), E, idx)
    offsets, src = synth.sort_rows_by_expert(key, E + 1)
    return offsets[: E + 1], src


def pin_cross_form(o):
    """The grouped fold over expert-sorted rows equals the gather fold over flat rows."""
    w = synth.custom_gather(8, n_tokens=11, top_k=4, n_experts=9, k_in=40, n_out=56,
                            max_rank=8, adapted_frac=0.7, base_frac=0.25, bad_ids=2)
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    ra = o.build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, 0, True)
    ref_g, fold_g = o.gather_fold(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank,
                                  w.n_out, w.top_k)
    offsets, src = _grouped_from_gather(w)
    n_exp = at.size
    ref_s, fold_s = o.grouped_fold(w.x, offsets[: n_exp + 1], src, ra, at, bt, st, w.base[src],
                                   w.k_in, w.max_rank, w.n_out, w.top_k, 0, src.size)
    assert np.array_equal(fold_s, fold_g[src])
    assert np.array_equal(ref_s, ref_g[src])


def pin_window_split(o):
    """Folding window by window, each on the previous result, equals one window
    over all rows; rows outside a window keep their input."""
    w = synth.custom_grouped(4, [13, 29, 7], top_k=3, n_experts=12, k_in=32, n_out=24,
                             max_rank=8, cap=17, adapted_frac=0.75, stream_base=[0, 1, 0])
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    n_exp = at.size
    ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
    R = w.rows
    full, ffull = o.grouped_fold(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base, w.k_in,
                                 w.max_rank, w.n_out, w.top_k, 0, R)
    assert ffull.any() and (~ffull).any()
    for cap in (1, 5, 17, 64):
        acc = np.zeros((R, w.n_out))
        seen = np.zeros(R, bool)
        for s, e in o.grouped_down_windows(R, cap):
            ref, fold = o.grouped_fold(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base,
                                       w.k_in, w.max_rank, w.n_out, w.top_k, s, e)
            assert not fold[:s].any() and not fold[e:].any()
            assert np.array_equal(ref[:s], _f(w.base[:s])) and np.array_equal(ref[e:],
                                                                              _f(w.base[e:]))
            acc[s:e] = ref[s:e]
            seen[s:e] = True
        assert seen.all() and np.array_equal(acc, full)
    # rows past expert_offsets[n_experts] (experts beyond the table) never fold
    assert not ffull[w.expert_offsets[n_exp]:].any()


def pin_router_is_one_entry_route(o):
    w = synth.custom_router(9, n_tokens=6, k_in=32, n_out=20, max_rank=8)
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    ra = np.array([0, -1, 0, 0, -1, 0], np.int32)
    ref_r, fold_r = o.router_fold(w.x, ra, at, bt, st, w.base, w.k_in, w.max_rank, w.n_out)
    ref_g, fold_g = o.gather_fold(w.x, np.zeros(6, np.int32), ra, at, bt, st, w.base, w.k_in,
                                  w.max_rank, w.n_out, 1)
    assert np.array_equal(ref_r, ref_g) and np.array_equal(fold_r, fold_g)
    assert fold_r.tolist() == [True, False, True, True, False, True]
    ref_n, fold_n = o.router_fold(w.x, None, at, bt, st, w.base, w.k_in, w.max_rank, w.n_out)
    assert fold_n.all()
    # a zero cell makes the route a no-op
    ref_z, fold_z = o.router_fold(w.x, None, np.zeros(1, np.uint64), bt, st, w.base, w.k_in,
                                  w.max_rank, w.n_out)
    assert not fold_z.any() and np.array_equal(ref_z, _f(w.base))


def pin_sampled_rows_match_full(o):
    """The row-sampled entry points equal the corresponding rows of the full folds."""
    w = synth.custom_gather(12, n_tokens=7, top_k=2, n_experts=5, k_in=24, n_out=16,
                            max_rank=8, adapted_frac=0.8, base_frac=0.3, bad_ids=1)
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    ra = o.build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, 0, True)
    ref, fold = o.gather_fold(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank,
                              w.n_out, w.top_k)
    rows = np.array([13, 0, 5, 6, 2], np.int32)
    ref_s, fold_s = o.gather_fold_rows(w.x, w.indices, ra, at, bt, st, w.base[rows], rows,
                                       w.k_in, w.max_rank, w.n_out, w.top_k)
    assert np.array_equal(ref_s, ref[rows]) and np.array_equal(fold_s, fold[rows])
    g = synth.custom_grouped(6, [9, 4], top_k=2, n_experts=6, k_in=16, n_out=24, max_rank=8,
                             cap=8, adapted_frac=0.7)
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in g.experts])
    at, bt, st = he.tables(o)
    ref, fold = o.grouped_fold(g.x, g.expert_offsets, g.src, None, at, bt, st, g.base, g.k_in,
                               g.max_rank, g.n_out, g.top_k, 3, 20)
    rows = np.array([0, 3, 19, 20, 25, 11], np.int32)
    ref_s, fold_s = o.grouped_fold_rows(g.x, g.expert_offsets, g.src, None, at, bt, st,
                                        g.base[rows], rows, g.k_in, g.max_rank, g.n_out,
                                        g.top_k, 3, 20)
    assert np.array_equal(ref_s, ref[rows]) and np.array_equal(fold_s, fold[rows])


def pin_xrows_forms(o):
    """The per-row x grouped fold (sorted row r reads x_rows[r]) equals the
    token form when x_rows[r] is the row's token, and equals a top_k = 1 gather
    fold over the sorted rows (row r as its own token, its span's expert as its
    id, its token's row-map entry as its entry) for arbitrary x_rows."""
    w = synth.custom_grouped(14, [11, 23, 6], top_k=3, n_experts=10, k_in=40, n_out=32,
                             max_rank=8, cap=19, adapted_frac=0.7, stream_base=[0, 1, 0])
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    n_exp = at.size
    ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
    R = w.rows
    tok_rows = w.x[w.src // w.top_k]
    for s, e in [(0, R), (5, 40), (R - 3, R)]:
        ref_t, fold_t = o.grouped_fold(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base,
                                       w.k_in, w.max_rank, w.n_out, w.top_k, s, e)
        ref_x, fold_x = o.grouped_fold_xrows(tok_rows, w.expert_offsets, w.src, ra, at, bt, st,
                                             w.base, w.k_in, w.max_rank, w.n_out, w.top_k, s, e)
        assert np.array_equal(fold_x, fold_t) and np.array_equal(ref_x, ref_t)
    rng = np.random.default_rng(3)
    x_rows = _bits(rng.standard_normal((R, w.k_in)))
    ids = np.full(R, n_exp + 7, np.int32)
    for e in range(n_exp):
        ids[w.expert_offsets[e]:w.expert_offsets[e + 1]] = e
    ra_rows = ra[w.src // w.top_k]
    ref_g, fold_g = o.gather_fold(x_rows, ids, ra_rows, at, bt, st, w.base, w.k_in, w.max_rank,
                                  w.n_out, 1)
    ref_x, fold_x = o.grouped_fold_xrows(x_rows, w.expert_offsets, w.src, ra, at, bt, st,
                                         w.base, w.k_in, w.max_rank, w.n_out, w.top_k, 0, R)
    assert fold_x.any() and (~fold_x).any()
    assert np.array_equal(fold_x, fold_g) and np.array_equal(ref_x, ref_g)
    # the row-sampled entry point equals the corresponding rows of a windowed fold
    ref_w, fold_w = o.grouped_fold_xrows(x_rows, w.expert_offsets, w.src, ra, at, bt, st,
                                         w.base, w.k_in, w.max_rank, w.n_out, w.top_k, 4, R - 6)
    rows = np.array([0, 3, 4, R - 7, R - 6, 17, R - 1, 30], np.int32)
    ref_s, fold_s = o.grouped_fold_xrows_rows(x_rows, w.expert_offsets, w.src, ra, at, bt, st,
                                              w.base[rows], rows, w.k_in, w.max_rank, w.n_out,
                                              w.top_k, 4, R - 6)
    assert np.array_equal(ref_s, ref_w[rows]) and np.array_equal(fold_s, fold_w[rows])


def pin_multi_adapter(o):
    """The multi-adapter fold: with one adapter it is the gather fold; in
    general it is, row for row, the gather fold of the row's own adapter's
    table slice (each row folds through exactly one set); and its decode map
    keeps installed slots, blanks base requests and padding, refuses a slot
    with no set, and folds nothing without MoE LoRA."""
    E, S = 9, 3
    w = synth.custom_gather_multi(21, n_tokens=13, top_k=3, n_experts=E, k_in=40, n_out=24,
                                  max_rank=8, n_adapters=S, adapted_frac=0.7, base_frac=0.2,
                                  bad_ids=2)
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o, length=S * E)
    status, ra = o.build_moe_row_adapter_decode_multi(w.adapter_slots, w.padded_n, S, True)
    assert status == 0 and np.array_equal(ra, np.where(w.adapter_slots >= 0, w.adapter_slots, -1))
    ref_m, fold_m = o.gather_fold_multi(w.x, w.indices, ra, at, bt, st, w.base, w.k_in,
                                        w.max_rank, w.n_out, w.top_k, E, S)
    assert fold_m.any() and (~fold_m).any()
    tok = np.arange(w.rows) // w.top_k
    acc = _f(w.base)
    seen = np.zeros(w.rows, bool)
    for s in range(S):
        sl = slice(s * E, (s + 1) * E)
        ra_s = np.where(ra == s, 0, -1).astype(np.int32)
        ref_s, fold_s = o.gather_fold(w.x, w.indices, ra_s, at[sl], bt[sl], st[sl], w.base,
                                      w.k_in, w.max_rank, w.n_out, w.top_k)
        mine = ra[tok] == s
        assert not (fold_s & ~mine).any()
        acc[mine] = ref_s[mine]
        seen |= fold_s
    assert np.array_equal(seen, fold_m) and np.array_equal(acc, ref_m)
    # one adapter: the gather fold itself
    ra1 = np.where(ra >= 0, 0, -1).astype(np.int32)
    ref_1, fold_1 = o.gather_fold_multi(w.x, w.indices, ra1, at[:E], bt[:E], st[:E], w.base,
                                        w.k_in, w.max_rank, w.n_out, w.top_k, E, 1)
    ref_g, fold_g = o.gather_fold(w.x, w.indices, ra1, at[:E], bt[:E], st[:E], w.base, w.k_in,
                                  w.max_rank, w.n_out, w.top_k)
    assert np.array_equal(ref_1, ref_g) and np.array_equal(fold_1, fold_g)
    # decode map cases
    st_, m = o.build_moe_row_adapter_decode_multi([2, -1, 0, 1, -7], 6, 3, True)
    assert st_ == 0 and m.tolist() == [2, -1, 0, 1, -1, -1]
    st_, m = o.build_moe_row_adapter_decode_multi([0, 3, -1], 4, 3, True)
    assert st_ == -4 and np.all(m == 0x5A5A5A5A)  # refused, nothing written
    st_, m = o.build_moe_row_adapter_decode_multi([0, 3, 1], 4, 3, False)
    assert st_ == 0 and m.tolist() == [-1, -1, -1, -1]
    slots = np.array([0, -1, 0, 0, -1], np.int32)
    st_, m = o.build_moe_row_adapter_decode_multi(slots, 7, 1, True)
    assert st_ == 0 and np.array_equal(m, o.build_moe_row_adapter_decode(slots, 7, 0, True))


class _Weights:
    """Host copies of expert GEMM weights W_e [n_out, k_in] (bf16 bits) and the
    table of their host addresses (0 = no weight for that expert)."""

    def __init__(self, mats, n_table):
        self.keep = []
        self.table = np.zeros(n_table, np.uint64)
        for e, m in mats.items():
            m = np.ascontiguousarray(m, np.uint16)
            self.keep.append(m)
            self.table[e] = m.ctypes.data


def pin_gemm_fold(o):
    """The expert GEMM with the fold in its epilogue.  With the LoRA cells
    zeroed it is numpy's float64 matmul of x_rows and W_e^T on the rows of
    spans with a weight; with small integers (every GEMM value an exact bf16)
    it equals the per-row x fold run on base = that GEMM result; with W_e a
    permutation (out column n picks x column perm_e[n]) it equals the per-row
    x fold on base = x_rows[:, perm_e]; rows of a span without a weight, and
    rows outside the window, keep their prior bits."""
    w = synth.custom_grouped(15, [13, 21, 7], top_k=3, n_experts=9, k_in=48, n_out=48,
                             max_rank=8, cap=17, adapted_frac=0.7, stream_base=[0, 1, 0],
                             per_row_x=True)
    he = HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o, length=w.n_experts_model)
    E, R, K, N = w.n_experts_model, w.rows, w.k_in, w.n_out
    ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
    rng = np.random.default_rng(8)
    counts = np.diff(w.expert_offsets)
    no_w = int(np.argmax(counts))  # the fullest span gets no weight
    span = np.full(R, -1)
    for e in range(E):
        span[w.expert_offsets[e]:w.expert_offsets[e + 1]] = e
    z = np.zeros(E, np.uint64)
    # (a) LoRA off: a plain grouped matmul, rows without a weight untouched
    mats = {e: _bits(rng.standard_normal((N, K)) / np.sqrt(K)) for e in range(E) if e != no_w}
    W = _Weights(mats, E)
    lo, hi = 2, R - 3
    ref, written, folded = o.grouped_gemm_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra,
                                                     W.table, z, z, st, w.base, K, w.max_rank,
                                                     N, w.top_k, lo, hi)
    assert not folded.any()
    for r in range(R):
        e = span[r]
        if lo <= r < hi and e >= 0 and e != no_w:
            assert written[r]
            exp = _f(w.x_rows[r:r + 1]) @ _f(mats[e]).T
            assert np.allclose(ref[r], exp[0], rtol=1e-12, atol=1e-12), r
        else:
            assert not written[r] and np.array_equal(ref[r], _f(w.base[r])), r
    # (b) small integers: GEMM exact in bf16, then the fold on that base
    xi = _bits(rng.integers(-2, 3, (R, K)).astype(np.float32))
    mats_i = {e: _bits(rng.integers(-1, 2, (N, K)).astype(np.float32)) for e in range(E)
              if e != no_w}
    Wi = _Weights(mats_i, E)
    gemm = np.zeros((R, N), np.float64)
    for r in range(R):
        if span[r] >= 0 and span[r] != no_w:
            gemm[r] = _f(xi[r:r + 1]) @ _f(mats_i[span[r]]).T
    assert np.abs(gemm).max() < 256
    base_g = np.where((span >= 0) & (span != no_w), 1, 0)[:, None] * gemm
    base_bits = np.where(((span >= 0) & (span != no_w))[:, None], _bits(base_g), w.base)
    ref, written, folded = o.grouped_gemm_fold_xrows(xi, w.expert_offsets, w.src, ra, Wi.table,
                                                     at, bt, st, w.base, K, w.max_rank, N,
                                                     w.top_k, 0, R)
    ref_f, fold_f = o.grouped_fold_xrows(xi, w.expert_offsets, w.src, ra, at, bt, st, base_bits,
                                         K, w.max_rank, N, w.top_k, 0, R)
    assert folded.any() and (written & ~folded).any()
    assert np.array_equal(folded, fold_f & written)
    assert np.array_equal(ref[written], ref_f[written])
    assert np.array_equal(ref[~written], _f(w.base[~written]))
    # (c) permutation weights: out column n is x column perm_e[n] plus the delta
    perms = {e: rng.permutation(K) for e in range(E) if e != no_w}
    for p in perms.values():
        assert np.any(p[p] != np.arange(K))  # not an involution, so a transpose shows
    mats_p = {}
    for e, p in perms.items():
        m = np.zeros((N, K), np.float32)
        m[np.arange(N), p] = 1.0
        mats_p[e] = _bits(m)
    Wp = _Weights(mats_p, E)
    base_p = w.base.copy()
    for r in range(R):
        if span[r] >= 0 and span[r] != no_w:
            base_p[r] = w.x_rows[r, perms[span[r]]]
    ref, written, folded = o.grouped_gemm_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra,
                                                     Wp.table, at, bt, st, w.base, K,
                                                     w.max_rank, N, w.top_k, 0, R)
    ref_f, fold_f = o.grouped_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra, at, bt, st,
                                         base_p, K, w.max_rank, N, w.top_k, 0, R)
    assert np.array_equal(ref[written], ref_f[written])
    assert np.array_equal(folded, fold_f & written)
    # the row-sampled entry point equals the corresponding rows of a windowed call
    lo, hi = 3, R - 5
    ref_w, wr_w, fo_w = o.grouped_gemm_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra,
                                                  W.table, at, bt, st, w.base, K, w.max_rank, N,
                                                  w.top_k, lo, hi)
    rows = np.array([0, 2, 3, 7, R - 6, R - 5, R - 1, 19, int(w.expert_offsets[no_w])], np.int32)
    ref_s, wr_s, fo_s = o.grouped_gemm_fold_xrows_rows(w.x_rows, w.expert_offsets, w.src, ra,
                                                       W.table, at, bt, st, w.base[rows], rows, K,
                                                       w.max_rank, N, w.top_k, lo, hi)
    assert np.array_equal(ref_s, ref_w[rows])
    assert np.array_equal(wr_s, wr_w[rows]) and np.array_equal(fo_s, fo_w[rows])


ALL_PINS = [
    pin_route_truth_table,
    pin_decode_maps,
    pin_host_maps,
    pin_pack,
    pin_windows,
    pin_wc,
    pin_row_token,
    pin_fold_unit_vectors,
    pin_fold_exact_integers,
    pin_fold_dense_matmul,
    pin_fold_skips_keep_input,
    pin_fold_linear_in_scale,
    pin_cross_form,
    pin_window_split,
    pin_router_is_one_entry_route,
    pin_sampled_rows_match_full,
    pin_xrows_forms,
    pin_multi_adapter,
    pin_gemm_fold,
]
