"""GPU parity of mlg_grouped_down (prefill fold) and mlg_router_fold against the
fp64 oracle: every element of every row, the 163840-row prefill included,
folded elements within 4e-3 * max(1, |ref|), everything else bit-identical."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import fold_harness as fh  # noqa: E402
import oracle  # noqa: E402
import lora_moe_expert_gb300 as mlg  # noqa: E402
from lora_moe_expert_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mlg.lib()
    mlg.mlg_read_device_errors(clear=True)
    yield
    torch.cuda.synchronize()
    assert mlg.mlg_read_device_errors(clear=True) == 0


def _run_and_check(w, guard_rows=3):
    from lora_moe_expert_gb300.device import FoldProblem

    prob = FoldProblem(w, guard_rows=guard_rows)
    ref, folded, keep = fh.oracle_reference(w)
    assert keep[1] == prob.n_experts
    prob.run()
    torch.cuda.synchronize()
    stats = fh.check_fold(prob.base_bits(), w.base, ref, folded)
    assert np.all(prob.guard_bits() == 0x7FC1), "guard rows changed"
    return prob, stats, folded


def test_small_grouped_multiple_windows():
    w = synth.custom_grouped(5, [70, 130, 60], 4, 16, 256, 512, 32, cap=300, adapted_frac=0.8)
    _, stats, folded = _run_and_check(w)
    assert 0 < folded.sum() < folded.size


def test_prefill_down_full():
    _, stats, folded = _run_and_check(synth.prefill_down())
    assert folded.all()


GROUPED_SHAPES = [
    # (lengths, top_k, experts, k_in, n_out, max_rank, cap, adapted, stream_base)
    ([5, 9], 2, 4, 64, 64, 8, 1000, 1.0, None),
    ([33, 17, 80], 3, 7, 72, 72, 24, 50, 0.6, [0, 1, 0]),
    ([200], 4, 5, 200, 1000, 40, 128, 1.0, None),
    ([64, 64], 2, 3, 1000, 8, 48, 97, 1.0, None),
    ([150, 40], 6, 30, 520, 328, 64, 256, 0.5, [1, 0]),
    ([300], 8, 64, 128, 136, 16, 1 << 20, 0.9, None),
    ([1], 1, 1, 64, 64, 8, 1, 1.0, None),
]


@pytest.mark.parametrize("shape", GROUPED_SHAPES, ids=lambda s: f"{sum(s[0])}x{s[1]}_{s[3]}_{s[4]}_r{s[5]}")
def test_grouped_shapes(shape):
    lengths, K, E, k_in, n_out, r, cap, adapted, sb = shape
    w = synth.custom_grouped(200 + k_in, lengths, K, E, k_in, n_out, r, cap=cap,
                             adapted_frac=adapted, stream_base=sb)
    _run_and_check(w)


def test_smaller_true_rank_zero_padded():
    w = synth.custom_grouped(31, [100, 50], 4, 8, 256, 256, 64, cap=90, rank=20)
    _run_and_check(w)


def test_window_split_is_bit_exact():
    """Any window split gives the bits of one window (each row's arithmetic is
    independent of which tile it lands in)."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(8, [120, 260, 90], 4, 12, 192, 384, 32, cap=1 << 20,
                             adapted_frac=0.75, stream_base=[0, 1, 0])
    outs = []
    for cap in (1 << 20, 128, 77, 5):
        w.cap = cap
        prob = FoldProblem(w)
        prob.run(per_window=True)
        torch.cuda.synchronize()
        outs.append(prob.base_bits())
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    ref, folded, _ = fh.oracle_reference(w)
    fh.check_fold(outs[0], w.base, ref, folded)


@pytest.mark.parametrize("cap", [1 << 20, 8192, 300, 128, 77])
def test_all_windows_launch_matches_per_window(cap):
    """One launch over all windows gives the bits of one launch per window."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(14, [400, 700, 250], 8, 40, 256, 512, 32, cap=cap,
                             adapted_frac=0.8, stream_base=[0, 0, 1])
    outs = []
    for per_window in (True, False):
        prob = FoldProblem(w)
        prob.run(per_window=per_window)
        torch.cuda.synchronize()
        outs.append(prob.base_bits())
    assert np.array_equal(outs[0], outs[1])
    ref, folded, _ = fh.oracle_reference(w)
    fh.check_fold(outs[1], w.base, ref, folded)


def test_negative_zero_and_repeat():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(12, [90, 70], 4, 10, 128, 256, 16, cap=100, adapted_frac=0.6,
                             stream_base=[1, 0])
    w.base[::2] = 0x8000
    ref, folded, _ = fh.oracle_reference(w)
    prob = FoldProblem(w)
    prob.run()
    torch.cuda.synchronize()
    first = prob.base_bits()
    fh.check_fold(first, w.base, ref, folded)
    prob.reset()
    prob.run()
    torch.cuda.synchronize()
    assert np.array_equal(prob.base_bits(), first)


def test_router_small_and_row_map():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_router(6, 200, 512, 256, 32)
    _run_and_check(w)
    # with a row map: negative tokens keep their input
    prob = FoldProblem(w)
    ra_host = np.where(np.arange(200) % 3 == 0, -1, 0).astype(np.int32)
    ra = torch.from_numpy(ra_host).cuda()
    mlg.mlg_router_fold(prob.x, ra, prob.a_table, prob.b_table, prob.scale_table, prob.base,
                        w.rows, w.k_in, w.max_rank, w.n_out)
    torch.cuda.synchronize()
    o = oracle.get()
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    ref, folded = o.router_fold(w.x, ra_host, at, bt, st, w.base, w.k_in, w.max_rank, w.n_out)
    fh.check_fold(prob.base_bits(), w.base, ref, folded)


@pytest.mark.parametrize("shape", [(77, 72, 64, 8), (300, 200, 264, 16), (1000, 1000, 128, 32),
                                   (153, 520, 96, 64)], ids=lambda s: "x".join(map(str, s)))
def test_router_shapes(shape):
    """Ragged k tails (the x boxes read zeros past k_in), token counts that are
    not a multiple of the tile height, every rank bucket."""
    T, k_in, n_out, r = shape
    _run_and_check(synth.custom_router(40 + T, T, k_in, n_out, r))


def test_router_zero_cell_is_noop():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_router(7, 64, 128, 64, 16)
    prob = FoldProblem(w)
    zero = torch.zeros(1, dtype=torch.int64, device="cuda")
    mlg.mlg_router_fold(prob.x, None, zero, prob.b_table, prob.scale_table, prob.base, w.rows,
                        w.k_in, w.max_rank, w.n_out)
    torch.cuda.synchronize()
    assert np.array_equal(prob.base_bits(), w.base)


def test_router_full():
    _, stats, folded = _run_and_check(synth.router())
    assert folded.all()


def test_prefill_large_full():
    """The 163840-row prefill at full size, in the window split and launch
    configuration the benchmark uses, checked in every element: the oracle
    (all host cores) folds every sorted row in chunks, each chunk compared
    with the GPU rows (every row folds here)."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.prefill_large()
    prob = FoldProblem(w, guard_rows=2)
    prob.run()
    torch.cuda.synchronize()
    got_all = prob.base_bits()
    assert np.all(prob.guard_bits() == 0x7FC1), "guard rows changed"
    o = oracle.get()
    o.set_threads(0)
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
    chunk = 16384
    n_checked = 0
    for r0 in range(0, w.rows, chunk):
        rows = np.arange(r0, min(r0 + chunk, w.rows), dtype=np.int32)
        ref, folded = o.grouped_fold_rows(w.x, w.expert_offsets, w.src, ra, at, bt, st,
                                          w.base[rows], rows, w.k_in, w.max_rank, w.n_out,
                                          w.top_k, 0, w.rows)
        assert folded.all()
        fh.check_fold(got_all[rows], w.base[rows], ref, folded)
        n_checked += rows.size
    assert n_checked == w.rows


def test_cuda_graph_replay_matches_eager():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(3, [300, 200, 100], 8, 32, 256, 512, 32, cap=1000)
    prob = FoldProblem(w)
    prob.run()
    torch.cuda.synchronize()
    eager = prob.base_bits()
    prob.reset()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            prob.run(stream=s)
    prob.reset()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(prob.base_bits(), eager)


def test_grouped_matches_gather_form():
    """Cross-form: the same decode batch folded through the grouped kernel on
    expert-sorted rows equals the gather kernel's result un-permuted, within
    the tolerance (the two kernels sum in different orders)."""
    from lora_moe_expert_gb300.device import FoldProblem

    g = synth.custom_gather(41, 96, 4, 16, 256, 384, 32, adapted_frac=0.7, base_frac=0.2)
    gp = FoldProblem(g)
    gp.run()
    torch.cuda.synchronize()
    gather_out = gp.base_bits()
    offsets, src = synth.sort_rows_by_expert(g.indices, g.n_experts_model)
    row_map = gp.row_map_host
    sp = FoldProblem(g)  # reuse allocations for x / tables; sorted base below
    sorted_base = torch.from_numpy(g.base[src].view(np.int16)).cuda().view(torch.bfloat16)
    mlg.mlg_grouped_down(sp.x, torch.from_numpy(offsets).cuda(), torch.from_numpy(src).cuda(),
                         torch.from_numpy(row_map).cuda(), sp.a_table, sp.b_table,
                         sp.scale_table, sorted_base, g.k_in, g.max_rank, g.n_out, g.top_k,
                         sp.n_experts, 0, src.size)
    torch.cuda.synchronize()
    grouped_out = np.empty_like(gather_out)
    grouped_out[src] = sorted_base.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, folded, _ = fh.oracle_reference(g)
    fh.check_fold(grouped_out, g.base, ref, folded)
    fh.check_fold(gather_out, g.base, ref, folded)


# ------------------------------------------------ per-row x form (x_rows[r])
@pytest.mark.parametrize("shape", GROUPED_SHAPES, ids=lambda s: f"{sum(s[0])}x{s[1]}_{s[3]}_{s[4]}_r{s[5]}")
def test_xrows_shapes(shape):
    lengths, K, E, k_in, n_out, r, cap, adapted, sb = shape
    w = synth.custom_grouped(300 + k_in, lengths, K, E, k_in, n_out, r, cap=cap,
                             adapted_frac=adapted, stream_base=sb, per_row_x=True)
    _run_and_check(w)


def test_prefill_down_xrows_full():
    """The benchmark's per-row x workload at full size, every row checked."""
    _, stats, folded = _run_and_check(synth.prefill_down_xrows())
    assert folded.all()


def test_xrows_token_rows_match_token_form_bits():
    """x_rows holding each sorted row's token row gives the token form's bits
    (same tiles, same arithmetic; only the address of each X row differs)."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(16, [210, 90, 333], 6, 24, 320, 512, 32, cap=400,
                             adapted_frac=0.75, stream_base=[0, 1, 0])
    tok = FoldProblem(w)
    tok.run()
    torch.cuda.synchronize()
    w.x_rows = w.x[w.src // w.top_k]
    per_row = FoldProblem(w)
    per_row.run()
    torch.cuda.synchronize()
    assert np.array_equal(per_row.base_bits(), tok.base_bits())
    ref, folded, _ = fh.oracle_reference(w)
    fh.check_fold(per_row.base_bits(), w.base, ref, folded)


@pytest.mark.parametrize("lo_hi_cap", [(17, -9, 50), (0, -1, 1 << 20), (128, 0, 128), (3, -200, 7)])
def test_xrows_row_range_and_windows(lo_hi_cap):
    """A sub-range [row_offset, row_end) in windows of cap rows: rows outside
    keep their input (guard rows and all), rows inside match the oracle."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(18, [150, 260], 4, 12, 192, 256, 16, cap=64, adapted_frac=0.8,
                             stream_base=[1, 0], per_row_x=True)
    lo, hi, cap = lo_hi_cap
    hi = w.rows + hi if hi <= 0 else hi
    prob = FoldProblem(w, guard_rows=2)
    mlg.mlg_grouped_down_xrows(prob.x_rows, prob.expert_offsets, prob.src, prob.row_adapter,
                               prob.a_table, prob.b_table, prob.scale_table, prob.base, w.k_in,
                               w.max_rank, w.n_out, w.top_k, prob.n_experts, lo, hi, cap)
    torch.cuda.synchronize()
    ref, folded, _ = fh.oracle_reference(w, row_offset=lo, row_end=hi)
    assert not folded[:lo].any() and not folded[hi:].any()
    fh.check_fold(prob.base_bits(), w.base, ref, folded)
    assert np.all(prob.guard_bits() == 0x7FC1)


def test_xrows_negative_src_and_no_row_map():
    """Without a row map every row of a span folds; a negative src entry folds
    nothing (its row keeps its input)."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(19, [120], 3, 6, 128, 128, 8, cap=1000, per_row_x=True)
    prob = FoldProblem(w)
    src = w.src.copy()
    neg = np.array([0, 5, 77, w.rows - 1])
    src[neg] = -1
    mlg.mlg_grouped_down_xrows(prob.x_rows, prob.expert_offsets, torch.from_numpy(src).cuda(),
                               None, prob.a_table, prob.b_table, prob.scale_table, prob.base,
                               w.k_in, w.max_rank, w.n_out, w.top_k, prob.n_experts, 0, w.rows,
                               1000)
    torch.cuda.synchronize()
    o = oracle.get()
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    ref, folded = o.grouped_fold_xrows(w.x_rows, w.expert_offsets, w.src, None, at, bt, st,
                                       w.base, w.k_in, w.max_rank, w.n_out, w.top_k, 0, w.rows)
    folded[neg] = False
    ref[neg] = synth.bf16_to_f32(w.base[neg]).astype(np.float64)
    fh.check_fold(prob.base_bits(), w.base, ref, folded)


def test_multi_adapter_prefill_through_cell_sort():
    """The prefill form of the multi-adapter fold needs no kernel of its own:
    rows sorted by cell (slot * n_experts + expert) and the grouped fold over
    the n_adapters * n_experts spans of slot-major tables give the oracle's
    multi-adapter fold, row for row."""
    from lora_moe_expert_gb300.device import FoldProblem

    E, S = 12, 3
    w = synth.custom_gather_multi(61, 150, 4, E, 256, 320, 32, S, adapted_frac=0.75,
                                  base_frac=0.2, bad_ids=3)
    prob = FoldProblem(w)  # x, slot-major tables (S * E cells), per-token slots as the row map
    slots = w.adapter_slots.astype(np.int64)
    tok = np.arange(w.rows) // w.top_k
    idx = w.indices.astype(np.int64)
    ok = (slots[tok] >= 0) & (idx >= 0) & (idx < E)
    key = np.where(ok, slots[tok] * E + idx, S * E)  # rows of no cell sort past the table
    offsets, src = synth.sort_rows_by_expert(key, S * E + 1)
    sorted_base = torch.from_numpy(w.base[src].view(np.int16)).cuda().view(torch.bfloat16)
    row_map = torch.from_numpy(w.adapter_slots.astype(np.int32)).cuda()
    mlg.mlg_grouped_down(prob.x, torch.from_numpy(offsets).cuda(), torch.from_numpy(src).cuda(),
                         row_map, prob.a_table, prob.b_table, prob.scale_table, sorted_base,
                         w.k_in, w.max_rank, w.n_out, w.top_k, prob.n_experts, 0, w.rows)
    torch.cuda.synchronize()
    got = np.empty_like(w.base)
    got[src] = sorted_base.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, folded, _ = fh.oracle_reference(w)
    assert 0 < folded.sum() < folded.size
    fh.check_fold(got, w.base, ref, folded)


@pytest.mark.parametrize("per_row_x", [False, True], ids=["token_x", "row_x"])
def test_inputs_written_by_the_preceding_kernel(per_row_x):
    """x and the expert spans are rewritten on the stream right before the
    fold (by kernels the fold may overlap): the fold uses the new values."""
    import copy

    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(71, [300, 180, 250], 6, 24, 256, 512, 32, cap=400,
                             adapted_frac=0.8, per_row_x=per_row_x)
    w2 = copy.deepcopy(w)
    rng = np.random.default_rng(5)
    if per_row_x:
        w2.x_rows = synth.bf16_bits(rng.standard_normal(w.x_rows.shape).astype(np.float32))
    else:
        w2.x = synth.bf16_bits(rng.standard_normal(w.x.shape).astype(np.float32))
    prob = FoldProblem(w)
    xt = prob.x_rows if per_row_x else prob.x
    x_new = torch.from_numpy((w2.x_rows if per_row_x else w2.x).view(np.int16)).cuda()
    off_new = prob.expert_offsets.clone()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    for _ in range(3):
        prob.reset()
        xt.view(torch.int16).zero_()
        xt.view(torch.int16).add_(x_new)
        prob.expert_offsets.zero_()
        prob.expert_offsets.add_(off_new)
        prob.run(stream=s)
    torch.cuda.synchronize()
    ref, folded, _ = fh.oracle_reference(w2)
    fh.check_fold(prob.base_bits(), w2.base, ref, folded)
