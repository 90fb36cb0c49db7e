"""GPU parity of mlg_gather_bgmv (decode fold) against the fp64 oracle.

Every element of every row is compared: folded elements within
4e-3 * max(1, |ref|), all other elements bit-identical, guard rows untouched.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import fold_harness as fh  # noqa: E402
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


def _run_and_check(w, guard_rows=3, tol=fh.TOL):
    from lora_moe_expert_gb300.device import FoldProblem

    prob = FoldProblem(w, guard_rows=guard_rows)
    ref, folded, keep = fh.oracle_reference(w)
    assert keep[1] == prob.n_experts  # both sides packed the same table length
    prob.run()
    torch.cuda.synchronize()
    stats = fh.check_fold(prob.base_bits(), w.base, ref, folded, tol)
    assert np.all(prob.guard_bits() == 0x7FC1), "guard rows changed"
    return prob, stats, folded


def test_tiny_decode():
    w = synth.tiny_decode()
    _, stats, folded = _run_and_check(w)
    # rows of token 0 slot 1 and token 2 slot 0 fold; id 9, ids 1/3 and the
    # Skip / Refuse tokens keep their input
    assert stats["folded_rows"] == int(folded.sum()) > 0


def test_decode_down_full():
    _, stats, folded = _run_and_check(synth.decode_down())
    assert folded.all()


def test_decode_gate_up_full():
    w = synth.decode_gate_up()
    _, stats, folded = _run_and_check(w)
    assert 0 < folded.sum() < folded.size


SHAPES = [
    # (tokens, top_k, experts, k_in, n_out, max_rank, adapted, base, pad, bad_ids)
    (7, 3, 5, 8, 8, 8, 1.0, 0.0, 0, 0),
    (13, 2, 6, 24, 40, 24, 0.7, 0.3, 2, 3),
    (33, 4, 4, 776, 136, 16, 1.0, 0.2, 0, 0),  # > 32 rows per expert, k tail
    (64, 2, 2, 200, 1000, 40, 1.0, 0.0, 0, 0),  # many row groups per expert
    (5, 8, 700, 264, 72, 56, 0.5, 0.0, 0, 2),  # table longer than the cluster cap
    (20, 6, 40, 4104, 48, 64, 0.6, 0.1, 3, 2),
    (9, 1, 4, 2048, 8200, 32, 1.0, 0.0, 0, 0),
    (1, 1, 1, 64, 64, 8, 1.0, 0.0, 0, 0),
    (64, 4, 8, 512, 256, 64, 1.0, 0.1, 0, 0),  # ~30 rows per expert: helper clusters
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:6])))
def test_gather_shapes(shape):
    T, K, E, k_in, n_out, r, adapted, base, pad, bad = shape
    w = synth.custom_gather(100 + T, T, K, E, k_in, n_out, r, adapted_frac=adapted,
                            base_frac=base, pad=pad, bad_ids=bad)
    _run_and_check(w)


def test_smaller_true_rank_zero_padded():
    w = synth.custom_gather(5, 16, 4, 8, 512, 256, 64, rank=20)
    _run_and_check(w)


@pytest.mark.parametrize("cs,ns2", [(1, 1), (2, 1), (4, 1), (8, 1), (1, 2), (1, 4), (1, 8),
                                    (2, 2), (4, 2)])
def test_split_configurations(cs, ns2):
    """Every split of an expert over CTAs (cluster k split cs, independent n
    split ns2) meets the tolerance, and repeats of one split are bit-exact
    (fixed-order reductions; only the k split, hence the fp32 summation
    order, differs between splits)."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_gather(77, 24, 8, 32, 1024, 512, 32, adapted_frac=0.8, base_frac=0.2)
    ref, folded, _ = fh.oracle_reference(w)
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_CLUSTER, cs)
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_NSPLIT, ns2)
        prob = FoldProblem(w)
        outs = []
        for _ in range(2):
            prob.reset()
            prob.run()
            torch.cuda.synchronize()
            outs.append(prob.base_bits())
        fh.check_fold(outs[0], w.base, ref, folded)
        assert np.array_equal(outs[0], outs[1])
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_CLUSTER, 0)
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_NSPLIT, 0)


def test_repeat_is_deterministic_and_negative_zero_kept():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_gather(9, 16, 4, 16, 256, 128, 16, adapted_frac=0.5, base_frac=0.4)
    w.base[::3] = 0x8000  # -0.0 in a third of the rows
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
    assert np.all(first[~folded][::3] == w.base[~folded][::3])


def test_cuda_graph_replay_matches_eager():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.decode_down()
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


def test_device_side_errors_are_status_codes():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.tiny_decode()
    prob = FoldProblem(w)
    with pytest.raises(mlg.MlgError) as ei:
        mlg.mlg_gather_bgmv(prob.x.data_ptr() + 2, prob.indices, prob.row_adapter, prob.a_table,
                            prob.b_table, prob.scale_table, prob.base, w.rows, w.k_in,
                            w.max_rank, w.n_out, w.top_k, prob.n_experts)
    assert ei.value.status == mlg.MLG_ERR_UNSUPPORTED
    assert np.array_equal(prob.base_bits(), w.base)


# Shapes the resident-pair kernel takes (max_rank 16 or 32, n_out <= 2048, at
# most one expert per SM); each runs through both kernels.
RESIDENT_SHAPES = [
    # (tokens, top_k, experts, k_in, n_out, max_rank, adapted, base, pad, bad_ids)
    (33, 4, 4, 776, 136, 16, 1.0, 0.2, 0, 0),  # > 32 rows per expert, k and n tails
    (40, 6, 12, 200, 1000, 32, 0.7, 0.2, 3, 2),  # zero cells, skipped and padded tokens
    (3, 2, 152, 64, 2048, 16, 1.0, 0.0, 0, 0),  # one expert per SM, most without rows
    (50, 4, 9, 1032, 40, 32, 0.5, 0.3, 1, 1),  # one partial 32-column quad
    (1, 1, 1, 32, 8, 16, 1.0, 0.0, 0, 0),  # smallest
    (96, 8, 128, 1024, 512, 16, 0.9, 0.1, 2, 3),  # long k, many rows
    (64, 2, 8, 256, 512, 16, 1.0, 0.0, 0, 0),  # 16 rows per expert: a helper CTA each
    (96, 4, 6, 128, 264, 32, 0.8, 0.1, 1, 1),  # ~64 rows per expert: many passes
]


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("shape", RESIDENT_SHAPES, ids=lambda s: "x".join(map(str, s[:6])))
def test_resident_and_cluster_kernels(shape, path):
    T, K, E, k_in, n_out, r, adapted, base, pad, bad = shape
    w = synth.custom_gather(300 + T, T, K, E, k_in, n_out, r, adapted_frac=adapted,
                            base_frac=base, pad=pad, bad_ids=bad)
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, path)
        _run_and_check(w)
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 0)


@pytest.mark.parametrize("multi", [False, True], ids=["single", "multi"])
@pytest.mark.parametrize("mode", [1, 2])
def test_speculation_modes_give_the_same_bits(mode, multi):
    """Row lists (multi-adapter form: first cells) picked before the preceding
    kernel completes are checked after it: with no early scan (1) or an early
    scan that always disagrees (2, everything requested again) the bits are
    those of the default mode."""
    from lora_moe_expert_gb300.device import FoldProblem

    if multi:
        w = synth.custom_gather_multi(24, 48, 8, 64, 768, 1024, 16, 3, adapted_frac=0.9,
                                      base_frac=0.2)
    else:
        w = synth.custom_gather(21, 48, 8, 64, 768, 1024, 16, adapted_frac=0.9, base_frac=0.2)
    outs = []
    try:
        for m in (0, mode):
            mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_SPECULATION, m)
            prob = FoldProblem(w)
            prob.run()
            torch.cuda.synchronize()
            outs.append(prob.base_bits())
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_SPECULATION, 0)
    assert np.array_equal(outs[0], outs[1])
    ref, folded, _ = fh.oracle_reference(w)
    fh.check_fold(outs[1], w.base, ref, folded)


@pytest.mark.parametrize("multi", [False, True], ids=["single", "multi"])
def test_routing_written_by_the_preceding_kernel(multi):
    """The routing is rewritten on the stream right before the fold (by a
    kernel the fold may overlap): the fold uses the new routing."""
    import copy

    from lora_moe_expert_gb300.device import FoldProblem

    if multi:
        w = synth.custom_gather_multi(25, 64, 8, 128, 768, 2048, 16, 4)
    else:
        w = synth.custom_gather(22, 64, 8, 128, 768, 2048, 16)
    w2 = copy.deepcopy(w)
    w2.indices = np.roll(w.indices, 8 * 5).copy()  # another token order
    prob = FoldProblem(w)
    new_idx = torch.from_numpy(w2.indices.astype(np.int32)).cuda()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    for _ in range(3):
        prob.reset()
        prob.indices.fill_(-1)
        prob.indices.copy_(new_idx)
        prob.run(stream=s)
    torch.cuda.synchronize()
    ref, folded, _ = fh.oracle_reference(w2)
    fh.check_fold(prob.base_bits(), w2.base, ref, folded)


def test_resident_kernel_rejects_other_shapes():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_gather(23, 8, 2, 4, 128, 128, 64)
    prob = FoldProblem(w)
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 1)
        with pytest.raises(mlg.MlgError) as ei:
            prob.run()
        assert ei.value.status == mlg.MLG_ERR_UNSUPPORTED
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 0)
    assert np.array_equal(prob.base_bits(), w.base)


# ------------------------------------------------ multi-adapter tables
MULTI_SHAPES = [
    # (tokens, top_k, experts, k_in, n_out, rank, adapters, adapted, base_frac, bad_ids)
    (24, 4, 32, 256, 512, 16, 4, 0.8, 0.2, 2),
    (40, 4, 20, 192, 264, 32, 3, 0.7, 0.1, 1),
    (96, 6, 64, 1024, 512, 64, 3, 0.6, 0.15, 2),
    (32, 2, 8, 128, 96, 8, 5, 1.0, 0.0, 0),
    (7, 3, 16, 64, 64, 16, 2, 0.5, 0.3, 1),
]


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("shape", MULTI_SHAPES, ids=lambda s: "x".join(map(str, s[:7])))
def test_gather_multi(shape, path):
    T, K, E, k_in, n_out, r, S, adapted, bf, bad = shape
    w = synth.custom_gather_multi(500 + T, T, K, E, k_in, n_out, r, S, adapted_frac=adapted,
                                  base_frac=bf, bad_ids=bad)
    if path == 1 and r not in (16, 32):
        pytest.skip("the resident-pair kernel takes rank 16 or 32")
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, path)
        _, stats, folded = _run_and_check(w)
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 0)
    assert 0 < folded.sum()


def test_decode_down_multi_full():
    w = synth.decode_down_multi()
    _, stats, folded = _run_and_check(w)
    assert folded.all()


def test_multi_one_adapter_matches_single_bits():
    """One installed set: the multi-adapter call gives the single-set call's bits."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_gather(77, 48, 4, 24, 256, 320, 16, adapted_frac=0.8, base_frac=0.2,
                            bad_ids=2)
    single = FoldProblem(w)
    single.run()
    torch.cuda.synchronize()
    multi = FoldProblem(w)
    mlg.mlg_gather_bgmv_multi(multi.x, multi.indices, multi.row_adapter, multi.a_table,
                              multi.b_table, multi.scale_table, multi.base, w.rows, w.k_in,
                              w.max_rank, w.n_out, w.top_k, multi.n_experts, 1)
    torch.cuda.synchronize()
    assert np.array_equal(multi.base_bits(), single.base_bits())


def test_multi_large_tables_fall_back_to_the_cluster_kernel():
    """More cells than the multi-cell form takes (6 adapters x 300 experts):
    the cluster kernel folds them (no compaction past 512 cells), and forcing
    the resident-pair kernel is refused without touching base_out."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_gather_multi(81, 24, 4, 300, 128, 256, 16, 6, adapted_frac=0.3,
                                  base_frac=0.2, bad_ids=2)
    _run_and_check(w)
    prob = FoldProblem(w)
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 1)
        with pytest.raises(mlg.MlgError) as ei:
            prob.run()
        assert ei.value.status == mlg.MLG_ERR_UNSUPPORTED
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 0)
    assert np.array_equal(prob.base_bits(), w.base)


@pytest.mark.parametrize("n_out", [1024, 264], ids=["halves", "whole"])
def test_multi_second_round_cells(n_out):
    """More hit cells than CTAs: past the first round the cells are split into
    two column halves over two CTAs (n_out a multiple of 128) or dealt whole."""
    w = synth.custom_gather_multi(91, 96, 8, 128, 256, n_out, 16, 4, adapted_frac=0.9)
    _, stats, folded = _run_and_check(w)
    assert folded.sum() > 0


@pytest.mark.parametrize("case", ["all_base", "zero_tables", "multi_all_base", "grouped_all_base"])
def test_degenerate_batches_fold_nothing(case):
    """Batches where no row folds still launch and leave every bit of base_out
    (and the guard rows) as it was."""
    from lora_moe_expert_gb300.device import FoldProblem

    if case == "all_base":
        w = synth.custom_gather(61, 24, 4, 16, 256, 512, 16, base_frac=1.0)
    elif case == "multi_all_base":
        w = synth.custom_gather_multi(62, 24, 4, 16, 256, 512, 16, 3, base_frac=1.0)
    elif case == "grouped_all_base":
        w = synth.custom_grouped(63, [40, 70], 4, 12, 256, 512, 32, cap=64,
                                 stream_base=[1, 1])
    else:
        w = synth.custom_gather(64, 24, 4, 16, 256, 512, 16)
    prob = FoldProblem(w, guard_rows=2)
    if case == "zero_tables":
        prob.a_table.zero_()
        prob.b_table.zero_()
    ref, folded, _ = fh.oracle_reference(w)
    if case != "zero_tables":
        assert not folded.any()
    prob.run()
    torch.cuda.synchronize()
    assert np.array_equal(prob.base_bits(), w.base)
    assert np.all(prob.guard_bits() == 0x7FC1)
