"""GPU parity of mlg_grouped_gemm_fold_xrows (the expert GEMM with the fold in
its epilogue) against the fp64 oracle: every element of every row the call
writes within 4e-3 * max(1, |ref|) and the correctly rounded value away from
bf16 rounding boundaries, every other row (outside the range) bit-identical, guard rows
untouched."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import fold_harness as fh  # noqa: E402
import lora_moe_expert_gb300 as mlg  # noqa: E402
import oracle  # noqa: E402
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


def _check(w, prob, row_offset=None, row_end=None):
    ref, written, _ = fh.oracle_reference(w, row_offset=row_offset, row_end=row_end)
    stats = fh.check_fold(prob.base_bits(), w.base, ref, written)
    assert np.all(prob.guard_bits() == 0x7FC1), "guard rows changed"
    return stats, written


SHAPES = [
    # (lengths, top_k, experts, k_in, n_out, max_rank, cap, lora_frac, stream_base)
    ([37, 50], 2, 6, 72, 200, 8, 1000, 0.7, [0, 1]),
    ([300], 4, 5, 256, 512, 32, 128, 1.0, None),
    ([64, 64], 2, 3, 1000, 8, 48, 97, 1.0, None),
    ([150, 40], 6, 30, 520, 328, 64, 256, 0.5, [1, 0]),
    ([200, 300], 8, 64, 128, 136, 16, 1 << 20, 0.9, None),
    ([1], 1, 1, 64, 64, 8, 1, 1.0, None),
    ([600, 700], 8, 16, 768, 2048, 16, 8192, 1.0, None),
    ([90, 333], 4, 9, 136, 264, 24, 150, 0.8, [0, 1]),
    ([257, 129], 2, 5, 200, 520, 56, 4096, 1.0, None),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{sum(s[0])}x{s[1]}_{s[3]}_{s[4]}_r{s[5]}")
def test_gemm_fold_shapes(shape):
    from lora_moe_expert_gb300.device import FoldProblem

    lengths, K, E, k_in, n_out, r, cap, lora, sb = shape
    w = synth.custom_grouped(400 + k_in, lengths, K, E, k_in, n_out, r, cap=cap,
                             adapted_frac=lora, stream_base=sb, per_row_x=True, gemm_weights=True)
    prob = FoldProblem(w, guard_rows=3)
    prob.run()
    torch.cuda.synchronize()
    _, written = _check(w, prob)
    assert written.any()


def test_prefill_down_fused_full():
    """The benchmark's fused workload (the ~30K-row down projection with every
    expert's weight), every element."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.prefill_down_fused()
    prob = FoldProblem(w, guard_rows=2)
    prob.run()
    torch.cuda.synchronize()
    stats, written = _check(w, prob)
    assert written.all()


def test_plain_gemm_with_zero_lora_cells():
    """With every LoRA cell zero the call is the plain grouped expert GEMM."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(41, [120, 90], 4, 12, 256, 384, 16, cap=100, per_row_x=True,
                             gemm_weights=True)
    prob = FoldProblem(w, guard_rows=2)
    prob.run(lora=False)
    torch.cuda.synchronize()
    ref, written, _ = fh.oracle_reference(_without_lora(w))
    fh.check_fold(prob.base_bits(), w.base, ref, written)
    assert written.any()


def _without_lora(w):
    import copy

    w2 = copy.copy(w)
    w2.experts = [synth.Expert(e.expert_id, e.A * 0, e.B * 0, e.scale) for e in w.experts]
    return w2


def test_range_and_windows_bit_exact_in_cap():
    """A sub-range keeps every row outside it; the result does not depend on
    the window length (each row's arithmetic is independent of its tile)."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(43, [150, 110], 4, 10, 192, 264, 32, cap=64, adapted_frac=0.8,
                             stream_base=[0, 1], per_row_x=True, gemm_weights=True)
    lo, hi = 37, w.rows - 29
    outs = []
    for cap in (64, 1000, 7):
        prob = FoldProblem(w, guard_rows=2)
        mlg.mlg_grouped_gemm_fold_xrows(prob.x_rows, prob.expert_offsets, prob.src,
                                        prob.row_adapter, prob.w_experts, prob.a_table,
                                        prob.b_table, prob.scale_table, prob.base, w.k_in,
                                        w.max_rank, w.n_out, w.top_k, prob.n_experts, lo, hi, cap)
        torch.cuda.synchronize()
        _, written = _check(w, prob, row_offset=lo, row_end=hi)
        assert not written[:lo].any() and not written[hi:].any()
        outs.append(prob.base_bits())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_negative_src_rows_get_the_gemm_only():
    """A negative src entry folds no delta, but its row still gets the GEMM."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(44, [120], 3, 6, 128, 128, 8, cap=1000, per_row_x=True,
                             gemm_weights=True)
    neg = np.array([0, 5, 77, w.rows - 1])
    w.src = w.src.copy()
    w.src[neg] = -1
    prob = FoldProblem(w)
    prob.run(use_row_map=False)
    torch.cuda.synchronize()
    o = oracle.get()
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o, length=prob.n_experts)
    wt, keep = fh.weight_table(w, prob.n_experts)
    ref, written, folded = o.grouped_gemm_fold_xrows(w.x_rows, w.expert_offsets, w.src, None,
                                                     wt, at, bt, st, w.base, w.k_in, w.max_rank,
                                                     w.n_out, w.top_k, 0, w.rows)
    assert written[neg].all() and not folded[neg].any() and folded.sum() > 100
    fh.check_fold(prob.base_bits(), w.base, ref, written)


def test_exact_integers_bit_identical():
    """Small integers everywhere, a power-of-two scale: every value is exact in
    fp32, so each output is the correctly rounded exact value, bit for bit."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(45, [90, 70], 4, 8, 128, 160, 16, cap=64, adapted_frac=0.75,
                             stream_base=[0, 1], per_row_x=True, gemm_weights=True)
    rng = np.random.default_rng(46)
    b16 = lambda a: synth.bf16_bits(np.asarray(a, np.float32))  # noqa: E731
    w.x_rows = b16(rng.integers(-2, 3, w.x_rows.shape))
    w.weights = b16(rng.integers(-1, 2, w.weights.shape))
    for e in w.experts:
        e.A = b16(rng.integers(-1, 2, e.A.shape))
        e.B = b16(rng.integers(-1, 2, e.B.shape))
        e.scale = 0.25
    w.base = b16(rng.integers(-50, 50, w.base.shape))
    prob = FoldProblem(w)
    prob.run()
    torch.cuda.synchronize()
    ref, written, _ = fh.oracle_reference(w)
    rne, _ = fh.rne_bf16_f64(ref[written])
    got = prob.base_bits()
    assert np.array_equal(got[written], rne)
    assert np.array_equal(got[~written], w.base[~written])


def test_graph_replay_matches_eager():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_grouped(47, [300, 200], 8, 32, 256, 512, 32, cap=1000, per_row_x=True,
                             gemm_weights=True)
    prob = FoldProblem(w)
    prob.run()
    torch.cuda.synchronize()
    eager = prob.base_bits()
    prob.reset()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            prob.run(stream=s)
    prob.reset()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(prob.base_bits(), eager)


def test_prefill_large_fused_full():
    """The expert GEMM with the fold at the large prefill's scale (163840 sorted
    rows, 512 experts, W_e 2048 x 512, rank 32), in the benchmark's launch
    configuration, checked in every element: the oracle (all host cores)
    computes every sorted row in chunks."""
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.prefill_large_fused()
    prob = FoldProblem(w, guard_rows=2)
    prob.run()
    torch.cuda.synchronize()
    got = prob.base_bits()
    assert np.all(prob.guard_bits() == 0x7FC1), "guard rows changed"
    o = oracle.get()
    o.set_threads(0)
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o, length=prob.n_experts)
    wt, keep = fh.weight_table(w, prob.n_experts)
    ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
    chunk = 16384
    for r0 in range(0, w.rows, chunk):
        rows = np.arange(r0, min(r0 + chunk, w.rows), dtype=np.int32)
        ref, written, folded = o.grouped_gemm_fold_xrows_rows(
            w.x_rows, w.expert_offsets, w.src, ra, wt, at, bt, st, w.base[rows], rows, w.k_in,
            w.max_rank, w.n_out, w.top_k, 0, w.rows)
        assert written.all() and folded.all()
        fh.check_fold(got[rows], w.base[rows], ref, written)
