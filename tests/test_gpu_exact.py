"""Exactly checkable folds on the GPU: bit-identical to the oracle.

x, A_e and B_e hold small integers (sparse +-1 rows) and every scale is a
power of two, so h, the expand sum and base + scale * delta are exact in fp32
and representable in bf16; the fold then has one correct bf16 answer and every
kernel must produce it bit for bit (no tolerance), in every folded element,
while unfolded elements keep their input bits.
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


def _sparse_pm1(rng, rows, cols, nnz):
    m = np.zeros((rows, cols), np.float32)
    for i in range(rows):
        pos = rng.choice(cols, size=min(nnz, cols), replace=False)
        m[i, pos] = rng.choice([-1.0, 1.0], size=pos.size)
    return m


def integerize(w, seed):
    """Make a workload exactly checkable: |h| <= 2, |delta| <= 4, scale in
    {1/2, 2}, base integers in [-64, 64] -> every result is a bf16 value."""
    rng = np.random.default_rng(seed)
    w.x = synth.bf16_bits(rng.integers(-1, 2, w.x.shape).astype(np.float32))
    if w.x_rows is not None:
        w.x_rows = synth.bf16_bits(rng.integers(-1, 2, w.x_rows.shape).astype(np.float32))
    w.base = synth.bf16_bits(rng.integers(-64, 65, w.base.shape).astype(np.float32))
    for i, e in enumerate(w.experts):
        e.A = synth.bf16_bits(_sparse_pm1(rng, w.max_rank, w.k_in, 2))
        e.B = synth.bf16_bits(_sparse_pm1(rng, w.n_out, w.max_rank, 2))
        e.scale = 0.5 if i % 2 else 2.0
    return w


def _check_exact(w, run):
    from lora_moe_expert_gb300.device import FoldProblem

    prob = FoldProblem(w, guard_rows=2)
    run(prob)
    torch.cuda.synchronize()
    ref, folded, _ = fh.oracle_reference(w)
    want = synth.bf16_bits(ref.astype(np.float32))
    # every reference value is exactly a bf16 value (a small multiple of 1/2)
    assert np.array_equal(synth.bf16_to_f32(want).astype(np.float64), ref)
    got = prob.base_bits()
    assert folded.any()
    assert np.array_equal(got[folded], want[folded])
    assert np.array_equal(got[~folded], w.base[~folded])
    assert np.all(prob.guard_bits() == 0x7FC1)


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("shape", [(64, 8, 128, 256, 512, 16), (40, 4, 24, 192, 264, 32),
                                   (24, 4, 8, 128, 96, 64), (64, 4, 8, 128, 96, 64)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gather_exact(shape, path):
    T, K, E, k_in, n_out, r = shape
    w = integerize(synth.custom_gather(400 + T, T, K, E, k_in, n_out, r, adapted_frac=0.8,
                                       base_frac=0.2, bad_ids=2), 11)
    if path == 1 and r not in (16, 32):
        pytest.skip("the resident-pair kernel takes rank 16 or 32")
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, path)
        _check_exact(w, lambda prob: prob.run())
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 0)


@pytest.mark.parametrize("path", [0, 1, 2])
def test_gather_multi_exact(path):
    w = integerize(synth.custom_gather_multi(45, 40, 4, 32, 256, 264, 16, 4, adapted_frac=0.8,
                                             base_frac=0.2, bad_ids=2), 15)
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, path)
        _check_exact(w, lambda prob: prob.run())
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 0)


def test_gather_multi_halves_exact():
    """The multi-adapter form's second-round cells folded in column halves, bit-exact."""
    w = integerize(synth.custom_gather_multi(46, 96, 8, 128, 256, 512, 16, 4, adapted_frac=0.9),
                   16)
    _check_exact(w, lambda prob: prob.run())


def test_grouped_exact():
    w = integerize(synth.custom_grouped(31, [120, 70, 90], 4, 10, 192, 320, 32, cap=100,
                                        adapted_frac=0.7, stream_base=[0, 1, 0]), 12)
    _check_exact(w, lambda prob: prob.run())


def test_grouped_xrows_exact():
    w = integerize(synth.custom_grouped(33, [150, 60, 110], 6, 12, 256, 192, 32, cap=90,
                                        adapted_frac=0.7, stream_base=[1, 0, 0],
                                        per_row_x=True), 14)
    _check_exact(w, lambda prob: prob.run())


def test_router_exact():
    w = integerize(synth.custom_router(32, 300, 256, 192, 32), 13)
    _check_exact(w, lambda prob: prob.run())
