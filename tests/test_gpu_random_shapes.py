"""Seeded random shape sweep of every fold form against the fp64 oracle.

The hand-picked shapes of the other GPU tests cover the edges each kernel is
known to have; this sweep draws further shapes from a fixed seed (k_in and
n_out multiples of 8 up to 1024, max_rank 8..64, ragged row counts, window
caps from one row to none, partial adapter coverage, base requests, padding
and out-of-range ids) so that ring plans, tile heights and fallback paths
chosen at run time meet shapes nobody chose.  Every element is checked as in
the other parity tests: folded elements within 4e-3 * max(1, |ref|) and
correctly rounded away from bf16 rounding boundaries, everything else
bit-identical, guard rows untouched."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import fold_harness as fh  # noqa: E402
import lora_moe_expert_gb300 as mlg  # noqa: E402
from lora_moe_expert_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

N_DRAWS = 16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mlg.lib()
    mlg.mlg_read_device_errors(clear=True)
    yield
    torch.cuda.synchronize()
    assert mlg.mlg_read_device_errors(clear=True) == 0


def _dims(rng):
    k_in = 8 * int(rng.integers(1, 129))
    n_out = 8 * int(rng.integers(1, 129))
    r = 8 * int(rng.integers(1, 9))
    return k_in, n_out, r


def _run(w, row_offset=None, row_end=None):
    from lora_moe_expert_gb300.device import FoldProblem

    prob = FoldProblem(w, guard_rows=2)
    ref, folded, keep = fh.oracle_reference(w, row_offset=row_offset, row_end=row_end)
    prob.run()
    torch.cuda.synchronize()
    fh.check_fold(prob.base_bits(), w.base, ref, folded)
    assert np.all(prob.guard_bits() == 0x7FC1), "guard rows changed"
    return folded


def _gather_shape(i):
    rng = np.random.default_rng(7100 + i)
    k_in, n_out, r = _dims(rng)
    T = int(rng.integers(1, 97))
    E = int(rng.integers(1, 161))
    return dict(seed=7200 + i, n_tokens=T, top_k=int(rng.integers(1, min(8, E) + 1)),
                n_experts=E, k_in=k_in, n_out=n_out, max_rank=r,
                adapted_frac=float(rng.uniform(0.3, 1.0)), base_frac=float(rng.uniform(0, 0.3)),
                pad=int(rng.integers(0, min(3, T - 1) + 1)), bad_ids=int(rng.integers(0, 3)))


def _multi_shape(i):
    rng = np.random.default_rng(7300 + i)
    k_in, n_out, r = _dims(rng)
    E = int(rng.integers(4, 49))
    return dict(seed=7400 + i, n_tokens=int(rng.integers(1, 97)),
                top_k=int(rng.integers(1, min(8, E) + 1)), n_experts=E, k_in=k_in, n_out=n_out,
                max_rank=r, n_adapters=int(rng.integers(2, 6)),
                adapted_frac=float(rng.uniform(0.4, 1.0)),
                base_frac=float(rng.uniform(0, 0.3)), bad_ids=int(rng.integers(0, 3)))


def _grouped_shape(i, base_seed):
    rng = np.random.default_rng(base_seed + i)
    k_in, n_out, r = _dims(rng)
    n_streams = int(rng.integers(1, 5))
    lengths = [int(v) for v in rng.integers(1, 401, n_streams)]
    cap = int(rng.choice([int(rng.integers(1, 2001)), 1 << 20]))
    sb = [int(v) for v in rng.integers(0, 2, n_streams)] if rng.random() < 0.5 else None
    E = int(rng.integers(1, 65))
    return dict(seed=base_seed + 100 + i, lengths=lengths,
                top_k=int(rng.integers(1, min(8, E) + 1)), n_experts=E, k_in=k_in, n_out=n_out,
                max_rank=r, cap=cap,
                adapted_frac=float(rng.uniform(0.4, 1.0)), stream_base=sb)


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_gather(i):
    _run(synth.custom_gather(**_gather_shape(i)))


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_gather_multi(i):
    _run(synth.custom_gather_multi(**_multi_shape(i)))


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_grouped_token_x(i):
    _run(synth.custom_grouped(**_grouped_shape(i, 7500)))


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_grouped_per_row_x(i):
    _run(synth.custom_grouped(**_grouped_shape(i, 7700), per_row_x=True))


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_router(i):
    rng = np.random.default_rng(7900 + i)
    k_in, n_out, r = _dims(rng)
    _run(synth.custom_router(8000 + i, int(rng.integers(1, 3001)), k_in, n_out, r))


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_gemm_fold(i):
    w = synth.custom_grouped(**_grouped_shape(i, 8100), per_row_x=True, gemm_weights=True)
    written = _run(w)
    assert written.any()
