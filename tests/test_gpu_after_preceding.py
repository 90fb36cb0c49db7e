"""Decode folds after a KERNEL that rewrites their tables or pair weights.

The decode folds read the expert tables and the A_e / B_e pairs before the
kernel ahead of them in the stream has completed (early start), so a caller
whose preceding kernel writes those must launch them with
MLG_FOLD_AFTER_PRECEDING.  Here elementwise torch kernels (not copies, which
are never overlapped) rewrite, right before the fold on the same stream,
(a) the tables, to point at another adapter's pairs, or (b) the pair weights
in place and the scales; the fold with the flag must match the oracle for
the new adapter.  Covers the resident-pair kernel, the cluster kernel and
the multi-adapter form."""
import copy

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


def _workload(case):
    if case == "resident":
        return synth.custom_gather(71, 64, 8, 96, 768, 2048, 16, base_frac=0.1), 1
    if case == "cluster":
        return synth.custom_gather(72, 48, 4, 24, 1024, 256, 64, base_frac=0.1), 2
    return synth.custom_gather_multi(73, 48, 8, 32, 512, 1024, 16, 3, adapted_frac=0.9,
                                     base_frac=0.2), 0


def _new_adapter(w, seed, same_ids):
    rng = np.random.default_rng(seed)
    ids = np.array([e.expert_id for e in w.experts])
    if not same_ids:
        n_table = int(ids.max()) + 1
        ids = np.sort(rng.choice(n_table, size=max(1, (2 * n_table) // 3), replace=False))
    w2 = copy.copy(w)
    w2.experts = synth._experts(rng, ids, w.k_in, w.max_rank, w.n_out)
    return w2


def _fold_ex(prob, stream):
    w = prob.w
    flags = mlg.MLG_FOLD_AFTER_PRECEDING
    if w.n_adapters:
        mlg.mlg_gather_bgmv_multi_ex(prob.x, prob.indices, prob.row_adapter, prob.a_table,
                                     prob.b_table, prob.scale_table, prob.base, w.rows, w.k_in,
                                     w.max_rank, w.n_out, w.top_k, w.n_experts_model,
                                     w.n_adapters, flags, stream=stream)
    else:
        mlg.mlg_gather_bgmv_ex(prob.x, prob.indices, prob.row_adapter, prob.a_table,
                               prob.b_table, prob.scale_table, prob.base, w.rows, w.k_in,
                               w.max_rank, w.n_out, w.top_k, prob.n_experts, flags,
                               stream=stream)


def _dev_tables(prob, pool):
    from lora_moe_expert_gb300.device import pad_tables

    a, b, sc = mlg.mlg_pack_expert_tables(pool.ids, pool.a_addr, pool.b_addr, pool.scale)
    a, b, sc = pad_tables(a, b, sc, prob.n_experts)
    dev = lambda v: torch.from_numpy(v.view(np.int64) if v.dtype == np.uint64 else v).cuda()  # noqa: E731
    return dev(a), dev(b), dev(sc)


@pytest.mark.parametrize("what", ["tables", "weights"])
@pytest.mark.parametrize("case", ["resident", "cluster", "multi"])
def test_fold_after_a_kernel_that_rewrites_tables_or_weights(case, what):
    from lora_moe_expert_gb300.device import ExpertPool, FoldProblem

    w, path = _workload(case)
    w2 = _new_adapter(w, 80 + len(case), same_ids=(what == "weights"))
    try:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, path)
        prob = FoldProblem(w)
        prob.run()  # a first fold with the old adapter (kernels loaded, caches warm)
        pool2 = ExpertPool(w2.experts, prob.device)
        a2, b2, s2 = _dev_tables(prob, pool2 if what == "tables" else prob.pool)
        if what == "weights":  # same cells, new scales
            s2 = torch.from_numpy(np.asarray(
                mlg.mlg_pack_expert_tables(pool2.ids, pool2.a_addr, pool2.b_addr,
                                           pool2.scale)[2])).cuda()
            s2 = torch.cat([s2, torch.zeros(prob.n_experts - s2.numel(), device=s2.device)])
            assert pool2.buffer.numel() == prob.pool.buffer.numel()
        torch.cuda.synchronize()
        prob.reset()
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            # elementwise kernels on the fold's stream, right before it
            if what == "tables":
                torch.bitwise_or(a2, 0, out=prob.a_table)
                torch.bitwise_or(b2, 0, out=prob.b_table)
            else:
                torch.bitwise_or(pool2.buffer, 0, out=prob.pool.buffer)
            torch.mul(s2, 1.0, out=prob.scale_table)
            _fold_ex(prob, s)
        s.synchronize()
    finally:
        mlg.mlg_test_set_knob(mlg.MLG_TEST_GATHER_PATH, 0)
    ref, folded, _ = fh.oracle_reference(w2)
    fh.check_fold(prob.base_bits(), w.base, ref, folded)
    assert folded.any()


def test_unknown_flag_is_rejected():
    from lora_moe_expert_gb300.device import FoldProblem

    w = synth.custom_gather(74, 8, 2, 8, 64, 64, 8)
    prob = FoldProblem(w)
    with pytest.raises(mlg.MlgError) as ei:
        mlg.mlg_gather_bgmv_ex(prob.x, prob.indices, prob.row_adapter, prob.a_table,
                               prob.b_table, prob.scale_table, prob.base, w.rows, w.k_in,
                               w.max_rank, w.n_out, w.top_k, prob.n_experts, 2)
    assert ei.value.status == mlg.MLG_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert np.array_equal(prob.base_bits(), w.base)
