"""Graph-stable adapter rotation: the expert tables are rewritten in place on
the device between replays of a captured CUDA graph, and the replay folds with
the new pairs without recapture (the kernels read table cells as data at run
time; nothing about the adapter is baked into the launch).  Each replay is
checked against the oracle run on that replay's experts."""
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


def _rotated(w, seed):
    """The same batch with another adapter: a different subset of expert ids
    (within the original table length) and fresh pairs and scales."""
    rng = np.random.default_rng(seed)
    n_table = max(e.expert_id for e in w.experts) + 1
    ids = np.sort(rng.choice(n_table, size=max(1, (2 * n_table) // 3), replace=False))
    if w.kind == "router":
        ids = np.array([0])
    w2 = copy.copy(w)
    w2.experts = synth._experts(rng, ids, w.k_in, w.max_rank, w.n_out)
    return w2


def _check(prob, w):
    ref, folded, _ = fh.oracle_reference(w)
    fh.check_fold(prob.base_bits(), w.base, ref, folded)


@pytest.mark.parametrize("case", ["decode_resident", "decode_cluster", "grouped", "router"])
def test_graph_replay_picks_up_rewritten_tables(case):
    from lora_moe_expert_gb300.device import ExpertPool, FoldProblem

    if case == "decode_resident":
        w = synth.custom_gather(51, 64, 8, 96, 512, 1024, 16, base_frac=0.1)
    elif case == "decode_cluster":
        w = synth.custom_gather(52, 48, 4, 24, 1024, 256, 64, base_frac=0.1)
    elif case == "grouped":
        w = synth.custom_grouped(53, [150, 90], 4, 12, 256, 384, 32, cap=200)
    else:
        w = synth.custom_router(54, 300, 512, 256, 32)
    prob = FoldProblem(w)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            prob.run(stream=s)
    keep = []
    for turn in range(3):
        cur = w if turn == 0 else _rotated(w, 60 + turn)
        if turn > 0:
            # new pairs in a new allocation; tables rewritten in place, same length
            pool = ExpertPool(cur.experts, prob.device)
            keep.append(pool)
            a, b, sc = mlg.mlg_pack_expert_tables(pool.ids, pool.a_addr, pool.b_addr, pool.scale)
            n = prob.n_experts
            assert a.size <= n
            pad = lambda v, dt: np.concatenate([v, np.zeros(n - v.size, dt)])  # noqa: E731
            mlg.mlg_upload_expert_tables(pad(a, np.uint64), pad(b, np.uint64),
                                         pad(sc, np.float32), prob.a_table, prob.b_table,
                                         prob.scale_table, stream=s)
        prob.reset()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        _check(prob, cur)
