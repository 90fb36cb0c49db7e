"""Host arithmetic of bench.py on CPU: the algorithmic bytes and FLOPs of a
step, counted by hand on small workloads (each term of the count is built
independently here from the workload's arrays)."""
import numpy as np
import pytest

import bench
import oracle
from lora_moe_expert_gb300 import synth


def _tables(w, o):
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    n = w.n_adapters * w.n_experts_model if w.n_adapters else None
    return he.tables(o, length=n), he


def test_gather_bytes_count_hit_experts_and_active_tokens():
    o = oracle.get()
    w = synth.custom_gather(5, 12, 4, 10, 64, 96, 16, adapted_frac=0.6, base_frac=0.3, bad_ids=2)
    (at, bt, st), _ = _tables(w, o)
    ra = o.build_moe_row_adapter_decode(w.adapter_slots, w.padded_n, w.active, w.has_moe_lora)
    rows, folded, nbytes, flops = bench.algorithmic(w, ra, (at, bt, st))
    _, fold = o.gather_fold(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank, w.n_out,
                            w.top_k)
    f_rows = np.flatnonzero(fold)
    experts = np.unique(w.indices[f_rows]).size
    tokens = np.unique(f_rows // w.top_k).size
    E = at.size
    exp_bytes = (tokens * w.k_in * 2 + experts * w.max_rank * (w.k_in + w.n_out) * 2
                 + fold.sum() * w.n_out * 4 + rows * 4 + ra.size * 4 + E * 20)
    assert rows == w.rows and folded == fold.sum()
    assert nbytes == exp_bytes
    assert flops == 2 * fold.sum() * w.max_rank * (w.k_in + w.n_out)


def test_multi_adapter_bytes_count_hit_cells():
    o = oracle.get()
    E, S = 8, 3
    w = synth.custom_gather_multi(6, 10, 4, E, 64, 96, 16, S, adapted_frac=0.6, base_frac=0.2,
                                  bad_ids=1)
    (at, bt, st), _ = _tables(w, o)
    _, ra = o.build_moe_row_adapter_decode_multi(w.adapter_slots, w.padded_n, S, True)
    rows, folded, nbytes, _ = bench.algorithmic(w, ra, (at, bt, st))
    _, fold = o.gather_fold_multi(w.x, w.indices, ra, at, bt, st, w.base, w.k_in, w.max_rank,
                                  w.n_out, w.top_k, E, S)
    f_rows = np.flatnonzero(fold)
    cells = np.unique(ra[f_rows // w.top_k].astype(np.int64) * E + w.indices[f_rows]).size
    tokens = np.unique(f_rows // w.top_k).size
    exp_bytes = (tokens * w.k_in * 2 + cells * w.max_rank * (w.k_in + w.n_out) * 2
                 + fold.sum() * w.n_out * 4 + rows * 4 + ra.size * 4 + at.size * 20)
    assert folded == fold.sum() and nbytes == exp_bytes


@pytest.mark.parametrize("per_row_x", [False, True])
def test_grouped_bytes_count_x_per_token_or_per_row(per_row_x):
    o = oracle.get()
    w = synth.custom_grouped(7, [30, 20], 4, 6, 64, 96, 16, cap=40, adapted_frac=0.7,
                             stream_base=[0, 1], per_row_x=per_row_x)
    (at, bt, st), _ = _tables(w, o)
    ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
    rows, folded, nbytes, _ = bench.algorithmic(w, ra, (at, bt, st))
    if per_row_x:
        _, fold = o.grouped_fold_xrows(w.x_rows, w.expert_offsets, w.src, ra, at, bt, st, w.base,
                                       w.k_in, w.max_rank, w.n_out, w.top_k, 0, w.rows)
    else:
        _, fold = o.grouped_fold(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base, w.k_in,
                                 w.max_rank, w.n_out, w.top_k, 0, w.rows)
    f_rows = np.flatnonzero(fold)
    expert_of_row = np.repeat(np.arange(w.n_experts_model), np.diff(w.expert_offsets))
    experts = np.unique(expert_of_row[f_rows]).size
    n_x = fold.sum() if per_row_x else np.unique(w.src[f_rows] // w.top_k).size
    exp_bytes = (n_x * w.k_in * 2 + experts * w.max_rank * (w.k_in + w.n_out) * 2
                 + fold.sum() * w.n_out * 4 + rows * 4 + ra.size * 4 + at.size * 20
                 + (w.n_experts_model + 1) * 4)
    assert folded == fold.sum() and nbytes == exp_bytes
