"""The oracle's row loops run on OpenMP threads; this checks that the thread
count changes no bit of any result.

Each output row is computed by one thread in the serial order of operations,
so a threaded run must give exactly the single-threaded fp64 values (and the
same folded flags) on the tiny decode batch, the 64 x top-8 down-projection
decode batch and the ~30K-row prefill.  The sampled-row entry points are
checked the same way."""
import numpy as np
import pytest

import fold_harness as fh
import oracle
from lora_moe_expert_gb300 import synth


@pytest.fixture(scope="module")
def o():
    orc = oracle.get()
    yield orc
    orc.set_threads(0)


def _run(o, w, threads):
    assert o.set_threads(threads) >= 1
    ref, folded, keep = fh.oracle_reference(w, o)
    return ref, folded, keep


@pytest.mark.parametrize("gen", [synth.tiny_decode, synth.decode_down, synth.prefill_down],
                         ids=["tiny_decode", "decode_down", "prefill_down"])
def test_threaded_oracle_is_bit_identical(o, gen):
    w = gen()
    ref1, f1, _ = _run(o, w, 1)
    ref_n, f_n, _ = _run(o, w, 0)
    assert np.array_equal(f1, f_n)
    assert np.array_equal(ref1.view(np.uint64), ref_n.view(np.uint64))


def test_threaded_sampled_rows_bit_identical(o):
    w = synth.custom_grouped(12, [300, 200, 150], 6, 40, 256, 384, 32, cap=200,
                             adapted_frac=0.7)
    he = oracle.HostExperts([(e.expert_id, e.A, e.B, e.scale) for e in w.experts])
    at, bt, st = he.tables(o)
    ra = o.build_moe_row_adapter_host(w.cu_seqlens, w.stream_slots)
    rows = np.arange(w.rows, dtype=np.int32)
    out = []
    for threads in (1, 0):
        o.set_threads(threads)
        out.append(o.grouped_fold_rows(w.x, w.expert_offsets, w.src, ra, at, bt, st, w.base,
                                       rows, w.k_in, w.max_rank, w.n_out, w.top_k, 0, w.rows))
    assert np.array_equal(out[0][1], out[1][1])
    assert np.array_equal(out[0][0].view(np.uint64), out[1][0].view(np.uint64))
