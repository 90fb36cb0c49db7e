"""Planted mistakes in copies of the oracle must each trip at least one pin.

Every mutant below is a plausible slip (a transposed operand, a dropped term,
a wrong sign or index, a wrong rule order).  The copy is compiled on the CPU
into a temporary directory; the real oracle source is never modified.
Mutants that would read or write out of bounds are deliberately not planted.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "A transposed": ("A[(int64_t)j * k_in + k]", "A[(int64_t)k * max_rank + j]"),
    "B transposed": ("B[(int64_t)n * max_rank + j]", "B[(int64_t)j * n_out + n]"),
    "scale dropped": ("bf16_value(base_row[n]) + scale * d", "bf16_value(base_row[n]) + d"),
    "delta sign": ("bf16_value(base_row[n]) + scale * d", "bf16_value(base_row[n]) - scale * d"),
    "base dropped": ("ref_row[n] = bf16_value(base_row[n]) + scale * d", "ref_row[n] = scale * d"),
    "last k dropped": ("for (int32_t k = 0; k < k_in; ++k)", "for (int32_t k = 0; k + 1 < k_in; ++k)"),
    "last rank dropped": ("for (int32_t j = 0; j < max_rank; ++j) d +=",
                          "for (int32_t j = 0; j + 1 < max_rank; ++j) d +="),
    "token = row % top_k": ("int32_t t = row / top_k;", "int32_t t = row % top_k;"),
    "row map sign": ("if (row_adapter[t] < 0 || !expert_folds", "if (row_adapter[t] > 0 || !expert_folds"),
    "grouped x row unsorted": ("int32_t t = src[r] / top_k;\n            if (row_adapter != NULL && row_adapter[t] < 0) continue;\n            const",
                               "int32_t t = (int32_t)(r / top_k);\n            if (row_adapter != NULL && row_adapter[t] < 0) continue;\n            const"),
    "span start shifted": ("expert_offsets[e] > row_offset ? expert_offsets[e] : row_offset",
                           "expert_offsets[e] >= row_offset ? expert_offsets[e] + 1 : row_offset"),
    "bf16 decode": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "skip on slot <= 0": ("if (adapter_slot < 0) return ROUTE_SKIP;", "if (adapter_slot <= 0) return ROUTE_SKIP;"),
    "rule order": ("    if (!has_moe_lora) return ROUTE_FOLD;\n    if (adapter_slot < 0) return ROUTE_SKIP;",
                   "    if (adapter_slot < 0) return ROUTE_SKIP;\n    if (!has_moe_lora) return ROUTE_FOLD;"),
    "map writes slot": ("out[i] = (route == ROUTE_FOLD) ? active : -1;",
                        "out[i] = (route == ROUTE_FOLD) ? adapter_slots[i] : -1;"),
    "equal boundary rejected": ("cu[b + 1] < cu[b]) return OR_NONE;", "cu[b + 1] <= cu[b]) return OR_NONE;"),
    "first duplicate wins": ("for (int64_t i = 0; i < n; ++i) { /* in input order",
                             "for (int64_t i = n - 1; i >= 0; --i) { /* in input order"),
    "window not clipped": ("if (end > total_rows) end = total_rows;", ";"),
    "wc not at least 1": ("return wc < 1 ? 1u : (uint32_t)wc;", "return (uint32_t)wc;"),
    "x_rows read by token": ("fold_one_row(x_rows + r * k_in", "fold_one_row(x_rows + (int64_t)(src[r] / top_k) * k_in"),
    "x_rows row map by sorted row": ("row_adapter[src[r] / top_k] < 0) continue;\n            fold_one_row(x_rows",
                                     "row_adapter[r / top_k] < 0) continue;\n            fold_one_row(x_rows"),
    "sampled x_rows by token": ("fold_one_row(x_rows + (int64_t)r * k_in",
                                "fold_one_row(x_rows + (int64_t)(src[r] / top_k) * k_in"),
    "multi cell expert-major": ("int64_t cell = (int64_t)s * n_experts + e;",
                                "int64_t cell = (int64_t)e * n_adapters + s;"),
    "multi map writes slot 0": ("adapter_slots[i] >= 0) entry = adapter_slots[i];",
                                "adapter_slots[i] >= 0) entry = 0;"),
    "multi refusal dropped": ("if (adapter_slots[i] >= n_adapters) return OR_REFUSE;", ";"),
    "multi base requests kept": ("if (has_moe_lora && i < n_slots && adapter_slots[i] >= 0)",
                                 "if (has_moe_lora && i < n_slots)"),
    "gemm W transposed": ("g += bf16_value(xr[k]) * bf16_value(W[(int64_t)n * k_in + k]);",
                          "g += bf16_value(xr[k]) * bf16_value(W[(int64_t)k * n_out + n]);"),
    "gemm last k dropped": ("for (int32_t k = 0; k < k_in; ++k)\n                    g +=",
                            "for (int32_t k = 0; k + 1 < k_in; ++k)\n                    g +="),
    "gemm delta unscaled": ("ref_row[n] += scale * d;", "ref_row[n] += d;"),
    "gemm row map slot 0 skipped": ("row_adapter[src[r] / top_k] >= 0);",
                                    "row_adapter[src[r] / top_k] > 0);"),
    "gemm weightless rows zeroed": (
        "if (w_table[e] == 0) continue;",
        "if (w_table[e] == 0) { for (int64_t q = lo; q < hi; ++q) "
        "for (int32_t n = 0; n < n_out; ++n) ref_out[q * n_out + n] = 0.0; continue; }"),
    "padding gets active": ("        } else {\n            out[i] = -1;\n        }",
                            "        } else {\n            out[i] = active;\n        }"),
}


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="mlg_oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


def _build(workdir, name, text):
    tag = "".join(c if c.isalnum() else "_" for c in name)
    src = os.path.join(workdir, f"{tag}.c")
    lib = os.path.join(workdir, f"lib{tag}.so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", lib, src], check=True)
    return oracle.Oracle(lib)


def _failing_pins(o):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


def test_unmutated_copy_passes(workdir):
    with open(oracle.SOURCE) as f:
        text = f.read()
    assert _failing_pins(_build(workdir, "clean", text)) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(workdir, name):
    with open(oracle.SOURCE) as f:
        text = f.read()
    old, new = MUTANTS[name]
    assert text.count(old) >= 1, f"mutation site not found: {old!r}"
    mutated = text.replace(old, new)
    failed = _failing_pins(_build(workdir, name, mutated))
    assert failed, f"no pin caught mutant {name!r}"
