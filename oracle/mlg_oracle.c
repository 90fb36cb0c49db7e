/*
 * mlg_oracle.c -- plain, slow, fp64 CPU oracle for the MoE expert LoRA fold.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is
 * compared against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load it.  The product library
 * (libmlg) never links, loads or calls it, and it shares no source with the
 * product: every rule below is restated here from the documentation pages.
 *
 * Sources (documentation pages of the "metrale" inference engine):
 *   [P1] moe_row_adapter.rs (metrale_model_layers/lora): resolve_moe_lora_route,
 *        ensure_decode_route_servable, build_moe_row_adapter_host,
 *        build_moe_row_adapter_decode.
 *   [P2] metrale_model_layers::layers::ops::moe_lora_grouped (module index):
 *        the module invariant on zero table cells and out-of-range ids,
 *        MoeExpertRoute (router fold = one-entry route), gather_row_token,
 *        grouped_down_wc, grouped_down_windows, moe_lora_gather_bgmv,
 *        moe_lora_grouped_down, pack_expert_tables.
 *
 * Arithmetic: every floating-point value is widened exactly to double and the
 * fold is evaluated as the plain definition
 *     ref[row, n] = base[row, n] + scale_e * sum_j (sum_k x[t,k] A_e[j,k]) B_e[n,j]
 * with no blocking, fusion or reordering.  The result is left unrounded so a
 * test can measure the distance of a rounded bf16 output from it.
 *
 * Expert tables hold addresses: a_table[e] / b_table[e] point at the expert's
 * A_e [max_rank, k_in] and B_e [n_out, max_rank] bf16 arrays (row-major, bf16
 * given as raw uint16 bit patterns).  For the oracle these are host
 * addresses of host copies; 0 means "no adapter for this expert".
 *
 * Status codes follow the library ABI's numbering so tests can compare them
 * directly: 0 ok, -1 invalid argument (the pages' None), -2 empty input,
 * -3 cap == 0 (the pages' panic), -4 refuse, -6 buffer too small.
 *
 * Threads: built with -fopenmp, the loops over output rows run in parallel
 * (OpenMP, oracle_set_threads).  Every row is computed by one thread with the
 * same sequence of operations as in a serial run, so the results are the same
 * bits for any thread count; only the wall time changes.  Built without
 * OpenMP the pragmas are ignored and the oracle is single-threaded.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_NONE (-1)
#define OR_EMPTY (-2)
#define OR_CAP_ZERO (-3)
#define OR_REFUSE (-4)
#define OR_TOO_SMALL (-6)

#define ROUTE_FOLD 0
#define ROUTE_SKIP 1
#define ROUTE_REFUSE 2

/* Threads used by the row loops (1 without OpenMP).  n < 1 selects every
 * core OpenMP reports.  Returns the thread count now in force. */
int32_t oracle_set_threads(int32_t n) {
#ifdef _OPENMP
    omp_set_num_threads(n >= 1 ? n : omp_get_num_procs());
    return (int32_t)omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* bf16 -> double, exact: a bf16 is the top half of an IEEE binary32. */
static double bf16_value(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* [P1] resolve_moe_lora_route, doc comment: the fold decision for one request.
 *   no MoE LoRA loaded -> Fold; base request (slot < 0) -> Skip;
 *   slot equal to the active adapter -> Fold; any other slot -> Refuse. */
int32_t oracle_resolve_moe_lora_route(int32_t adapter_slot, int32_t active, int32_t has_moe_lora) {
    if (!has_moe_lora) return ROUTE_FOLD;
    if (adapter_slot < 0) return ROUTE_SKIP;
    if (adapter_slot == active) return ROUTE_FOLD;
    return ROUTE_REFUSE;
}

/* [P1] ensure_decode_route_servable: an error exactly when the route is Refuse. */
int32_t oracle_ensure_decode_route_servable(int32_t route) {
    return route == ROUTE_REFUSE ? OR_REFUSE : OR_OK;
}

/* [P1] build_moe_row_adapter_decode: the [padded_n] decode map.  Entry i is
 * `active` when slot i exists and routes to Fold, and -1 for Skip, Refuse
 * and for padding entries (i at or past the number of slots). */
void oracle_build_moe_row_adapter_decode(const int32_t *adapter_slots, int64_t n_slots,
                                         int64_t padded_n, int32_t active, int32_t has_moe_lora,
                                         int32_t *out) {
    for (int64_t i = 0; i < padded_n; ++i) {
        if (i < n_slots) {
            int32_t route = oracle_resolve_moe_lora_route(adapter_slots[i], active, has_moe_lora);
            out[i] = (route == ROUTE_FOLD) ? active : -1;
        } else {
            out[i] = -1;
        }
    }
}

/* Multi-adapter decode map.  [P1] resolve_moe_lora_route refuses any slot
 * other than the active one because only the active adapter's pairs are
 * installed (ensure_decode_route_servable's message: one adapter per batch).
 * With one table set installed per slot 0 .. n_adapters - 1, the entry of a
 * request is its own slot when that slot has a set, and -1 for base requests
 * (slot < 0) and padding entries.  A slot at or past n_adapters has no set:
 * the whole batch is refused (OR_REFUSE) with nothing written, the same
 * refusal moved to the slots without tables.  With no MoE LoRA loaded
 * (has_moe_lora == 0) nothing folds: every entry is -1. */
int32_t oracle_build_moe_row_adapter_decode_multi(const int32_t *adapter_slots, int64_t n_slots,
                                                  int64_t padded_n, int32_t n_adapters,
                                                  int32_t has_moe_lora, int32_t *out) {
    if (has_moe_lora) {
        for (int64_t i = 0; i < n_slots && i < padded_n; ++i) {
            if (adapter_slots[i] >= n_adapters) return OR_REFUSE;
        }
    }
    for (int64_t i = 0; i < padded_n; ++i) {
        int32_t entry = -1;
        if (has_moe_lora && i < n_slots && adapter_slots[i] >= 0) entry = adapter_slots[i];
        out[i] = entry;
    }
    return OR_OK;
}

/* [P1] build_moe_row_adapter_host: the [total_tokens] prefill map.  `cu` is the
 * [batch + 1] prefix sum of stream lengths; stream b's slot is written
 * unchanged over rows cu[b] .. cu[b+1].  None (OR_NONE, nothing written) when
 * cu has fewer than two entries, the slot count is not batch, cu[0] != 0, or
 * any boundary is negative or decreasing -- all checked before sizing.
 * The size of the map is returned through *total_out on success; a buffer
 * shorter than that is OR_TOO_SMALL (nothing written). */
int32_t oracle_build_moe_row_adapter_host(const int32_t *cu, int64_t n_cu,
                                          const int32_t *adapter_slots, int64_t n_slots,
                                          int32_t *out, int64_t out_cap, int64_t *total_out) {
    if (n_cu < 2) return OR_NONE;
    int64_t batch = n_cu - 1;
    if (n_slots != batch) return OR_NONE;
    if (cu[0] != 0) return OR_NONE;
    for (int64_t b = 0; b < batch; ++b) {
        if (cu[b] < 0 || cu[b + 1] < cu[b]) return OR_NONE;
    }
    int64_t total = cu[batch];
    *total_out = total;
    if (out_cap < total) return OR_TOO_SMALL;
    for (int64_t r = 0; r < total; ++r) out[r] = -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t r = cu[b]; r < cu[b + 1]; ++r) out[r] = adapter_slots[b];
    }
    return OR_OK;
}

/* [P2] pack_expert_tables: dense tables indexed by expert id.  n_experts is
 * the largest id + 1, every id without an entry gets 0 / 0 / 0.0, a
 * duplicated id keeps its last entry, and empty input gives None (OR_EMPTY). */
int32_t oracle_pack_expert_tables(const uint32_t *ids, const uint64_t *a_addr,
                                  const uint64_t *b_addr, const float *scale, int64_t n,
                                  uint64_t *a_out, uint64_t *b_out, float *scale_out,
                                  int64_t out_cap, int64_t *n_experts_out) {
    if (n == 0) return OR_EMPTY;
    uint32_t max_id = 0;
    for (int64_t i = 0; i < n; ++i)
        if (ids[i] > max_id) max_id = ids[i];
    int64_t n_experts = (int64_t)max_id + 1;
    *n_experts_out = n_experts;
    if (out_cap < n_experts) return OR_TOO_SMALL;
    for (int64_t e = 0; e < n_experts; ++e) {
        a_out[e] = 0;
        b_out[e] = 0;
        scale_out[e] = 0.0f;
    }
    for (int64_t i = 0; i < n; ++i) { /* in input order, so the last duplicate wins */
        a_out[ids[i]] = a_addr[i];
        b_out[ids[i]] = b_addr[i];
        scale_out[ids[i]] = scale[i];
    }
    return OR_OK;
}

/* [P2] grouped_down_windows: contiguous [start, end) windows of at most `cap`
 * rows covering 0 .. total_rows; cap == 0 is the pages' panic (OR_CAP_ZERO).
 * Read: window i is [i*cap, min((i+1)*cap, total)).  Returns the number of
 * windows, or a negative status.  Windows past out_cap are counted, not
 * written. */
int64_t oracle_grouped_down_windows(uint32_t total_rows, uint32_t cap, uint32_t *starts,
                                    uint32_t *ends, int64_t out_cap) {
    if (cap == 0) return OR_CAP_ZERO;
    int64_t count = 0;
    uint64_t start = 0;
    while (start < total_rows) {
        uint64_t end = start + cap;
        if (end > total_rows) end = total_rows;
        if (count < out_cap) {
            starts[count] = (uint32_t)start;
            ends[count] = (uint32_t)end;
        }
        ++count;
        start = end;
    }
    return count;
}

/* [P2] grouped_down_wc: grid.y of the grouped fold for a window,
 * ceil((row_end - row_offset) / m_tile), at least 1.  The tile height is a
 * parameter here: the pages do not print MLG_M_TILE's value. */
uint32_t oracle_grouped_down_wc(uint32_t row_offset, uint32_t row_end, uint32_t m_tile) {
    uint64_t len = (row_end > row_offset) ? (uint64_t)(row_end - row_offset) : 0;
    uint64_t wc = 0;
    while (wc * m_tile < len) ++wc; /* ceil by counting, no division shortcut */
    return wc < 1 ? 1u : (uint32_t)wc;
}

/* [P2] gather_row_token: the token owning flat (token, slot) row `row`. */
uint32_t oracle_gather_row_token(uint32_t row, uint32_t top_k) { return row / top_k; }

/* [P2] module invariant: an expert folds nothing when its id is at or above
 * the table length or either table cell is 0.  A negative id is read as out
 * of range as well. */
static int expert_folds(int64_t e, int32_t n_experts, const uint64_t *a_table,
                        const uint64_t *b_table) {
    if (e < 0 || e >= n_experts) return 0;
    return a_table[e] != 0 && b_table[e] != 0;
}

/* The fold of one output row: ref[n] = base[n] + scale * sum_j h_j * B[n, j],
 * h_j = sum_k x[k] * A[j, k]  ([P2] moe_lora_gather_bgmv / moe_lora_grouped_down). */
static void fold_one_row(const uint16_t *x_row, const uint16_t *A, const uint16_t *B, double scale,
                         const uint16_t *base_row, double *ref_row, int32_t k_in, int32_t max_rank,
                         int32_t n_out) {
    double h[1024];
    for (int32_t j = 0; j < max_rank; ++j) {
        double acc = 0.0;
        for (int32_t k = 0; k < k_in; ++k)
            acc += bf16_value(x_row[k]) * bf16_value(A[(int64_t)j * k_in + k]);
        h[j] = acc;
    }
    for (int32_t n = 0; n < n_out; ++n) {
        double d = 0.0;
        for (int32_t j = 0; j < max_rank; ++j) d += h[j] * bf16_value(B[(int64_t)n * max_rank + j]);
        ref_row[n] = bf16_value(base_row[n]) + scale * d;
    }
}

static void copy_row(const uint16_t *base_row, double *ref_row, int32_t n_out) {
    for (int32_t n = 0; n < n_out; ++n) ref_row[n] = bf16_value(base_row[n]);
}

/* [P2] moe_lora_gather_bgmv: for every flat (token, slot) row < n_slots,
 * e = indices[row], token t = row / top_k; the row folds x[t] through expert
 * e unless row_adapter[t] < 0 ([P1] build_moe_row_adapter_decode: the kernel
 * skips a negative entry) or expert e folds nothing.  `folded[row]` is set to
 * 1 for rows that fold, 0 for rows that keep their input. */
int32_t oracle_gather_fold(const uint16_t *x, const int32_t *indices, const int32_t *row_adapter,
                           const uint64_t *a_table, const uint64_t *b_table,
                           const float *scale_table, const uint16_t *base_in, double *ref_out,
                           uint8_t *folded, int32_t n_slots, int32_t k_in, int32_t max_rank,
                           int32_t n_out, int32_t top_k, int32_t n_experts) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t row = 0; row < n_slots; ++row) {
        const uint16_t *base_row = base_in + (int64_t)row * n_out;
        double *ref_row = ref_out + (int64_t)row * n_out;
        int32_t t = row / top_k;
        int32_t e = indices[row];
        folded[row] = 0;
        if (row_adapter[t] < 0 || !expert_folds(e, n_experts, a_table, b_table)) {
            copy_row(base_row, ref_row, n_out);
            continue;
        }
        const uint16_t *A = (const uint16_t *)(uintptr_t)a_table[e];
        const uint16_t *B = (const uint16_t *)(uintptr_t)b_table[e];
        fold_one_row(x + (int64_t)t * k_in, A, B, (double)scale_table[e], base_row, ref_row, k_in,
                     max_rank, n_out);
        folded[row] = 1;
    }
    return OR_OK;
}

/* Multi-adapter gather fold.  The tables hold one set of n_experts cells per
 * adapter slot, slot-major: cell s * n_experts + e is adapter s's pair for
 * expert e.  The row map entry of a row's token names the set:
 * s = row_adapter[row / top_k]; a row folds nothing when s < 0, when
 * s >= n_adapters, when e = indices[row] is outside [0, n_experts), or when
 * its cell is zero; otherwise it folds as the [P2] moe_lora_gather_bgmv row
 * does, through its cell. */
int32_t oracle_gather_fold_multi(const uint16_t *x, const int32_t *indices,
                                 const int32_t *row_adapter, const uint64_t *a_table,
                                 const uint64_t *b_table, const float *scale_table,
                                 const uint16_t *base_in, double *ref_out, uint8_t *folded,
                                 int32_t n_slots, int32_t k_in, int32_t max_rank, int32_t n_out,
                                 int32_t top_k, int32_t n_experts, int32_t n_adapters) {
    if (max_rank > 1024 || top_k < 1 || n_adapters < 1) return OR_NONE;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t row = 0; row < n_slots; ++row) {
        const uint16_t *base_row = base_in + (int64_t)row * n_out;
        double *ref_row = ref_out + (int64_t)row * n_out;
        int32_t t = row / top_k;
        int32_t s = row_adapter[t];
        int32_t e = indices[row];
        folded[row] = 0;
        copy_row(base_row, ref_row, n_out);
        if (s < 0 || s >= n_adapters || e < 0 || e >= n_experts) continue;
        int64_t cell = (int64_t)s * n_experts + e;
        if (!expert_folds(cell, n_adapters * n_experts, a_table, b_table)) continue;
        fold_one_row(x + (int64_t)t * k_in, (const uint16_t *)(uintptr_t)a_table[cell],
                     (const uint16_t *)(uintptr_t)b_table[cell], (double)scale_table[cell],
                     base_row, ref_row, k_in, max_rank, n_out);
        folded[row] = 1;
    }
    return OR_OK;
}

/* [P2] moe_lora_grouped_down: sorted rows r in the window [row_offset,
 * row_end); e is the expert whose span expert_offsets[e] .. expert_offsets[e+1]
 * holds r, and the row's input is x[src[r] / top_k] (read of the pages'
 * row(r): src maps a sorted row to its flat (token, slot) row).  When
 * row_adapter is given, a row whose token has a negative entry is skipped.
 * Rows outside the window or outside every span e < n_experts keep their
 * input.  ref_out / folded cover all total_rows sorted rows. */
int32_t oracle_grouped_fold(const uint16_t *x, const int32_t *expert_offsets, const int32_t *src,
                            const int32_t *row_adapter, const uint64_t *a_table,
                            const uint64_t *b_table, const float *scale_table,
                            const uint16_t *base_in, double *ref_out, uint8_t *folded,
                            int64_t total_rows, int32_t k_in, int32_t max_rank, int32_t n_out,
                            int32_t top_k, int32_t n_experts, int32_t row_offset, int32_t row_end) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
    for (int64_t r = 0; r < total_rows; ++r) {
        copy_row(base_in + r * n_out, ref_out + r * n_out, n_out);
        folded[r] = 0;
    }
    for (int32_t e = 0; e < n_experts; ++e) {
        int64_t lo = expert_offsets[e] > row_offset ? expert_offsets[e] : row_offset;
        int64_t hi = expert_offsets[e + 1] < row_end ? expert_offsets[e + 1] : row_end;
        if (!expert_folds(e, n_experts, a_table, b_table)) continue;
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t r = lo; r < hi; ++r) {
            int32_t t = src[r] / top_k;
            if (row_adapter != NULL && row_adapter[t] < 0) continue;
            const uint16_t *A = (const uint16_t *)(uintptr_t)a_table[e];
            const uint16_t *B = (const uint16_t *)(uintptr_t)b_table[e];
            fold_one_row(x + (int64_t)t * k_in, A, B, (double)scale_table[e], base_in + r * n_out,
                         ref_out + r * n_out, k_in, max_rank, n_out);
            folded[r] = 1;
        }
    }
    return OR_OK;
}

/* Per-row x variant of the grouped fold.  [P2] moe_lora_grouped_down leaves
 * the x row of a sorted row undefined; the token reading above takes
 * x[src[r] / top_k].  In a real down projection the input is the expert's
 * intermediate activation, one row per sorted row, so this variant takes
 * x_rows[r] ([total_rows, k_in]) for sorted row r.  Everything else -- spans,
 * window, zero cells, the row map read through src[r] / top_k -- is the
 * grouped fold's. */
int32_t oracle_grouped_fold_xrows(const uint16_t *x_rows, const int32_t *expert_offsets,
                                  const int32_t *src, const int32_t *row_adapter,
                                  const uint64_t *a_table, const uint64_t *b_table,
                                  const float *scale_table, const uint16_t *base_in,
                                  double *ref_out, uint8_t *folded, int64_t total_rows,
                                  int32_t k_in, int32_t max_rank, int32_t n_out, int32_t top_k,
                                  int32_t n_experts, int32_t row_offset, int32_t row_end) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
    for (int64_t r = 0; r < total_rows; ++r) {
        copy_row(base_in + r * n_out, ref_out + r * n_out, n_out);
        folded[r] = 0;
    }
    for (int32_t e = 0; e < n_experts; ++e) {
        int64_t lo = expert_offsets[e] > row_offset ? expert_offsets[e] : row_offset;
        int64_t hi = expert_offsets[e + 1] < row_end ? expert_offsets[e + 1] : row_end;
        if (!expert_folds(e, n_experts, a_table, b_table)) continue;
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t r = lo; r < hi; ++r) {
            if (row_adapter != NULL && row_adapter[src[r] / top_k] < 0) continue;
            fold_one_row(x_rows + r * k_in, (const uint16_t *)(uintptr_t)a_table[e],
                         (const uint16_t *)(uintptr_t)b_table[e], (double)scale_table[e],
                         base_in + r * n_out, ref_out + r * n_out, k_in, max_rank, n_out);
            folded[r] = 1;
        }
    }
    return OR_OK;
}

/* [P2] MoeExpertRoute: the router fold is a one-entry route whose expert 0 is
 * the router pair, so every token t folds x[t] through entry 0 (top_k = 1,
 * identity rows).  A row map, when given, skips tokens with a negative entry. */
int32_t oracle_router_fold(const uint16_t *x, const int32_t *row_adapter, const uint64_t *a_table,
                           const uint64_t *b_table, const float *scale_table,
                           const uint16_t *base_in, double *ref_out, uint8_t *folded,
                           int32_t n_tokens, int32_t k_in, int32_t max_rank, int32_t n_out) {
    if (max_rank > 1024) return OR_NONE;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t t = 0; t < n_tokens; ++t) {
        const uint16_t *base_row = base_in + (int64_t)t * n_out;
        double *ref_row = ref_out + (int64_t)t * n_out;
        folded[t] = 0;
        if ((row_adapter != NULL && row_adapter[t] < 0) ||
            !expert_folds(0, 1, a_table, b_table)) {
            copy_row(base_row, ref_row, n_out);
            continue;
        }
        fold_one_row(x + (int64_t)t * k_in, (const uint16_t *)(uintptr_t)a_table[0],
                     (const uint16_t *)(uintptr_t)b_table[0], (double)scale_table[0], base_row,
                     ref_row, k_in, max_rank, n_out);
        folded[t] = 1;
    }
    return OR_OK;
}

/* Sampled variant for full-size checks: fold only the listed rows of a
 * gather-form problem (rows are flat rows), writing one ref row per entry. */
int32_t oracle_gather_fold_rows(const uint16_t *x, const int32_t *indices,
                                const int32_t *row_adapter, const uint64_t *a_table,
                                const uint64_t *b_table, const float *scale_table,
                                const uint16_t *base_rows, const int32_t *rows, int32_t n_rows,
                                double *ref_out, uint8_t *folded, int32_t k_in, int32_t max_rank,
                                int32_t n_out, int32_t top_k, int32_t n_experts) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t i = 0; i < n_rows; ++i) {
        int32_t row = rows[i];
        int32_t t = row / top_k;
        int32_t e = indices[row];
        const uint16_t *base_row = base_rows + (int64_t)i * n_out;
        double *ref_row = ref_out + (int64_t)i * n_out;
        folded[i] = 0;
        if ((row_adapter != NULL && row_adapter[t] < 0) ||
            !expert_folds(e, n_experts, a_table, b_table)) {
            copy_row(base_row, ref_row, n_out);
            continue;
        }
        fold_one_row(x + (int64_t)t * k_in, (const uint16_t *)(uintptr_t)a_table[e],
                     (const uint16_t *)(uintptr_t)b_table[e], (double)scale_table[e], base_row,
                     ref_row, k_in, max_rank, n_out);
        folded[i] = 1;
    }
    return OR_OK;
}

/* Sampled variant of the grouped fold: the listed sorted rows only. */
int32_t oracle_grouped_fold_rows(const uint16_t *x, const int32_t *expert_offsets,
                                 const int32_t *src, const int32_t *row_adapter,
                                 const uint64_t *a_table, const uint64_t *b_table,
                                 const float *scale_table, const uint16_t *base_rows,
                                 const int32_t *rows, int32_t n_rows, double *ref_out,
                                 uint8_t *folded, int32_t k_in, int32_t max_rank, int32_t n_out,
                                 int32_t top_k, int32_t n_experts, int32_t row_offset,
                                 int32_t row_end) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t i = 0; i < n_rows; ++i) {
        int32_t r = rows[i];
        const uint16_t *base_row = base_rows + (int64_t)i * n_out;
        double *ref_row = ref_out + (int64_t)i * n_out;
        folded[i] = 0;
        copy_row(base_row, ref_row, n_out);
        if (r < row_offset || r >= row_end) continue;
        /* the expert whose span holds r, by walking the spans in order */
        int32_t owner = -1;
        for (int32_t e = 0; e < n_experts; ++e) {
            if (expert_offsets[e] <= r && r < expert_offsets[e + 1]) {
                owner = e;
                break;
            }
        }
        if (owner < 0 || !expert_folds(owner, n_experts, a_table, b_table)) continue;
        int32_t t = src[r] / top_k;
        if (row_adapter != NULL && row_adapter[t] < 0) continue;
        fold_one_row(x + (int64_t)t * k_in, (const uint16_t *)(uintptr_t)a_table[owner],
                     (const uint16_t *)(uintptr_t)b_table[owner], (double)scale_table[owner],
                     base_row, ref_row, k_in, max_rank, n_out);
        folded[i] = 1;
    }
    return OR_OK;
}

/* Sampled variant of the per-row x grouped fold: the listed sorted rows only,
 * row r reading x_rows[r]. */
int32_t oracle_grouped_fold_xrows_rows(const uint16_t *x_rows, const int32_t *expert_offsets,
                                       const int32_t *src, const int32_t *row_adapter,
                                       const uint64_t *a_table, const uint64_t *b_table,
                                       const float *scale_table, const uint16_t *base_rows,
                                       const int32_t *rows, int32_t n_rows, double *ref_out,
                                       uint8_t *folded, int32_t k_in, int32_t max_rank,
                                       int32_t n_out, int32_t top_k, int32_t n_experts,
                                       int32_t row_offset, int32_t row_end) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t i = 0; i < n_rows; ++i) {
        int32_t r = rows[i];
        const uint16_t *base_row = base_rows + (int64_t)i * n_out;
        double *ref_row = ref_out + (int64_t)i * n_out;
        folded[i] = 0;
        copy_row(base_row, ref_row, n_out);
        if (r < row_offset || r >= row_end) continue;
        int32_t owner = -1;
        for (int32_t e = 0; e < n_experts; ++e) {
            if (expert_offsets[e] <= r && r < expert_offsets[e + 1]) {
                owner = e;
                break;
            }
        }
        if (owner < 0 || !expert_folds(owner, n_experts, a_table, b_table)) continue;
        if (row_adapter != NULL && row_adapter[src[r] / top_k] < 0) continue;
        fold_one_row(x_rows + (int64_t)r * k_in, (const uint16_t *)(uintptr_t)a_table[owner],
                     (const uint16_t *)(uintptr_t)b_table[owner], (double)scale_table[owner],
                     base_row, ref_row, k_in, max_rank, n_out);
        folded[i] = 1;
    }
    return OR_OK;
}

/* The expert GEMM with the LoRA fold in its epilogue (per-row x form).
 * [P2] moe_lora_grouped_down folds into base_out, which is the expert
 * projection's output: base_out[r] = x_rows[r] @ W_e^T for a down projection
 * whose input is the expert's intermediate row.  Computing both in one pass
 * gives, for sorted row r in [row_offset, row_end) held by span e < n_experts
 * whose weight cell w_table[e] is non-zero (W_e [n_out, k_in] bf16):
 *     out[r, n] = sum_k x_rows[r, k] W_e[n, k]
 *                 + [row folds] scale_e * sum_j h_j B_e[n, j],
 *     h_j = sum_k x_rows[r, k] A_e[j, k],
 * where the row folds under the per-row x fold's rules: expert e's a / b
 * cells non-zero, src[r] >= 0, and (when given) row_adapter[src[r] / top_k]
 * >= 0.  A row of a span whose weight cell is 0, or outside the window or
 * every span, is not an output of this call and keeps its prior value
 * (out_in).  `written[r]` marks rows given the GEMM result, `folded[r]` the
 * rows that also took the delta.  Unrounded, like every fold here. */
int32_t oracle_grouped_gemm_fold_xrows(const uint16_t *x_rows, const int32_t *expert_offsets,
                                       const int32_t *src, const int32_t *row_adapter,
                                       const uint64_t *w_table, const uint64_t *a_table,
                                       const uint64_t *b_table, const float *scale_table,
                                       const uint16_t *out_in, double *ref_out, uint8_t *written,
                                       uint8_t *folded, int64_t total_rows, int32_t k_in,
                                       int32_t max_rank, int32_t n_out, int32_t top_k,
                                       int32_t n_experts, int32_t row_offset, int32_t row_end) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
    for (int64_t r = 0; r < total_rows; ++r) {
        copy_row(out_in + r * n_out, ref_out + r * n_out, n_out);
        written[r] = 0;
        folded[r] = 0;
    }
    for (int32_t e = 0; e < n_experts; ++e) {
        int64_t lo = expert_offsets[e] > row_offset ? expert_offsets[e] : row_offset;
        int64_t hi = expert_offsets[e + 1] < row_end ? expert_offsets[e + 1] : row_end;
        if (w_table[e] == 0) continue;
        const uint16_t *W = (const uint16_t *)(uintptr_t)w_table[e];
        int lora = expert_folds(e, n_experts, a_table, b_table);
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t r = lo; r < hi; ++r) {
            const uint16_t *xr = x_rows + r * k_in;
            double *ref_row = ref_out + r * n_out;
            for (int32_t n = 0; n < n_out; ++n) {
                double g = 0.0;
                for (int32_t k = 0; k < k_in; ++k)
                    g += bf16_value(xr[k]) * bf16_value(W[(int64_t)n * k_in + k]);
                ref_row[n] = g;
            }
            written[r] = 1;
            int row_folds = lora && src[r] >= 0 &&
                            (row_adapter == NULL || row_adapter[src[r] / top_k] >= 0);
            if (!row_folds) continue;
            const uint16_t *A = (const uint16_t *)(uintptr_t)a_table[e];
            const uint16_t *B = (const uint16_t *)(uintptr_t)b_table[e];
            double h[1024];
            for (int32_t j = 0; j < max_rank; ++j) {
                double acc = 0.0;
                for (int32_t k = 0; k < k_in; ++k)
                    acc += bf16_value(xr[k]) * bf16_value(A[(int64_t)j * k_in + k]);
                h[j] = acc;
            }
            double scale = (double)scale_table[e];
            for (int32_t n = 0; n < n_out; ++n) {
                double d = 0.0;
                for (int32_t j = 0; j < max_rank; ++j)
                    d += h[j] * bf16_value(B[(int64_t)n * max_rank + j]);
                ref_row[n] += scale * d;
            }
            folded[r] = 1;
        }
    }
    return OR_OK;
}

/* Sampled variant of the expert GEMM with the fold: the listed sorted rows
 * only (one ref row per entry; `prior_rows` holds their prior values, which a
 * row that is not an output keeps), each computed exactly as in
 * oracle_grouped_gemm_fold_xrows. */
int32_t oracle_grouped_gemm_fold_xrows_rows(const uint16_t *x_rows, const int32_t *expert_offsets,
                                            const int32_t *src, const int32_t *row_adapter,
                                            const uint64_t *w_table, const uint64_t *a_table,
                                            const uint64_t *b_table, const float *scale_table,
                                            const uint16_t *prior_rows, const int32_t *rows,
                                            int32_t n_rows, double *ref_out, uint8_t *written,
                                            uint8_t *folded, int32_t k_in, int32_t max_rank,
                                            int32_t n_out, int32_t top_k, int32_t n_experts,
                                            int32_t row_offset, int32_t row_end) {
    if (max_rank > 1024 || top_k < 1) return OR_NONE;
#pragma omp parallel for schedule(dynamic, 8)
    for (int32_t i = 0; i < n_rows; ++i) {
        int32_t r = rows[i];
        double *ref_row = ref_out + (int64_t)i * n_out;
        copy_row(prior_rows + (int64_t)i * n_out, ref_row, n_out);
        written[i] = 0;
        folded[i] = 0;
        if (r < row_offset || r >= row_end) continue;
        int32_t owner = -1;
        for (int32_t e = 0; e < n_experts; ++e) {
            if (expert_offsets[e] <= r && r < expert_offsets[e + 1]) {
                owner = e;
                break;
            }
        }
        if (owner < 0 || w_table[owner] == 0) continue;
        const uint16_t *W = (const uint16_t *)(uintptr_t)w_table[owner];
        const uint16_t *xr = x_rows + (int64_t)r * k_in;
        for (int32_t n = 0; n < n_out; ++n) {
            double g = 0.0;
            for (int32_t k = 0; k < k_in; ++k)
                g += bf16_value(xr[k]) * bf16_value(W[(int64_t)n * k_in + k]);
            ref_row[n] = g;
        }
        written[i] = 1;
        if (!expert_folds(owner, n_experts, a_table, b_table) || src[r] < 0 ||
            (row_adapter != NULL && row_adapter[src[r] / top_k] < 0))
            continue;
        const uint16_t *A = (const uint16_t *)(uintptr_t)a_table[owner];
        const uint16_t *B = (const uint16_t *)(uintptr_t)b_table[owner];
        double h[1024];
        for (int32_t j = 0; j < max_rank; ++j) {
            double acc = 0.0;
            for (int32_t k = 0; k < k_in; ++k)
                acc += bf16_value(xr[k]) * bf16_value(A[(int64_t)j * k_in + k]);
            h[j] = acc;
        }
        double scale = (double)scale_table[owner];
        for (int32_t n = 0; n < n_out; ++n) {
            double d = 0.0;
            for (int32_t j = 0; j < max_rank; ++j) d += h[j] * bf16_value(B[(int64_t)n * max_rank + j]);
            ref_row[n] += scale * d;
        }
        folded[i] = 1;
    }
    return OR_OK;
}
