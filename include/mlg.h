/*
 * mlg.h -- C ABI of libmlg, the GB300 (sm_103a) MoE expert LoRA fold.
 *
 * The fold, for every row it covers:
 *
 *     base_out[row] += scale_e * (x[x_row] @ A_e^T) @ B_e^T
 *
 * with A_e [max_rank, k_in] and B_e [n_out, max_rank] the LoRA pair of expert
 * e.  Source: the "metrale" documentation pages -- the module index of
 * metrale_model_layers::layers::ops::moe_lora_grouped (items
 * moe_lora_gather_bgmv, moe_lora_grouped_down, MoeExpertRoute,
 * pack_expert_tables, grouped_down_windows, grouped_down_wc,
 * gather_row_token, MLG_M_TILE and the module invariant on zero table cells)
 * and the source page moe_row_adapter.rs (resolve_moe_lora_route,
 * ensure_decode_route_servable, build_moe_row_adapter_host,
 * build_moe_row_adapter_decode).
 *
 * Three widened forms sit beside the pages' calls: a per-row x grouped fold
 * (mlg_grouped_down_xrows: sorted row r reads x_rows[r], the input a down
 * projection has), the expert GEMM with that fold in its epilogue
 * (mlg_grouped_gemm_fold_xrows: base_out produced and folded in one pass)
 * and a multi-adapter decode fold (mlg_gather_bgmv_multi, with
 * mlg_build_moe_row_adapter_decode_multi: one table set per adapter slot,
 * each token's row-map entry naming its set).  Each states the reading of
 * the pages it rests on.
 *
 * Conventions shared by every call:
 *  - Every call that can fail returns an mlg_status; the library never
 *    aborts, asserts or prints.  The pages' `None` becomes MLG_ERR_EMPTY or
 *    MLG_ERR_INVALID_ARG, their panic MLG_ERR_CAP_ZERO, their `Err`
 *    MLG_ERR_REFUSE.
 *  - The caller owns every buffer, host and device.  The fold entry points
 *    allocate no memory, never synchronise the device or the host, and
 *    enqueue only on the stream they are given, so each can be captured in a
 *    CUDA graph.  `stream` is a cudaStream_t passed as void* (0 = the legacy
 *    default stream).
 *  - Early start (programmatic dependent launch).  Every fold kernel may
 *    start while the kernel before it in the stream is still running and
 *    waits for that kernel's completion (and the visibility of its writes)
 *    before it reads the routing (indices, expert_offsets, src), the row map,
 *    x or base_out, so those may be written by the preceding kernel.  The
 *    grouped and router folds read everything else after that wait too.  The
 *    decode folds (mlg_gather_bgmv, mlg_gather_bgmv_multi) do NOT: they may
 *    read a_table, b_table, scale_table and the A_e / B_e pairs those tables
 *    point to BEFORE the wait, to overlap the pair traffic with the preceding
 *    kernel.  Tables and pairs written by a copy (cudaMemcpy*, as the upload
 *    helpers do) are safe, because a copy is never overlapped; a caller whose
 *    preceding KERNEL writes the tables or the pair weights (a device-side
 *    adapter install or rotation, a dequantisation kernel) must call
 *    mlg_gather_bgmv_ex / mlg_gather_bgmv_multi_ex with
 *    MLG_FOLD_AFTER_PRECEDING, which launches the fold without early start,
 *    or it may fold stale tables or weights with no error reported.
 *  - All arguments are validated on the host before anything is enqueued or
 *    written; on any error nothing is launched and no output is written.
 *  - Device arrays are row-major.  bf16 values are raw IEEE bfloat16 bit
 *    patterns (uint16).  Device pointers must come from the CUDA allocator
 *    of the current device (or be offsets into such allocations).
 *  - Table cells are data: an expert folds nothing when its id is negative,
 *    at or above n_experts, or either of its table cells is 0.  A non-zero
 *    cell that is not 16-byte aligned is also treated as 0 (the kernels never
 *    fault on table contents they can check).  A non-zero, aligned cell must
 *    hold the device address of an array of the stated shape.
 *  - Rows that do not fold keep their input bits exactly (including -0.0).
 *  - Arithmetic: bf16 inputs, fp32 products and sums, and one
 *    round-to-nearest-even to bf16 of base + scale * delta per element.  The
 *    rank-r intermediate h is accumulated in fp32 and enters the expand
 *    (a bf16 tensor-core product) as the sum of two bf16 values, hi = bf16(h)
 *    and lo = bf16(h - hi): |h - hi - lo| <= 2^-18 |h|, so h is never
 *    rounded to a single bf16 and the expand sees it at about fp32's
 *    precision (2^-18 against fp32's 2^-24 relative).
 */
#ifndef MLG_H_
#define MLG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mlg_status;

#if defined(__GNUC__)
#define MLG_API __attribute__((visibility("default")))
#else
#define MLG_API
#endif

#define MLG_OK 0
#define MLG_ERR_INVALID_ARG (-1)      /* bad pointer, size or relation; the pages' None */
#define MLG_ERR_EMPTY (-2)            /* empty input where the pages return None */
#define MLG_ERR_CAP_ZERO (-3)         /* window cap of 0: the pages' panic */
#define MLG_ERR_REFUSE (-4)           /* a decode batch the installed adapter(s) cannot serve */
#define MLG_ERR_UNSUPPORTED (-5)      /* alignment or size limit of this implementation */
#define MLG_ERR_BUFFER_TOO_SMALL (-6) /* output buffer shorter than the result */
#define MLG_ERR_CUDA (-7)             /* a CUDA runtime call failed; see mlg_last_cuda_error() */

/* Route values of resolve_moe_lora_route (moe_row_adapter.rs). */
#define MLG_ROUTE_FOLD 0
#define MLG_ROUTE_SKIP 1
#define MLG_ROUTE_REFUSE 2

/* Largest max_rank the fold kernels accept.  max_rank must also be a
 * multiple of 8 so that every row of B_e starts on a 16-byte boundary; a
 * smaller true rank is stored zero-padded to max_rank. */
#define MLG_MAX_RANK 64

typedef uint16_t mlg_bf16;

/* One (expert_id, a_addr, b_addr, scale) entry of pack_expert_tables. */
typedef struct mlg_expert_entry {
  uint32_t expert_id;
  uint32_t reserved0; /* ignored */
  uint64_t a_addr;    /* device address of A_e [max_rank, k_in] bf16, or 0 */
  uint64_t b_addr;    /* device address of B_e [n_out, max_rank] bf16, or 0 */
  float scale;        /* scale_e */
  uint32_t reserved1; /* ignored */
} mlg_expert_entry;

/* One [start, end) window of grouped_down_windows. */
typedef struct mlg_window {
  uint32_t start;
  uint32_t end;
} mlg_window;

/* ------------------------------------------------------------------------
 * Fold entry points (device work; enqueue on `stream`, return immediately).
 * ------------------------------------------------------------------------ */

/* moe_lora_gather_bgmv (moe_lora_grouped module index): the decode-side fold
 * over flat (token, slot) rows, row = token * top_k + slot.  For every row in
 * [0, n_slots): e = indices[row], t = row / top_k (gather_row_token); the row
 * folds x[t] through expert e unless row_adapter[t] < 0 (the decode row map of
 * build_moe_row_adapter_decode) or expert e folds nothing (see above).
 *
 *   x            device, [ceil(n_slots / top_k), k_in] bf16, 16-byte aligned
 *   indices      device, [n_slots] int32 expert ids (any value: invalid ids fold nothing)
 *   row_adapter  device, [ceil(n_slots / top_k)] int32, required (non-NULL)
 *   a_table      device, [n_experts] uint64 addresses of A_e (0 = unadapted)
 *   b_table      device, [n_experts] uint64 addresses of B_e (0 = unadapted)
 *   scale_table  device, [n_experts] float scale_e
 *   base_out     device, [n_slots, n_out] bf16, updated in place, 16-byte aligned
 *   k_in         >= 8, multiple of 8;  n_out >= 8, multiple of 8
 *   max_rank     1..MLG_MAX_RANK, multiple of 8
 *   top_k        >= 1;  n_experts >= 0 (0: nothing folds, nothing is launched)
 * n_slots == 0 is a no-op.  Errors: INVALID_ARG (NULL pointer, negative size,
 * top_k < 1), UNSUPPORTED (alignment, k_in / n_out / max_rank limits),
 * CUDA (the launch failed). */
MLG_API mlg_status mlg_gather_bgmv(const mlg_bf16 *x, const int32_t *indices, const int32_t *row_adapter,
                           const uint64_t *a_table, const uint64_t *b_table,
                           const float *scale_table, mlg_bf16 *base_out, int32_t n_slots,
                           int32_t k_in, int32_t max_rank, int32_t n_out, int32_t top_k,
                           int32_t n_experts, void *stream);

/* Multi-adapter gather fold.  The single-active rule of resolve_moe_lora_route
 * and ensure_decode_route_servable (moe_row_adapter.rs) refuses a batch that
 * mixes adapters because only the active adapter's pairs are installed.  Here
 * one table set per adapter slot is installed at once, slot-major: cell
 * s * n_experts + e holds adapter s's pair for expert e.  A row's token names
 * its set through the row map, s = row_adapter[row / top_k], and the row folds
 *     base_out[row] += scale[c] * (x[row / top_k] @ A_c^T) @ B_c^T,
 *     c = s * n_experts + indices[row],
 * unless s < 0, s >= n_adapters, indices[row] is outside [0, n_experts) or
 * cell c is zero (those rows keep their input).
 *
 *   tables       device, [n_adapters * n_experts] each, slot-major; every
 *                set packed by mlg_pack_expert_tables with cap n_experts
 *                (holes are zero cells)
 *   row_adapter  device, [ceil(n_slots / top_k)] int32 slot per token
 *                (mlg_build_moe_row_adapter_decode_multi), required
 *   n_adapters   >= 1; n_adapters * n_experts <= 2^30
 *   others       as for mlg_gather_bgmv
 * Errors as for mlg_gather_bgmv, plus INVALID_ARG for n_adapters < 1 and
 * UNSUPPORTED for more than 2^30 cells.
 * The prefill form needs no call of its own: sort the flat rows by cell
 * (slot * n_experts + expert; rows of no cell after the last) into
 * expert_offsets / src and call mlg_grouped_down or
 * mlg_grouped_down_all_windows with n_experts = n_adapters * n_experts, the
 * slot-major tables and the prefill row map of slots. */
MLG_API mlg_status mlg_gather_bgmv_multi(const mlg_bf16 *x, const int32_t *indices,
                                         const int32_t *row_adapter, const uint64_t *a_table,
                                         const uint64_t *b_table, const float *scale_table,
                                         mlg_bf16 *base_out, int32_t n_slots, int32_t k_in,
                                         int32_t max_rank, int32_t n_out, int32_t top_k,
                                         int32_t n_experts, int32_t n_adapters, void *stream);

/* Launch flags of the _ex decode entry points.
 *   MLG_FOLD_AFTER_PRECEDING  launch without early start: the fold begins
 *                             only once the preceding work in the stream has
 *                             completed, so it may read tables and A_e / B_e
 *                             pairs that the preceding kernel wrote (see
 *                             "Early start" above).  Costs the overlap of
 *                             the pair traffic with that kernel. */
#define MLG_FOLD_AFTER_PRECEDING 1u

/* mlg_gather_bgmv and mlg_gather_bgmv_multi with launch flags (0 or
 * MLG_FOLD_AFTER_PRECEDING); with flags == 0 they are exactly the calls
 * above.  Errors as for those calls, plus INVALID_ARG for an unknown flag. */
MLG_API mlg_status mlg_gather_bgmv_ex(const mlg_bf16 *x, const int32_t *indices,
                                      const int32_t *row_adapter, const uint64_t *a_table,
                                      const uint64_t *b_table, const float *scale_table,
                                      mlg_bf16 *base_out, int32_t n_slots, int32_t k_in,
                                      int32_t max_rank, int32_t n_out, int32_t top_k,
                                      int32_t n_experts, uint32_t flags, void *stream);
MLG_API mlg_status mlg_gather_bgmv_multi_ex(const mlg_bf16 *x, const int32_t *indices,
                                            const int32_t *row_adapter, const uint64_t *a_table,
                                            const uint64_t *b_table, const float *scale_table,
                                            mlg_bf16 *base_out, int32_t n_slots, int32_t k_in,
                                            int32_t max_rank, int32_t n_out, int32_t top_k,
                                            int32_t n_experts, int32_t n_adapters,
                                            uint32_t flags, void *stream);

/* moe_lora_grouped_down (moe_lora_grouped module index): the prefill-side fold
 * over expert-sorted rows r in the window [row_offset, row_end).  e is the
 * expert whose span expert_offsets[e] <= r < expert_offsets[e + 1] holds r
 * (e < n_experts); the row's input is x[src[r] / top_k].  base_out is indexed
 * by sorted row.  Rows outside the window, rows in no span below n_experts
 * (at or past expert_offsets[n_experts]) and rows whose token has a negative
 * row_adapter entry keep their input.
 *
 *   x              device, [n_tokens, k_in] bf16, 16-byte aligned
 *   expert_offsets device, >= n_experts + 1 int32, non-decreasing; read on the
 *                  device only (no host copy), so the call is graph-capturable
 *   src            device, int32 sorted row -> flat (token, slot) row; every
 *                  src[r] in the window must be < n_tokens * top_k (a negative
 *                  entry folds nothing)
 *   row_adapter    device, [n_tokens] int32 prefill row map, or NULL (every row folds)
 *   tables         as for mlg_gather_bgmv
 *   base_out       device, [>= row_end, n_out] bf16, in place, 16-byte aligned
 *   0 <= row_offset <= row_end; an empty window is a no-op
 * Errors as for mlg_gather_bgmv, plus INVALID_ARG for row_end < row_offset. */
MLG_API mlg_status mlg_grouped_down(const mlg_bf16 *x, const int32_t *expert_offsets, const int32_t *src,
                            const int32_t *row_adapter, const uint64_t *a_table,
                            const uint64_t *b_table, const float *scale_table,
                            mlg_bf16 *base_out, int32_t k_in, int32_t max_rank, int32_t n_out,
                            int32_t top_k, int32_t n_experts, int32_t row_offset,
                            int32_t row_end, void *stream);

/* All windows of grouped_down_windows(total_rows, cap) folded in ONE launch:
 * the same result, bit for bit, as calling mlg_grouped_down for each window
 * [i*cap, min((i+1)*cap, total_rows)) in turn, because every tile of the
 * kernel lies inside one window and one expert span and each row's arithmetic
 * does not depend on its tile.  One persistent launch instead of one per
 * window removes the per-window pipeline fill and tail.  Arguments as for
 * mlg_grouped_down with row_offset = 0, row_end = total_rows.  Errors as for
 * mlg_grouped_down, plus CAP_ZERO for cap == 0. */
MLG_API mlg_status mlg_grouped_down_all_windows(const mlg_bf16 *x, const int32_t *expert_offsets,
                                                const int32_t *src, const int32_t *row_adapter,
                                                const uint64_t *a_table, const uint64_t *b_table,
                                                const float *scale_table, mlg_bf16 *base_out,
                                                int32_t k_in, int32_t max_rank, int32_t n_out,
                                                int32_t top_k, int32_t n_experts,
                                                int32_t total_rows, uint32_t cap, void *stream);

/* Per-row x form of moe_lora_grouped_down (moe_lora_grouped module index).
 * The page leaves open which x row a sorted row reads; in a down projection
 * the input is the expert's own intermediate row, one per sorted row, so here
 * sorted row r reads x_rows[r]:
 *     base_out[r] += scale_e * (x_rows[r] @ A_e^T) @ B_e^T
 * for r in [row_offset, row_end) held by span e < n_experts.  src serves the
 * row map only: a row whose token src[r] / top_k has a negative row_adapter
 * entry, or whose src[r] is negative, keeps its input, as do rows outside the
 * range or outside every span.  The range is folded in windows of cap rows
 * (starting at row_offset) in ONE launch; the result does not depend on cap.
 *
 *   x_rows         device, [>= row_end, k_in] bf16, indexed by sorted row,
 *                  16-byte aligned; read only
 *   expert_offsets, src, row_adapter, tables, base_out
 *                  as for mlg_grouped_down (src must be non-NULL)
 *   cap            window length in rows, >= 1
 * Errors as for mlg_grouped_down, plus CAP_ZERO for cap == 0. */
MLG_API mlg_status mlg_grouped_down_xrows(const mlg_bf16 *x_rows, const int32_t *expert_offsets,
                                          const int32_t *src, const int32_t *row_adapter,
                                          const uint64_t *a_table, const uint64_t *b_table,
                                          const float *scale_table, mlg_bf16 *base_out,
                                          int32_t k_in, int32_t max_rank, int32_t n_out,
                                          int32_t top_k, int32_t n_experts, int32_t row_offset,
                                          int32_t row_end, uint32_t cap, void *stream);

/* The expert GEMM with the fold in its epilogue (per-row x form).  The
 * moe_lora_grouped module index folds into base_out (moe_lora_grouped_down),
 * and base_out is the expert projection's output; computing both in one pass
 * means base_out is written once instead of written, read back and written
 * again.  For every sorted row r in [row_offset, row_end) held by span
 * e < n_experts:
 *     out[r] = RNE_bf16( x_rows[r] @ W_e^T
 *                        + [row folds] scale_e * (x_rows[r] @ A_e^T) @ B_e^T )
 * with W_e [n_out, k_in] the expert's slice of the stacked weights, the
 * products and sums in fp32 (tensor cores) and one rounding.  A row folds
 * under the rules of mlg_grouped_down_xrows (LoRA cells non-zero, src[r] >= 0,
 * row-map entry of its token not negative); a row that does not fold still
 * gets the GEMM.  Rows outside the range and rows past
 * expert_offsets[n_experts] are not outputs of this call: out keeps their
 * bits.  The range is processed in windows of cap rows in ONE launch; the
 * result does not depend on cap.
 *
 *   x_rows         device, [>= row_end, k_in] bf16, 16-byte aligned
 *   w_experts      device, [n_experts, n_out, k_in] bf16 (the experts' weights
 *                  stacked, each row-major), 16-byte aligned; read only
 *   expert_offsets, src, row_adapter, a/b/scale tables
 *                  as for mlg_grouped_down_xrows (src non-NULL); the tables
 *                  have n_experts cells
 *   out            device, [>= row_end, n_out] bf16, written (not read), 16-byte aligned
 * With every LoRA cell 0 this is a plain grouped expert GEMM.  Errors as for
 * mlg_grouped_down_xrows. */
MLG_API mlg_status mlg_grouped_gemm_fold_xrows(const mlg_bf16 *x_rows,
                                               const int32_t *expert_offsets, const int32_t *src,
                                               const int32_t *row_adapter,
                                               const mlg_bf16 *w_experts, const uint64_t *a_table,
                                               const uint64_t *b_table, const float *scale_table,
                                               mlg_bf16 *out, int32_t k_in, int32_t max_rank,
                                               int32_t n_out, int32_t top_k, int32_t n_experts,
                                               int32_t row_offset, int32_t row_end, uint32_t cap,
                                               void *stream);

/* The router fold (MoeExpertRoute, moe_lora_grouped module index): a one-entry
 * route whose expert 0 is the router pair, so every token t folds
 * base_out[t] += scale_0 * (x[t] @ A_0^T) @ B_0^T.  The tables have one entry;
 * a zero cell makes the call a no-op on the device.
 *
 *   x            device, [n_tokens, k_in] bf16;  base_out device, [n_tokens, n_out] bf16
 *   row_adapter  device, [n_tokens] int32 or NULL (negative entries skip the token)
 * Limits and errors as for mlg_grouped_down. */
MLG_API mlg_status mlg_router_fold(const mlg_bf16 *x, const int32_t *row_adapter, const uint64_t *a_table,
                           const uint64_t *b_table, const float *scale_table, mlg_bf16 *base_out,
                           int32_t n_tokens, int32_t k_in, int32_t max_rank, int32_t n_out,
                           void *stream);

/* ------------------------------------------------------------------------
 * Host helpers (pure CPU unless stated; no device work).
 * ------------------------------------------------------------------------ */

/* resolve_moe_lora_route (moe_row_adapter.rs): the fold decision for one
 * request.  Returns MLG_ROUTE_FOLD when has_moe_lora is 0; else SKIP for a
 * negative slot; else FOLD when slot == active; else REFUSE. */
MLG_API int32_t mlg_resolve_moe_lora_route(int32_t adapter_slot, int32_t active, int32_t has_moe_lora);

/* ensure_decode_route_servable (moe_row_adapter.rs): MLG_ERR_REFUSE when
 * route is MLG_ROUTE_REFUSE (a decode batch cannot serve a non-active adapter
 * under the single-active fold), MLG_OK for FOLD / SKIP, INVALID_ARG for any
 * other value. */
MLG_API mlg_status mlg_ensure_decode_route_servable(int32_t route);

/* build_moe_row_adapter_decode (moe_row_adapter.rs): writes the [padded_n]
 * decode row map to out: entry i is `active` when i < n_slots and slot i
 * routes to FOLD, else -1 (Skip, Refuse and padding).  out must hold padded_n
 * entries.  Errors: INVALID_ARG for out == NULL with padded_n > 0, or
 * adapter_slots == NULL with n_slots > 0. */
MLG_API mlg_status mlg_build_moe_row_adapter_decode(const int32_t *adapter_slots, size_t n_slots,
                                            size_t padded_n, int32_t active,
                                            int32_t has_moe_lora, int32_t *out);

/* Decode map of the multi-adapter fold (see mlg_gather_bgmv_multi): entry i
 * is adapter_slots[i] when 0 <= slot < n_adapters, -1 for a base request
 * (slot < 0) and for padding (i >= n_slots), and -1 everywhere when
 * has_moe_lora is 0.  A slot >= n_adapters has no table set: the call
 * returns MLG_ERR_REFUSE and writes nothing (the single-active refusal, moved
 * to the slots without tables).  Errors: INVALID_ARG for out == NULL with
 * padded_n > 0, adapter_slots == NULL with n_slots > 0, or n_adapters < 1. */
MLG_API mlg_status mlg_build_moe_row_adapter_decode_multi(const int32_t *adapter_slots,
                                                          size_t n_slots, size_t padded_n,
                                                          int32_t n_adapters,
                                                          int32_t has_moe_lora, int32_t *out);

/* build_moe_row_adapter_host (moe_row_adapter.rs): the [total_tokens] prefill
 * row map.  cu_seqlens holds n_cu = batch + 1 prefix sums; stream b's slot is
 * written over rows cu[b]..cu[b+1].  INVALID_ARG (nothing written) when
 * n_cu < 2, n_slots != n_cu - 1, cu[0] != 0, or a boundary is negative or
 * decreasing -- the pages' None.  *total_out receives cu[n_cu-1] whenever the
 * boundaries are valid; BUFFER_TOO_SMALL (nothing written) when cap is below
 * it, so a caller may size the buffer with a first call of cap 0. */
MLG_API mlg_status mlg_build_moe_row_adapter_host(const int32_t *cu_seqlens, size_t n_cu,
                                          const int32_t *adapter_slots, size_t n_slots,
                                          int32_t *out, size_t cap, size_t *total_out);

/* pack_expert_tables (moe_lora_grouped module index): dense tables indexed by
 * expert id with n_experts = max id + 1, 0 / 0 / 0.0f at every id without an
 * entry, and the last entry winning for a duplicated id.  EMPTY for n == 0.
 * *n_experts_out is set whenever n > 0; BUFFER_TOO_SMALL (nothing written)
 * when cap < n_experts.  UNSUPPORTED (nothing written) when a non-zero
 * address is not 16-byte aligned.  The tables are host arrays; upload them
 * with mlg_upload_expert_tables. */
MLG_API mlg_status mlg_pack_expert_tables(const mlg_expert_entry *entries, size_t n, uint64_t *a_out,
                                  uint64_t *b_out, float *scale_out, size_t cap,
                                  uint32_t *n_experts_out);

/* Table upload: three cudaMemcpyAsync host-to-device copies of n_experts
 * entries on `stream`.  Staging in pinned memory is the caller's choice; with
 * pageable memory the copies are synchronous with respect to the host.  A
 * fold enqueued after these copies always sees the new tables (copies are
 * never overlapped by a fold's early start); tables written by a kernel need
 * MLG_FOLD_AFTER_PRECEDING on the decode folds.
 * Errors: INVALID_ARG (NULL), CUDA. */
MLG_API mlg_status mlg_upload_expert_tables(const uint64_t *a_host, const uint64_t *b_host,
                                    const float *scale_host, uint32_t n_experts,
                                    uint64_t *a_dev, uint64_t *b_dev, float *scale_dev,
                                    void *stream);

/* Row-map upload (the engine's upload_moe_row_adapter): one cudaMemcpyAsync
 * of n int32 entries, host to device, on `stream`. */
MLG_API mlg_status mlg_upload_row_adapter(const int32_t *map_host, size_t n, int32_t *map_dev,
                                  void *stream);

/* grouped_down_windows (moe_lora_grouped module index): contiguous windows
 * [i*cap, min((i+1)*cap, total_rows)) covering 0..total_rows.  CAP_ZERO for
 * cap == 0.  *n_windows receives the window count; BUFFER_TOO_SMALL (nothing
 * written) when out_cap is below it. */
MLG_API mlg_status mlg_grouped_down_windows(uint32_t total_rows, uint32_t cap, mlg_window *out,
                                    size_t out_cap, size_t *n_windows);

/* grouped_down_wc (moe_lora_grouped module index): the tile count of a
 * window, max(1, ceil((row_end - row_offset) / MLG_M_TILE)); 1 when
 * row_end <= row_offset. */
MLG_API uint32_t mlg_grouped_down_wc(uint32_t row_offset, uint32_t row_end);

/* gather_row_token (moe_lora_grouped module index): row / top_k; 0 when
 * top_k == 0. */
MLG_API uint32_t mlg_gather_row_token(uint32_t row, uint32_t top_k);

/* MLG_M_TILE: sorted rows per grouped-fold tile (the tensor-core M of the
 * grouped kernel).  mlg_grouped_down_wc uses the same value. */
MLG_API uint32_t mlg_m_tile(void);

/* A static, NUL-terminated description of a status code. */
MLG_API const char *mlg_status_string(mlg_status status);

/* The cudaError_t of the last failing CUDA call made by this library on the
 * calling thread (0 when none). */
MLG_API int32_t mlg_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
MLG_API int32_t mlg_version(void);

/* Device error bits the fold kernels recorded on the current device instead
 * of trapping: MLG_DEVERR_WAIT_TIMEOUT (a wait for a copy or an MMA ran past
 * its one-second limit; the kernel stopped issuing work and the affected rows
 * may be unfolded), MLG_DEVERR_TMEM_ALLOC (tensor memory could not be
 * allocated; the affected tiles were not folded), MLG_DEVERR_UNIT_DROPPED (a
 * multi-adapter decode CTA was dealt more cells than it holds and left the
 * excess unfolded; the launch-time shape check is meant to rule this out).
 * Reads the OR of all bits
 * since the last clear into *flags_out and clears them when `clear` is
 * non-zero.  Synchronous (a device-to-host copy); not for the hot path. */
#define MLG_DEVERR_WAIT_TIMEOUT 1u
#define MLG_DEVERR_TMEM_ALLOC 2u
#define MLG_DEVERR_UNIT_DROPPED 4u
MLG_API mlg_status mlg_read_device_errors(uint32_t *flags_out, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* MLG_H_ */
