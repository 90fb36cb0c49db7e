// mlg_decode.cu -- decode-side MoE expert LoRA fold (moe_lora_gather_bgmv of
// the moe_lora_grouped module index) for expert pairs that fit one CTA:
//     base_out[row] += scale_e * (x[row / top_k] @ A_e^T) @ B_e^T,  e = indices[row],
// rows whose token has a negative row-map entry skipped (moe_row_adapter.rs,
// build_moe_row_adapter_decode), experts with a zero table cell or an id at or
// above n_experts folding nothing.
//
// GB300 design.  A decode fold moves few bytes (a 64-token down projection is
// ~16 MB), so its time is set by dependent round trips, not by bandwidth.  The
// kernel is built so that consecutive folds in a stream overlap:
//  * one CTA per expert holds the whole pair: A_e and B_e are bulk-copied into
//    shared memory before griddepcontrol.wait (tables and weights are never
//    written by the preceding kernel), and a CTA takes under half of an SM, so
//    the next fold's CTAs are resident and load their pairs while this fold
//    finishes (programmatic dependent launch);
//  * the rows of the expert are found before the wait by a speculative scan of
//    the routing (L2 loads only; the values may still change), and their x
//    and base_out lines are prefetched into L2.  After the wait the x rows and
//    base_out rows of that row list are requested at once with the fresh
//    routing loads; the first pass's x is shrunk while those are in flight.
//    A routing of one scan chunk is compared value for value with what the
//    speculation read (kept in registers): unchanged, the speculative rows,
//    counts and roles stand; else the routing is scanned again and rows that
//    differ are requested again.  The round trip on the routing thus overlaps
//    the one on x and the shrink;
//  * shrink h = x A_e^T with mma.sync m16n8k16 (M = rank, N = 8 rows, k split
//    over the warps, partial sums added in a fixed order), h split into bf16
//    hi + lo halves (h enters the expand at ~2^-17 relative precision);
//  * expand with swapped operands, M = 16 rows of B_e, N = the 8 rows, K =
//    rank; each lane takes adjacent rank words of B_e and h (the same physical
//    rank assignment for both operands), and the B_e rows are dealt to the M
//    rows so that every lane ends with 8 adjacent output columns of two rows:
//    base_out is read (into registers, right after the wait) and written with
//    16-byte accesses, rounded once: RNE(base + scale * delta).  B_e sits in
//    shared memory with its rows XOR-permuted for conflict-free loads: every
//    thread copies its 16-byte pieces of B_e (cp.async) straight into their
//    rows' slots, so no permutation pass follows the copy;
//  * an expert with more than 6 rows gets a helper CTA (the SMs left over by
//    the experts): the owner folds the first half of its rows, the helper the
//    second, both deciding the split from the same per-expert row counts
//    (the rows a CTA stores bound its time: one SM writes ~32 B per cycle).
// Rows are folded 8 at a time; an expert with more rows runs several passes.
// Multi-adapter tables (one set of cells per adapter slot) take a second form
// of the kernel, described at decode_fold_kernel.
#include <cuda_bf16.h>

#include <mutex>

#include "mlg_internal.h"
#include "mlg_ptx.cuh"

namespace mlg {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 8;         // rows per pass: expand M rows g = 0..7
constexpr int kMaxBlocks = 4;    // 64-column output blocks per warp (n_out <= 2048)
constexpr int kScanPer = 2;      // rows per thread per scan chunk (small code)
constexpr int kScanChunk = kScanPer * kThreads;
constexpr int kSpecRows = 32;    // rows of the speculative scan kept for L2 prefetch
constexpr int kMaxCtas = 160;    // owner + helper CTAs (and table entries) at most
constexpr int kSplitRows = 6;    // an expert with more folding rows than this gets a helper
constexpr int kMaxUnits = 8;     // cells one CTA takes in the multi-adapter form
constexpr int kMaxCells = 1280;  // table cells of the multi-adapter form at most

static __device__ uint32_t g_decode_errors;

struct DecodeParams {
  const uint16_t *x;
  const int32_t *indices;
  const int32_t *row_adapter;
  const uint64_t *a_table;
  const uint64_t *b_table;
  const float *scale_table;
  uint16_t *base_out;
  int32_t n_slots, k_in, n_out, top_k, n_experts;  // n_experts: table cells
  int32_t e_model, n_adapters;  // multi-adapter tables (n_adapters > 0): cell = slot * e_model + id
  int32_t spec_mode;  // 0: speculative row scan, 1: none, 2: scan a different expert (tests)
  uint32_t stride_a;  // bytes per A_e / x row in shared memory
  uint32_t off_a, off_x, off_b, off_p, off_h, zero_bytes, smem_bytes;
};

__device__ __forceinline__ void record_error(uint32_t bit) { atomicOr(&g_decode_errors, bit); }

// L2-only loads: never served from a line this SM cached before the wait.
__device__ __forceinline__ int ld_cg_s32(const int32_t *p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_cg_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_v4(void *p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Issue the routing loads of one scan chunk (rows base + i*256 + tid).
__device__ __forceinline__ void scan_load(const DecodeParams &p, int base, int (&idx)[kScanPer],
                                          int (&ra)[kScanPer]) {
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    const int row = base + i * kThreads + threadIdx.x;
    idx[i] = -1;
    ra[i] = -1;
    if (row < p.n_slots) {
      idx[i] = ld_cg_s32(p.indices + row);
      ra[i] = ld_cg_s32(p.row_adapter + row / p.top_k);
    }
    if (p.n_adapters > 0)  // the row map names the table set: fold through its cell
      idx[i] = (ra[i] >= 0 && ra[i] < p.n_adapters && idx[i] >= 0 && idx[i] < p.e_model)
                   ? ra[i] * p.e_model + idx[i]
                   : -1;
  }
}

// Ordered list of the rows that fold through expert e: writes ranks
// [g0, g0 + cap) of the list to s_rows and returns the list's length.  The
// order (chunk, i, warp, lane) is the same in every call.  Block-uniform.
// When have0, the loads of the first chunk were issued by the caller.  With
// s_hist, also adds every folding row to its expert's count (e = -1 collects
// only the counts).
__device__ int scan_expert_rows(const DecodeParams &p, int e, int g0, int cap, int *s_rows,
                                int (*s_cnt)[kWarps], const int (&idx0)[kScanPer],
                                const int (&ra0)[kScanPer], bool have0, int *s_hist) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int count = 0;
  for (int base = 0; base < p.n_slots; base += kScanChunk) {
    int idx[kScanPer], ra[kScanPer];
    if (base == 0 && have0) {
#pragma unroll
      for (int i = 0; i < kScanPer; ++i) {
        idx[i] = idx0[i];
        ra[i] = ra0[i];
      }
    } else {
      scan_load(p, base, idx, ra);
    }
    if (s_hist != nullptr) {  // folding rows per expert (ids in the table only)
#pragma unroll
      for (int i = 0; i < kScanPer; ++i)
        if (ra[i] >= 0 && idx[i] >= 0 && idx[i] < p.n_experts) atomicAdd(&s_hist[idx[i]], 1);
    }
    unsigned mask[kScanPer];
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      mask[i] = __ballot_sync(0xffffffffu, e >= 0 && idx[i] == e && ra[i] >= 0);
      if (lane == 0) s_cnt[i][warp] = __popc(mask[i]);
    }
    __syncthreads();
    int run = count;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      int mine = run;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mine += (w < warp) ? s_cnt[i][w] : 0;
      const int rank = mine + __popc(mask[i] & ((1u << lane) - 1u));
      if (((mask[i] >> lane) & 1u) && rank >= g0 && rank < g0 + cap)
        s_rows[rank - g0] = base + i * kThreads + tid;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) run += s_cnt[i][w];
    }
    count = run;
    __syncthreads();
  }
  return count;
}

// One pass's x rows into shared memory: warp 0, bulk copies on bar_x.
__device__ __forceinline__ void request_x(const DecodeParams &p, int warp, int lane, int n_g,
                                          uint32_t row_bytes_x, bool bad, const int *s_rows,
                                          uint8_t *sX, uint32_t bar_x) {
  if (warp == 0 && !bad) {
    if (lane == 0) mbar_arrive_expect_tx(bar_x, n_g * row_bytes_x);
    __syncwarp();
    if (lane < n_g)
      bulk_g2s(smem_addr(sX + lane * p.stride_a),
               p.x + static_cast<size_t>(s_rows[lane] / p.top_k) * p.k_in, row_bytes_x, bar_x);
  }
}

// This lane's base_out rows (rows 2c and 2c+1 of the pass) in 16-byte chunks:
// columns blk*64 + 8g .. +7 of the warp's 64-column blocks, into registers.
// Of the columns [col0, col0 + n_cols) only (the whole row in the single-table form).
__device__ __forceinline__ void request_base(const DecodeParams &p, int warp, int g, int c,
                                             int n_g, const int *s_rows,
                                             uint4 (&base_v)[kMaxBlocks][2], int (&my_row)[2],
                                             int col0, int n_cols) {
  my_row[0] = 2 * c < n_g ? s_rows[2 * c] : -1;
  my_row[1] = 2 * c + 1 < n_g ? s_rows[2 * c + 1] : -1;
#pragma unroll
  for (int i = 0; i < kMaxBlocks; ++i) {
    const int col = (warp + i * kWarps) * 64 + 8 * g;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      base_v[i][r] = make_uint4(0, 0, 0, 0);
      if (my_row[r] >= 0 && col < n_cols)
        base_v[i][r] =
            ld_cg_v4(p.base_out + static_cast<size_t>(my_row[r]) * p.n_out + col0 + col);
    }
  }
}

template <int N>
__device__ __forceinline__ void load_words(uint32_t (&w)[N], const uint8_t *s) {
  if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2 *>(s);
    w[0] = v.x;
    w[1] = v.y;
  } else {
    const uint4 v = *reinterpret_cast<const uint4 *>(s);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
}

__device__ __forceinline__ uint32_t fold_pair(uint32_t base2, float d0, float d1, float scale) {
  const float r0 = fmaf(scale, d0, __uint_as_float(base2 << 16));
  const float r1 = fmaf(scale, d1, __uint_as_float(base2 & 0xffff0000u));
  uint32_t o;  // round both to nearest even; r1 into the upper half
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(r1), "f"(r0));
  return o;
}

// Row slot of B_e row r in shared memory: within each 128-byte group of rows,
// the slots are XOR-permuted by bits 3.. of r, so that the rows one expand
// load touches (8g + 2t for g = 0..7) fall on distinct banks.
template <int RP>
__device__ __forceinline__ int b_slot(int r) {
  constexpr int RPC = 64 / RP;  // rows per 128 bytes
  return r ^ ((r >> 3) & (RPC - 1));
}

// The expand of one 64-column block: swapped operands, M = 16 B_e rows, N =
// the 8 rows of the pass, K = rank, h as hi + lo, four m-tiles t.  M-row g of
// tile t takes B_e row blk*64 + 8g + 2t and M-row g+8 the next one, so lane
// (g, c) -- whose D holds M-rows g, g+8 of rows 2c, 2c+1 -- ends with output
// columns blk*64 + 8g .. +7 of both rows: tile t gives columns 8g + 2t (d[t][0]
// row 2c, d[t][1] row 2c+1) and 8g + 2t + 1 (d[t][2], d[t][3]).  No transpose
// before the 16-byte base_out accesses.  B_e rows at or past n_out read as 0.
template <int RP>
__device__ __forceinline__ void expand_block(float (&d)[4][4], const uint8_t *sB,
                                             const uint32_t (&hh)[RP / 8],
                                             const uint32_t (&hl)[RP / 8], int blk, int n_out) {
  constexpr int WPL = RP / 8, KST = RP / 16;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int row0 = blk * 64 + 8 * g;
  const bool ok = row0 < n_out;  // n_out % 8 == 0: all 8 rows or none
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint32_t b0[WPL], b1[WPL];
#pragma unroll
    for (int w = 0; w < WPL; ++w) b0[w] = b1[w] = 0u;
    if (ok) {
      load_words<WPL>(b0, sB + (b_slot<RP>(row0 + 2 * t) * RP + c * WPL * 2) * 2);
      load_words<WPL>(b1, sB + (b_slot<RP>(row0 + 2 * t + 1) * RP + c * WPL * 2) * 2);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) d[t][u] = 0.f;
#pragma unroll
    for (int st = 0; st < KST; ++st) {
      mma_bf16_16816(d[t], b0[2 * st], b1[2 * st], b0[2 * st + 1], b1[2 * st + 1], hh[2 * st],
                     hh[2 * st + 1]);
      mma_bf16_16816(d[t], b0[2 * st], b1[2 * st], b0[2 * st + 1], b1[2 * st + 1], hl[2 * st],
                     hl[2 * st + 1]);
    }
  }
}

// Which expert a helper CTA takes, or whether an owner has a helper, from the
// per-expert counts of folding rows: an expert with more than kSplitRows rows
// is "heavy"; the i-th heavy expert (by id) gets helper CTA i, if there is one.
// Warp 0 computes it; the result is in *s_out after the next barrier.
__device__ __forceinline__ void assign_helper(const int *s_hist, int n_experts, int n_helpers,
                                              bool helper, int who, int *s_out) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) != 0) return;
  int run = 0, found = helper ? -1 : 0;
  for (int b = 0; b < n_experts; b += 32) {
    const int e = b + lane;
    const bool heavy = e < n_experts && s_hist[e] > kSplitRows;
    const unsigned mask = __ballot_sync(0xffffffffu, heavy);
    const int rank = run + __popc(mask & ((1u << lane) - 1u));
    if (heavy && rank < n_helpers) {
      if (helper && rank == who) found = e;
      if (!helper && e == who) found = 1;
    }
    run += __popc(mask);
  }
  // at most one lane found something; combine over the warp
  const int v = __reduce_max_sync(0xffffffffu, found);
  if (lane == 0) *s_out = v;
}

// MULTI = false: one CTA per table entry, its pair requested before the grid
// dependency wait (plus helper CTAs for heavy experts).  MULTI = true (the
// multi-adapter tables, where a batch hits few of many cells): the cells the
// routing hits are dealt round-robin to the CTAs, each folding its cells one
// after another; the first cell is picked from a speculative (L2-only) read
// of the routing before the wait, so its pair loads while the preceding
// kernel runs, and is kept only if the fresh routing deals the same cell.
template <int RP, bool MULTI>  // max_rank: 16 or 32
__global__ void __launch_bounds__(kThreads, 2) decode_fold_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2];  // 0: the pair, 1: x rows
  __shared__ int s_spec[kSpecRows];
  __shared__ int s_rows[kSpecRows];  // ranks [list0, list0 + 32) of the row list
  __shared__ int s_cnt[kScanPer][kWarps];
  __shared__ int s_hist[kMaxCtas];   // folding rows per expert
  __shared__ int s_role;
  __shared__ int s_units[kMaxUnits];  // MULTI: this CTA's cells
  __shared__ uint32_t s_fold[MULTI ? kMaxCells / 32 : 1];  // MULTI: foldable cells, one bit each

  constexpr int MT = RP / 16;   // rank m-tiles of the shrink
  constexpr int WPL = RP / 8;   // rank words (bf16 pairs) per lane in the expand
  constexpr int PS = RP + 4;    // fp32 row stride of the shrink partials

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;

  uint8_t *sA = smem + p.off_a;
  uint8_t *sX = smem + p.off_x;
  const uint8_t *sB = smem + p.off_b;
  float *sP = reinterpret_cast<float *>(smem + p.off_p);
  uint8_t *sHhi = smem + p.off_h;
  uint8_t *sHlo = sHhi + kRows * RP * 2;

  // The k tail of the A_e / x rows (up to the next 32 columns) is read by the
  // MMAs but never written by a copy: zero it once.
  for (uint32_t i = tid * 16; i < p.zero_bytes; i += kThreads * 16)
    *reinterpret_cast<uint4 *>(smem + i) = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < kMaxCtas; i += kThreads) s_hist[i] = 0;
  const uint32_t bar_w = smem_addr(&bars[0]), bar_x = smem_addr(&bars[1]);
  if (tid == 0) {
    mbar_init(bar_w, 1 + kThreads);  // the A_e copies' expect_tx + every thread's B_e copies
    mbar_init(bar_x, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // The next fold in the stream may start its prologue now: before its own
  // wait it reads tables and weights, and the routing through L2 only.
  griddep_launch_dependents();

  const int no_idx[kScanPer] = {};
  const int kblocks = (p.k_in + 31) / 32;
  const uint32_t row_bytes_x = static_cast<uint32_t>(p.k_in) * 2u;
  uint32_t ph_w = 0, ph_x = 0;
  bool bad = false;

  // Owner CTA e folds expert e; helper CTA h (blockIdx >= n_experts) folds the
  // second half of the rows of the h-th heavy expert, whose owner folds the first.
  const bool helper = !MULTI && static_cast<int>(blockIdx.x) >= p.n_experts;
  const int who = helper ? static_cast<int>(blockIdx.x) - p.n_experts : static_cast<int>(blockIdx.x);
  const int n_helpers = MULTI ? 0 : static_cast<int>(gridDim.x) - p.n_experts;
  const bool spec = p.spec_mode != 1;
  int e = helper ? -1 : who;
  int total = 0;
  float scale = 0.f;
  bool pair = false;  // the pair of expert e was requested on bar_w

  // Columns of this CTA's current unit: [col0, col0 + n_cols).  The
  // single-table form always takes whole rows; the multi-adapter form may
  // split a cell's columns over two CTAs.
  int col0_v = 0, n_cols_v = p.n_out;
  auto col0 = [&]() { return MULTI ? col0_v : 0; };
  auto n_cols = [&]() { return MULTI ? n_cols_v : p.n_out; };

  // Table entry of expert ex; on a foldable pair, request it (CTA-uniform):
  // all of A_e and the B_e rows of this unit's columns.
  auto request_pair = [&](int ex) -> bool {
    const uint64_t a_addr = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + ex);
    const uint64_t b_addr = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + ex);
    scale = __ldg(p.scale_table + ex);
    if (a_addr == 0 || b_addr == 0 || ((a_addr | b_addr) & 15u) != 0) return false;
    if (!bad) {
      if (warp == 0) {  // one bulk copy per A_e row
        if (lane == 0) mbar_arrive_expect_tx(bar_w, RP * row_bytes_x);
        __syncwarp();
        const uint8_t *A = reinterpret_cast<const uint8_t *>(a_addr);
        for (int j = lane; j < RP; j += 32)
          bulk_g2s(smem_addr(sA + j * p.stride_a), A + static_cast<size_t>(j) * row_bytes_x,
                   row_bytes_x, bar_w);
      }
      // The B_e rows of this unit's columns, each 16-byte piece straight into
      // its row's bank-spread slot (no permutation pass after it lands); every
      // thread's copies complete on bar_w through cp.async.mbarrier.arrive.
      constexpr int RB = 2 * RP;  // bytes per B_e row
      const uint8_t *B = reinterpret_cast<const uint8_t *>(b_addr) + static_cast<size_t>(col0()) * RB;
      const int pieces = n_cols() * RB / 16;
      uint8_t *sBw = smem + p.off_b;
      for (int i = tid; i < pieces; i += kThreads) {
        const int r = (i * 16) / RB, off = (i * 16) % RB;
        cp_async_16(smem_addr(sBw + b_slot<RP>(r) * RB + off), B + i * 16, 16u);
      }
      cp_async_arrive_noinc(bar_w);
    }
    return true;
  };
  auto spec_target = [&](int ex) { return p.spec_mode == 2 ? (ex + 1) % p.n_experts : ex; };

  // State of the passes over one expert's rows (set by each form below).
  uint4 base_v[kMaxBlocks][2];
  int my_row[2] = {-1, -1};
  bool have_pair = false;
  bool issued = false;  // the next pass's x copies and base_out loads are in flight
  int list0 = 0;        // rank of s_rows[0] in the row list
  int g_begin = 0, g_end = 0;
  bool h_ready = false;  // the first pass's h is already split into sHhi / sHlo

  // ---- shrink: h[row][j] = sum_k x[row][k] A_e[j][k] over the pass's x rows
  // in sX, k split over warps, into the warps' partials.  Lane column c feeds
  // physical k = 8c .. 8c+7 of every 32-wide k block to both operands, so the
  // contraction covers every k once.
  auto shrink_pass = [&]() {
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    for (int kb = warp; kb < kblocks; kb += kWarps) {
      const uint32_t kbyte = (kb * 32 + 8 * c) * 2;
      const uint4 sx = *reinterpret_cast<const uint4 *>(sX + g * p.stride_a + kbyte);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint4 pa = *reinterpret_cast<const uint4 *>(sA + (mt * 16 + g) * p.stride_a + kbyte);
        const uint4 qa = *reinterpret_cast<const uint4 *>(sA + (mt * 16 + g + 8) * p.stride_a + kbyte);
        mma_bf16_16816(acc[mt], pa.x, qa.x, pa.y, qa.y, sx.x, sx.y);
        mma_bf16_16816(acc[mt], pa.z, qa.z, pa.w, qa.w, sx.z, sx.w);
      }
    }
    // acc[mt] = (j mt*16+g, row 2c), (j, row 2c+1), (j+8, row 2c), (j+8, row 2c+1)
    float *part = sP + warp * (kRows * PS);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int j = mt * 16 + g, row = 2 * c;
      part[row * PS + j] = acc[mt][0];
      part[(row + 1) * PS + j] = acc[mt][1];
      part[row * PS + j + 8] = acc[mt][2];
      part[(row + 1) * PS + j + 8] = acc[mt][3];
    }
    __syncthreads();
  };
  // Sum the warps' partials in warp order; split h into bf16 hi + lo.
  auto split_h = [&]() {
    if (tid < kRows * RP / 2) {
      const int row = (2 * tid) / RP, j = (2 * tid) % RP;
      float h0 = 0.f, h1 = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        h0 += sP[w * (kRows * PS) + row * PS + j];
        h1 += sP[w * (kRows * PS) + row * PS + j + 1];
      }
      float a0, b0, a1, b1;
      split_hi_lo(h0, a0, b0);
      split_hi_lo(h1, a1, b1);
      *reinterpret_cast<uint32_t *>(sHhi + (row * RP + j) * 2) = pack_bf16x2(a0, a1);
      *reinterpret_cast<uint32_t *>(sHlo + (row * RP + j) * 2) = pack_bf16x2(b0, b1);
    }
    __syncthreads();
  };

  // Fold rows [g_begin, g_end) of expert e's row list, kRows per pass.
  auto run_passes = [&]() {
    bool timed_out = false;
    for (int g0 = g_begin; g0 < g_end && !bad; g0 += kRows) {
      if (g0 + kRows > list0 + kSpecRows) {  // this pass's rows are past the list
        scan_expert_rows(p, e, g0, kSpecRows, s_rows, s_cnt, no_idx, no_idx, false, nullptr);
        list0 = g0;
      }
      const int *rows = s_rows + (g0 - list0);
      const int n_g = min(kRows, g_end - g0);
      if (!issued) {
        request_x(p, warp, lane, n_g, row_bytes_x, bad, rows, sX, bar_x);
        request_base(p, warp, g, c, n_g, rows, base_v, my_row, col0(), n_cols());
      }
      issued = false;
      timed_out = false;
      if (!have_pair) {  // the pair lands (B_e already in its bank-spread row slots)
        timed_out = tid == 0 && !mbar_wait_bounded(bar_w, ph_w);
        ph_w ^= 1u;
        have_pair = true;
        if (__syncthreads_or(timed_out)) {
          if (tid == 0) record_error(kErrWaitTimeout);
          bad = true;
          break;
        }
      }
      if (!h_ready) {
        // One thread polls; the barrier passes what it observed to the others.
        timed_out = tid == 0 && !mbar_wait_bounded(bar_x, ph_x);
        ph_x ^= 1u;
        if (__syncthreads_or(timed_out)) {  // (also orders the landed B_e before its reads)
          if (tid == 0) record_error(kErrWaitTimeout);
          bad = true;
          break;
        }
        shrink_pass();
      }
      // The next pass of this CTA (its rows already in s_rows): its x rows are
      // requested now that sX is free, its base_out rows as the quads of this
      // pass retire, so neither round trip is exposed.
      const int g1 = g0 + kRows;
      const bool pre = g1 < g_end && g1 + kRows <= list0 + kSpecRows;  // CTA-uniform
      const int *rows1 = s_rows + (g1 - list0);
      const int n_g1 = pre ? min(kRows, g_end - g1) : 0;
      int my_row1[2];
      my_row1[0] = 2 * c < n_g1 ? rows1[2 * c] : -1;
      my_row1[1] = 2 * c + 1 < n_g1 ? rows1[2 * c + 1] : -1;
      if (pre) request_x(p, warp, lane, n_g1, row_bytes_x, bad, rows1, sX, bar_x);
      if (!h_ready) split_h();
      h_ready = false;

      // ---- expand + epilogue (see expand_block).  Lane c takes rank words
      // c*WPL .. c*WPL+WPL-1 of h and of B_e: k-step st uses word c*WPL + 2st
      // (logical k 2c, 2c+1) and the next (logical 2c+8, 2c+9).
      {
        uint32_t hh[WPL], hl[WPL];
        load_words<WPL>(hh, sHhi + (g * RP + c * WPL * 2) * 2);
        load_words<WPL>(hl, sHlo + (g * RP + c * WPL * 2) * 2);
        // base_v[0] is always the current block: the registers rotate down and
        // the next pass's loads enter at the top.
#pragma unroll
        for (int i = 0; i < kMaxBlocks; ++i) {
          const int blk = warp + i * kWarps;
          uint4 nv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
          if (blk * 64 < n_cols()) {  // warp-uniform
            float d[4][4];
            expand_block<RP>(d, sB, hh, hl, blk, n_cols());
            const int col = col0() + blk * 64 + 8 * g;
            const bool col_ok = col < col0() + n_cols();
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              if (my_row[r] >= 0 && col_ok) {
                const uint4 b = base_v[0][r];
                uint4 o;
                o.x = fold_pair(b.x, d[0][r], d[0][r + 2], scale);
                o.y = fold_pair(b.y, d[1][r], d[1][r + 2], scale);
                o.z = fold_pair(b.z, d[2][r], d[2][r + 2], scale);
                o.w = fold_pair(b.w, d[3][r], d[3][r + 2], scale);
                st_v4(p.base_out + static_cast<size_t>(my_row[r]) * p.n_out + col, o);
              }
              if (pre && my_row1[r] >= 0 && col_ok)
                nv[r] = ld_cg_v4(p.base_out + static_cast<size_t>(my_row1[r]) * p.n_out + col);
            }
          }
#pragma unroll
          for (int k = 0; k + 1 < kMaxBlocks; ++k) {
            base_v[k][0] = base_v[k + 1][0];
            base_v[k][1] = base_v[k + 1][1];
          }
          base_v[kMaxBlocks - 1][0] = nv[0];
          base_v[kMaxBlocks - 1][1] = nv[1];
        }
      }
      __syncthreads();  // sP / sH are rewritten by the next pass
      if (pre) {
        my_row[0] = my_row1[0];
        my_row[1] = my_row1[1];
        issued = true;
      }
    }
  };
  auto drain = [&]() {
    // Let every copy still in flight land before leaving (a pair requested but
    // never waited for when no pass ran; after a timeout, whatever was issued).
    if (pair && !have_pair) {
      const bool t = tid == 0 && !mbar_wait_bounded(bar_w, ph_w);
      if (t && tid == 0) record_error(kErrWaitTimeout);
    }
    if (issued) {
      const bool t = tid == 0 && !mbar_wait_bounded(bar_x, ph_x);
      if (t && tid == 0) record_error(kErrWaitTimeout);
    }
  };

  if constexpr (!MULTI) {
    // ---- before the wait: the pair, and a speculative row list (L2 loads only)
    // When the routing is one scan chunk, the values read here are kept, so
    // that after the wait an unchanged routing confirms everything derived
    // from them without a second scan.
    int idx_s[kScanPer] = {}, ra_s[kScanPer] = {};
    const bool snap = spec && p.n_slots <= kScanChunk;
    if (snap) scan_load(p, 0, idx_s, ra_s);
    // An owner knows its expert without the routing: its table entry and pair
    // are requested while the routing loads are in flight.
    if (!helper) pair = request_pair(e);
    if (spec) {
      total = scan_expert_rows(p, helper ? -1 : spec_target(e), 0, kSpecRows, s_spec, s_cnt, idx_s,
                               ra_s, snap, s_hist);
      if (helper) {
        // (spec_mode 2: a different heavy expert, so that the check after the wait fails)
        assign_helper(s_hist, p.n_experts, n_helpers + 1, true, p.spec_mode == 2 ? who + 1 : who,
                      &s_role);
        __syncthreads();
        e = s_role;
        if (e >= 0)
          total = scan_expert_rows(p, spec_target(e), 0, kSpecRows, s_spec, s_cnt, idx_s, ra_s,
                                   snap, nullptr);
      }
    }
    int spec_role = 0;  // owner: 1 if the speculative counts give it a helper
    if (spec && !helper) {
      assign_helper(s_hist, p.n_experts, n_helpers, false, who, &s_role);
      __syncthreads();
      spec_role = s_role;
    }
    if (helper && e >= 0) pair = request_pair(e);
    // Rows of a split expert: the owner folds ranks [0, half), the helper
    // [half, total), half = ceil(total / 2); passes of up to 8 rows each.
    const bool spec_split = helper || spec_role == 1;
    const int spec_g0 = helper ? (total + 1) / 2 : 0;
    const int spec_end = (spec_split && !helper) ? (total + 1) / 2 : total;
    int n_spec = (spec && pair && spec_g0 < kSpecRows - kRows)
                     ? max(0, min(kRows, spec_end - spec_g0)) : 0;
    if (warp == 1 && lane < n_spec) {
      const int row = s_spec[spec_g0 + lane];
      prefetch_l2(p.x + static_cast<size_t>(row / p.top_k) * p.k_in, row_bytes_x);
      prefetch_l2(p.base_out + static_cast<size_t>(row) * p.n_out, static_cast<uint32_t>(p.n_out) * 2u);
    }
    for (int i = tid; i < kMaxCtas; i += kThreads) s_hist[i] = 0;
    __syncthreads();
    griddep_wait();  // routing, x and base_out may be written by the preceding kernel

    // ---- after the wait: the speculative first pass's x and base_out rows, the
    // fresh scan's loads and its base_out loads are all in flight together,
    // and only then is the pair (requested at the start) waited for, so that
    // none of these round trips queues behind it when nothing ran before.
    if (n_spec > 0) request_x(p, warp, lane, n_spec, row_bytes_x, bad, s_spec + spec_g0, sX, bar_x);
    int idx0[kScanPer], ra0[kScanPer];
    scan_load(p, 0, idx0, ra0);
    if (n_spec > 0)
      request_base(p, warp, g, c, n_spec, s_spec + spec_g0, base_v, my_row, 0, p.n_out);
    if (pair) {  // the pair has landed (B_e straight into its bank-spread row slots)
      const bool t = tid == 0 && !mbar_wait_bounded(bar_w, ph_w);
      ph_w ^= 1u;
      have_pair = true;
      if (__syncthreads_or(t)) {
        if (tid == 0) record_error(kErrWaitTimeout);
        bad = true;
      }
    }
    // The speculative first pass's h, while the fresh routing loads are in
    // flight: its x rows land and are shrunk before the scan is read, and the
    // h is kept only if the scan confirms the rows (h_ready below).
    bool x_landed = false;
    if (n_spec > 0 && have_pair && !bad) {
      const bool t = tid == 0 && !mbar_wait_bounded(bar_x, ph_x);
      ph_x ^= 1u;
      x_landed = true;
      if (__syncthreads_or(t)) {
        if (tid == 0) record_error(kErrWaitTimeout);
        bad = true;
      } else {
        shrink_pass();
        split_h();
      }
    }
    // The speculation stands as a whole when the routing it read (one chunk,
    // its own expert) is unchanged: its rows, counts and roles are then the
    // fresh ones.  Otherwise scan again and check the first pass's rows.
    int fresh = total;
    int role = helper ? e : spec_role;  // helper: its expert; owner: 1 if it has a helper
    bool timed_out = false;
    bool same = snap && p.spec_mode == 0;
    if (same) {
#pragma unroll
      for (int i = 0; i < kScanPer; ++i) same = same && idx0[i] == idx_s[i] && ra0[i] == ra_s[i];
      same = !__syncthreads_or(!same);
    }
    if (same) {
      if (tid < kSpecRows) s_rows[tid] = s_spec[tid];
      __syncthreads();
    } else {
      fresh = scan_expert_rows(p, e, 0, kSpecRows, s_rows, s_cnt, idx0, ra0, true, s_hist);
      assign_helper(s_hist, p.n_experts, n_helpers, helper, who, &s_role);
      __syncthreads();
      role = s_role;
      if (helper && role != e) {  // the speculation picked another expert (or none)
        if (n_spec > 0 && !x_landed) {
          timed_out = !bad && tid == 0 && !mbar_wait_bounded(bar_x, ph_x);
          ph_x ^= 1u;
        }
        if (pair && !have_pair) {
          timed_out = (!bad && tid == 0 && !mbar_wait_bounded(bar_w, ph_w)) || timed_out;
          ph_w ^= 1u;
        }
        have_pair = false;
        if (__syncthreads_or(timed_out)) {
          if (!bad && tid == 0) record_error(kErrWaitTimeout);
          bad = true;
        }
        n_spec = 0;
        my_row[0] = my_row[1] = -1;
        e = role;
        pair = false;
        if (e >= 0 && !bad) {
          fence_proxy_async_smem();  // the old pair's buffers were read by no one; order anyway
          pair = request_pair(e);
          if (pair)
            fresh = scan_expert_rows(p, e, 0, kSpecRows, s_rows, s_cnt, no_idx, no_idx, false,
                                     nullptr);
        }
      } else if (n_spec > 0) {
        // The speculative rows stand if the fresh scan agrees.
        // (equal totals and roles give the same first pass [spec_g0, spec_g0 + n_spec))
        bool differ = tid == 0 && (fresh != total || (!helper && role != spec_role));
        if (tid < n_spec && s_rows[spec_g0 + tid] != s_spec[spec_g0 + tid]) differ = true;
        if (__syncthreads_or(differ)) {  // let the copies of the stale rows land first
          if (!x_landed) {
            timed_out = !bad && tid == 0 && !mbar_wait_bounded(bar_x, ph_x);
            ph_x ^= 1u;
          }
          if (__syncthreads_or(timed_out)) {
            if (!bad && tid == 0) record_error(kErrWaitTimeout);
            bad = true;
          }
          n_spec = 0;
          my_row[0] = my_row[1] = -1;
        }
      }
    }
    total = pair ? fresh : 0;
    const bool split = helper || role == 1;
    g_begin = helper ? (total + 1) / 2 : 0;
    g_end = (split && !helper) ? (total + 1) / 2 : total;
    issued = n_spec > 0;  // the first pass's x copies and base_out loads are in flight
    h_ready = issued && x_landed && !bad;  // ... and its x already shrunk into h
    list0 = 0;
    run_passes();
    drain();
  } else {
    // ---- before the wait: which cells fold (the tables are never written by
    // the preceding kernel), a speculative unit list from an L2-only routing
    // scan, and the pair of this CTA's first speculative cell.
    int *hist = reinterpret_cast<int *>(smem + p.off_p);  // free until the first shrink
    for (int b = 0; b < p.n_experts; b += kThreads) {
      const int ex = b + tid;
      bool f = false;
      if (ex < p.n_experts) {
        const uint64_t a = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + ex);
        const uint64_t bb = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + ex);
        f = a != 0 && bb != 0 && ((a | bb) & 15u) == 0;
      }
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (lane == 0) s_fold[(b >> 5) + warp] = m;
    }
    // Units: the foldable cells with a folding row, in cell order; the one of
    // rank k < G goes to CTA k.  Cells past the first round of G are split by
    // columns into two halves (when n_out is a multiple of 128), half j of
    // the extra ones going to CTA j mod G, so no CTA folds a second whole
    // cell while the rest wait.  An entry of s_units is cell | (half + 1) << 28
    // (0: the whole cell).  Returns this CTA's count.
    const int G = static_cast<int>(gridDim.x);
    const bool halves = p.n_out % 128 == 0;
    auto deal_units = [&](int me, const int (&idx0)[kScanPer], const int (&ra0)[kScanPer],
                          bool have0) -> int {
      for (int i = tid; i < p.n_experts; i += kThreads) hist[i] = 0;
      __syncthreads();
      scan_expert_rows(p, -1, 0, 0, s_rows, s_cnt, idx0, ra0, have0, hist);
      int n_hit = 0;
      for (int b = 0; b < p.n_experts; b += kThreads) {
        const int ex = b + tid;
        const bool f = ex < p.n_experts && hist[ex] > 0 && ((s_fold[ex >> 5] >> (ex & 31)) & 1u);
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (lane == 0) s_cnt[0][warp] = __popc(m);
        __syncthreads();
        int before = n_hit;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          before += (w < warp) ? s_cnt[0][w] : 0;
          n_hit += s_cnt[0][w];
        }
        const int rank = before + __popc(m & ((1u << lane) - 1u));
        if (f && (!halves || rank < G)) {
          if (rank % G == me && rank / G < kMaxUnits) s_units[rank / G] = ex;
        } else if (f) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = 2 * (rank - G) + h;
            if (j % G == me && 1 + j / G < kMaxUnits) s_units[1 + j / G] = ex | ((h + 1) << 28);
          }
        }
        __syncthreads();
      }
      // The count before clamping to s_units: the host's eligibility check
      // keeps it within kMaxUnits; a larger one is recorded, not hidden.
      if (!halves) return n_hit > me ? (n_hit - 1 - me) / G + 1 : 0;
      const int extra = 2 * max(0, n_hit - G);  // half units past the first round
      return (n_hit > me ? 1 : 0) + (extra > me ? (extra - 1 - me) / G + 1 : 0);
    };
    // (spec_mode 1: no speculation; 2: another CTA's first cell, so that the
    // check after the wait fails)
    const int me = static_cast<int>(blockIdx.x);
    // When the routing is one scan chunk, the values read here are kept: if
    // they are unchanged after the wait, the units and the first cell's rows
    // dealt from them stand without a second read.
    int idx_s[kScanPer] = {}, ra_s[kScanPer] = {};
    const bool snap = spec && p.spec_mode == 0 && p.n_slots <= kScanChunk;
    if (snap) scan_load(p, 0, idx_s, ra_s);
    int n_mine = spec ? deal_units(p.spec_mode == 2 ? (me + 1) % G : me, idx_s, ra_s, snap) : 0;
    const int n_mine_spec = n_mine;
    n_mine = min(kMaxUnits, n_mine);
    const int e_spec = n_mine > 0 ? s_units[0] : -1;
    bool spec_pair = false;
    int ns = 0;  // rows of the first cell (first kSpecRows of them in s_spec)
    if (e_spec >= 0) {
      spec_pair = request_pair(e_spec);
      ns = scan_expert_rows(p, e_spec, 0, kSpecRows, s_spec, s_cnt, idx_s, ra_s, snap, nullptr);
      if (warp == 1 && lane < min(ns, kRows)) {
        const int row = s_spec[lane];
        prefetch_l2(p.x + static_cast<size_t>(row / p.top_k) * p.k_in, row_bytes_x);
        prefetch_l2(p.base_out + static_cast<size_t>(row) * p.n_out,
                    static_cast<uint32_t>(p.n_out) * 2u);
      }
      if (spec_pair) {  // one thread polls, pausing; the others sleep in the barrier
        const bool t = tid == 0 && !mbar_wait_bounded_sleep(bar_w, ph_w, 128);
        ph_w ^= 1u;
        if (__syncthreads_or(t)) {
          if (tid == 0) record_error(kErrWaitTimeout);
          bad = true;
        }
      }
    }
    __syncthreads();
    griddep_wait();  // the routing, x and base_out may be written by the preceding kernel

    // ---- after the wait: the fresh unit list; the first cell's pair is kept
    // when the speculation picked it.
    bool same = snap;
    if (same) {
      int idx0[kScanPer], ra0[kScanPer];
      scan_load(p, 0, idx0, ra0);
#pragma unroll
      for (int i = 0; i < kScanPer; ++i) same = same && idx0[i] == idx_s[i] && ra0[i] == ra_s[i];
      same = !__syncthreads_or(!same);
    }
    const int n_dealt = same ? n_mine_spec : deal_units(me, no_idx, no_idx, false);
    if (n_dealt > kMaxUnits && tid == 0) record_error(kErrUnitDropped);
    n_mine = min(kMaxUnits, n_dealt);
    for (int u = 0; u < n_mine && !bad; ++u) {
      e = s_units[u] & 0x0fffffff;
      const int half = (s_units[u] >> 28) - 1;  // -1: the whole cell
      col0_v = half < 0 ? 0 : half * (p.n_out / 2);
      n_cols_v = half < 0 ? p.n_out : p.n_out / 2;
      if (u == 0 && spec_pair && e == e_spec && half < 0) {
        pair = true;  // landed before the wait; scale set by its request
        have_pair = true;
      } else {
        fence_proxy_async_smem();  // the last unit's buffers were read: order before new copies
        __syncthreads();
        pair = request_pair(e);
        have_pair = false;
      }
      if (u == 0 && same && e == e_spec && half < 0) {  // the speculative rows stand
        if (tid < kSpecRows) s_rows[tid] = s_spec[tid];
        __syncthreads();
        total = pair ? ns : 0;
      } else {
        total = pair ? scan_expert_rows(p, e, 0, kSpecRows, s_rows, s_cnt, no_idx, no_idx, false,
                                        nullptr)
                     : 0;
      }
      g_begin = 0;
      g_end = total;
      issued = false;
      list0 = 0;
      my_row[0] = my_row[1] = -1;
      run_passes();
      drain();
    }
  }
}

int g_path_override = 0;  // 0 auto, 1 this kernel, 2 the cluster kernel
int g_spec_mode = 0;
constexpr uint32_t kSmemTwoPerSm = 113 * 1024 - 2048;  // with ~1.3 KB static and 1 KB reserved

uint32_t round_up(uint32_t v, uint32_t m) { return (v + m - 1) / m * m; }

int decode_grid() { return sm_count() < kMaxCtas ? sm_count() : kMaxCtas; }

uint32_t layout(DecodeParams &p, int rp) {
  const uint32_t kpad = round_up(static_cast<uint32_t>(p.k_in), 32) * 2;
  uint32_t sa = kpad;
  if (sa % 128 == 0) sa += 64;  // 16-byte operand loads of 8 rows conflict-free
  p.stride_a = sa;
  uint32_t off = 0;
  p.off_a = off;
  off += rp * sa;
  p.off_x = off;
  off += kRows * sa;
  p.zero_bytes = round_up(off, 16);
  off = round_up(off, 128);
  p.off_b = off;
  off += round_up(static_cast<uint32_t>(p.n_out) * rp * 2, 128);
  p.off_p = off;  // shrink partials
  off += kWarps * kRows * (rp + 4) * 4;
  p.off_h = off;
  off += 2 * kRows * rp * 2;
  p.smem_bytes = round_up(off, 128);
  return p.smem_bytes;
}

template <int RP, bool MULTI>
cudaError_t launch(const DecodeParams &p, int grid, bool early, cudaStream_t stream) {
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [d = dev & 63] {
    attr_err[d] = cudaFuncSetAttribute(decode_fold_kernel<RP, MULTI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemTwoPerSm));
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;  // without early start griddepcontrol.wait returns at once
  return cudaLaunchKernelEx(&cfg, decode_fold_kernel<RP, MULTI>, p);
}

}  // namespace

uint32_t decode_read_errors(bool clear) {
  uint32_t v = 0;
  cudaMemcpyFromSymbol(&v, g_decode_errors, sizeof v);
  if (clear) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(g_decode_errors, &z, sizeof z);
  }
  return v;
}

void gather_set_path_override(int path) { g_path_override = path; }
void gather_set_speculation(int mode) { g_spec_mode = mode; }
int gather_path_override() { return g_path_override; }

// Whether the resident-pair kernel takes this problem (shapes already
// validated): rank 16 or 32, n_out <= 2048, the pair, 8 x rows and the
// buffers within half an SM, and at most one expert per SM.
bool decode_fold_eligible(int32_t k_in, int32_t max_rank, int32_t n_out, int32_t n_cells) {
  if (max_rank != 16 && max_rank != 32) return false;
  if (n_out > kMaxBlocks * kWarps * 64) return false;
  if (n_cells > decode_grid()) return false;
  DecodeParams p = {};
  p.k_in = k_in;
  p.n_out = n_out;
  return layout(p, max_rank) <= kSmemTwoPerSm;
}

// The multi-cell form: the same pair limits, two CTAs on every SM, at most
// kMaxUnits cells per CTA, and the per-cell counts within the shrink
// partials' space.
bool decode_multi_eligible(int32_t k_in, int32_t max_rank, int32_t n_out, int32_t n_cells) {
  if (max_rank != 16 && max_rank != 32) return false;
  if (n_out > kMaxBlocks * kWarps * 64) return false;
  if (n_cells > kMaxCells) return false;
  // Units of one CTA when every cell is hit: one cell per CTA in the first
  // round, then (n_out a multiple of 128) two column halves per further cell
  // dealt round-robin, else whole cells round-robin.
  const int64_t G = 2 * static_cast<int64_t>(sm_count());
  const int64_t worst = n_out % 128 == 0
                            ? (n_cells > G ? 1 + (2 * (n_cells - G) + G - 1) / G : 1)
                            : (n_cells + G - 1) / G;
  if (worst > kMaxUnits) return false;
  if (static_cast<int64_t>(n_cells) * 4 > kWarps * kRows * (max_rank + 4) * 4) return false;
  DecodeParams p = {};
  p.k_in = k_in;
  p.n_out = n_out;
  return layout(p, max_rank) <= kSmemTwoPerSm;
}

cudaError_t decode_fold_launch(const uint16_t *x, const int32_t *indices,
                               const int32_t *row_adapter, const uint64_t *a_table,
                               const uint64_t *b_table, const float *scale_table,
                               uint16_t *base_out, int32_t n_slots, int32_t k_in,
                               int32_t max_rank, int32_t n_out, int32_t top_k,
                               int32_t n_cells, int32_t e_model, int32_t n_adapters,
                               bool early, cudaStream_t stream) {
  DecodeParams p = {};
  p.x = x;
  p.indices = indices;
  p.row_adapter = row_adapter;
  p.a_table = a_table;
  p.b_table = b_table;
  p.scale_table = scale_table;
  p.base_out = base_out;
  p.n_slots = n_slots;
  p.k_in = k_in;
  p.n_out = n_out;
  p.top_k = top_k;
  p.n_experts = n_cells;
  p.e_model = e_model;
  p.n_adapters = n_adapters;
  p.spec_mode = g_spec_mode;
  layout(p, max_rank);
  if (n_adapters > 0) {  // cells dealt to two CTAs per SM
    const int grid = 2 * sm_count();
    return max_rank == 16 ? launch<16, true>(p, grid, early, stream)
                          : launch<32, true>(p, grid, early, stream);
  }
  const int grid = decode_grid();  // owners, then helpers for experts with many rows
  return max_rank == 16 ? launch<16, false>(p, grid, early, stream)
                        : launch<32, false>(p, grid, early, stream);
}

}  // namespace mlg
