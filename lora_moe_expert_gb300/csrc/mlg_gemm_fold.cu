// mlg_gemm_fold.cu -- the MoE expert GEMM with the LoRA fold in its epilogue
// (per-row x form of the down projection).
//
// moe_lora_grouped_down (moe_lora_grouped module index) folds into base_out,
// and base_out is the expert projection's output.  Producing both in one
// kernel removes base_out's round trip through HBM: for every expert-sorted
// row r in [row_offset, row_end) held by span e < n_experts (W_e [n_out, k_in]
// bf16, slice e of the stacked expert weights),
//     out[r] = RNE_bf16( x_rows[r] @ W_e^T + [row folds] scale_e * (x_rows[r] @ A_e^T) @ B_e^T ),
// a row folding under the per-row x fold's rules (non-zero, aligned LoRA
// cells, src[r] >= 0 and a non-negative row-map entry for its token).
//
// GB300 design (one CTA per SM, persistent over expert-aligned tiles of <= 128
// rows that never cross a row window, dealt round-robin; the tiles of a last,
// partial round are split into pieces of their output chunks so that no CTA
// idles for a whole tile time):
//  * one shared-memory ring of stages, each an X box (128 rows x 64 k, TMA,
//    128-byte swizzle) and a Y tile (up to 256 rows x 64 k in the same
//    swizzle); per tile the ring carries, in order, the shrink's stages
//    [X | A_e chunk], then for every 256-column output chunk the GEMM stages
//    [X | W_e chunk] and one expand stage [- | B_e chunk].  X and W_e come in
//    as TMA boxes (W_e through one 3-D tensor map over the stacked weights);
//    A_e and B_e, found through the tables at run time, by 16-byte cp.async;
//  * warp 0 issues tcgen05.mma (kind::f16, cta_group::1): per output chunk
//    ACC = X W_e^T (M 128, N <= 256, K 64 a stage) into one of two TMEM
//    accumulators (all 512 columns), then ACC += [H_hi | H_lo] [B_e | B_e]^T
//    with h split into two bf16 halves (about 2^-18 relative), so h enters
//    the expand at about fp32 precision; h = X A_e^T itself is computed at
//    the start of the tile into the first columns of the accumulator that
//    the tile's first chunk then overwrites;
//  * warps 1-2 fill the ring (warp 1 lane 0 issues the TMA boxes);
//  * warps 4-11 split h (scaled, zero for rows that do not fold) into shared
//    memory, and per output chunk read their 32 rows x 128 columns of the
//    accumulator, release it, round once to bf16 and store: a warp whose 32
//    rows all belong to the tile writes 32 x 32 boxes into shared memory and
//    TMA-stores them; a partial box is stored row by row from registers
//    (32-byte stores when rows are 32-byte aligned); rows past the tile and
//    columns past n_out are never written.
// Every wait is bounded; a timeout sets an error bit and the CTA drains its
// copies and exits instead of hanging.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "mlg_internal.h"
#include "mlg_ptx.cuh"
#include "mlg_tiles.cuh"

namespace mlg {
namespace {

constexpr int kThreadsF = 384;     // warp 0 MMA, warps 1-2 ring fill, warp 3 idle, 4-11 epilogue
constexpr int kEpiWarpsF = 8;
constexpr int kTileMF = MLG_M_TILE;  // 128 rows per tile (the MMA M)
constexpr int kNch = 256;            // output columns per accumulator chunk (the MMA N)
constexpr int kMaxStagesF = 4;
constexpr int kMyTilesMaxF = 16;
constexpr uint32_t kTmemColsF = 512;
// TMEM: two 256-column accumulators; a tile's h is computed into the first
// columns of the accumulator its first output chunk will use.
__device__ __forceinline__ uint32_t acc_col(int b) { return b ? 256u : 0u; }
constexpr uint32_t kXBytes = kTileMF * 128;      // X box: 128 rows x 128 bytes
constexpr uint32_t kYBytes = kNch * 128;         // Y tile: 256 rows x 128 bytes

static __device__ uint32_t g_gemm_fold_errors;

struct FusedParams {
  const uint8_t *x;              // x_rows, bf16 [>= row_end, k_in]
  const int32_t *offsets;        // [n_experts + 1]
  const int32_t *src;            // sorted row -> flat row (row map only)
  const int32_t *row_adapter;    // [n_tokens] or null
  const uint64_t *a_table, *b_table;
  const float *scale_table;
  uint8_t *out;                  // bf16 [>= row_end, n_out], written
  int32_t k_in, rank, n_out, top_k, n_experts, row_offset, row_end;
  int32_t win, tile_m;           // window length, rows per tile
  int32_t r_pad, k_exp;          // rank rounded up to 16; expand K of [hi | lo], padded to 64
  int32_t kc_count, nc_count;    // 64-wide k chunks, 256-column output chunks
  int32_t nst;                   // ring stages
  int32_t v8;                    // 1: output rows 32-byte aligned (32-byte stores)
  int32_t staged;                // 1: whole 32-row boxes stored through shared memory by TMA
  uint32_t stage_bytes;
  uint32_t off_ring, off_h, off_stage, off_tab, off_my, smem_bytes;
};

constexpr uint32_t kStageBox = 32 * 64;  // one 32-row x 32-column bf16 output box (64B swizzle)

struct FCtl {
  uint64_t full[kMaxStagesF], empty[kMaxStagesF];
  uint64_t h_full, hs_full, hs_empty, acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  volatile int abort_flag;
};

// Per-CTA tile list entry: expert, rows, scale, and whether its LoRA pair folds.
struct FTile {
  int e, r0, r1;
  float scale;
  int lora;
  int nc0, nc1;  // the output chunks this CTA computes: [nc0, nc1)
};

__device__ __forceinline__ bool wait_f(FCtl &ctl, uint64_t &bar, uint32_t parity) {
  const uint32_t a = smem_addr(&bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (ctl.abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_gemm_fold_errors, kErrWaitTimeout);
      ctl.abort_flag = 1;
      return false;
    }
  }
}

// 3-D TMA load (x innermost, then y, then z) into shared memory, completion
// counted on `bar` in bytes, with an L2 cache hint.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void *tmap, int32_t x,
                                                 int32_t y, int32_t z, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st_global_v4(void *p, const uint32_t *v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}
// One whole 32-byte sector (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// RP: rank rounded up to a multiple of 16.
template <int RP>
__global__ void __launch_bounds__(kThreadsF, 1)
    gemm_fold_kernel(const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_out, const FusedParams p) {
  constexpr int KEXP = (2 * RP + 63) / 64 * 64;  // expand K: [hi | lo | zero pad]
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ FCtl ctl;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_e = p.n_experts;
  int *tile_start = reinterpret_cast<int *>(smem + p.off_tab);  // [n_e + 1]

  // ---- prologue: barriers and TMEM (overlaps the preceding kernel) --------
  if (tid == 0) {
    for (int s = 0; s < kMaxStagesF; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), 64);  // the 64 lanes of warps 1-2
      mbar_init(smem_addr(&ctl.empty[s]), 1);
    }
    mbar_init(smem_addr(&ctl.h_full), 1);
    mbar_init(smem_addr(&ctl.hs_full), 4);
    mbar_init(smem_addr(&ctl.hs_empty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&ctl.acc_full[b]), 1);
      mbar_init(smem_addr(&ctl.acc_empty[b]), kEpiWarpsF);
    }
    mbar_init(smem_addr(&ctl.drain), 1);
    ctl.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_x);
    prefetch_tmap(&tmap_w);
    if (p.staged) prefetch_tmap(&tmap_out);
  }
  __syncthreads();
  if (warp == 0) {
    tmem_alloc(smem_addr(&ctl.tmem_base), kTmemColsF);
    tmem_relinquish();
  }
  // Every input may be written by the preceding kernel: wait before the
  // first read of any of them.  The next kernel may start its own setup now.
  griddep_launch_dependents();
  griddep_wait();

  // Tile table: expert e contributes ceil(rows in window / 128) tiles;
  // exclusive prefix over experts.
  {
    int carry = 0;
    for (int base = 0; base < n_e; base += kThreadsF) {
      const int e = base + tid;
      int n = 0;
      if (e < n_e) n = span_tiles(p, span_lo(p, e), span_hi(p, e));
      int incl = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      __shared__ int warp_tot[kThreadsF / 32];
      if (lane == 31) warp_tot[warp] = incl;
      __syncthreads();
      int before = carry, total = 0;
#pragma unroll
      for (int w = 0; w < kThreadsF / 32; ++w) {
        before += (w < warp) ? warp_tot[w] : 0;
        total += warp_tot[w];
      }
      if (e < n_e) tile_start[e] = before + incl - n;
      carry += total;
      __syncthreads();
    }
    if (tid == 0) tile_start[n_e] = carry;
  }
  __syncthreads();
  // This CTA's work: tile c + i G of every full round i (all output chunks).
  // A tile costs about the same whatever its rows (its MMAs are per 128-row
  // tile), so a last round of R < G tiles would leave G - R CTAs idle for a
  // whole tile time (the 163840-row prefill: 1526 tiles on 152 SMs, 11 tile
  // times where 10.04 would do).  Its tiles are split instead into P pieces
  // of their output chunks, P = min(chunks, G / R), piece u going to CTA u
  // (each piece recomputes its tile's h; rows and results are unchanged).
  FTile *my_tiles = reinterpret_cast<FTile *>(smem + p.off_my);
  const int n_tiles_all = tile_start[n_e];
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const int q_full = n_tiles_all / G, rest = n_tiles_all % G;
  const int pieces = rest > 0 ? max(1, min(p.nc_count, G / rest)) : 1;
  const bool has_piece = cta < rest * pieces;
  const int my_count = min(kMyTilesMaxF, q_full + (has_piece ? 1 : 0));
  if (tid < my_count) {
    int t = cta + tid * G, nc0 = 0, nc1 = p.nc_count;
    if (tid == q_full) {  // this CTA's piece of a last-round tile
      const int j = cta % pieces;
      t = q_full * G + cta / pieces;
      nc0 = j * p.nc_count / pieces;
      nc1 = (j + 1) * p.nc_count / pieces;
    }
    const TileInfo ti = tile_info(p, tile_start, n_e, t);
    const uint64_t a = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + ti.e);
    const uint64_t b = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + ti.e);
    my_tiles[tid].e = ti.e;
    my_tiles[tid].r0 = ti.r0;
    my_tiles[tid].r1 = ti.r1;
    my_tiles[tid].scale = __ldg(p.scale_table + ti.e);
    my_tiles[tid].lora = cells_fold(a, b) ? 1 : 0;
    my_tiles[tid].nc0 = nc0;
    my_tiles[tid].nc1 = nc1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const int n_tiles = my_count;
  const uint32_t ring = smem_addr(smem + p.off_ring);
  const uint32_t h_base = smem_addr(smem + p.off_h);

  if (warp == 0) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_shrink = umma_idesc_bf16(kTileMF, RP);
      uint32_t it = 0, acc_it = 0, h_it = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const FTile mt = my_tiles[t];
        const int b0 = acc_it & 1;  // the accumulator of the tile's first chunk
        if (mt.lora) {
          // H = X A_e^T into the first columns of accumulator b0, once it is free
          if (!wait_f(ctl, ctl.acc_empty[b0], ((acc_it >> 1) & 1) ^ 1)) goto mma_done;
          tc_fence_after();
          for (int kc = 0; kc < p.kc_count; ++kc, ++it) {
            const int st = it % p.nst;
            if (!wait_f(ctl, ctl.full[st], (it / p.nst) & 1)) goto mma_done;
            fence_proxy_async_smem();  // A_e came in by cp.async (generic proxy)
            tc_fence_after();
            const uint32_t xs = ring + st * p.stage_bytes, ys = xs + kXBytes;
            const uint64_t ad = umma_desc_sw128(xs), bd = umma_desc_sw128(ys);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_bf16(tmem + acc_col(b0), ad + 2 * k, bd + 2 * k, idesc_shrink, (kc | k) != 0);
            umma_commit(smem_addr(&ctl.empty[st]));
          }
          umma_commit(smem_addr(&ctl.h_full));
          // the first chunk overwrites those columns: wait until the epilogue
          // has read h out of them (and written its split to shared memory)
          if (!wait_f(ctl, ctl.hs_full, h_it & 1)) goto mma_done;
          tc_fence_after();
        }
        for (int nc = mt.nc0; nc < mt.nc1; ++nc, ++acc_it) {
          const int b = acc_it & 1;
          const uint32_t d = tmem + acc_col(b);
          const int ncols = min(kNch, (p.n_out - nc * kNch + 15) / 16 * 16);
          const uint32_t idesc = umma_idesc_bf16(kTileMF, ncols);
          if (!(mt.lora && nc == mt.nc0)) {  // (the lora tile's first buffer was waited for above)
            if (!wait_f(ctl, ctl.acc_empty[b], ((acc_it >> 1) & 1) ^ 1)) goto mma_done;
            tc_fence_after();
          }
          for (int kc = 0; kc < p.kc_count; ++kc, ++it) {  // ACC = X W_e^T
            const int st = it % p.nst;
            if (!wait_f(ctl, ctl.full[st], (it / p.nst) & 1)) goto mma_done;
            tc_fence_after();
            const uint32_t xs = ring + st * p.stage_bytes, ys = xs + kXBytes;
            const uint64_t ad = umma_desc_sw128(xs), bd = umma_desc_sw128(ys);
#pragma unroll
            for (int k = 0; k < 4; ++k) umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kc | k) != 0);
            umma_commit(smem_addr(&ctl.empty[st]));
          }
          if (mt.lora) {  // ACC += [H_hi | H_lo] [B_e | B_e]^T
            const int st = it % p.nst;
            if (!wait_f(ctl, ctl.full[st], (it / p.nst) & 1)) goto mma_done;
            fence_proxy_async_smem();  // B_e came in by cp.async (generic proxy)
            tc_fence_after();
            const uint32_t ys = ring + st * p.stage_bytes + kXBytes;
#pragma unroll
            for (int kk = 0; kk < RP; kk += 16) {
              const uint64_t bdesc = umma_desc_sw128(ys + kk * 2);
              umma_bf16(d, umma_desc_sw128(h_base + (kk >> 6) * (kTileMF * 128) + (kk & 63) * 2),
                        bdesc, idesc, true);
              const int kl = RP + kk;
              umma_bf16(d, umma_desc_sw128(h_base + (kl >> 6) * (kTileMF * 128) + (kl & 63) * 2),
                        bdesc, idesc, true);
            }
            umma_commit(smem_addr(&ctl.empty[st]));
            ++it;
          }
          umma_commit(smem_addr(&ctl.acc_full[b]));
        }
        if (mt.lora) {
          umma_commit(smem_addr(&ctl.hs_empty));
          ++h_it;
        }
      }
    mma_done:
      umma_commit(smem_addr(&ctl.drain));
      mbar_wait_bounded(smem_addr(&ctl.drain), 0);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ================================================================ ring fill
    // The two warps split the Y rows (warp 1 the first half); lane c & 7 takes
    // 16-byte chunk c of a 128-byte row segment, four rows per instruction,
    // so every copy instruction covers whole 128-byte segments.  Every lane
    // arrives on a stage's full barrier through cp.async.mbarrier.arrive, so
    // the arrival lands when that lane's copies have; the TMA boxes complete
    // on the same barrier by their bytes.  A stage is therefore ready as soon
    // as its own data is, however far ahead the ring is filled.
    const int pw = warp - 1;
    const int c = lane & 7, rq = lane >> 3;
    // x_rows of a tile are re-read for every output chunk (evict last); a W_e
    // box is re-read only by the expert's other tiles, which run at the same
    // time (evict normal); A_e / B_e are small and re-read (evict last).
    const uint64_t keep = l2_evict_last();
    const uint64_t wpol = l2_evict_normal_policy();
    uint32_t it = 0;
    // Begin a stage: wait for it to be free; lane 0 of warp 1 issues the X box
    // and, for a GEMM stage (e >= 0), the W_e box of rows n0.. .
    auto begin = [&](int r0, int k0, bool with_x, int e, int n0) -> int {
      const int st = it % p.nst;
      if (!wait_f(ctl, ctl.empty[st], ((it / p.nst) & 1) ^ 1)) return -1;
      if (with_x && pw == 0 && lane == 0) {
        const uint32_t full = smem_addr(&ctl.full[st]);
        const uint32_t xs = ring + st * p.stage_bytes;
        mbar_expect_tx(full, e >= 0 ? kXBytes + kYBytes : kXBytes);
        tma_load_2d_hint(xs, &tmap_x, k0, r0, full, keep);
        if (e >= 0) tma_load_3d_hint(xs + kXBytes, &tmap_w, k0, n0, e, full, wpol);
      }
      return st;
    };
    auto finish = [&](int st) {
      cp_async_arrive_noinc(smem_addr(&ctl.full[st]));
      ++it;
    };
    for (int t = 0; t < n_tiles; ++t) {
      const FTile mt = my_tiles[t];
      const uint8_t *A = reinterpret_cast<const uint8_t *>(
          __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + mt.e));
      const uint8_t *B = reinterpret_cast<const uint8_t *>(
          __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + mt.e));
      if (mt.lora) {  // [X | A_e rows 0..RP)
        for (int kc = 0; kc < p.kc_count; ++kc) {
          const int st = begin(mt.r0, kc * 64, true, -1, 0);
          if (st < 0) goto fill_done;
          const uint32_t ys = ring + st * p.stage_bytes + kXBytes;
          const int kk = kc * 64 + 8 * c;
#pragma unroll
          for (int i = 0; i < RP / 8; ++i) {
            const int j = pw * (RP / 2) + 4 * i + rq;
            const bool in = j < p.rank && kk < p.k_in;
            cp_async_16_hint(ys + sw128(j, c), A + (in ? (static_cast<size_t>(j) * p.k_in + kk) * 2 : 0),
                             in ? 16u : 0u, keep);
          }
          finish(st);
        }
      }
      for (int nc = mt.nc0; nc < mt.nc1; ++nc) {
        const int n0 = nc * kNch;
        for (int kc = 0; kc < p.kc_count; ++kc) {  // [X | W_e rows n0.., k chunk kc]: TMA only
          const int st = begin(mt.r0, kc * 64, true, mt.e, n0);
          if (st < 0) goto fill_done;
          finish(st);
        }
        if (mt.lora) {  // [- | B_e rows n0.., rank columns (zero past rank)]
          const int st = begin(0, 0, false, -1, 0);
          if (st < 0) goto fill_done;
          const uint32_t ys = ring + st * p.stage_bytes + kXBytes;
          if (c < RP / 8) {
            const bool cin = 8 * c < p.rank;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
              const int row = pw * 128 + 4 * i + rq;
              const int n = n0 + row;
              const bool in = cin && n < p.n_out;
              cp_async_16_hint(ys + sw128(row, c),
                               B + (in ? (static_cast<size_t>(n) * p.rank + 8 * c) * 2 : 0),
                               in ? 16u : 0u, keep);
            }
          }
          finish(st);
        }
      }
    }
  fill_done:
    cp_async_wait_group<0>();
    if (pw == 0 && lane == 0) {  // TMA boxes of stages issued but never consumed: let them land
      for (uint32_t k = 0; k < static_cast<uint32_t>(p.nst) && k < it; ++k) {
        const uint32_t j = it - 1 - k;
        mbar_wait_bounded(smem_addr(&ctl.full[j % p.nst]), (j / p.nst) & 1);
      }
    }
  } else if (warp >= 4) {
    // ================================================================ epilogue
    // Warp w reads TMEM lanes [32 (w % 4), +32) -- its 32 rows of the tile --
    // and the two warps of a lane quarter take the two 128-column halves of
    // each 256-column chunk.
    const int ew = warp - 4, quarter = warp & 3, sub = ew >> 2;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int row = quarter * 32 + lane;
    uint32_t fold_bits = 0;
    {
      int sr[kMyTilesMaxF];
#pragma unroll
      for (int t = 0; t < kMyTilesMaxF; ++t) {
        sr[t] = -1;
        if (t < n_tiles) {
          const FTile mt = my_tiles[t];
          const int r = mt.r0 + row;
          if (r < mt.r1) sr[t] = __ldg(p.src + r);
        }
      }
#pragma unroll
      for (int t = 0; t < kMyTilesMaxF; ++t) {
        const bool f = sr[t] >= 0 && (p.row_adapter == nullptr ||
                                      __ldg(p.row_adapter + sr[t] / p.top_k) >= 0);
        fold_bits |= f ? (1u << t) : 0u;
      }
    }
    uint32_t acc_it = 0, h_it = 0;
    for (int t = 0; t < n_tiles; ++t) {
      const FTile mt = my_tiles[t];
      const int rg = mt.r0 + row;
      const bool valid = rg < mt.r1;
      if (mt.lora) {
        // ---- h: tensor memory -> scaled, split into bf16 hi / lo -> shared memory
        if (!wait_f(ctl, ctl.h_full, h_it & 1)) goto epi_done;
        if (sub == 0) {
          tc_fence_after();
          float h[RP];
#pragma unroll
          for (int qq = 0; qq < RP / 16; ++qq) {
            float v[16];
            tmem_ld16(lane_addr + acc_col(acc_it & 1) + qq * 16, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) h[qq * 16 + i] = v[i];
          }
          tmem_wait_ld();
          if (!wait_f(ctl, ctl.hs_empty, (h_it & 1) ^ 1)) goto epi_done;
          const bool folds = valid && ((fold_bits >> t) & 1u);
          float hi[RP], lo[RP];
#pragma unroll
          for (int jj = 0; jj < RP; ++jj)
            split_hi_lo(folds ? h[jj] * mt.scale : 0.f, hi[jj], lo[jj]);
          uint8_t *hrow = smem + p.off_h;
#pragma unroll
          for (int kk = 0; kk < KEXP; kk += 8) {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (kk < 2 * RP) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int jj = (kk < RP ? kk : kk - RP) + 2 * i;
                w[i] = kk < RP ? pack_bf16x2(hi[jj], hi[jj + 1]) : pack_bf16x2(lo[jj], lo[jj + 1]);
              }
            }
            const uint32_t off = (kk >> 6) * (kTileMF * 128) + sw128(row, (kk & 63) >> 3);
            *reinterpret_cast<uint4 *>(hrow + off) = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&ctl.hs_full));
        }
        ++h_it;
      }
      // ---- output chunks: accumulator -> registers -> one rounding -> global
      for (int nc = mt.nc0; nc < mt.nc1; ++nc, ++acc_it) {
        const int b = acc_it & 1;
        if (!wait_f(ctl, ctl.acc_full[b], (acc_it >> 1) & 1)) goto epi_done;
        tc_fence_after();
        const int col0 = nc * kNch + sub * 128;
        uint32_t packed[64];
        if (col0 < p.n_out) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[64];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              float u[16];
              tmem_ld16(lane_addr + acc_col(b) + sub * 128 + half * 64 + qq * 16, u);
#pragma unroll
              for (int i = 0; i < 16; ++i) v[qq * 16 + i] = u[i];
            }
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) packed[half * 32 + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl.acc_empty[b]));
        // A warp whose 32 rows all belong to the tile stores its boxes through
        // shared memory (TMA clips columns past n_out); a partial box is stored
        // row by row, so no row of another tile is written.
        const bool whole = p.staged && mt.r0 + quarter * 32 + 32 <= mt.r1;
        if (whole && col0 < p.n_out) {
          uint8_t *stage = smem + p.off_stage + ew * kStageBox;
          const uint32_t stage_addr = smem_addr(stage);
#pragma unroll
          for (int bx = 0; bx < 4; ++bx) {  // 32-column boxes of this warp's 128 columns
            if (col0 + bx * 32 >= p.n_out) break;
            if (lane == 0) bulk_wait_read_all();  // the previous box has left the buffer
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)  // 16-byte chunk cc of this lane's row, 64B swizzle
              *reinterpret_cast<uint4 *>(stage + lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(packed[bx * 16 + 4 * cc], packed[bx * 16 + 4 * cc + 1],
                             packed[bx * 16 + 4 * cc + 2], packed[bx * 16 + 4 * cc + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_out, col0 + bx * 32, mt.r0 + quarter * 32, stage_addr);
              bulk_commit();
            }
          }
        } else if (valid && col0 < p.n_out) {
          uint8_t *orow = p.out + (static_cast<size_t>(rg) * p.n_out + col0) * 2;
          if (p.v8) {  // whole sectors: each store is a full 32-byte sector of the row
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              if (col0 + 16 * cc < p.n_out) st_global_v8(orow + cc * 32, packed + 8 * cc);
          } else {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              if (col0 + 8 * cc < p.n_out) st_global_v4(orow + cc * 16, packed + 4 * cc);
          }
        }
      }
    }
  epi_done:
    if (lane == 0) bulk_wait_all();  // this warp's output boxes have been written
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemColsF);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFnF = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnF encode_fn_f() {
  static EncodeTiledFnF fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFnF>(ptr);
  });
  return fn;
}

constexpr uint32_t kSmemLimitF = 227 * 1024 - 1024;  // less the kernel's static part

uint32_t rup_f(uint32_t v, uint32_t m) { return (v + m - 1) / m * m; }

uint32_t plan_f(FusedParams &p, int nst, bool staged) {
  p.nst = nst;
  p.staged = staged ? 1 : 0;
  p.stage_bytes = kXBytes + kYBytes;
  uint32_t off = 0;
  p.off_ring = off;
  off += nst * p.stage_bytes;
  p.off_h = off;
  off += kTileMF * p.k_exp * 2;
  p.off_stage = off;  // 1024-aligned (the ring and h are multiples of 1 KB)
  off += staged ? kEpiWarpsF * kStageBox : 0;
  p.off_tab = off;
  off += rup_f((p.n_experts + 1) * 4, 16);
  p.off_my = off;
  off += rup_f(kMyTilesMaxF * sizeof(FTile), 16);
  p.smem_bytes = off;
  return off + 1024;  // 1 KB alignment slack
}

}  // namespace

uint32_t gemm_fold_read_errors(bool clear) {
  uint32_t v = 0;
  cudaMemcpyFromSymbol(&v, g_gemm_fold_errors, sizeof v);
  if (clear) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(g_gemm_fold_errors, &z, sizeof z);
  }
  return v;
}

}  // namespace mlg

extern "C" mlg_status mlg_grouped_gemm_fold_xrows(
    const mlg_bf16 *x_rows, const int32_t *expert_offsets, const int32_t *src,
    const int32_t *row_adapter, const mlg_bf16 *w_experts, const uint64_t *a_table,
    const uint64_t *b_table, const float *scale_table, mlg_bf16 *out, int32_t k_in,
    int32_t max_rank, int32_t n_out, int32_t top_k, int32_t n_experts, int32_t row_offset,
    int32_t row_end, uint32_t cap, void *stream) {
  using namespace mlg;
  if (cap == 0) return MLG_ERR_CAP_ZERO;
  if (top_k < 1 || n_experts < 0 || row_offset < 0 || row_end < row_offset)
    return MLG_ERR_INVALID_ARG;
  const mlg_status shape = check_shapes(k_in, max_rank, n_out);
  if (shape != MLG_OK) return shape;
  if (!x_rows || !expert_offsets || !src || !w_experts || !a_table || !b_table || !scale_table ||
      !out)
    return MLG_ERR_INVALID_ARG;
  if (!aligned16(x_rows) || !aligned16(out) || !aligned16(w_experts)) return MLG_ERR_UNSUPPORTED;
  if (row_end == row_offset || n_experts == 0) return MLG_OK;
  FusedParams p = {};
  p.x = reinterpret_cast<const uint8_t *>(x_rows);
  p.offsets = expert_offsets;
  p.src = src;
  p.row_adapter = row_adapter;
  p.a_table = a_table;
  p.b_table = b_table;
  p.scale_table = scale_table;
  p.out = reinterpret_cast<uint8_t *>(out);
  p.k_in = k_in;
  p.rank = max_rank;
  p.n_out = n_out;
  p.top_k = top_k;
  p.n_experts = n_experts;
  p.row_offset = row_offset;
  p.row_end = row_end;
  const int32_t len = row_end - row_offset;
  p.win = cap < static_cast<uint32_t>(len) ? static_cast<int32_t>(cap) : len;
  p.tile_m = kTileMF;
  p.r_pad = static_cast<int32_t>(rup_f(max_rank, 16));
  p.k_exp = static_cast<int32_t>(rup_f(2 * p.r_pad, 64));
  p.kc_count = (k_in + 63) / 64;
  p.nc_count = (n_out + kNch - 1) / kNch;
  p.v8 = (n_out % 16 == 0 && (reinterpret_cast<uintptr_t>(out) & 31u) == 0) ? 1 : 0;
  // Deepest ring first, output staging when it fits beside it.
  static const int kPlans[][2] = {{4, 1}, {4, 0}, {3, 1}, {3, 0}, {2, 0}};
  uint32_t total = 0;
  bool fits = false;
  for (const auto &pl : kPlans) {
    total = plan_f(p, pl[0], pl[1] != 0);
    if ((fits = total <= kSmemLimitF)) break;
  }
  if (!fits) return MLG_ERR_UNSUPPORTED;

  EncodeTiledFnF enc = encode_fn_f();
  if (enc == nullptr) return MLG_ERR_CUDA;
  CUtensorMap tmap_x;
  const cuuint64_t xdims[2] = {static_cast<cuuint64_t>(k_in), static_cast<cuuint64_t>(row_end)};
  const cuuint64_t xstrides[1] = {static_cast<cuuint64_t>(k_in) * 2};
  const cuuint32_t xbox[2] = {64, static_cast<cuuint32_t>(kTileMF)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tmap_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<mlg_bf16 *>(x_rows), xdims,
          xstrides, xbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLG_ERR_CUDA;
  // W: the stacked expert weights [n_experts, n_out, k_in], boxes of 64 k x
  // 256 rows of one expert (rows past n_out and k past k_in read as zero).
  CUtensorMap tmap_w;
  const cuuint64_t wdims[3] = {static_cast<cuuint64_t>(k_in), static_cast<cuuint64_t>(n_out),
                               static_cast<cuuint64_t>(n_experts)};
  const cuuint64_t wstrides[2] = {static_cast<cuuint64_t>(k_in) * 2,
                                  static_cast<cuuint64_t>(k_in) * n_out * 2};
  const cuuint32_t wbox[3] = {64, static_cast<cuuint32_t>(kNch), 1};
  const cuuint32_t estr3[3] = {1, 1, 1};
  if (enc(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<mlg_bf16 *>(w_experts), wdims,
          wstrides, wbox, estr3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLG_ERR_CUDA;

  // out: [row_end, n_out], 32 x 32 boxes, 64-byte swizzle (the staging layout)
  CUtensorMap tmap_out;
  const cuuint64_t odims[2] = {static_cast<cuuint64_t>(n_out), static_cast<cuuint64_t>(row_end)};
  const cuuint64_t ostrides[1] = {static_cast<cuuint64_t>(n_out) * 2};
  const cuuint32_t obox[2] = {32, 32};
  if (enc(&tmap_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, odims, ostrides, obox, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLG_ERR_CUDA;

  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [d = dev & 63] {
    const int lim = static_cast<int>(kSmemLimitF);
    const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    const void *fns[] = {reinterpret_cast<const void *>(gemm_fold_kernel<16>),
                         reinterpret_cast<const void *>(gemm_fold_kernel<32>),
                         reinterpret_cast<const void *>(gemm_fold_kernel<48>),
                         reinterpret_cast<const void *>(gemm_fold_kernel<64>)};
    cudaError_t e = cudaSuccess;
    for (const void *fn : fns)
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, attr, lim);
    attr_err[d] = e;
  });
  if (attr_err[dev & 63] != cudaSuccess) return cuda_status(attr_err[dev & 63]);

  // Persistent: one CTA per SM, more only when a CTA's tile list would
  // overflow, fewer when there are fewer tiles.
  const int64_t rows = len;
  const int64_t n_win = (rows + p.win - 1) / p.win;
  const int64_t full = rows / p.win, rest = rows % p.win;
  const int64_t T = p.tile_m;
  const int64_t max_tiles = full * ((p.win + T - 1) / T) + (rest + T - 1) / T + n_experts + n_win;
  int grid = sm_count();
  const int64_t need = (max_tiles + kMyTilesMaxF - 1) / kMyTilesMaxF;
  if (grid < need) grid = static_cast<int>(need);
  if (grid > max_tiles) grid = static_cast<int>(max_tiles);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreadsF, 1, 1);
  cfg.dynamicSmemBytes = total;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, FusedParams);
  KernelFn fn;
  switch (p.r_pad) {
    case 16: fn = gemm_fold_kernel<16>; break;
    case 32: fn = gemm_fold_kernel<32>; break;
    case 48: fn = gemm_fold_kernel<48>; break;
    default: fn = gemm_fold_kernel<64>; break;
  }
  const cudaError_t err = cudaLaunchKernelEx(&cfg, fn, tmap_x, tmap_w, tmap_out, p);
  if (err != cudaSuccess) return cuda_status(err);
  return cuda_status(cudaGetLastError());
}
