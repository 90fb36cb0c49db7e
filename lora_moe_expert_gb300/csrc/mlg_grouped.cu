// mlg_grouped.cu -- prefill-side grouped fold (moe_lora_grouped_down of the
// moe_lora_grouped module index) and the router fold (MoeExpertRoute: a
// one-entry route whose expert 0 is the router pair).
//
// For every expert-sorted row r of the window [row_offset, row_end) held by
// expert e's span expert_offsets[e] .. expert_offsets[e+1]:
//     base_out[r] += scale_e * (x[src[r] / top_k] @ A_e^T) @ B_e^T.
// The per-row x variant reads x_rows[r] instead of x[src[r] / top_k] (the
// down projection's input is the expert's own intermediate row); src then
// serves the row map only.
//
// GB300 design (not the pages' MLG_M_TILE grid):
//  * tiles are expert-aligned runs of <= 128 sorted rows (one tcgen05 M), so
//    a tile never mixes experts and every output row has one owner; the tile
//    list is built on the device from expert_offsets and the tables (no host
//    copy), and persistent CTAs (one per SM) walk it round-robin (the tiles
//    of a last, partial round split into pieces of their expand chunks over
//    the idle CTAs).  The setup that reads none of the fold's inputs runs
//    before griddepcontrol.wait, so it overlaps the preceding kernel
//    (programmatic dependent launch);
//  * warp 0 issues the tensor-core work: shrink H = X A_e^T (M=128, N=rank,
//    K=k_in in 64-wide chunks) into tensor memory, then expand
//    ACC = [H_hi | H_lo] [B_e | B_e]^T (M=128, N=64/128 columns per chunk) into
//    a double-buffered TMEM accumulator -- h is split into two bf16 halves so
//    it enters the expand at ~2^-17 relative precision (kept fp32 in effect);
//  * warps 1 and 3 gather the X rows via src and A_e chunks, warp 2 the B_e
//    chunks, with 16-byte cp.async into swizzled K-major tiles (X and A_e in
//    128-byte rows; B_e in rows of 2 * rank bytes, 32- or 64-byte swizzle for
//    rank 16 / 32, so a B_e stage takes a quarter / half the space); when
//    a tile's x rows are rows r0.. of x (router, per-row x) they come in as
//    64 x 64 TMA boxes instead.  Each producer lane arrives on a stage's full
//    barrier through cp.async.mbarrier.arrive (landing when its copies have)
//    and the boxes complete on it by their bytes, so a stage is ready as soon
//    as its own data is;
//  * warps 4-11 (two per TMEM lane quarter) scale and split h, then stream
//    base_out: the pair owns the quarter's 32 rows of the tile, each warp
//    takes every other 64-column box and runs its own ring of 32x64 TMA
//    boxes (prefetch depth D-1), adds the accumulator, rounds once
//    to bf16 (RNE) and TMA-stores boxes it owns whole; rows of a box it owns
//    only in part are stored row by row, so no row of another tile is written.
//  Every wait is bounded; a timeout sets an error bit and the CTA drains and
//  exits instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "mlg_internal.h"
#include "mlg_ptx.cuh"
#include "mlg_tiles.cuh"

namespace mlg {
namespace {

constexpr int kGThreads = 384;      // 4 role warps + 8 epilogue warps
constexpr int kEpiWarps = 8;
constexpr int kTileM = MLG_M_TILE;   // 128 rows per tile
constexpr int kBoxRows = 32;         // rows per TMA box (one epilogue warp)
constexpr int kBoxCols = 64;         // bf16 columns per TMA box (128 bytes)
constexpr int kMaxDepth = 8;         // base-ring stages per epilogue warp
constexpr int kMaxStages = 6;        // operand ring stages
constexpr int kMyTilesMax = 16;      // per-CTA tile list capacity
constexpr uint32_t kTmemCols = 512;
// TMEM columns: two h buffers (tile parity), two expand accumulators.
constexpr uint32_t kTmemH0 = 0, kTmemH1 = 64, kTmemAcc0 = 128, kTmemAcc1 = 256;

static __device__ uint32_t g_grouped_errors;

struct GroupedParams {
  const uint8_t *x;              // bf16 [n_tokens, k_in], or [rows, k_in] when x_per_row
  const int32_t *offsets;        // [n_experts + 1] or null (router: one span)
  const int32_t *src;            // sorted row -> flat row, or null (identity)
  const int32_t *row_adapter;    // [n_tokens] or null
  const uint64_t *a_table;
  const uint64_t *b_table;
  const float *scale_table;
  uint8_t *base_out;             // bf16 [>= row_end, n_out]
  int32_t k_in, rank, n_out, top_k, n_experts, row_offset, row_end;
  int32_t win;                   // window length (windows start at row_offset + i * win)
  int32_t r_pad;                 // rank rounded up to 16 (shrink N)
  int32_t k_exp;                 // expand K: [hi | lo] padded to a multiple of 64
  int32_t n_ch;                  // expand N per accumulator chunk (64 or 128)
  int32_t kc_count, nc_count, nbx;  // k chunks, n chunks, 64-column boxes per row
  int32_t nxa, nbs, depth;       // ring stages
  uint32_t xa_stage, b_stage;    // bytes per stage
  uint32_t off_xa, off_b, off_h, off_base, off_tab, off_my, smem_bytes;
  int32_t my_cap;                // tiles per CTA the tile list holds
  int32_t x_per_row;             // 1: sorted row r reads x row r (not its token's)
  int32_t tile_m;                // rows per tile (<= kTileM; the MMA M stays kTileM)
  int32_t x_tma;                 // 1: a tile's x rows are rows r0.. of x (router, per-row x)
};

struct Ctl {
  uint64_t xa_full[kMaxStages], xa_empty[kMaxStages];
  uint64_t b_full[kMaxStages], b_empty[kMaxStages];
  uint64_t h_full[2], hs_full, hs_empty, drain;
  uint64_t acc_full[2], acc_empty[2];
  uint64_t base_full[kEpiWarps][kMaxDepth];
  uint32_t tmem_base;
  volatile int abort_flag;
};

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(Ctl &ctl, uint64_t &bar, uint32_t parity) {
  const uint32_t a = smem_addr(&bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (ctl.abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_grouped_errors, kErrWaitTimeout);
      ctl.abort_flag = 1;
      return false;
    }
  }
}

// Per-CTA tile list entry, built once in the prologue: expert and rows.
// Which rows fold is decided where it is needed: the X producers gather every
// row of the tile (no round trip on the row map before the first copy), and
// each epilogue lane reads its own rows' row-map entries once, up front.
struct MyTile {
  int e, r0, r1;
  int nc0, nc1;  // the expand chunks this CTA folds: [nc0, nc1)
};


// out = RNE_bf16(base + v) for 8 consecutive elements (base given as bf16 bits).
__device__ __forceinline__ uint4 add8_bf16(const uint4 b, const float *v) {
  const uint32_t w[4] = {b.x, b.y, b.z, b.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = pack_bf16x2(bf16lo_to_f32(w[i]) + v[2 * i], bf16hi_to_f32(w[i]) + v[2 * i + 1]);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// RP: rank rounded up to a multiple of 16.  XTMA: a tile's x rows are rows
// r0.. of x (router, per-row x) and come in as TMA boxes; else they are
// gathered row by row through src.
template <int RP, bool XTMA>
__global__ void __launch_bounds__(kGThreads, 1)
    grouped_fold_kernel(const __grid_constant__ CUtensorMap tmap_base,
                        const __grid_constant__ CUtensorMap tmap_x, const GroupedParams p) {
  constexpr int KEXP = (2 * RP + 63) / 64 * 64;  // expand K: [hi | lo | zero pad]
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ Ctl ctl;
  // 1024-byte alignment for the swizzled tiles.
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_e = p.offsets ? p.n_experts : 1;
  int *tile_start = reinterpret_cast<int *>(smem + p.off_tab);  // [n_e + 1]

  // ---- prologue: barriers, zeroed operand padding, tile table, TMEM ------
  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(smem_addr(&ctl.xa_full[s]), 64);
      mbar_init(smem_addr(&ctl.xa_empty[s]), 1);
      mbar_init(smem_addr(&ctl.b_full[s]), 32);
      mbar_init(smem_addr(&ctl.b_empty[s]), 1);
    }
    mbar_init(smem_addr(&ctl.h_full[0]), 1);
    mbar_init(smem_addr(&ctl.h_full[1]), 1);
    mbar_init(smem_addr(&ctl.hs_full), 4);
    mbar_init(smem_addr(&ctl.hs_empty), 1);
    mbar_init(smem_addr(&ctl.drain), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&ctl.acc_full[s]), 1);
      mbar_init(smem_addr(&ctl.acc_empty[s]), kEpiWarps);
    }
    for (int w = 0; w < kEpiWarps; ++w)
      for (int s = 0; s < kMaxDepth; ++s) mbar_init(smem_addr(&ctl.base_full[w][s]), 1);
    ctl.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_base);
  }
  // Operand padding read by the MMAs but never written by a copy: A_e rows
  // [rank, r_pad) of every X/A stage and the B positions outside the two
  // copies of B_e's rank columns.
  for (uint32_t i = tid * 16; i < p.off_h; i += kGThreads * 16)
    *reinterpret_cast<uint4 *>(smem + i) = make_uint4(0, 0, 0, 0);
  __syncthreads();  // barriers initialised (and visible) before anyone waits on them
  if (warp == 0) {
    tmem_alloc(smem_addr(&ctl.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  // Everything above runs while the preceding kernel finishes (programmatic
  // dependent launch); the routing, x, the row map and base_out may be written
  // by it, so every thread waits before its first read of them.  The next
  // fold may start its own setup now.
  griddep_launch_dependents();
  griddep_wait();
  // Tile table: tiles of expert e = ceil(rows of e in the window / 128), 0 if
  // the expert folds nothing; exclusive prefix over experts.  One expert per
  // thread per pass, its four loads issued together.
  {
    int carry = 0;
    for (int base = 0; base < n_e; base += kGThreads) {
      const int e = base + tid;
      int n = 0;
      if (e < n_e) {
        const int lo = span_lo(p, e), hi = span_hi(p, e);
        const uint64_t a = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + e);
        const uint64_t b = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + e);
        if (hi > lo && cells_fold(a, b)) n = span_tiles(p, lo, hi);
      }
      // block exclusive scan
      int incl = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      __shared__ int warp_tot[kGThreads / 32];
      if (lane == 31) warp_tot[warp] = incl;
      __syncthreads();
      int before = carry, total = 0;
#pragma unroll
      for (int w = 0; w < kGThreads / 32; ++w) {
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
  // This CTA's tiles (t = blockIdx.x + i * gridDim.x): expert and rows.  (The
  // scale is read by the epilogue, which needs it only for the first h split,
  // so its round trip is not on the prologue's path.)
  // Full rounds: tile c + i G, all expand chunks.  The tiles of a last,
  // partial round of R < G tiles are split into P = min(chunks, G / R) pieces
  // of their expand chunks, piece u to CTA u (each piece recomputes its
  // tile's h and folds its own columns), so the CTAs holding one tile more
  // than the rest do not set the step alone (the 163840-row prefill: 1526
  // tiles on 152 SMs, and its last CTAs to finish were those with 11 tiles).
  MyTile *my_tiles = reinterpret_cast<MyTile *>(smem + p.off_my);
  const int n_tiles_all = tile_start[n_e];
  const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const int q_full = n_tiles_all / G, rest = n_tiles_all % G;
  const int pieces = rest > 0 ? max(1, min(p.nc_count, G / rest)) : 1;
  const int my_count = min(p.my_cap, q_full + (cta < rest * pieces ? 1 : 0));
  if (tid < my_count) {
    int t = cta + tid * G, nc0 = 0, nc1 = p.nc_count;
    if (tid == q_full) {  // this CTA's piece of a last-round tile
      const int j = cta % pieces;
      t = q_full * G + cta / pieces;
      nc0 = j * p.nc_count / pieces;
      nc1 = (j + 1) * p.nc_count / pieces;
    }
    const TileInfo ti = tile_info(p, tile_start, n_e, t);
    my_tiles[tid].e = ti.e;
    my_tiles[tid].r0 = ti.r0;
    my_tiles[tid].r1 = ti.r1;
    my_tiles[tid].nc0 = nc0;
    my_tiles[tid].nc1 = nc1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const int n_tiles = my_count;  // tiles of this CTA, indexed 0 .. my_count-1
  const uint32_t idesc_shrink = umma_idesc_bf16(kTileM, RP);
  const uint32_t idesc_expand = umma_idesc_bf16(kTileM, p.n_ch);
  const uint32_t xa_base = smem_addr(smem + p.off_xa);
  const uint32_t b_base = smem_addr(smem + p.off_b);
  const uint32_t h_base = smem_addr(smem + p.off_h);

  if (warp == 0) {
    // ================================================================ MMA issuer
    // Shrink chunks of tile t+1 are issued, as their X / A_e stages arrive,
    // between the expand chunks of tile t (h of consecutive tiles alternates
    // between two TMEM buffers), so h is ready when the epilogue needs it.
    if (lane == 0) {
      uint32_t xa_it = 0, b_it = 0, acc_it = 0;
      int sh_t = 0, sh_kc = 0;  // next shrink chunk to issue: tile, k chunk
      auto issue_shrink_chunk = [&]() {
        const int st = xa_it % p.nxa;
        fence_proxy_async_smem();  // A_e (and gathered x) came in by cp.async (generic proxy)
        tc_fence_after();
        const uint32_t xs = xa_base + st * p.xa_stage;
        const uint32_t as = xs + kTileM * 128;
        const uint32_t hd = tmem + ((sh_t & 1) ? kTmemH1 : kTmemH0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_bf16(hd, umma_desc_sw128(xs + k * 32), umma_desc_sw128(as + k * 32), idesc_shrink,
                    (sh_kc | k) != 0);
        umma_commit(smem_addr(&ctl.xa_empty[st]));
        ++xa_it;
        if (++sh_kc == p.kc_count) {
          umma_commit(smem_addr(&ctl.h_full[sh_t & 1]));
          sh_kc = 0;
          ++sh_t;
        }
      };
      for (int t = 0; t < n_tiles; ++t) {
        while (sh_t <= t) {  // finish tile t's shrink (blocking)
          if (!wait_bar(ctl, ctl.xa_full[xa_it % p.nxa], (xa_it / p.nxa) & 1)) goto mma_done;
          issue_shrink_chunk();
        }
        if (!wait_bar(ctl, ctl.hs_full, t & 1)) goto mma_done;
        tc_fence_after();
        for (int nc = my_tiles[t].nc0; nc < my_tiles[t].nc1; ++nc, ++b_it, ++acc_it) {
          const int st = b_it % p.nbs;
          const int ab = acc_it & 1;
          if (!wait_bar(ctl, ctl.b_full[st], (b_it / p.nbs) & 1)) goto mma_done;
          if (!wait_bar(ctl, ctl.acc_empty[ab], ((acc_it >> 1) & 1) ^ 1)) goto mma_done;
          fence_proxy_async_smem();  // B_e came in by cp.async (generic proxy)
          tc_fence_after();
          const uint32_t bs = b_base + st * p.b_stage;
          const uint32_t d = tmem + (ab ? kTmemAcc1 : kTmemAcc0);
#pragma unroll
          for (int kk = 0; kk < RP; kk += 16) {
            // hi half: H columns [0, RP); lo half: H columns [RP, 2 RP); both
            // against B_e's rank columns kk .. kk+15.
            const uint64_t bdesc = umma_desc_k<b_row_bytes(RP)>(bs + kk * 2);
            umma_bf16(d, umma_desc_sw128(h_base + (kk >> 6) * (kTileM * 128) + (kk & 63) * 2),
                      bdesc, idesc_expand, kk != 0);
            const int kl = RP + kk;
            umma_bf16(d, umma_desc_sw128(h_base + (kl >> 6) * (kTileM * 128) + (kl & 63) * 2),
                      bdesc, idesc_expand, true);
          }
          umma_commit(smem_addr(&ctl.b_empty[st]));
          umma_commit(smem_addr(&ctl.acc_full[ab]));
          // next tile's shrink chunks that have already arrived (no blocking)
          while (sh_t == t + 1 && sh_t < n_tiles &&
                 mbar_try_wait(smem_addr(&ctl.xa_full[xa_it % p.nxa]), (xa_it / p.nxa) & 1))
            issue_shrink_chunk();
        }
        umma_commit(smem_addr(&ctl.hs_empty));
      }
    mma_done:
      umma_commit(smem_addr(&ctl.drain));
      mbar_wait_bounded(smem_addr(&ctl.drain), 0);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ================================================================ X / A_e producers
    // Warp 1 gathers tile rows 0-63 and A_e rows 0-31, warp 3 rows 64-127 and
    // A_e rows 32-63.  Every lane arrives on a stage's full barrier through
    // cp.async.mbarrier.arrive (the arrival lands when that lane's copies have)
    // and x boxes complete on it by their bytes, so a stage is ready as soon as
    // its own data is, however many stages are in flight.
    const int half = warp == 1 ? 0 : 1;
    const uint64_t keep = l2_evict_last();  // A_e (and token x rows) are re-read by other tiles
    // a per-row x row (and a router row) is read once
    const uint64_t xpol = (p.x_per_row || XTMA) ? l2_evict_first() : keep;
    uint32_t it = 0;
    // x token of this lane's two rows, loaded one tile ahead
    auto tokens = [&](int t, int (&tok)[2]) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        tok[u] = -1;
        if (t >= n_tiles) continue;
        const MyTile mt = my_tiles[t];
        const int row = half * 64 + lane + 32 * u;
        const int r = mt.r0 + row;
        if (r < mt.r1) {
          const int sr = p.src ? __ldg(p.src + r) : r;
          tok[u] = sr < 0 ? -1 : (p.x_per_row ? r : sr / p.top_k);
        }
      }
    };
    int tok_next[2] = {-1, -1};
    if constexpr (!XTMA) tokens(0, tok_next);
    for (int t = 0; t < n_tiles; ++t) {
      const MyTile ti = my_tiles[t];
      const uint8_t *A = reinterpret_cast<const uint8_t *>(
          __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + ti.e));
      const uint8_t *xrow[2];
      bool xv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        xv[u] = tok_next[u] >= 0;
        xrow[u] = p.x + static_cast<size_t>(tok_next[u] >= 0 ? tok_next[u] : 0) * p.k_in * 2;
      }
      if constexpr (!XTMA) tokens(t + 1, tok_next);
      for (int kc = 0; kc < p.kc_count; ++kc, ++it) {
        const int st = it % p.nxa;
        if (!wait_bar(ctl, ctl.xa_empty[st], ((it / p.nxa) & 1) ^ 1)) goto prod_a_done;
        const uint32_t xs = xa_base + st * p.xa_stage;
        const uint32_t as = xs + kTileM * 128;
        const int k0 = kc * 64;
        // Each copy instruction takes 4 whole 128-byte row segments (8 lanes
        // per row), so every request is a full line.
        const int c = lane & 7;
        const int kk = k0 + 8 * c;
        const bool in = kk < p.k_in;
        if constexpr (XTMA) {
          // This warp's 64 rows of the chunk in one box (rows past the tensor
          // and columns past k_in read as zero); its bytes complete on the
          // stage's barrier beside the lanes' arrivals for the A_e copies.
          if (lane == 0) {
            const uint32_t full = smem_addr(&ctl.xa_full[st]);
            mbar_expect_tx(full, 64 * 128);
            tma_load_2d_hint(xs + half * 64 * 128, &tmap_x, k0, ti.r0 + half * 64, full, xpol);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int rl = 4 * i + (lane >> 3);  // row of this warp's 64
            const uint8_t *xr = reinterpret_cast<const uint8_t *>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(xrow[rl >> 5]), rl & 31));
            const bool v = __shfl_sync(0xffffffffu, xv[rl >> 5], rl & 31);
            if (v)
              cp_async_16_hint(xs + sw128(half * 64 + rl, c), xr + (in ? kk * 2 : 0), in ? 16u : 0u,
                               xpol);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ja = half * 32 + 4 * i + (lane >> 3);  // A_e row
          if (ja < p.rank)
            cp_async_16_hint(as + sw128(ja, c),
                             A + (static_cast<size_t>(ja) * p.k_in + (in ? kk : 0)) * 2,
                             in ? 16u : 0u, keep);
        }
        cp_async_arrive_noinc(smem_addr(&ctl.xa_full[st]));
      }
    }
  prod_a_done:
    cp_async_wait_group<0>();
    if constexpr (XTMA) {  // this warp's boxes of the last stages: let them land
      if (lane == 0) {
        const uint32_t nl = it < static_cast<uint32_t>(p.nxa) ? it : static_cast<uint32_t>(p.nxa);
        for (uint32_t j = 0; j < nl; ++j) {
          const uint32_t k = it - nl + j;
          mbar_wait_bounded(smem_addr(&ctl.xa_full[k % p.nxa]), (k / p.nxa) & 1);
        }
      }
    }
  } else if (warp == 2) {
    // ================================================================ B_e producer
    // One B_e tile [n_ch rows x rank] per accumulator chunk; each lane's
    // arrival on the stage's full barrier lands when its copies have.
    uint32_t it = 0;
    const int rc = p.rank / 8;  // 16-byte chunks per B_e row
    const uint64_t keep = l2_evict_last();
    for (int t = 0; t < n_tiles; ++t) {
      const MyTile ti = my_tiles[t];
      const uint8_t *B = reinterpret_cast<const uint8_t *>(
          __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + ti.e));
      for (int nc = ti.nc0; nc < ti.nc1; ++nc, ++it) {
        const int st = it % p.nbs;
        if (!wait_bar(ctl, ctl.b_empty[st], ((it / p.nbs) & 1) ^ 1)) goto prod_b_done;
        const uint32_t bs = b_base + st * p.b_stage;
        const int n0 = nc * p.n_ch;
        // Lanes take whole B_e rows: rc lanes per row, 32 / rc rows per copy.
        {
          const int per = 32 / rc, c = lane % rc;
          for (int i = lane / rc; lane < per * rc && i < p.n_ch; i += per) {
            const int n = n0 + i;
            const bool in = n < p.n_out;
            const uint8_t *brow = B + static_cast<size_t>(in ? n : 0) * p.rank * 2;
            cp_async_16_hint(bs + swk<b_row_bytes(RP)>(i, c), brow + c * 16, in ? 16u : 0u,
                             keep);
          }
        }
        cp_async_arrive_noinc(smem_addr(&ctl.b_full[st]));
      }
    }
  prod_b_done:
    cp_async_wait_group<0>();
  } else if (warp >= 4) {
    // ================================================================ epilogue
    // Eight warps: warp w reads TMEM lanes [32 (w % 4), +32) (its tile rows);
    // the two warps of a lane quarter split the 64-column boxes (even / odd).
    const int ew = warp - 4;
    const int quarter = warp & 3;
    const int sub = ew >> 2;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint8_t *ring = smem + p.off_base + ew * p.depth * 4096;
    const uint32_t ring_addr = smem_addr(ring);
    const uint64_t stream_policy = l2_evict_first();  // base_out is touched once
    uint32_t tile_it = 0, acc_it = 0;
    // box sequence of this warp: (tile, box column) over tiles with rows here
    // (a tile's boxes: the 64-column boxes of its expand chunks [nc0, nc1))
    int ld_t = 0, ld_b = sub, ld_y = 0;
    uint32_t ld_count = 0, box_it = 0;
    auto box_hi = [&](const MyTile &ti) { return min(p.nbx, ti.nc1 * (p.n_ch / kBoxCols)); };
    auto ld_advance = [&](bool first) {
      if (!first) {
        ld_b += 2;
        if (ld_b < box_hi(my_tiles[ld_t])) return;
        ++ld_t;
      }
      for (; ld_t < n_tiles; ++ld_t) {
        const MyTile ti = my_tiles[ld_t];
        const int b0 = ti.nc0 * (p.n_ch / kBoxCols);
        ld_b = b0 + ((sub - b0) & 1);  // this warp's first box (its column parity)
        if (ld_b < box_hi(ti) && ti.r1 > ti.r0 + quarter * kBoxRows) {
          ld_y = ti.r0 + quarter * kBoxRows;
          return;
        }
      }
    };
    auto ld_issue = [&]() {  // lane 0 only
      if (ld_t >= n_tiles) return;
      const int st = ld_count % p.depth;
      const uint32_t bar = smem_addr(&ctl.base_full[ew][st]);
      mbar_arrive_expect_tx(bar, kBoxRows * kBoxCols * 2);
      tma_load_2d_hint(ring_addr + st * 4096, &tmap_base, ld_b * kBoxCols, ld_y, bar,
                       stream_policy);
      ++ld_count;
      ld_advance(false);
    };
    ld_advance(true);
    if (lane == 0)
      for (int i = 0; i < p.depth - 1; ++i) ld_issue();
    // Which of this lane's rows fold, one bit per tile of this CTA: a row of
    // the tile whose src is valid and whose token's row-map entry is not
    // negative.  Loads of all tiles issued together (two round trips in all).
    uint32_t fold_bits = 0;
    {
      int sr[kMyTilesMax];
#pragma unroll
      for (int t = 0; t < kMyTilesMax; ++t) {
        sr[t] = -1;
        if (t < n_tiles) {
          const MyTile mt = my_tiles[t];
          const int r = mt.r0 + quarter * kBoxRows + lane;
          if (r < mt.r1) sr[t] = p.src ? __ldg(p.src + r) : r;
        }
      }
#pragma unroll
      for (int t = 0; t < kMyTilesMax; ++t) {
        const bool f = sr[t] >= 0 && (p.row_adapter == nullptr ||
                                      __ldg(p.row_adapter + sr[t] / p.top_k) >= 0);
        fold_bits |= f ? (1u << t) : 0u;
      }
    }

    for (int t = 0; t < n_tiles; ++t, ++tile_it) {
      const MyTile ti = my_tiles[t];
      const int row = quarter * kBoxRows + lane;
      const int rg = ti.r0 + row;
      const bool folds = (fold_bits >> t) & 1u;
      const float scale = __ldg(p.scale_table + ti.e);
      const int owned = min(max(ti.r1 - (ti.r0 + quarter * kBoxRows), 0), kBoxRows);

      // ---- h: tensor memory -> scaled, split into bf16 hi / lo -> shared memory
      if (!wait_bar(ctl, ctl.h_full[tile_it & 1], (tile_it >> 1) & 1)) goto epi_done;
      if (sub == 0) {
        tc_fence_after();
        float h[RP];
#pragma unroll
        for (int qq = 0; qq < RP / 16; ++qq) {
          float v[16];
          tmem_ld16(lane_addr + ((tile_it & 1) ? kTmemH1 : kTmemH0) + qq * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) h[qq * 16 + i] = v[i];
        }
        tmem_wait_ld();
        if (!wait_bar(ctl, ctl.hs_empty, (tile_it & 1) ^ 1)) goto epi_done;
        float hi[RP], lo[RP];
#pragma unroll
        for (int jj = 0; jj < RP; ++jj) split_hi_lo(folds ? h[jj] * scale : 0.f, hi[jj], lo[jj]);
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
          const uint32_t off = (kk >> 6) * (kTileM * 128) + sw128(row, (kk & 63) >> 3);
          *reinterpret_cast<uint4 *>(hrow + off) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl.hs_full));
      }

      // ---- expand epilogue: base_out boxes of this warp's rows -------------
      for (int nc = ti.nc0; nc < ti.nc1; ++nc, ++acc_it) {
        const int ab = acc_it & 1;
        if (!wait_bar(ctl, ctl.acc_full[ab], (acc_it >> 1) & 1)) goto epi_done;
        tc_fence_after();
        for (int jb = 0; jb < p.n_ch / kBoxCols; ++jb) {
          const int bcol = nc * (p.n_ch / kBoxCols) + jb;
          if ((bcol & 1) != sub || owned == 0 || bcol >= p.nbx) continue;
          const int st = box_it % p.depth;
          if (!wait_bar(ctl, ctl.base_full[ew][st], (box_it / p.depth) & 1)) goto epi_done;
          float v[64];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            float u[16];
            tmem_ld16(lane_addr + (ab ? kTmemAcc1 : kTmemAcc0) + jb * kBoxCols + qq * 16, u);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[qq * 16 + i] = u[i];
          }
          tmem_wait_ld();
          uint8_t *boxp = ring + st * 4096 + lane * 128;
          const bool whole = owned == kBoxRows;
          if (folds) {
            const int col0 = bcol * kBoxCols;
            uint4 bb[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              bb[c] = *reinterpret_cast<const uint4 *>(boxp + ((c ^ (lane & 7)) << 4));
#pragma unroll
            for (int c = 0; c < 8; ++c) bb[c] = add8_bf16(bb[c], v + 8 * c);
            if (whole) {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(boxp + ((c ^ (lane & 7)) << 4)) = bb[c];
            } else {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                if (col0 + 8 * c < p.n_out)
                  *reinterpret_cast<uint4 *>(
                      p.base_out + (static_cast<size_t>(rg) * p.n_out + col0 + 8 * c) * 2) = bb[c];
            }
          }
          if (whole) fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (whole)
              tma_store_2d_hint(&tmap_base, bcol * kBoxCols, ti.r0 + quarter * kBoxRows,
                                ring_addr + st * 4096, stream_policy);
            bulk_commit();
            bulk_wait_read_1();  // the previous box's store has left its stage
            ld_issue();
          }
          __syncwarp();
          ++box_it;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&ctl.acc_empty[ab]));
      }
    }
  epi_done:
    if (lane == 0) {
      bulk_wait_all();
      // loads issued but not consumed (only after an abort): let them land
      for (uint32_t k = box_it; k < ld_count; ++k)
        mbar_wait_bounded(smem_addr(&ctl.base_full[ew][k % p.depth]), (k / p.depth) & 1);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int g_grouped_ctas = 0;
// Dynamic shared memory cap: 227 KB per block minus room for the static part.
constexpr uint32_t kGSmemLimit = 227 * 1024 - 2048;

uint32_t rup(uint32_t v, uint32_t m) { return (v + m - 1) / m * m; }

// Shared-memory plan; returns total dynamic bytes (including 1 KB alignment slack).
uint32_t plan(GroupedParams &p, int n_ch, int nxa, int nbs, int depth, int n_e) {
  p.n_ch = n_ch;
  p.nxa = nxa;
  p.nbs = nbs;
  p.depth = depth;
  p.nc_count = (p.n_out + n_ch - 1) / n_ch;
  p.xa_stage = rup(kTileM * 128 + p.r_pad * 128, 1024);
  // K = rank, in rows of b_row_bytes (32, 64 or 128 bytes)
  p.b_stage = rup(static_cast<uint32_t>(n_ch * b_row_bytes(p.r_pad)), 1024);
  uint32_t off = 0;
  p.off_xa = off;
  off += nxa * p.xa_stage;
  p.off_b = off;
  off += nbs * p.b_stage;
  p.off_h = off;
  off += kTileM * p.k_exp * 2;
  p.off_base = off;
  off += kEpiWarps * depth * 4096;
  p.off_tab = off;
  off += rup((n_e + 1) * 4, 16);
  p.off_my = off;
  off += rup(kMyTilesMax * sizeof(MyTile), 16);
  p.smem_bytes = off;
  return off + 1024;
}

mlg_status launch_grouped(GroupedParams &p, cudaStream_t stream) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return MLG_ERR_CUDA;
  const int n_e = p.offsets ? p.n_experts : 1;
  p.r_pad = static_cast<int>(rup(p.rank, 16));
  p.k_exp = static_cast<int>(rup(2 * p.r_pad, 64));
  p.kc_count = (p.k_in + 63) / 64;
  p.nbx = (p.n_out + kBoxCols - 1) / kBoxCols;
  // Deepest rings that fit, as {X/A stages, B_e stages, base_out boxes per
  // warp}.  Rows whose x is wider than their base_out read-modify-write
  // (router-like shapes) take {4, 2, 3}: the 16384-token router measured
  // 26.5 us with {6, 2, 2} and 25.3 us with {4, 2, 3}; three X/A stages or
  // four boxes were slower.  The rest take four B_e stages (a tile's expand
  // needs a fresh B_e chunk per accumulator chunk; with two stages that
  // stream set the pace of the 163840-row prefill) beside a base_out ring
  // four boxes deep per warp, which the compact B_e rows (b_row_bytes) leave
  // room for: 305 us with {2, 2, 4}, 274 us with {2, 4, 3}, 258 us with
  // {2, 4, 4}; a ring two deep measured far slower (350 us).  Where a third
  // X/A stage fits beside them (rank <= 16) it shortens the first tile's
  // shrink: the 30K-row per-row x prefill 56.8 -> 55.3 us.
  static const int cand_base[][3] = {{3, 4, 4}, {2, 4, 4}, {2, 4, 3}, {2, 2, 4}, {3, 3, 3},
                                     {2, 3, 3}, {2, 2, 3}, {2, 2, 2}};
  static const int cand_x[][3] = {{4, 2, 3}, {6, 2, 2}, {5, 2, 2}, {4, 2, 2}, {3, 2, 3},
                                  {3, 2, 2}, {2, 2, 2}};
  const bool x_heavy = static_cast<int64_t>(p.k_in) * 2 > static_cast<int64_t>(p.n_out) * 4;
  bool ok = false;
  uint32_t total = 0;
  const int n_chs[2] = {128, 64};
  for (int a = 0; a < 2 && !ok; ++a) {
    const int(*cand)[3] = x_heavy ? cand_x : cand_base;
    const int nc = x_heavy ? static_cast<int>(sizeof(cand_x) / sizeof(cand_x[0]))
                           : static_cast<int>(sizeof(cand_base) / sizeof(cand_base[0]));
    for (int i = 0; i < nc; ++i) {
      total = plan(p, n_chs[a], cand[i][0], cand[i][1], cand[i][2], n_e);
      if ((ok = total <= kGSmemLimit)) break;
    }
  }
  if (!ok) return MLG_ERR_UNSUPPORTED;

  CUtensorMap tmap;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.n_out), static_cast<cuuint64_t>(p.row_end)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.n_out) * 2};
  const cuuint32_t box[2] = {kBoxCols, kBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.base_out, dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLG_ERR_CUDA;
  CUtensorMap tmap_x = tmap;  // unused unless x_tma
  if (p.x_tma) {  // x rows [row_end, k_in], 64 x 64 boxes in the X tile's 128-byte swizzle
    const cuuint64_t xdims[2] = {static_cast<cuuint64_t>(p.k_in),
                                 static_cast<cuuint64_t>(p.row_end)};
    const cuuint64_t xstrides[1] = {static_cast<cuuint64_t>(p.k_in) * 2};
    const cuuint32_t xbox[2] = {64, 64};
    if (enc(&tmap_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t *>(p.x), xdims,
            xstrides, xbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLG_ERR_CUDA;
  }

  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [d = dev & 63] {
    const int lim = static_cast<int>(kGSmemLimit);
    const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    const void *fns[] = {
        reinterpret_cast<const void *>(grouped_fold_kernel<16, false>),
        reinterpret_cast<const void *>(grouped_fold_kernel<32, false>),
        reinterpret_cast<const void *>(grouped_fold_kernel<48, false>),
        reinterpret_cast<const void *>(grouped_fold_kernel<64, false>),
        reinterpret_cast<const void *>(grouped_fold_kernel<16, true>),
        reinterpret_cast<const void *>(grouped_fold_kernel<32, true>),
        reinterpret_cast<const void *>(grouped_fold_kernel<48, true>),
        reinterpret_cast<const void *>(grouped_fold_kernel<64, true>)};
    cudaError_t e = cudaSuccess;
    for (const void *fn : fns)
      if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, attr, lim);
    attr_err[d] = e;
  });
  if (attr_err[dev & 63] != cudaSuccess) return cuda_status(attr_err[dev & 63]);
  // Persistent: one CTA per SM (more only when a CTA's tile list would
  // overflow), fewer when there are fewer tiles.  Tile bound: whole-window
  // tiles plus one split per expert span and per window boundary.
  const int64_t rows = p.row_end - p.row_offset;
  const int64_t n_win = (rows + p.win - 1) / p.win;
  const int64_t full = rows / p.win, rest = rows % p.win;
  const int64_t T = p.tile_m;
  const int64_t max_tiles = full * ((p.win + T - 1) / T) + (rest + T - 1) / T + n_e + n_win;
  int grid = sm_count();
  if (g_grouped_ctas > 0) grid = g_grouped_ctas;
  const int64_t need = (max_tiles + kMyTilesMax - 1) / kMyTilesMax;
  if (grid < need) grid = static_cast<int>(need);
  if (grid > max_tiles) grid = static_cast<int>(max_tiles);
  p.my_cap = kMyTilesMax;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kGThreads, 1, 1);
  cfg.dynamicSmemBytes = total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  using KernelFn = void (*)(CUtensorMap, CUtensorMap, GroupedParams);
  KernelFn fn;
  switch (p.r_pad) {
    case 16: fn = p.x_tma ? grouped_fold_kernel<16, true> : grouped_fold_kernel<16, false>; break;
    case 32: fn = p.x_tma ? grouped_fold_kernel<32, true> : grouped_fold_kernel<32, false>; break;
    case 48: fn = p.x_tma ? grouped_fold_kernel<48, true> : grouped_fold_kernel<48, false>; break;
    default: fn = p.x_tma ? grouped_fold_kernel<64, true> : grouped_fold_kernel<64, false>; break;
  }
  const cudaError_t err = cudaLaunchKernelEx(&cfg, fn, tmap, tmap_x, p);
  if (err != cudaSuccess) return cuda_status(err);
  return cuda_status(cudaGetLastError());
}

mlg_status fill_common(GroupedParams &p, const mlg_bf16 *x, const int32_t *row_adapter,
                       const uint64_t *a_table, const uint64_t *b_table, const float *scale_table,
                       mlg_bf16 *base_out, int32_t k_in, int32_t max_rank, int32_t n_out) {
  const mlg_status shape = check_shapes(k_in, max_rank, n_out);
  if (shape != MLG_OK) return shape;
  if (!x || !a_table || !b_table || !scale_table || !base_out) return MLG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(base_out)) return MLG_ERR_UNSUPPORTED;
  p.x = reinterpret_cast<const uint8_t *>(x);
  p.row_adapter = row_adapter;
  p.a_table = a_table;
  p.b_table = b_table;
  p.scale_table = scale_table;
  p.base_out = reinterpret_cast<uint8_t *>(base_out);
  p.k_in = k_in;
  p.rank = max_rank;
  p.n_out = n_out;
  p.tile_m = kTileM;
  return MLG_OK;
}

}  // namespace

uint32_t grouped_read_errors(bool clear) {
  uint32_t v = 0;
  cudaMemcpyFromSymbol(&v, g_grouped_errors, sizeof v);
  if (clear) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(g_grouped_errors, &z, sizeof z);
  }
  return v;
}

void grouped_set_ctas(int ctas) { g_grouped_ctas = ctas; }

}  // namespace mlg

extern "C" mlg_status mlg_grouped_down(const mlg_bf16 *x, const int32_t *expert_offsets,
                                       const int32_t *src, const int32_t *row_adapter,
                                       const uint64_t *a_table, const uint64_t *b_table,
                                       const float *scale_table, mlg_bf16 *base_out,
                                       int32_t k_in, int32_t max_rank, int32_t n_out,
                                       int32_t top_k, int32_t n_experts, int32_t row_offset,
                                       int32_t row_end, void *stream) {
  using namespace mlg;
  if (top_k < 1 || n_experts < 0 || row_offset < 0 || row_end < row_offset)
    return MLG_ERR_INVALID_ARG;
  GroupedParams p = {};
  const mlg_status st = fill_common(p, x, row_adapter, a_table, b_table, scale_table, base_out,
                                    k_in, max_rank, n_out);
  if (st != MLG_OK) return st;
  if (!expert_offsets || !src) return MLG_ERR_INVALID_ARG;
  if (row_end == row_offset || n_experts == 0) return MLG_OK;
  p.offsets = expert_offsets;
  p.src = src;
  p.top_k = top_k;
  p.n_experts = n_experts;
  p.row_offset = row_offset;
  p.row_end = row_end;
  p.win = row_end - row_offset;  // one window
  return launch_grouped(p, static_cast<cudaStream_t>(stream));
}

extern "C" mlg_status mlg_grouped_down_all_windows(
    const mlg_bf16 *x, const int32_t *expert_offsets, const int32_t *src,
    const int32_t *row_adapter, const uint64_t *a_table, const uint64_t *b_table,
    const float *scale_table, mlg_bf16 *base_out, int32_t k_in, int32_t max_rank, int32_t n_out,
    int32_t top_k, int32_t n_experts, int32_t total_rows, uint32_t cap, void *stream) {
  using namespace mlg;
  if (cap == 0) return MLG_ERR_CAP_ZERO;
  if (top_k < 1 || n_experts < 0 || total_rows < 0) return MLG_ERR_INVALID_ARG;
  GroupedParams p = {};
  const mlg_status st = fill_common(p, x, row_adapter, a_table, b_table, scale_table, base_out,
                                    k_in, max_rank, n_out);
  if (st != MLG_OK) return st;
  if (!expert_offsets || !src) return MLG_ERR_INVALID_ARG;
  if (total_rows == 0 || n_experts == 0) return MLG_OK;
  p.offsets = expert_offsets;
  p.src = src;
  p.top_k = top_k;
  p.n_experts = n_experts;
  p.row_offset = 0;
  p.row_end = total_rows;
  p.win = cap < static_cast<uint32_t>(total_rows) ? static_cast<int32_t>(cap) : total_rows;
  return launch_grouped(p, static_cast<cudaStream_t>(stream));
}

extern "C" mlg_status mlg_grouped_down_xrows(
    const mlg_bf16 *x_rows, const int32_t *expert_offsets, const int32_t *src,
    const int32_t *row_adapter, const uint64_t *a_table, const uint64_t *b_table,
    const float *scale_table, mlg_bf16 *base_out, int32_t k_in, int32_t max_rank, int32_t n_out,
    int32_t top_k, int32_t n_experts, int32_t row_offset, int32_t row_end, uint32_t cap,
    void *stream) {
  using namespace mlg;
  if (cap == 0) return MLG_ERR_CAP_ZERO;
  if (top_k < 1 || n_experts < 0 || row_offset < 0 || row_end < row_offset)
    return MLG_ERR_INVALID_ARG;
  GroupedParams p = {};
  const mlg_status st = fill_common(p, x_rows, row_adapter, a_table, b_table, scale_table,
                                    base_out, k_in, max_rank, n_out);
  if (st != MLG_OK) return st;
  if (!expert_offsets || !src) return MLG_ERR_INVALID_ARG;
  if (row_end == row_offset || n_experts == 0) return MLG_OK;
  p.offsets = expert_offsets;
  p.src = src;
  p.top_k = top_k;
  p.n_experts = n_experts;
  p.row_offset = row_offset;
  p.row_end = row_end;
  const int32_t len = row_end - row_offset;
  p.win = cap < static_cast<uint32_t>(len) ? static_cast<int32_t>(cap) : len;
  p.x_per_row = 1;
  p.x_tma = 1;
  return launch_grouped(p, static_cast<cudaStream_t>(stream));
}

extern "C" mlg_status mlg_router_fold(const mlg_bf16 *x, const int32_t *row_adapter,
                                      const uint64_t *a_table, const uint64_t *b_table,
                                      const float *scale_table, mlg_bf16 *base_out,
                                      int32_t n_tokens, int32_t k_in, int32_t max_rank,
                                      int32_t n_out, void *stream) {
  using namespace mlg;
  if (n_tokens < 0) return MLG_ERR_INVALID_ARG;
  GroupedParams p = {};
  const mlg_status st = fill_common(p, x, row_adapter, a_table, b_table, scale_table, base_out,
                                    k_in, max_rank, n_out);
  if (st != MLG_OK) return st;
  if (n_tokens == 0) return MLG_OK;
  p.offsets = nullptr;  // one span [0, n_tokens): expert 0 of a one-entry table
  p.src = nullptr;      // identity rows, x_row = t
  p.top_k = 1;
  p.n_experts = 1;
  p.row_offset = 0;
  p.row_end = n_tokens;
  p.win = n_tokens;
  // One span: tiles just tall enough that every SM gets at most one (whole
  // 4-row steps, so that nearly every SM gets one), so no SM idles while
  // others fold a second tile.
  const int64_t per_sm = (static_cast<int64_t>(n_tokens) + sm_count() - 1) / sm_count();
  p.tile_m = static_cast<int32_t>(
      std::min<int64_t>(kTileM, std::max<int64_t>(16, (per_sm + 3) / 4 * 4)));
  p.x_tma = 1;
  return launch_grouped(p, static_cast<cudaStream_t>(stream));
}
