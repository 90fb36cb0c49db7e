// mlg_gather.cu -- decode-side MoE expert LoRA fold (moe_lora_gather_bgmv of
// the moe_lora_grouped module index): for every flat (token, slot) row,
//     base_out[row] += scale_e * (x[row / top_k] @ A_e^T) @ B_e^T,  e = indices[row],
// skipping rows whose token has a negative row-map entry (moe_row_adapter.rs,
// build_moe_row_adapter_decode) and experts that fold nothing.
//
// GB300 design (not the pages' two-launch shrink/expand layout).  Decode is
// bound by latency and by the bytes of the expert pairs, so each expert's A_e
// and B_e leave HBM once and every CTA gets all of its bytes in flight at once:
//  * work unit = (expert, n slice).  Two ways to split an expert over CTAs:
//      - cs == 1 ("full shrink"): each CTA computes all of h (A_e is read once
//        from HBM and again from L2 by the other n slices) and folds its own
//        n slice -- no communication between CTAs; chosen when A_e is small
//        next to B_e (down projections);
//      - cs > 1 (a thread-block cluster of cs CTAs): rank q computes h over k
//        columns [q*ks, (q+1)*ks); the partial h are summed through
//        distributed shared memory in a fixed rank order; chosen when A_e
//        dominates (gate / up projections);
//  * loads and stores are TMA bulk copies with mbarrier completion (the A_e
//    rows spread over every warp); the B_e fragments of the expand are loaded
//    straight into registers;
//  * programmatic dependent launch: the table read and the compaction of the
//    experts that fold happen before griddepcontrol.wait, so they overlap the
//    preceding kernel; after it the routing loads go out first, then the
//    weight copies, so the routing scan does not wait behind the pair stream;
//    x, base_out and the B_e fragments follow the scan;
//  * shrink h = x A_e^T on the tensor cores (mma.sync m16n8k16 bf16 -> fp32,
//    M = rank, N = rows; decode has 1..32 rows per expert, below any tcgen05
//    M); expand with swapped operands (M = 16 rows of B_e, N = rows, K = rank)
//    against h split into bf16 hi + lo halves, so h enters at ~2^-17
//    relative precision (h stays fp32 in effect) and the expand cost does not
//    depend on how many rows an expert has;
//  * epilogue: out = RNE_bf16(base + scale * (h B^T)) in shared memory, then
//    bulk-stored; rows that do not fold are never loaded or stored;
//  * multi-adapter tables (one set of cells per adapter slot, the row map
//    naming the set) fold through the row's cell; for them the units are the
//    cells the routing hits (read first), and a CTA prefetches its next
//    unit's slices into L2 while it folds the current one.
#include <cuda_bf16.h>

#include <mutex>

#include "mlg_internal.h"
#include "mlg_ptx.cuh"

namespace mlg {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRowGroup = 32;                 // most rows of one expert folded per pass
constexpr int kScanPer = 8;                      // rows per thread per scan chunk
constexpr int kScanChunk = kScanPer * kThreads;  // 2048 rows
constexpr int kMaxMtPerPass = 8;  // B_e m-tiles x k-steps a warp holds in registers
constexpr int kMaxCompact = 512;  // tables up to this length are compacted to foldable experts

static __device__ uint32_t g_gather_errors;

struct GatherParams {
  const uint16_t *x;
  const int32_t *indices;
  const int32_t *row_adapter;
  const uint64_t *a_table;
  const uint64_t *b_table;
  const float *scale_table;
  uint16_t *base_out;
  int32_t n_slots, k_in, rank, n_out, top_k, n_experts;  // n_experts: table cells
  int32_t e_model, n_adapters;  // multi-adapter tables (n_adapters > 0): cell = slot * e_model + id
  int32_t hit_compact;          // units: only cells with a folding row (routing read first)
  int32_t ns2;            // n slices per cluster rank (independent CTAs, full shrink each)
  int32_t ks, ns;         // k columns per cluster rank, n columns per CTA
  int32_t rg;             // rows per pass (16 or 32)
  uint32_t stride_a;      // bytes per A_e / x row in shared memory
  uint32_t stride_base;   // bytes per base row in shared memory
  uint32_t off_a, off_x, off_base, off_p, off_hloc, hloc_bytes, smem_bytes;
};

__device__ __forceinline__ void record_error(uint32_t bit) { atomicOr(&g_gather_errors, bit); }

__device__ __forceinline__ uint32_t ld_nc_u32(const void *ptr) {
  uint32_t v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}

// Issue the index and row-map loads of one scan chunk (rows base + i*256 + tid).
__device__ __forceinline__ void scan_load(const GatherParams &p, int base, int (&idx)[kScanPer],
                                          int (&ra)[kScanPer]) {
#pragma unroll
  for (int i = 0; i < kScanPer; ++i) {
    const int row = base + i * kThreads + threadIdx.x;
    idx[i] = -1;
    ra[i] = -1;
    if (row < p.n_slots) {
      idx[i] = __ldg(p.indices + row);
      ra[i] = __ldg(p.row_adapter + row / p.top_k);
    }
    if (p.n_adapters > 0)  // the row map names the table set: fold through its cell
      idx[i] = (ra[i] >= 0 && ra[i] < p.n_adapters && idx[i] >= 0 && idx[i] < p.e_model)
                   ? ra[i] * p.e_model + idx[i]
                   : -1;
  }
}

// Collect the rows [g0, g0 + cap) of the rows that fold through expert e, in
// the order (chunk, i, warp, lane) -- the same in every CTA -- and return the
// total number of such rows.  Block-uniform; two barriers per 2048-row chunk.
// When have0, chunk 0's loads are passed in (already issued).  With s_hist,
// every folding row is also counted for its expert (e = -1 only counts).
__device__ int scan_rows(const GatherParams &p, int e, int g0, int cap, const int (&idx0)[kScanPer],
                         const int (&ra0)[kScanPer], bool have0, int *s_rows,
                         int (*s_cnt)[kWarps], int *s_hist = nullptr) {
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

// Experts with more folding rows than one pass takes (rg) are "heavy"; the
// i-th heavy expert by id gets the i-th helper cluster, if there is one.
// who >= 0: the expert helper `who` takes (-1 if none); who < 0: whether
// expert -1 - who has a helper (1 / 0).  Warp 0 computes, *s_out holds the
// result after the next barrier.
__device__ void heavy_assign(const int *s_hist, int n_experts, int rg, int n_helpers, int who,
                             int *s_out) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) != 0) return;
  int run = 0, found = who >= 0 ? -1 : 0;
  for (int b = 0; b < n_experts; b += 32) {
    const int ex = b + lane;
    const bool heavy = ex < n_experts && s_hist[ex] > rg;
    const unsigned m = __ballot_sync(0xffffffffu, heavy);
    const int rank = run + __popc(m & ((1u << lane) - 1u));
    if (heavy && rank < n_helpers) {
      if (who >= 0 && rank == who) found = ex;
      if (who < 0 && ex == -1 - who) found = 1;
    }
    run += __popc(m);
  }
  const int v = __reduce_max_sync(0xffffffffu, found);
  if (lane == 0) *s_out = v;
}

// B_e fragments of one 16-row m-tile for the swapped expand (A operand of
// m16n8k16): thread (g, c) holds B_e rows n and n+8, rank columns
// c*q + 4*st .. c*q + 4*st + 3 of every k-step st (q = rank / 4).  The same
// physical-column assignment is used for h, so the contraction covers every
// rank column once; slots at or past q are zero.
template <int KST>
__device__ __forceinline__ void load_b_frags(const uint8_t *B, int n, int n_out, int r, int c,
                                             uint32_t (&f)[KST][4]) {
  const int q4 = r / 4;
#pragma unroll
  for (int st = 0; st < KST; ++st) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int row = n + hr * 8;
      const bool in = row < n_out;
      const uint8_t *base = B + (static_cast<size_t>(in ? row : 0) * r + c * q4 + 4 * st) * 2;
      f[st][hr] = (in && 4 * st < q4) ? ld_nc_u32(base) : 0u;              // slots 0, 1
      f[st][2 + hr] = (in && 4 * st + 2 < q4) ? ld_nc_u32(base + 4) : 0u;  // slots 2, 3
    }
  }
}

template <int RP>  // max_rank rounded up to a multiple of 16
__global__ void __launch_bounds__(kThreads, 2) gather_fold_kernel(const GatherParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2];  // 0: weights, 1: rows
  __shared__ int s_rows[kMaxRowGroup];
  __shared__ int s_cnt[kScanPer][kWarps];
  __shared__ int s_ex[kMaxCompact];  // foldable experts, in id order

  constexpr int MT = RP / 16;   // rank m-tiles of the shrink
  constexpr int KST = RP / 16;  // k-steps of the expand
  constexpr int HS = RP + 4;    // fp32 row stride of the h buffers
  constexpr int HB = RP + 8;    // bf16 row stride of the hi / lo buffers
  constexpr int MPP = kMaxMtPerPass / KST > 0 ? kMaxMtPerPass / KST : 1;  // m-tiles per pass

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t q = cluster_ctarank();
  const uint32_t cs = gridDim.x / ncluster_x();

  const int k0 = static_cast<int>(q) * p.ks;
  const int ksv = max(0, min(p.ks, p.k_in - k0));
  const int r = p.rank;
  const int q4 = r / 4;

  uint8_t *sA = smem + p.off_a;
  uint8_t *sX = smem + p.off_x;
  uint8_t *sBase = smem + p.off_base;
  float *sP = reinterpret_cast<float *>(smem + p.off_p);
  // hi / lo bf16 copies of h (B operand of the expand) reuse the partials' space
  uint16_t *sHhi = reinterpret_cast<uint16_t *>(smem + p.off_p);
  uint16_t *sHlo = sHhi + kMaxRowGroup * HB;
  float *sHloc2[2] = {reinterpret_cast<float *>(smem + p.off_hloc),
                      reinterpret_cast<float *>(smem + p.off_hloc + p.hloc_bytes)};

  // A_e rows >= rank and the k tail of the A / x rows (up to the next 32) are
  // read by the MMAs but never written by a copy: zero them once.
  if (r < RP || (ksv & 31) != 0) {
    for (uint32_t i = tid * 16; i < p.off_base; i += kThreads * 16)
      *reinterpret_cast<uint4 *>(smem + i) = make_uint4(0, 0, 0, 0);
  }
  const uint32_t bar_w = smem_addr(&bars[0]), bar_x = smem_addr(&bars[1]);
  if (tid == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_x, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // The next fold in the stream may start its own prologue now: it reads only
  // tables and expert weights (never written by this kernel) before waiting.
  griddep_launch_dependents();
  uint32_t ph_w = 0, ph_x = 0, grp = 0;
  bool bad = false;
  bool waited = false;  // griddep_wait() done (before the first routing / x / base read)

  // Units are (expert, n slice) pairs over the experts whose cells fold
  // (tables are read before the wait: under early start the caller's contract
  // is that the preceding kernel does not write them),
  // so no cluster spends a round on an expert that folds nothing.  With
  // hit_compact (sparse tables: many cells, few rows each) the routing is
  // read first and only cells with a folding row become units, so no pair is
  // loaded that no row of this batch needs.
  const bool compact = p.n_experts <= kMaxCompact;
  int *s_hist = reinterpret_cast<int *>(smem + p.off_p);  // counts; free until a shrink
  const int no_idx[kScanPer] = {};
  const bool hits = compact && p.hit_compact;
  if (hits) {
    griddep_wait();
    waited = true;
    for (int i = tid; i < p.n_experts; i += kThreads) s_hist[i] = 0;
    __syncthreads();
    scan_rows(p, -1, 0, 0, no_idx, no_idx, false, s_rows, s_cnt, s_hist);
  }
  int n_fold = p.n_experts;
  if (compact) {
    n_fold = 0;
    for (int b = 0; b < p.n_experts; b += kThreads) {
      const int ex = b + tid;
      bool f = false;
      if (ex < p.n_experts) {
        const uint64_t a = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + ex);
        const uint64_t bb = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + ex);
        f = a != 0 && bb != 0 && ((a | bb) & 15u) == 0 && (!hits || s_hist[ex] > 0);
      }
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (lane == 0) s_cnt[0][warp] = __popc(m);
      __syncthreads();
      int before = n_fold, tot = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        before += (w < warp) ? s_cnt[0][w] : 0;
        tot += s_cnt[0][w];
      }
      if (f) s_ex[before + __popc(m & ((1u << lane) - 1u))] = ex;
      n_fold += tot;
      __syncthreads();
    }
  }
  const int n_units = n_fold * p.ns2;
  // Clusters left over once every unit has one become helpers: the i-th takes
  // the second half of the rows of the i-th heavy expert (its owner folds the
  // first half), so no cluster runs a second pass while others idle.  Both
  // sides decide from the same per-expert row counts, read after the wait.
  const int ncl = static_cast<int>(ncluster_x());
  const int n_helpers = (compact && p.ns2 == 1 && n_units < ncl) ? ncl - n_units : 0;
  for (int unit = static_cast<int>(cluster_id_x()); unit < n_units + n_helpers; unit += ncl) {
    const bool help = unit >= n_units;
    int e = help ? -1 : (compact ? s_ex[unit / p.ns2] : unit / p.ns2);
    if (help) {
      if (!waited) {
        griddep_wait();
        waited = true;
      }
      for (int i = tid; i < p.n_experts; i += kThreads) s_hist[i] = 0;
      __syncthreads();
      scan_rows(p, -1, 0, 0, no_idx, no_idx, false, s_rows, s_cnt, s_hist);
      heavy_assign(s_hist, p.n_experts, p.rg, n_helpers, unit - n_units, &s_cnt[0][0]);
      __syncthreads();
      e = s_cnt[0][0];
      __syncthreads();  // s_cnt is rewritten by the next scan
      if (e < 0) continue;
    }
    const int ni = (unit % p.ns2) * static_cast<int>(cs) + static_cast<int>(q);  // n slice
    const int n0 = ni * p.ns;
    const int nsv = max(0, min(p.ns, p.n_out - n0));
    const uint64_t a_addr = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + e);
    const uint64_t b_addr = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + e);
    const float scale = __ldg(p.scale_table + e);
    if (a_addr == 0 || b_addr == 0 || ((a_addr | b_addr) & 15u) != 0)
      continue;  // the expert folds nothing (uniform in the cluster)
    if (warp == 1 && lane == 0 && !help && unit + ncl < n_units) {
      // This CTA's slices of the next unit's pair, into L2 while this one runs.
      const int u2 = unit + ncl;
      const int e2 = compact ? s_ex[u2 / p.ns2] : u2 / p.ns2;
      const uint64_t a2 = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + e2);
      const uint64_t b2 = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + e2);
      const int n2 = ((u2 % p.ns2) * static_cast<int>(cs) + static_cast<int>(q)) * p.ns;
      const int nsv2 = max(0, min(p.ns, p.n_out - n2));
      if (a2 != 0 && b2 != 0 && ((a2 | b2) & 15u) == 0) {
        const uint8_t *A2 = reinterpret_cast<const uint8_t *>(a2);
        if (ksv > 0) {
          if (ksv == p.k_in) {  // whole rows: one contiguous run
            for (uint32_t o = 0; o < static_cast<uint32_t>(r * p.k_in * 2); o += 8192)
              prefetch_l2(A2 + o, min(8192u, static_cast<uint32_t>(r * p.k_in * 2) - o));
          } else {
            for (int j = 0; j < r; ++j)
              prefetch_l2(A2 + (static_cast<size_t>(j) * p.k_in + k0) * 2, ksv * 2u);
          }
        }
        const uint8_t *B2 = reinterpret_cast<const uint8_t *>(b2) + static_cast<size_t>(n2) * r * 2;
        const uint32_t bb = static_cast<uint32_t>(nsv2 * r * 2);
        for (uint32_t o = 0; o < bb; o += 8192) prefetch_l2(B2 + o, min(8192u, bb - o));
      }
    }
    // Routing, x and base_out may be written by the preceding kernel.  The
    // routing loads go out first: issued after the weight copies they would
    // queue behind the whole pair stream (~3 us) on their way back.
    if (!waited) {
      griddep_wait();
      waited = true;
    }
    int idx0[kScanPer], ra0[kScanPer];
    scan_load(p, 0, idx0, ra0);
    // A_e k slice: one bulk copy per rank row, issued by eight lanes of every
    // warp (a single warp issuing all of them stalls for ~2 us on the copy
    // engine's queue, and every warp then waits for it at the routing scan).
    // The byte count is posted before the barrier, so it precedes every copy.
    if (tid == 0 && !bad) mbar_arrive_expect_tx(bar_w, ksv > 0 ? r * ksv * 2u : 0u);
    fence_proxy_async_smem();  // earlier generic accesses before new async writes
    __syncthreads();
    if (!bad && ksv > 0 && lane < 8) {
      const uint8_t *A = reinterpret_cast<const uint8_t *>(a_addr);
      for (int j = warp * 8 + lane; j < r; j += kWarps * 8)
        bulk_g2s(smem_addr(sA + j * p.stride_a), A + (static_cast<size_t>(j) * p.k_in + k0) * 2,
                 ksv * 2u, bar_w);
    }
    // B_e fragments go straight into registers once the first row group's x
    // and base_out copies are out (their loads would delay the routing scan).
    const uint8_t *B = reinterpret_cast<const uint8_t *>(b_addr);
    const int mtn = (nsv + 15) / 16;
    uint32_t bf[MPP][KST][4];
    int bf_pass = -1;  // which pass of m-tiles bf holds (none yet)
    const bool count = n_helpers > 0 && !help;  // an owner also counts every expert's rows
    if (count) {
      for (int i = tid; i < p.n_experts; i += kThreads) s_hist[i] = 0;
      __syncthreads();
    }
    const int total = scan_rows(p, e, 0, kMaxRowGroup, idx0, ra0, true, s_rows, s_cnt,
                                count ? s_hist : nullptr);
    // Rows of this unit: [0, total), or a half of them when the expert is split.
    int lo = 0, hi = total;
    if (help) {
      lo = (total + 1) / 2;
    } else if (count) {
      heavy_assign(s_hist, p.n_experts, p.rg, n_helpers, -1 - e, &s_cnt[0][0]);
      __syncthreads();
      if (s_cnt[0][0] == 1) hi = (total + 1) / 2;
      __syncthreads();
    }
    if (hi <= lo) {  // an adapted expert with no folding row here: let its weights land
      const bool timed_out = !bad && !mbar_wait_bounded(bar_w, ph_w);
      ph_w ^= 1u;
      if (__syncthreads_or(timed_out)) {
        if (!bad && tid == 0) record_error(kErrWaitTimeout);
        bad = true;
      }
      continue;
    }
    bool have_weights = false;
    int list0 = 0;  // s_rows holds ranks [list0, list0 + kMaxRowGroup) of the row list

    for (int g0 = lo; g0 < hi; g0 += p.rg, ++grp) {
      const int n_g = min(p.rg, hi - g0);
      if (g0 + n_g > list0 + kMaxRowGroup) {
        scan_rows(p, e, g0, kMaxRowGroup, idx0, ra0, false, s_rows, s_cnt);
        list0 = g0;
      }
      const int *rows = s_rows + (g0 - list0);

      // Rows of this group: x slices and base slices.
      if (warp == 0 && !bad) {
        bulk_wait_read_all();  // earlier bulk stores of sBase have read it
        const uint32_t bytes = n_g * ((ksv > 0 ? ksv * 2u : 0u) + (nsv > 0 ? nsv * 2u : 0u));
        if (lane == 0) mbar_arrive_expect_tx(bar_x, bytes);
        __syncwarp();
        if (lane < n_g) {
          const int row = rows[lane];
          const int t = row / p.top_k;
          if (ksv > 0)
            bulk_g2s(smem_addr(sX + lane * p.stride_a),
                     p.x + static_cast<size_t>(t) * p.k_in + k0, ksv * 2u, bar_x);
          if (nsv > 0)
            bulk_g2s(smem_addr(sBase + lane * p.stride_base),
                     p.base_out + static_cast<size_t>(row) * p.n_out + n0, nsv * 2u, bar_x);
        }
      }
      if (bf_pass != 0) {  // B_e fragments of this warp's first m-tiles
#pragma unroll
        for (int i = 0; i < MPP; ++i) {
          const int m = warp + i * kWarps;
          if (m < mtn) load_b_frags<KST>(B, n0 + m * 16 + g, p.n_out, r, c, bf[i]);
        }
        bf_pass = 0;
      }
      bool timed_out = false;
      if (!bad && !have_weights) timed_out = !mbar_wait_bounded(bar_w, ph_w);
      if (!bad && !timed_out) timed_out = !mbar_wait_bounded(bar_x, ph_x);
      if (!have_weights) ph_w ^= 1u;
      ph_x ^= 1u;
      have_weights = true;
      // One thread's timeout stops the whole CTA's work (kept CTA-uniform).
      if (__syncthreads_or(timed_out)) {
        if (!bad && tid == 0) record_error(kErrWaitTimeout);
        bad = true;
      }

      // ---- shrink: partial h[row][j] over this CTA's k slice --------------
      // MMA M = rank (A_e rows), N = rows (x rows), K = k.  Each thread column
      // c feeds physical k = 8c .. 8c+7 of every 32-wide k block; A and B use
      // the same k assignment, so the contraction covers every k once.
      float *sHloc = sHloc2[grp & 1];
      const int ntr = (n_g + 7) / 8;
      const int units = MT * ntr;
      int ksplit = 1;
      while (units * ksplit * 2 <= kWarps) ksplit *= 2;
      const int kblocks = (ksv + 31) / 32;
      int my_units[2] = {-1, -1};
      int kq = 0;
      if (units >= kWarps) {
        my_units[0] = warp;
        my_units[1] = warp + kWarps < units ? warp + kWarps : -1;
      } else if (warp < units * ksplit) {
        my_units[0] = warp % units;
        kq = warp / units;
      }
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      // A warp with one unit spreads its MMAs over four accumulators (four
      // independent chains: the two MMAs of a k block, even and odd blocks),
      // added in a fixed order afterwards.
      const bool dual = my_units[1] < 0;
      if (!bad && my_units[0] >= 0) {
        const int kb_lo = kq * kblocks / ksplit, kb_hi = (kq + 1) * kblocks / ksplit;
        if (dual) {
          float ex[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          const int u = my_units[0], mt = u % MT, nt = u / MT;
          const uint8_t *ra = sA + (mt * 16 + g) * p.stride_a, *rb = ra + 8 * p.stride_a;
          const uint8_t *rx = sX + (nt * 8 + g) * p.stride_a;
#pragma unroll 2
          for (int kb = kb_lo; kb < kb_hi; kb += 2) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              if (kb + q >= kb_hi) continue;
              const uint32_t kbyte = ((kb + q) * 32 + 8 * c) * 2;
              const uint4 pa = *reinterpret_cast<const uint4 *>(ra + kbyte);
              const uint4 qa = *reinterpret_cast<const uint4 *>(rb + kbyte);
              const uint4 sx = *reinterpret_cast<const uint4 *>(rx + kbyte);
              mma_bf16_16816(acc[q], pa.x, qa.x, pa.y, qa.y, sx.x, sx.y);
              mma_bf16_16816(ex[q], pa.z, qa.z, pa.w, qa.w, sx.z, sx.w);
            }
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[0][v] = (acc[0][v] + ex[0][v]) + (acc[1][v] + ex[1][v]);
        } else {
#pragma unroll 4
          for (int kb = kb_lo; kb < kb_hi; ++kb) {
            const uint32_t kbyte = (kb * 32 + 8 * c) * 2;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int u = my_units[i];
              if (u < 0) continue;
              const int mt = u % MT, nt = u / MT;
              const uint4 pa =
                  *reinterpret_cast<const uint4 *>(sA + (mt * 16 + g) * p.stride_a + kbyte);
              const uint4 qa =
                  *reinterpret_cast<const uint4 *>(sA + (mt * 16 + g + 8) * p.stride_a + kbyte);
              const uint4 sx =
                  *reinterpret_cast<const uint4 *>(sX + (nt * 8 + g) * p.stride_a + kbyte);
              mma_bf16_16816(acc[i], pa.x, qa.x, pa.y, qa.y, sx.x, sx.y);
              mma_bf16_16816(acc[i], pa.z, qa.z, pa.w, qa.w, sx.z, sx.w);
            }
          }
        }
      }
      // acc[i] = (rank mt*16+g, row nt*8+2c), (.., +1), (rank +8, row), (rank +8, row +1)
      float *dst = (ksplit == 1) ? sHloc : sP + kq * (ntr * 8 * HS);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int u = my_units[i];
        if (u < 0) continue;
        const int mt = u % MT, nt = u / MT;
        const int j = mt * 16 + g, row = nt * 8 + 2 * c;
        dst[row * HS + j] = acc[i][0];
        dst[(row + 1) * HS + j] = acc[i][1];
        dst[row * HS + j + 8] = acc[i][2];
        dst[(row + 1) * HS + j + 8] = acc[i][3];
      }
      __syncthreads();
      if (ksplit > 1) {  // fixed-order sum of the k-split partials
        for (int idx = tid; idx < ntr * 8 * HS; idx += kThreads) {
          float sum = 0.f;
          for (int kk = 0; kk < ksplit; ++kk) sum += sP[kk * (ntr * 8 * HS) + idx];
          sHloc[idx] = sum;
        }
        __syncthreads();
      }
      // ---- h (summed over the cluster's k slices) -> bf16 hi / lo ----------
      // sHloc alternates between two buffers, so a peer still reading this
      // group's buffer is never overwritten before the next group's barrier.
      if (cs > 1) cluster_sync();
      {
        const uint32_t local = smem_addr(sHloc);
        const int n2 = ntr * 8 * RP / 2;  // pairs of h values
        for (int i2 = tid; i2 < n2; i2 += kThreads) {
          const int row = (2 * i2) / RP, j = (2 * i2) % RP;
          float h0 = 0.f, h1 = 0.f;
          if (cs > 1) {
            // Every rank's partial is requested before any is added, so the
            // remote round trips overlap; the sum is then taken in rank order.
            float v0[8], v1[8];
#pragma unroll
            for (uint32_t rk = 0; rk < 8; ++rk) {
              v0[rk] = v1[rk] = 0.f;
              if (rk < cs) {
                const uint32_t a = map_to_rank(local + (row * HS + j) * 4, rk);
                asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                             : "=f"(v0[rk]), "=f"(v1[rk])
                             : "r"(a)
                             : "memory");
              }
            }
#pragma unroll
            for (uint32_t rk = 0; rk < 8; ++rk) {
              if (rk < cs) {
                h0 += v0[rk];
                h1 += v1[rk];
              }
            }
          } else {
            h0 = sHloc[row * HS + j];
            h1 = sHloc[row * HS + j + 1];
          }
          float a0, b0, a1, b1;
          split_hi_lo(h0, a0, b0);
          split_hi_lo(h1, a1, b1);
          *reinterpret_cast<uint32_t *>(sHhi + row * HB + j) = pack_bf16x2(a0, a1);
          *reinterpret_cast<uint32_t *>(sHlo + row * HB + j) = pack_bf16x2(b0, b1);
        }
      }
      __syncthreads();

      // ---- expand + epilogue (swapped operands: M = B_e rows, N = rows) ----
      if (!bad && nsv > 0) {
        const int nte = (n_g + 7) / 8;  // row n-tiles
        for (int pass = 0; pass * MPP * kWarps < mtn; ++pass) {
          if (pass != bf_pass) {  // later passes, or pass 0 again for a later row group
#pragma unroll
            for (int i = 0; i < MPP; ++i) {
              const int m = warp + (pass * MPP + i) * kWarps;
              if (m < mtn) load_b_frags<KST>(B, n0 + m * 16 + g, p.n_out, r, c, bf[i]);
            }
            bf_pass = pass;
          }
          for (int nt = 0; nt < nte; ++nt) {
            // h^T fragments (B operand): rows nt*8 + g, same physical rank columns
            uint32_t hh[KST][2], hl[KST][2];
            const int hrow = nt * 8 + g;
#pragma unroll
            for (int st = 0; st < KST; ++st) {
              const int j = c * q4 + 4 * st;
              const bool v0 = 4 * st < q4, v1 = 4 * st + 2 < q4;
              hh[st][0] = v0 ? *reinterpret_cast<const uint32_t *>(sHhi + hrow * HB + j) : 0u;
              hh[st][1] = v1 ? *reinterpret_cast<const uint32_t *>(sHhi + hrow * HB + j + 2) : 0u;
              hl[st][0] = v0 ? *reinterpret_cast<const uint32_t *>(sHlo + hrow * HB + j) : 0u;
              hl[st][1] = v1 ? *reinterpret_cast<const uint32_t *>(sHlo + hrow * HB + j + 2) : 0u;
            }
            // All MMAs of the pass first, then every base element is read, then
            // every result written: the shared-memory round trips overlap instead
            // of forming one load -> store chain per element.
            // The hi and lo halves accumulate in separate registers (two
            // independent MMA chains per m-tile), summed in a fixed order.
            float d[MPP][4];
#pragma unroll
            for (int i = 0; i < MPP; ++i) {
              const int m = warp + (pass * MPP + i) * kWarps;
              float dl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int u = 0; u < 4; ++u) d[i][u] = 0.f;
              if (m >= mtn) continue;
#pragma unroll
              for (int st = 0; st < KST; ++st) {
                mma_bf16_16816(d[i], bf[i][st][0], bf[i][st][1], bf[i][st][2], bf[i][st][3],
                               hh[st][0], hh[st][1]);
                mma_bf16_16816(dl, bf[i][st][0], bf[i][st][1], bf[i][st][2], bf[i][st][3],
                               hl[st][0], hl[st][1]);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) d[i][u] += dl[u];
            }
            // d[i] = (n m*16+g, row nt*8+2c), (n, row+1), (n+8, row), (n+8, row+1)
            constexpr int CH = MPP < 4 ? MPP : 4;  // m-tiles per batch of loads (registers)
#pragma unroll
            for (int i0 = 0; i0 < MPP; i0 += CH) {
              uint32_t bv[CH][4];
#pragma unroll
              for (int i = 0; i < CH; ++i) {
                const int m = warp + (pass * MPP + i0 + i) * kWarps;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int nl = m * 16 + g + (u >> 1) * 8;
                  const int row = nt * 8 + 2 * c + (u & 1);
                  bv[i][u] = 0u;
                  if (m < mtn && nl < nsv && row < n_g)
                    bv[i][u] = *(reinterpret_cast<const uint16_t *>(sBase + row * p.stride_base) + nl);
                }
              }
#pragma unroll
              for (int i = 0; i < CH; ++i) {
                const int m = warp + (pass * MPP + i0 + i) * kWarps;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int nl = m * 16 + g + (u >> 1) * 8;
                  const int row = nt * 8 + 2 * c + (u & 1);
                  if (m < mtn && nl < nsv && row < n_g) {
                    const float base = __uint_as_float(bv[i][u] << 16);
                    *(reinterpret_cast<uint16_t *>(sBase + row * p.stride_base) + nl) =
                        __bfloat16_as_ushort(__float2bfloat16_rn(fmaf(scale, d[i0 + i][u], base)));
                  }
                }
              }
            }
          }
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (warp == 0 && !bad && nsv > 0 && lane < n_g) {
        const int row = rows[lane];
        bulk_s2g(p.base_out + static_cast<size_t>(row) * p.n_out + n0,
                 smem_addr(sBase + lane * p.stride_base), nsv * 2u);
        bulk_commit();
      }
    }
  }
  if (!waited) griddep_wait();  // complete only after the preceding kernel
  if (warp == 0) bulk_wait_all();
  if (cs > 1) cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

uint32_t round_up(uint32_t v, uint32_t m) { return (v + m - 1) / m * m; }

// Shared-memory layout for a split (cs, ns2); returns total bytes.
uint32_t layout(GatherParams &p, int cs, int ns2, int rp) {
  p.ns2 = ns2;
  p.ks = static_cast<int>(round_up((p.k_in + cs - 1) / cs, 32));
  p.ns = static_cast<int>(round_up((p.n_out + cs * ns2 - 1) / (cs * ns2), 8));
  uint32_t sa = p.ks * 2;
  if (sa % 128 == 0) sa += 64;  // 16-byte MMA operand loads conflict-free
  p.stride_a = sa;
  uint32_t sb = p.ns * 2;
  sb += (16 + 128 - sb % 128) % 128;  // row stride = 16 (mod 128) bytes
  p.stride_base = sb;
  const uint32_t hbytes = p.rg * (rp + 4) * 4;
  // k-split partials (<= 1280 floats), reused afterwards for the hi / lo h copies
  uint32_t pbytes = 1280 * 4;
  const uint32_t hilo = 2 * kMaxRowGroup * (rp + 8) * 2;
  if (hilo > pbytes) pbytes = hilo;
  uint32_t off = 0;
  p.off_a = off;
  off += round_up(rp * sa, 128);
  p.off_x = off;
  off += round_up(p.rg * sa, 128);
  p.off_base = off;
  off += round_up(p.rg * sb, 128);
  p.off_p = off;
  off += round_up(pbytes, 128);
  p.off_hloc = off;  // two buffers (alternating row groups)
  p.hloc_bytes = round_up(hbytes, 128);
  off += 2 * p.hloc_bytes;
  p.smem_bytes = off;
  return off;
}

int g_cluster_override = 0;
int g_nsplit_override = 0;
// Two CTAs per SM: each may use up to half of the 228 KB, less its ~2.5 KB of
// static shared memory and the 1 KB the driver reserves per CTA.
constexpr uint32_t kSmemTwoPerSm = 113 * 1024 - 3072;
constexpr uint32_t kSmemLimit = 227 * 1024 - 3072;  // leaves room for the static part

template <int RP>
cudaError_t launch(const GatherParams &p, int cs, int clusters, bool early, cudaStream_t stream) {
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [d = dev & 63] {
    attr_err[d] = cudaFuncSetAttribute(gather_fold_kernel<RP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemLimit));
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs * clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 2 : 1;  // without early start griddepcontrol.wait returns at once
  return cudaLaunchKernelEx(&cfg, gather_fold_kernel<RP>, p);
}

}  // namespace

int sm_count() {
  static int counts[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int &c = counts[dev & 63];
  if (c == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 148;
    c = v;
  }
  return c;
}

uint32_t gather_read_errors(bool clear) {
  uint32_t v = 0;
  cudaMemcpyFromSymbol(&v, g_gather_errors, sizeof v);
  if (clear) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(g_gather_errors, &z, sizeof z);
  }
  return v;
}

void gather_set_cluster_override(int cs) { g_cluster_override = cs; }
void gather_set_nsplit_override(int ns2) { g_nsplit_override = ns2; }

}  // namespace mlg

namespace mlg {
namespace {

// Both gather entry points: n_experts is the table length (cells); e_model /
// n_adapters describe multi-adapter tables (n_adapters == 0: single set).
mlg_status gather_dispatch(const mlg_bf16 *x, const int32_t *indices, const int32_t *row_adapter,
                           const uint64_t *a_table, const uint64_t *b_table,
                           const float *scale_table, mlg_bf16 *base_out, int32_t n_slots,
                           int32_t k_in, int32_t max_rank, int32_t n_out, int32_t top_k,
                           int32_t n_experts, int32_t e_model, int32_t n_adapters,
                           uint32_t flags, void *stream) {
  if ((flags & ~MLG_FOLD_AFTER_PRECEDING) != 0) return MLG_ERR_INVALID_ARG;
  const bool early = (flags & MLG_FOLD_AFTER_PRECEDING) == 0;
  if (n_slots == 0 || n_experts == 0) return MLG_OK;
  if (!x || !indices || !row_adapter || !a_table || !b_table || !scale_table || !base_out)
    return MLG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(base_out)) return MLG_ERR_UNSUPPORTED;

  // Expert pairs that fit half an SM go to the resident-pair kernel.
  const int path = gather_path_override();
  const bool resident = n_adapters > 0 ? decode_multi_eligible(k_in, max_rank, n_out, n_experts)
                                       : decode_fold_eligible(k_in, max_rank, n_out, n_experts);
  if (path == 1 && !resident) return MLG_ERR_UNSUPPORTED;
  if (path != 2 && resident)
    return cuda_status(decode_fold_launch(x, indices, row_adapter, a_table, b_table, scale_table,
                                          base_out, n_slots, k_in, max_rank, n_out, top_k,
                                          n_experts, e_model, n_adapters, early,
                                          static_cast<cudaStream_t>(stream)));

  GatherParams p = {};
  p.x = x;
  p.indices = indices;
  p.row_adapter = row_adapter;
  p.a_table = a_table;
  p.b_table = b_table;
  p.scale_table = scale_table;
  p.base_out = base_out;
  p.n_slots = n_slots;
  p.k_in = k_in;
  p.rank = max_rank;
  p.n_out = n_out;
  p.top_k = top_k;
  p.n_experts = n_experts;
  p.e_model = e_model;
  p.n_adapters = n_adapters;
  // Multi-adapter tables are sparse in a batch (a cell is one adapter's
  // expert): read the routing first and give units only to cells it hits.
  p.hit_compact = n_adapters > 0 ? 1 : 0;
  const int rp = static_cast<int>(round_up(max_rank, 16));
  // Rows per pass: decode batches spread ~n_slots / n_experts rows per expert.
  p.rg = (n_slots <= 16 * n_experts) ? 16 : 32;

  // Split: when A_e is at most half of B_e, every CTA computes the whole
  // shrink and the expert's n range is split over ns2 independent CTAs
  // (each CTA's share of the pair bounded to ~64 KB); else a cluster of cs
  // CTAs splits k (partial h summed in shared memory) and n, cs the smallest
  // that leaves room for two CTAs per SM.
  const double a_bytes = 2.0 * max_rank * k_in, b_bytes = 2.0 * max_rank * n_out;
  int cs = 1, ns2 = 1;
  if (2.0 * a_bytes <= b_bytes) {
    while (ns2 < 8 && a_bytes + b_bytes / ns2 > 64.0 * 1024) ns2 *= 2;
  }
  if (g_cluster_override > 0) cs = g_cluster_override;
  if (g_nsplit_override > 0) ns2 = g_nsplit_override;
  if (g_cluster_override == 0)
    while (layout(p, cs, ns2, rp) > kSmemTwoPerSm && cs < 8) cs *= 2;
  if (layout(p, cs, ns2, rp) > kSmemLimit) return MLG_ERR_UNSUPPORTED;

  // One cluster per (expert, n slice), looping when there are more than fit;
  // the grid is what can be resident at once (no second wave of CTAs).
  const int64_t units = static_cast<int64_t>(n_experts) * ns2;
  const int per_sm = layout(p, cs, ns2, rp) <= kSmemTwoPerSm ? 2 : 1;
  const int max_clusters = (per_sm * sm_count()) / cs > 0 ? (per_sm * sm_count()) / cs : 1;
  const int clusters = units < max_clusters ? static_cast<int>(units) : max_clusters;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  switch (rp) {
    case 16: err = launch<16>(p, cs, clusters, early, s); break;
    case 32: err = launch<32>(p, cs, clusters, early, s); break;
    case 48: err = launch<48>(p, cs, clusters, early, s); break;
    default: err = launch<64>(p, cs, clusters, early, s); break;
  }
  return cuda_status(err);
}

}  // namespace
}  // namespace mlg

namespace {

mlg_status gather_single(const mlg_bf16 *x, const int32_t *indices, const int32_t *row_adapter,
                         const uint64_t *a_table, const uint64_t *b_table,
                         const float *scale_table, mlg_bf16 *base_out, int32_t n_slots,
                         int32_t k_in, int32_t max_rank, int32_t n_out, int32_t top_k,
                         int32_t n_experts, uint32_t flags, void *stream) {
  using namespace mlg;
  if (n_slots < 0 || n_experts < 0 || top_k < 1) return MLG_ERR_INVALID_ARG;
  const mlg_status shape = check_shapes(k_in, max_rank, n_out);
  if (shape != MLG_OK) return shape;
  return gather_dispatch(x, indices, row_adapter, a_table, b_table, scale_table, base_out,
                         n_slots, k_in, max_rank, n_out, top_k, n_experts, n_experts, 0, flags,
                         stream);
}

mlg_status gather_multi(const mlg_bf16 *x, const int32_t *indices, const int32_t *row_adapter,
                        const uint64_t *a_table, const uint64_t *b_table, const float *scale_table,
                        mlg_bf16 *base_out, int32_t n_slots, int32_t k_in, int32_t max_rank,
                        int32_t n_out, int32_t top_k, int32_t n_experts, int32_t n_adapters,
                        uint32_t flags, void *stream) {
  using namespace mlg;
  if (n_slots < 0 || n_experts < 0 || n_adapters < 1 || top_k < 1) return MLG_ERR_INVALID_ARG;
  const int64_t cells = static_cast<int64_t>(n_experts) * n_adapters;
  if (cells > (1 << 30)) return MLG_ERR_UNSUPPORTED;
  const mlg_status shape = check_shapes(k_in, max_rank, n_out);
  if (shape != MLG_OK) return shape;
  return gather_dispatch(x, indices, row_adapter, a_table, b_table, scale_table, base_out,
                         n_slots, k_in, max_rank, n_out, top_k, static_cast<int32_t>(cells),
                         n_experts, n_adapters, flags, stream);
}

}  // namespace

extern "C" mlg_status mlg_gather_bgmv(const mlg_bf16 *x, const int32_t *indices,
                                      const int32_t *row_adapter, const uint64_t *a_table,
                                      const uint64_t *b_table, const float *scale_table,
                                      mlg_bf16 *base_out, int32_t n_slots, int32_t k_in,
                                      int32_t max_rank, int32_t n_out, int32_t top_k,
                                      int32_t n_experts, void *stream) {
  return gather_single(x, indices, row_adapter, a_table, b_table, scale_table, base_out, n_slots,
                       k_in, max_rank, n_out, top_k, n_experts, 0u, stream);
}

extern "C" mlg_status mlg_gather_bgmv_ex(const mlg_bf16 *x, const int32_t *indices,
                                         const int32_t *row_adapter, const uint64_t *a_table,
                                         const uint64_t *b_table, const float *scale_table,
                                         mlg_bf16 *base_out, int32_t n_slots, int32_t k_in,
                                         int32_t max_rank, int32_t n_out, int32_t top_k,
                                         int32_t n_experts, uint32_t flags, void *stream) {
  return gather_single(x, indices, row_adapter, a_table, b_table, scale_table, base_out, n_slots,
                       k_in, max_rank, n_out, top_k, n_experts, flags, stream);
}

extern "C" mlg_status mlg_gather_bgmv_multi(const mlg_bf16 *x, const int32_t *indices,
                                            const int32_t *row_adapter, const uint64_t *a_table,
                                            const uint64_t *b_table, const float *scale_table,
                                            mlg_bf16 *base_out, int32_t n_slots, int32_t k_in,
                                            int32_t max_rank, int32_t n_out, int32_t top_k,
                                            int32_t n_experts, int32_t n_adapters, void *stream) {
  return gather_multi(x, indices, row_adapter, a_table, b_table, scale_table, base_out, n_slots,
                      k_in, max_rank, n_out, top_k, n_experts, n_adapters, 0u, stream);
}

extern "C" mlg_status mlg_gather_bgmv_multi_ex(const mlg_bf16 *x, const int32_t *indices,
                                               const int32_t *row_adapter,
                                               const uint64_t *a_table, const uint64_t *b_table,
                                               const float *scale_table, mlg_bf16 *base_out,
                                               int32_t n_slots, int32_t k_in, int32_t max_rank,
                                               int32_t n_out, int32_t top_k, int32_t n_experts,
                                               int32_t n_adapters, uint32_t flags, void *stream) {
  return gather_multi(x, indices, row_adapter, a_table, b_table, scale_table, base_out, n_slots,
                      k_in, max_rank, n_out, top_k, n_experts, n_adapters, flags, stream);
}
