// mlg_gather.cu -- decode-side MoE expert LoRA fold (moe_lora_gather_bgmv of
// the moe_lora_grouped module index): for every flat (token, slot) row,
//     base_out[row] += scale_e * (x[row / top_k] @ A_e^T) @ B_e^T,  e = indices[row],
// skipping rows whose token has a negative row-map entry (moe_row_adapter.rs,
// build_moe_row_adapter_decode) and experts that fold nothing.
//
// GB300 design (not the pages' two-launch shrink/expand layout):
//  * one thread-block cluster of CS CTAs per expert: the expert's A_e and B_e
//    leave HBM exactly once, split over the cluster -- rank q holds the k
//    columns [q*ks, (q+1)*ks) of A_e and the n rows [q*ns, (q+1)*ns) of B_e;
//  * every load and store is a TMA bulk copy (cp.async.bulk) issued by one
//    warp, completion counted on an mbarrier, so all of a CTA's bytes are in
//    flight at once; the weight copies are issued before the row scan;
//  * rows of the expert are found on the device by a scan of `indices`
//    (ordered ballot compaction, identical in every CTA of the cluster);
//  * shrink h = x A_e^T and expand h B_e^T run on the tensor cores
//    (mma.sync m16n8k16 bf16 -> fp32; decode M is 1..32 rows, below the
//    smallest tcgen05 M), h stays fp32: each CTA's partial h over its k slice
//    is summed across the cluster through distributed shared memory in a
//    fixed rank order, and the expand multiplies B_e by h = hi + lo (two bf16
//    halves, so h is carried to ~2^-17 relative precision);
//  * epilogue: out = RNE_bf16(base + scale * (h B^T)), written in place in
//    shared memory and bulk-stored; rows that do not fold are never loaded
//    or stored.
#include <cuda_bf16.h>

#include <mutex>

#include "mlg_internal.h"
#include "mlg_ptx.cuh"

namespace mlg {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRowGroup = 32;  // most rows of one expert folded per pass

static __device__ uint32_t g_gather_errors;

struct GatherParams {
  const uint16_t *x;
  const int32_t *indices;
  const int32_t *row_adapter;
  const uint64_t *a_table;
  const uint64_t *b_table;
  const float *scale_table;
  uint16_t *base_out;
  int32_t n_slots, k_in, rank, n_out, top_k, n_experts;
  int32_t ks, ns;         // k columns / n rows per cluster rank
  int32_t rg;             // rows per pass (16 or 32)
  uint32_t stride_a;      // bytes per A_e / x row in shared memory
  uint32_t stride_base;   // bytes per base row in shared memory
  uint32_t off_a, off_x, off_b, off_base, off_p, off_hloc, off_h, smem_bytes;
};

__device__ __forceinline__ void record_error(uint32_t bit) { atomicOr(&g_gather_errors, bit); }

constexpr int kScanPer = 8;                       // rows per thread per scan chunk
constexpr int kScanChunk = kScanPer * kThreads;   // 2048 rows

// Collect the rows [g0, g0 + rg) of the rows that fold through expert e, in
// the order (chunk, i, warp, lane) -- the same in every CTA of a cluster --
// and return the total number of such rows.  Block-uniform.  Each chunk's
// index and row-map loads are all issued before any is used (one memory
// round trip per chunk), and a chunk costs two block barriers.
__device__ int scan_rows(const GatherParams &p, int e, int g0, int *s_rows,
                         int (*s_cnt)[kWarps]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int count = 0;
  for (int base = 0; base < p.n_slots; base += kScanChunk) {
    int idx[kScanPer], ra[kScanPer];
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      const int row = base + i * kThreads + tid;
      idx[i] = -1;
      ra[i] = -1;
      if (row < p.n_slots) {
        idx[i] = __ldg(p.indices + row);
        ra[i] = __ldg(p.row_adapter + row / p.top_k);
      }
    }
    unsigned mask[kScanPer];
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      mask[i] = __ballot_sync(0xffffffffu, idx[i] == e && ra[i] >= 0);
      if (lane == 0) s_cnt[i][warp] = __popc(mask[i]);
    }
    __syncthreads();
    int total = 0;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int v = s_cnt[i][w];
        total += v;
      }
    }
    int run = count;
#pragma unroll
    for (int i = 0; i < kScanPer; ++i) {
      int mine = run;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mine += (w < warp) ? s_cnt[i][w] : 0;
      const int rank = mine + __popc(mask[i] & ((1u << lane) - 1u));
      if (((mask[i] >> lane) & 1u) && rank >= g0 && rank < g0 + p.rg)
        s_rows[rank - g0] = base + i * kThreads + tid;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) run += s_cnt[i][w];
    }
    count += total;
    __syncthreads();
  }
  return count;
}

template <int RP>  // max_rank rounded up to a multiple of 16
__global__ void __launch_bounds__(kThreads, 2) gather_fold_kernel(const GatherParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2];  // 0: weights, 1: rows
  __shared__ int s_rows[kMaxRowGroup];
  __shared__ int s_cnt[kScanPer][kWarps];

  constexpr int MT = RP / 16;   // rank m-tiles of the shrink
  constexpr int KST = RP / 16;  // k-steps of the expand
  constexpr int HS = RP + 4;    // fp32 row stride of the h buffers

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t q = cluster_ctarank();
  const uint32_t cs = gridDim.x / ncluster_x();

  const int k0 = static_cast<int>(q) * p.ks;
  const int ksv = max(0, min(p.ks, p.k_in - k0));
  const int n0 = static_cast<int>(q) * p.ns;
  const int nsv = max(0, min(p.ns, p.n_out - n0));
  const int r = p.rank;
  const int q4 = r / 4;  // rank columns held by each MMA thread-column c

  uint8_t *sA = smem + p.off_a;
  uint8_t *sX = smem + p.off_x;
  const uint8_t *sB = smem + p.off_b;
  uint8_t *sBase = smem + p.off_base;
  float *sP = reinterpret_cast<float *>(smem + p.off_p);
  float *sHloc = reinterpret_cast<float *>(smem + p.off_hloc);
  float *sH = reinterpret_cast<float *>(smem + p.off_h);

  // A_e rows >= rank and the k tail of the A / x rows (up to the next 32) are
  // read by the MMAs but never written by a copy: zero them once.
  if (r < RP || (ksv & 31) != 0) {
    for (uint32_t i = tid * 16; i < p.off_b; i += kThreads * 16)
      *reinterpret_cast<uint4 *>(smem + i) = make_uint4(0, 0, 0, 0);
  }
  const uint32_t bar_w = smem_addr(&bars[0]), bar_x = smem_addr(&bars[1]);
  if (tid == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_x, 1);
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t ph_w = 0, ph_x = 0;
  bool bad = false;

  for (int e = static_cast<int>(cluster_id_x()); e < p.n_experts;
       e += static_cast<int>(ncluster_x())) {
    // Table loads first; the row scan's loads are issued before they are
    // needed, so both memory round trips overlap.
    const uint64_t a_addr = __ldg(reinterpret_cast<const unsigned long long *>(p.a_table) + e);
    const uint64_t b_addr = __ldg(reinterpret_cast<const unsigned long long *>(p.b_table) + e);
    const float scale = __ldg(p.scale_table + e);
    fence_proxy_async_smem();  // earlier generic accesses before new async writes
    int total = scan_rows(p, e, 0, s_rows, s_cnt);
    if (total == 0 || a_addr == 0 || b_addr == 0 || ((a_addr | b_addr) & 15u) != 0)
      continue;  // no folding row, or the expert folds nothing (uniform in the cluster)

    // Weights: A_e k slice (one bulk copy per rank row), B_e n slice (one copy).
    if (warp == 0 && !bad) {
      const uint32_t bytes = (ksv > 0 ? r * ksv * 2u : 0u) + (nsv > 0 ? nsv * r * 2u : 0u);
      if (lane == 0) mbar_arrive_expect_tx(bar_w, bytes);
      __syncwarp();
      const uint8_t *A = reinterpret_cast<const uint8_t *>(a_addr);
      if (ksv > 0)
        for (int j = lane; j < r; j += 32)
          bulk_g2s(smem_addr(sA + j * p.stride_a), A + (static_cast<size_t>(j) * p.k_in + k0) * 2,
                   ksv * 2u, bar_w);
      if (nsv > 0 && lane == 31)
        bulk_g2s(smem_addr(const_cast<uint8_t *>(sB)),
                 reinterpret_cast<const uint8_t *>(b_addr) + static_cast<size_t>(n0) * r * 2,
                 nsv * r * 2u, bar_w);
    }
    bool have_weights = false;

    for (int g0 = 0; g0 < total; g0 += p.rg) {
      if (g0 > 0) scan_rows(p, e, g0, s_rows, s_cnt);
      const int n_g = min(p.rg, total - g0);

      // Rows of this group: x slices and base slices.
      if (warp == 0 && !bad) {
        bulk_wait_read_all();  // earlier bulk stores of sBase have read it
        const uint32_t bytes = n_g * ((ksv > 0 ? ksv * 2u : 0u) + (nsv > 0 ? nsv * 2u : 0u));
        if (lane == 0) mbar_arrive_expect_tx(bar_x, bytes);
        __syncwarp();
        if (lane < n_g) {
          const int row = s_rows[lane];
          const int t = row / p.top_k;
          if (ksv > 0)
            bulk_g2s(smem_addr(sX + lane * p.stride_a),
                     p.x + static_cast<size_t>(t) * p.k_in + k0, ksv * 2u, bar_x);
          if (nsv > 0)
            bulk_g2s(smem_addr(sBase + lane * p.stride_base),
                     p.base_out + static_cast<size_t>(row) * p.n_out + n0, nsv * 2u, bar_x);
        }
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
      if (!bad && my_units[0] >= 0) {
        const int kb_lo = kq * kblocks / ksplit, kb_hi = (kq + 1) * kblocks / ksplit;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          const uint32_t kbyte = (kb * 32 + 8 * c) * 2;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int u = my_units[i];
            if (u < 0) continue;
            const int mt = u % MT, nt = u / MT;
            const uint4 pa = *reinterpret_cast<const uint4 *>(sA + (mt * 16 + g) * p.stride_a + kbyte);
            const uint4 qa =
                *reinterpret_cast<const uint4 *>(sA + (mt * 16 + g + 8) * p.stride_a + kbyte);
            const uint4 sx = *reinterpret_cast<const uint4 *>(sX + (nt * 8 + g) * p.stride_a + kbyte);
            mma_bf16_16816(acc[i], pa.x, qa.x, pa.y, qa.y, sx.x, sx.y);
            mma_bf16_16816(acc[i], pa.z, qa.z, pa.w, qa.w, sx.z, sx.w);
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
          float s = 0.f;
          for (int kk = 0; kk < ksplit; ++kk) s += sP[kk * (ntr * 8 * HS) + idx];
          sHloc[idx] = s;
        }
      }
      // ---- h = sum over the cluster's k slices (distributed shared memory) --
      cluster_sync();
      {
        const uint32_t local = smem_addr(sHloc);
        const int n4 = ntr * 8 * HS / 4;
        for (int i4 = tid; i4 < n4; i4 += kThreads) {
          float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
          for (uint32_t rk = 0; rk < cs; ++rk) {
            const float4 v = ld_dsmem_f4(map_to_rank(local + i4 * 16, rk));
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
          }
          reinterpret_cast<float4 *>(sH)[i4] = s;
        }
      }
      cluster_sync();  // peers are done reading sHloc; sH is complete

      // ---- expand + epilogue over this CTA's n slice ----------------------
      // MMA M = rows, N = n, K = rank; A = h split into bf16 hi and lo halves.
      const int mte = (n_g + 15) / 16;
      const int ntn = nsv / 8;
      if (!bad) {
        uint32_t ah[2][KST][4], al[2][KST][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
          for (int st = 0; st < KST; ++st) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
              for (int hr = 0; hr < 2; ++hr) {
                const int slot = st * 4 + half * 2;
                const int row = mt * 16 + g + hr * 8;
                float v0 = 0.f, v1 = 0.f;
                if (slot < q4 && mt < mte) {
                  v0 = sH[row * HS + c * q4 + slot];
                  v1 = sH[row * HS + c * q4 + slot + 1];
                }
                float h0, l0, h1, l1;
                split_hi_lo(v0, h0, l0);
                split_hi_lo(v1, h1, l1);
                ah[mt][st][half * 2 + hr] = pack_bf16x2(h0, h1);
                al[mt][st][half * 2 + hr] = pack_bf16x2(l0, l1);
              }
            }
          }
        }
        for (int nt = warp; nt < ntn; nt += kWarps) {
          const int nl = nt * 8 + g;  // B_e row within the slice
          const uint32_t *brow = reinterpret_cast<const uint32_t *>(sB + (nl * r + c * q4) * 2);
          uint32_t b[KST][2];
#pragma unroll
          for (int st = 0; st < KST; ++st) {
            b[st][0] = (st * 4 < q4) ? brow[st * 2] : 0u;
            b[st][1] = (st * 4 + 2 < q4) ? brow[st * 2 + 1] : 0u;
          }
          float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            if (mt >= mte) continue;
#pragma unroll
            for (int st = 0; st < KST; ++st) {
              mma_bf16_16816(d[mt], ah[mt][st][0], ah[mt][st][1], ah[mt][st][2], ah[mt][st][3],
                             b[st][0], b[st][1]);
              mma_bf16_16816(d[mt], al[mt][st][0], al[mt][st][1], al[mt][st][2], al[mt][st][3],
                             b[st][0], b[st][1]);
            }
          }
          const int col = nt * 8 + 2 * c;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int row = mt * 16 + g + hr * 8;
              if (mt >= mte || row >= n_g) continue;
              uint32_t *w = reinterpret_cast<uint32_t *>(sBase + row * p.stride_base + col * 2);
              const uint32_t bw = *w;
              const float o0 = fmaf(scale, d[mt][hr * 2 + 0], bf16lo_to_f32(bw));
              const float o1 = fmaf(scale, d[mt][hr * 2 + 1], bf16hi_to_f32(bw));
              *w = pack_bf16x2(o0, o1);
            }
          }
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (warp == 0 && !bad && nsv > 0 && lane < n_g) {
        const int row = s_rows[lane];
        bulk_s2g(p.base_out + static_cast<size_t>(row) * p.n_out + n0,
                 smem_addr(sBase + lane * p.stride_base), nsv * 2u);
        bulk_commit();
      }
    }
  }
  if (warp == 0) bulk_wait_all();
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
}

struct Plan {
  int cs, ks, ns, rp;
  GatherParams p;
};

uint32_t round_up(uint32_t v, uint32_t m) { return (v + m - 1) / m * m; }

// Shared-memory layout for a cluster size; returns total bytes.
uint32_t layout(GatherParams &p, int cs, int rp) {
  p.ks = static_cast<int>(round_up((p.k_in + cs - 1) / cs, 32));
  p.ns = static_cast<int>(round_up((p.n_out + cs - 1) / cs, 8));
  uint32_t sa = p.ks * 2;
  if (sa % 128 == 0) sa += 64;  // 16-byte MMA operand loads conflict-free
  p.stride_a = sa;
  uint32_t sb = p.ns * 2;
  sb += (16 + 128 - sb % 128) % 128;  // row stride = 16 (mod 128) bytes
  p.stride_base = sb;
  const uint32_t hbytes = p.rg * (rp + 4) * 4;
  // k-split partials: ksplit * ntr <= 8 / (rp / 16) slots of ntr * 8 rows -> <= 1280 floats
  const uint32_t pbytes = 1280 * 4 > hbytes ? 1280 * 4 : hbytes;
  uint32_t off = 0;
  p.off_a = off;
  off += round_up(rp * sa, 128);
  p.off_x = off;
  off += round_up(p.rg * sa, 128);
  p.off_b = off;
  off += round_up(p.ns * p.rank * 2, 128);
  p.off_base = off;
  off += round_up(p.rg * sb, 128);
  p.off_p = off;
  off += round_up(pbytes, 128);
  p.off_hloc = off;
  off += round_up(hbytes, 128);
  p.off_h = off;
  off += round_up(hbytes, 128);
  p.smem_bytes = off;
  return off;
}

int g_cluster_override = 0;
constexpr uint32_t kSmemLimit = 227 * 1024 - 2048;  // leaves room for static shared memory

template <int RP>
cudaError_t launch(const GatherParams &p, int cs, int clusters, cudaStream_t stream) {
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
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

}  // namespace mlg

extern "C" mlg_status mlg_gather_bgmv(const mlg_bf16 *x, const int32_t *indices,
                                      const int32_t *row_adapter, const uint64_t *a_table,
                                      const uint64_t *b_table, const float *scale_table,
                                      mlg_bf16 *base_out, int32_t n_slots, int32_t k_in,
                                      int32_t max_rank, int32_t n_out, int32_t top_k,
                                      int32_t n_experts, void *stream) {
  using namespace mlg;
  if (n_slots < 0 || n_experts < 0 || top_k < 1) return MLG_ERR_INVALID_ARG;
  const mlg_status shape = check_shapes(k_in, max_rank, n_out);
  if (shape != MLG_OK) return shape;
  if (n_slots == 0 || n_experts == 0) return MLG_OK;
  if (!x || !indices || !row_adapter || !a_table || !b_table || !scale_table || !base_out)
    return MLG_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(base_out)) return MLG_ERR_UNSUPPORTED;

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
  const int rp = static_cast<int>(round_up(max_rank, 16));
  // Rows per pass: decode batches spread ~n_slots / n_experts rows per expert.
  p.rg = (n_slots <= 8 * n_experts) ? 16 : 32;

  // Cluster size: the smallest power of two that bounds one CTA's share of an
  // expert's weights to ~48 KB, raised until the shared-memory layout fits.
  const double pair_bytes = 2.0 * max_rank * (static_cast<double>(k_in) + n_out);
  int cs = 1;
  while (cs < 8 && pair_bytes / cs > 48.0 * 1024) cs *= 2;
  if (g_cluster_override > 0) cs = g_cluster_override;
  while (layout(p, cs, rp) > kSmemLimit && cs < 8) cs *= 2;
  if (layout(p, cs, rp) > kSmemLimit) return MLG_ERR_UNSUPPORTED;

  // One cluster per expert, looping when the table is longer than the cap.
  const int max_clusters = (4 * sm_count()) / cs;
  const int clusters = n_experts < max_clusters ? n_experts : max_clusters;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  switch (rp) {
    case 16: err = launch<16>(p, cs, clusters, s); break;
    case 32: err = launch<32>(p, cs, clusters, s); break;
    case 48: err = launch<48>(p, cs, clusters, s); break;
    default: err = launch<64>(p, cs, clusters, s); break;
  }
  return cuda_status(err);
}
