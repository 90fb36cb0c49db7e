// mlg_tiles.cuh -- tile geometry of the grouped kernels (the grouped fold and
// the expert GEMM with the fold in its epilogue): expert-aligned tiles of
// expert-sorted rows that never cross a row window, and the 128-byte swizzle
// of their K-major operand tiles in shared memory.
//
// A params type P given to these templates has: offsets (int32 expert spans,
// or null for a single span [0, row_end)), row_offset, row_end, win (window
// length; windows start at row_offset + i * win) and tile_m (rows per tile).
#pragma once

#include <cstdint>

namespace mlg {

// Byte offset of 16-byte chunk `c` (of 8 per 128-byte row) of row `row` in a
// K-major 128-byte-swizzled tile whose 8-row atoms are 1024 bytes apart.
__device__ __forceinline__ uint32_t sw128(int row, int c) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4));
}

// The same for K-major tiles of RB-byte rows (RB = 32, 64 or 128) in the
// matching 32-, 64- or 128-byte swizzle: 8-row atoms of 8 * RB bytes, the
// 16-byte chunk index XORed with the address bits [7, ..) the swizzle mixes in.
template <int RB>
__device__ __forceinline__ uint32_t swk(int row, int c) {
  static_assert(RB == 32 || RB == 64 || RB == 128, "row bytes");
  const int x = RB == 128 ? (row & 7) : RB == 64 ? ((row >> 1) & 3) : ((row >> 2) & 1);
  return static_cast<uint32_t>((row >> 3) * (8 * RB) + (row & 7) * RB + ((c ^ x) << 4));
}

// tcgen05 shared-memory matrix descriptor of such a tile (K-major, version 1,
// start address in 16-byte units, SBO = one 8-row atom, layout code of the
// swizzle: 2 = 128-byte, 4 = 64-byte, 6 = 32-byte).
template <int RB>
__device__ __forceinline__ uint64_t umma_desc_k(uint32_t smem_byte_addr) {
  constexpr uint64_t kLayout = RB == 128 ? 2u : RB == 64 ? 4u : 6u;
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;                  // LBO (unused for swizzled K-major)
  d |= static_cast<uint64_t>((8u * RB) >> 4) << 32;      // SBO: 8 rows
  d |= static_cast<uint64_t>(1u) << 46;                  // descriptor version
  d |= kLayout << 61;
  return d;
}

// Bytes per B_e row in the grouped kernels' expand tiles: the rank columns in
// the narrowest swizzle that holds them (a rank of 48 takes 128-byte rows).
__host__ __device__ constexpr int b_row_bytes(int rp) { return rp <= 16 ? 32 : rp <= 32 ? 64 : 128; }

struct TileInfo {
  int e, r0, r1;
};

template <class P>
__device__ __forceinline__ int span_lo(const P &p, int e) {
  const int lo = p.offsets ? __ldg(p.offsets + e) : 0;
  return max(lo, p.row_offset);
}
template <class P>
__device__ __forceinline__ int span_hi(const P &p, int e) {
  const int hi = p.offsets ? __ldg(p.offsets + e + 1) : p.row_end;
  return min(hi, p.row_end);
}

// Tiles of one expert span [lo, hi): runs of <= tile_m rows that also never
// cross a window boundary (boundaries at row_offset + i * win).
template <class P>
__device__ __forceinline__ int span_tiles(const P &p, int lo, int hi) {
  if (hi <= lo) return 0;
  const int ro = p.row_offset, W = p.win, T = p.tile_m;
  const int w0 = (lo - ro) / W, w1 = (hi - 1 - ro) / W;
  if (w0 == w1) return (hi - lo + T - 1) / T;
  const int first = ro + (w0 + 1) * W - lo;
  const int last = hi - (ro + w1 * W);
  return (first + T - 1) / T + (w1 - w0 - 1) * ((W + T - 1) / T) + (last + T - 1) / T;
}

// Tile t: the expert owning it (tile_start is an exclusive prefix over
// experts) and its rows [r0, r1).
template <class P>
__device__ TileInfo tile_info(const P &p, const int *tile_start, int n_e, int t) {
  int lo = 0, hi = n_e - 1;  // largest e with tile_start[e] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int slo = span_lo(p, lo), shi = span_hi(p, lo);
  const int ro = p.row_offset, W = p.win, T = p.tile_m;
  int u = t - tile_start[lo];
  // walk the window pieces of the span (O(1) per piece type)
  const int w0 = (slo - ro) / W;
  int a = slo;
  int b = min(shi, ro + (w0 + 1) * W);
  int n = (b - a + T - 1) / T;
  if (u >= n) {
    u -= n;
    const int per = (W + T - 1) / T;  // tiles of one whole window
    const int w = w0 + 1 + u / per;
    u %= per;
    a = ro + w * W;
    b = min(shi, a + W);
  }
  ti.r0 = a + u * T;
  ti.r1 = min(ti.r0 + T, b);
  return ti;
}

// A LoRA pair folds when both table cells hold a non-zero, 16-byte-aligned
// address (a misaligned cell is treated as 0: the kernels never fault on
// table contents they can check).
__device__ __forceinline__ bool cells_fold(uint64_t a, uint64_t b) {
  return a != 0 && b != 0 && ((a | b) & 15u) == 0;
}

}  // namespace mlg
