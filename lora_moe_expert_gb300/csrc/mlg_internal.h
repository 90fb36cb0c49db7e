// mlg_internal.h -- declarations shared by the translation units of libmlg.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "mlg.h"

// Sorted rows per grouped-fold tile: the M of one tcgen05 MMA (cta_group::1).
#define MLG_M_TILE 128u

namespace mlg {

extern thread_local int32_t g_last_cuda_error;
mlg_status cuda_status(cudaError_t err);

// Device-side error word: kernels OR bits into it instead of trapping.  Read
// and cleared on the host by mlg_read_device_errors().
enum DeviceError : uint32_t {
  kErrWaitTimeout = 1u,   // an mbarrier wait ran past its time limit
  kErrTmemAlloc = 2u,     // tensor-memory allocation did not succeed
  kErrUnitDropped = 4u,   // a CTA was dealt more work units than it holds
};

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side validation shared by the fold entry points.
inline mlg_status check_shapes(int32_t k_in, int32_t max_rank, int32_t n_out) {
  if (k_in <= 0 || max_rank <= 0 || n_out <= 0) return MLG_ERR_INVALID_ARG;
  if (k_in % 8 != 0 || n_out % 8 != 0) return MLG_ERR_UNSUPPORTED;
  if (max_rank % 8 != 0 || max_rank > MLG_MAX_RANK) return MLG_ERR_UNSUPPORTED;
  return MLG_OK;
}

int sm_count();  // multiprocessors of the current device (cached per device)

// The resident-pair decode fold (mlg_decode.cu): eligibility and launch.
// n_cells is the table length; with n_adapters > 0 the tables hold
// n_adapters sets of e_model cells, slot-major, and a row's cell is
// row_adapter[token] * e_model + indices[row] (n_adapters == 0: the cell is
// indices[row] and the row map only gates).  A launch with n_adapters > 0
// takes the multi-cell form (decode_multi_eligible).
int gather_path_override();  // 0 auto, 1 resident-pair kernel, 2 cluster kernel
bool decode_fold_eligible(int32_t k_in, int32_t max_rank, int32_t n_out, int32_t n_cells);
bool decode_multi_eligible(int32_t k_in, int32_t max_rank, int32_t n_out, int32_t n_cells);
cudaError_t decode_fold_launch(const uint16_t *x, const int32_t *indices,
                               const int32_t *row_adapter, const uint64_t *a_table,
                               const uint64_t *b_table, const float *scale_table,
                               uint16_t *base_out, int32_t n_slots, int32_t k_in,
                               int32_t max_rank, int32_t n_out, int32_t top_k,
                               int32_t n_cells, int32_t e_model, int32_t n_adapters,
                               bool early, cudaStream_t stream);

}  // namespace mlg
