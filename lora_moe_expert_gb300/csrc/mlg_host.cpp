// mlg_host.cpp -- host helpers of libmlg: routing, row maps, table packing,
// windows, uploads and status strings.  Pure CPU except the two uploads.
//
// Rules restated from the "metrale" documentation pages:
//   moe_row_adapter.rs: resolve_moe_lora_route, ensure_decode_route_servable,
//     build_moe_row_adapter_host, build_moe_row_adapter_decode;
//   moe_lora_grouped module index: pack_expert_tables, grouped_down_windows,
//     grouped_down_wc, gather_row_token, MLG_M_TILE.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <vector>

#include "mlg.h"
#include "mlg_internal.h"
#include "mlg_test.h"

namespace mlg {
thread_local int32_t g_last_cuda_error = 0;

mlg_status cuda_status(cudaError_t err) {
  if (err == cudaSuccess) return MLG_OK;
  g_last_cuda_error = static_cast<int32_t>(err);
  return MLG_ERR_CUDA;
}
}  // namespace mlg

extern "C" {

int32_t mlg_resolve_moe_lora_route(int32_t adapter_slot, int32_t active, int32_t has_moe_lora) {
  // Order of the tests as in the doc comment: no pool, base request, active, other.
  if (has_moe_lora == 0) return MLG_ROUTE_FOLD;
  if (adapter_slot < 0) return MLG_ROUTE_SKIP;
  return adapter_slot == active ? MLG_ROUTE_FOLD : MLG_ROUTE_REFUSE;
}

mlg_status mlg_ensure_decode_route_servable(int32_t route) {
  switch (route) {
    case MLG_ROUTE_FOLD:
    case MLG_ROUTE_SKIP:
      return MLG_OK;
    case MLG_ROUTE_REFUSE:
      return MLG_ERR_REFUSE;
    default:
      return MLG_ERR_INVALID_ARG;
  }
}

mlg_status mlg_build_moe_row_adapter_decode(const int32_t *adapter_slots, size_t n_slots,
                                            size_t padded_n, int32_t active,
                                            int32_t has_moe_lora, int32_t *out) {
  if (padded_n > 0 && out == nullptr) return MLG_ERR_INVALID_ARG;
  if (n_slots > 0 && adapter_slots == nullptr) return MLG_ERR_INVALID_ARG;
  const size_t real = n_slots < padded_n ? n_slots : padded_n;
  for (size_t i = 0; i < real; ++i) {
    const int32_t route = mlg_resolve_moe_lora_route(adapter_slots[i], active, has_moe_lora);
    out[i] = route == MLG_ROUTE_FOLD ? active : -1;
  }
  for (size_t i = real; i < padded_n; ++i) out[i] = -1;  // padding rows never fold
  return MLG_OK;
}

mlg_status mlg_build_moe_row_adapter_decode_multi(const int32_t *adapter_slots, size_t n_slots,
                                                  size_t padded_n, int32_t n_adapters,
                                                  int32_t has_moe_lora, int32_t *out) {
  if (padded_n > 0 && out == nullptr) return MLG_ERR_INVALID_ARG;
  if (n_slots > 0 && adapter_slots == nullptr) return MLG_ERR_INVALID_ARG;
  if (n_adapters < 1) return MLG_ERR_INVALID_ARG;
  const size_t real = n_slots < padded_n ? n_slots : padded_n;
  if (has_moe_lora) {  // a slot without a table set refuses the batch, nothing written
    for (size_t i = 0; i < real; ++i)
      if (adapter_slots[i] >= n_adapters) return MLG_ERR_REFUSE;
  }
  for (size_t i = 0; i < real; ++i)
    out[i] = (has_moe_lora && adapter_slots[i] >= 0) ? adapter_slots[i] : -1;
  for (size_t i = real; i < padded_n; ++i) out[i] = -1;  // padding rows never fold
  return MLG_OK;
}

// build_moe_row_adapter_host (moe_row_adapter.rs): the prefill map gives
// every token of stream b the stream's adapter slot.  The boundaries must be
// a valid prefix sum -- at least two of them, one slot per stream, starting
// at 0 and never decreasing (so none is negative) -- or the page returns
// None, here INVALID_ARG with nothing written.
mlg_status mlg_build_moe_row_adapter_host(const int32_t *cu_seqlens, size_t n_cu,
                                          const int32_t *adapter_slots, size_t n_slots,
                                          int32_t *out, size_t cap, size_t *total_out) {
  if (cu_seqlens == nullptr || adapter_slots == nullptr) return MLG_ERR_INVALID_ARG;
  if (n_cu < 2 || n_slots + 1 != n_cu || cu_seqlens[0] != 0) return MLG_ERR_INVALID_ARG;
  int32_t prev = 0;
  for (size_t i = 1; i < n_cu; prev = cu_seqlens[i++])
    if (cu_seqlens[i] < prev) return MLG_ERR_INVALID_ARG;
  const size_t tokens = static_cast<size_t>(prev);
  if (total_out != nullptr) *total_out = tokens;
  if (cap < tokens) return MLG_ERR_BUFFER_TOO_SMALL;
  if (tokens > 0 && out == nullptr) return MLG_ERR_INVALID_ARG;
  size_t stream = 0;  // the stream whose [cu[b], cu[b+1]) holds token t
  for (size_t t = 0; t < tokens; ++t) {
    while (static_cast<size_t>(cu_seqlens[stream + 1]) <= t) ++stream;
    out[t] = adapter_slots[stream];
  }
  return MLG_OK;
}

mlg_status mlg_pack_expert_tables(const mlg_expert_entry *entries, size_t n, uint64_t *a_out,
                                  uint64_t *b_out, float *scale_out, size_t cap,
                                  uint32_t *n_experts_out) {
  if (n == 0) return MLG_ERR_EMPTY;
  if (entries == nullptr) return MLG_ERR_INVALID_ARG;
  uint64_t max_id = 0;
  for (size_t i = 0; i < n; ++i) {
    if (entries[i].expert_id > max_id) max_id = entries[i].expert_id;
    if ((entries[i].a_addr & 15u) != 0 || (entries[i].b_addr & 15u) != 0)
      return MLG_ERR_UNSUPPORTED;
  }
  const uint64_t n_experts = max_id + 1;
  if (n_experts > 0x7fffffffull) return MLG_ERR_UNSUPPORTED;  // ids feed int32 kernel args
  if (n_experts_out != nullptr) *n_experts_out = static_cast<uint32_t>(n_experts);
  if (cap < n_experts) return MLG_ERR_BUFFER_TOO_SMALL;
  if (a_out == nullptr || b_out == nullptr || scale_out == nullptr) return MLG_ERR_INVALID_ARG;
  std::memset(a_out, 0, n_experts * sizeof(uint64_t));
  std::memset(b_out, 0, n_experts * sizeof(uint64_t));
  for (uint64_t e = 0; e < n_experts; ++e) scale_out[e] = 0.0f;
  for (size_t i = 0; i < n; ++i) {  // input order: a later duplicate overwrites
    const uint32_t id = entries[i].expert_id;
    a_out[id] = entries[i].a_addr;
    b_out[id] = entries[i].b_addr;
    scale_out[id] = entries[i].scale;
  }
  return MLG_OK;
}

mlg_status mlg_upload_expert_tables(const uint64_t *a_host, const uint64_t *b_host,
                                    const float *scale_host, uint32_t n_experts,
                                    uint64_t *a_dev, uint64_t *b_dev, float *scale_dev,
                                    void *stream) {
  if (n_experts == 0) return MLG_OK;
  if (!a_host || !b_host || !scale_host || !a_dev || !b_dev || !scale_dev)
    return MLG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mlg_status st = mlg::cuda_status(
      cudaMemcpyAsync(a_dev, a_host, n_experts * sizeof(uint64_t), cudaMemcpyHostToDevice, s));
  if (st != MLG_OK) return st;
  st = mlg::cuda_status(
      cudaMemcpyAsync(b_dev, b_host, n_experts * sizeof(uint64_t), cudaMemcpyHostToDevice, s));
  if (st != MLG_OK) return st;
  return mlg::cuda_status(cudaMemcpyAsync(scale_dev, scale_host, n_experts * sizeof(float),
                                          cudaMemcpyHostToDevice, s));
}

mlg_status mlg_upload_row_adapter(const int32_t *map_host, size_t n, int32_t *map_dev,
                                  void *stream) {
  if (n == 0) return MLG_OK;
  if (map_host == nullptr || map_dev == nullptr) return MLG_ERR_INVALID_ARG;
  return mlg::cuda_status(cudaMemcpyAsync(map_dev, map_host, n * sizeof(int32_t),
                                          cudaMemcpyHostToDevice,
                                          static_cast<cudaStream_t>(stream)));
}

mlg_status mlg_grouped_down_windows(uint32_t total_rows, uint32_t cap, mlg_window *out,
                                    size_t out_cap, size_t *n_windows) {
  if (cap == 0) return MLG_ERR_CAP_ZERO;
  const size_t count = (static_cast<uint64_t>(total_rows) + cap - 1) / cap;
  if (n_windows != nullptr) *n_windows = count;
  if (out_cap < count) return MLG_ERR_BUFFER_TOO_SMALL;
  if (count > 0 && out == nullptr) return MLG_ERR_INVALID_ARG;
  for (size_t i = 0; i < count; ++i) {
    const uint64_t start = static_cast<uint64_t>(i) * cap;
    const uint64_t end = start + cap < total_rows ? start + cap : total_rows;
    out[i].start = static_cast<uint32_t>(start);
    out[i].end = static_cast<uint32_t>(end);
  }
  return MLG_OK;
}

uint32_t mlg_m_tile(void) { return MLG_M_TILE; }

uint32_t mlg_grouped_down_wc(uint32_t row_offset, uint32_t row_end) {
  if (row_end <= row_offset) return 1;
  const uint64_t len = static_cast<uint64_t>(row_end - row_offset);
  const uint64_t wc = (len + MLG_M_TILE - 1) / MLG_M_TILE;
  return wc < 1 ? 1u : static_cast<uint32_t>(wc);
}

uint32_t mlg_gather_row_token(uint32_t row, uint32_t top_k) { return top_k ? row / top_k : 0u; }

const char *mlg_status_string(mlg_status status) {
  switch (status) {
    case MLG_OK: return "ok";
    case MLG_ERR_INVALID_ARG: return "invalid argument";
    case MLG_ERR_EMPTY: return "empty input";
    case MLG_ERR_CAP_ZERO: return "window cap is 0";
    case MLG_ERR_REFUSE:
      return "MoE LoRA: a sequence routes to a non-active adapter under the single-active fold; "
             "refusing rather than folding the active adapter into it (one adapter per batch)";
    case MLG_ERR_UNSUPPORTED: return "unsupported size or alignment";
    case MLG_ERR_BUFFER_TOO_SMALL: return "output buffer too small";
    case MLG_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int32_t mlg_last_cuda_error(void) { return mlg::g_last_cuda_error; }

int32_t mlg_version(void) { return 10000; }

}  // extern "C"

namespace mlg {
uint32_t gather_read_errors(bool clear);
uint32_t grouped_read_errors(bool clear);
uint32_t gemm_fold_read_errors(bool clear);
void gather_set_cluster_override(int cs);
void gather_set_nsplit_override(int ns2);
void grouped_set_ctas(int ctas);
uint32_t decode_read_errors(bool clear);
void gather_set_path_override(int path);
void gather_set_speculation(int mode);
}  // namespace mlg

extern "C" mlg_status mlg_read_device_errors(uint32_t *flags_out, int32_t clear) {
  if (flags_out == nullptr) return MLG_ERR_INVALID_ARG;
  cudaGetLastError();
  const uint32_t v = mlg::gather_read_errors(clear != 0) | mlg::grouped_read_errors(clear != 0) |
                     mlg::decode_read_errors(clear != 0) | mlg::gemm_fold_read_errors(clear != 0);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return mlg::cuda_status(err);
  *flags_out = v;
  return MLG_OK;
}

extern "C" mlg_status mlg_test_set_knob(int32_t knob, int32_t value) {
  switch (knob) {
    case MLG_TEST_GATHER_CLUSTER:
      if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8)
        return MLG_ERR_INVALID_ARG;
      mlg::gather_set_cluster_override(value);
      return MLG_OK;
    case MLG_TEST_GATHER_NSPLIT:
      if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8)
        return MLG_ERR_INVALID_ARG;
      mlg::gather_set_nsplit_override(value);
      return MLG_OK;
    case MLG_TEST_GATHER_PATH:
      if (value < 0 || value > 2) return MLG_ERR_INVALID_ARG;
      mlg::gather_set_path_override(value);
      return MLG_OK;
    case MLG_TEST_GATHER_SPECULATION:
      if (value < 0 || value > 2) return MLG_ERR_INVALID_ARG;
      mlg::gather_set_speculation(value);
      return MLG_OK;
    case MLG_TEST_GROUPED_CTAS:
      if (value < 0 || value > 65535) return MLG_ERR_INVALID_ARG;
      mlg::grouped_set_ctas(value);
      return MLG_OK;
    default:
      return MLG_ERR_INVALID_ARG;
  }
}
