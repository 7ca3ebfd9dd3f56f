// pa_api.cu -- status strings, sizes and shared host helpers of the C ABI.

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdlib>
#include <cstring>

#include "pa_host.h"
#include "pagedkv.h"

namespace pa {

bool validating() {
  static const bool on = [] {
    const char* v = std::getenv("PA_VALIDATE");
    return v && v[0] && std::strcmp(v, "0") != 0;
  }();
  return on;
}

pa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

extern "C" int32_t pa_decode_num_splits(int32_t max_context, int32_t split_tokens) {
  if (split_tokens <= 0 || max_context <= 0) return 0;
  return (int32_t)(((long long)max_context + split_tokens - 1) / split_tokens);
}

extern "C" size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                            int32_t head_dim, int32_t max_splits) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_splits <= 0) return 0;
  const size_t rows = (size_t)num_seqs * num_q_heads * max_splits;
  const size_t out_bytes = (rows * head_dim * sizeof(float) + 255) & ~(size_t)255;
  return out_bytes + rows * sizeof(float);
}

extern "C" int64_t pa_kv_bytes_per_token(int32_t num_layers, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t bytes_per_value) {
  return 2ll * num_layers * num_kv_heads * head_dim * bytes_per_value;
}

extern "C" const char* pa_status_str(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
  }
  return "PA_ERR_UNKNOWN";
}

extern "C" const char* pa_version(void) { return "pagedkv 0.1.0 sm_103a"; }
