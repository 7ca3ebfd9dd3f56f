// pa_api.cu -- status strings, sizes and shared host helpers of the C ABI.

#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

pa_status prepare_kernel(const void* func, int threads, int smem_bytes, int* blocks_per_sm) {
  static std::mutex mu;
  // The dynamic shared-memory limit is one attribute per kernel and device:
  // it only ever grows here (to the largest size launched so far), so a
  // smaller launch in between never leaves it below a size cached earlier.
  static std::map<std::pair<const void*, int>, int> limit;
  static std::map<std::tuple<const void*, int, int, int>, int> occupancy;  // -> blocks per SM
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  int& lim = limit[std::make_pair(func, dev)];
  if (smem_bytes > lim) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
        cudaSuccess) {
      cudaGetLastError();  // reported here, not by a later launch check
      return PA_ERR_CUDA;
    }
    lim = smem_bytes;
  }
  const auto key = std::make_tuple(func, dev, threads, smem_bytes);
  auto it = occupancy.find(key);
  if (it == occupancy.end()) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, threads, smem_bytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    it = occupancy.emplace(key, per_sm < 1 ? 1 : per_sm).first;
  }
  if (blocks_per_sm) *blocks_per_sm = it->second;
  return PA_OK;
}

bool make_cache_map(CUtensorMap* map, const void* base, int hkv, int d, long long rows,
                    int box_rows, int elem_bytes) {
  auto enc = tensor_map_encoder();
  if (!enc || (elem_bytes != 1 && elem_bytes != 2)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)hkv * d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hkv * d * elem_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  // L2 fetches grow to 256 B only where one (token, KV head) row spans 256 B;
  // a 128-byte row (e4m3 at head_dim 128, bf16 at 64) would drag in its
  // neighbour head's row, which another block reads at another time.
  const CUtensorMapL2promotion promo = (long long)d * elem_bytes >= 256
                                           ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                           : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
  if ((long long)d * elem_bytes == 256 && box_rows >= 16) {
    // 3-D view (64 columns, rows, 128-byte column halves of all heads): one
    // box {64, box_rows, 2} lands both halves of a (token range, head) tile in
    // the [half][row] shared-memory layout the 2-D boxes produce, so a tile
    // costs one TMA instruction per K or V instead of two. (The halves' stride,
    // 128 B, is below the rows' stride.)
    cuuint64_t dims3[3] = {(cuuint64_t)(128 / elem_bytes), (cuuint64_t)rows,
                           (cuuint64_t)hkv * d * elem_bytes / 128};
    cuuint64_t strides3[2] = {(cuuint64_t)hkv * d * elem_bytes, 128};
    cuuint32_t box3[3] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows, 2};
    cuuint32_t estr3[3] = {1, 1, 1};
    CUresult r = enc(map, dt, 3, const_cast<void*>(base), dims3, strides3, box3, estr3,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  }
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

pa_status check_tables(const int32_t* block_tables, int mb, const int32_t* context_lens, int B,
                       int num_blocks, int bs, int split_tokens, int max_splits,
                       cudaStream_t stream) {
  std::vector<int32_t> lens(B), tab((size_t)B * mb);
  if (cudaMemcpyAsync(lens.data(), context_lens, sizeof(int32_t) * B, cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess ||
      cudaMemcpyAsync(tab.data(), block_tables, sizeof(int32_t) * tab.size(),
                      cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return PA_ERR_CUDA;
  for (int b = 0; b < B; ++b) {
    const long long ctx = lens[b];
    if (ctx < 0 || ctx > (long long)mb * bs) return PA_ERR_INVALID_ARG;
    if (split_tokens > 0 && ctx > (long long)max_splits * split_tokens) return PA_ERR_INVALID_ARG;
    const long long nblk = (ctx + bs - 1) / bs;
    for (long long i = 0; i < nblk; ++i) {
      const int32_t v = tab[(size_t)b * mb + i];
      if (v < 0 || v >= num_blocks) return PA_ERR_INVALID_ARG;
    }
  }
  return PA_OK;
}

pa_status check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, float scale, const void* out) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(block_size) || block_size > 256) return PA_ERR_UNSUPPORTED;
  if ((long long)num_blocks * block_size >= (1ll << 31)) return PA_ERR_INVALID_ARG;
  if ((long long)max_blocks_per_seq * block_size >= (1ll << 31)) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (!(scale == scale)) return PA_ERR_INVALID_ARG;
  return PA_OK;
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

extern "C" pa_status pa_last_device_error(int32_t* code) {
  if (!code) return PA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  const unsigned int v =
      pa::take_decode_errors() | pa::take_balanced_errors() | pa::take_multi_errors();
  *code = (int32_t)v;
  return v ? PA_ERR_DEVICE : PA_OK;
}

extern "C" const char* pa_status_str(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
    case PA_ERR_CAPACITY: return "PA_ERR_CAPACITY";
  }
  return "PA_ERR_UNKNOWN";
}

extern "C" const char* pa_version(void) { return "pagedkv 0.1.0 sm_103a"; }
