// pa_append.cu -- scatter new K/V rows into their paged slots (sm_103a).
//
// A new token's K and V vectors for every KV head go into the sequence's
// current block, at the slot the host allocator picked ("Text Generation
// Inference: Hugging Face's production-grade LLM inference server", section
// "Under the Hood: PagedAttention"). The pool row of slot s is one contiguous
// run of num_kv_heads*head_dim bf16 values, so each thread moves one 16-byte
// chunk of K and the same chunk of V: reads are fully coalesced over the
// token-major input, writes are coalesced within each destination row. Bytes
// are copied unchanged (bit-exact). Slots < 0 (padding) and slots outside the
// pool are skipped, never written.

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pagedkv.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     const int64_t* __restrict__ slot_mapping, long long total_chunks,
                     int chunks_per_token, long long num_slots, uint4* __restrict__ k_cache,
                     uint4* __restrict__ v_cache) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total_chunks;
       i += stride) {
    const long long t = i / chunks_per_token;
    const int c = (int)(i - t * chunks_per_token);
    const long long slot = slot_mapping[t];
    if (slot < 0 || slot >= num_slots) continue;
    const uint4 kv = k_new[i];
    const uint4 vv = v_new[i];
    const long long dst = slot * chunks_per_token + c;
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

// FP8 pool: each thread quantizes 8 values (one 16-byte bf16 chunk) of K and
// the same 8 of V to e4m3 codes, value / scale of its KV head computed in fp32
// (round to nearest) and rounded to the nearest even e4m3 code, saturating at
// +-448; the 8 codes go out as one 8-byte store.
__global__ void __launch_bounds__(256)
    kv_append_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                         const int64_t* __restrict__ slot_mapping, long long total_chunks,
                         int chunks_per_token, int chunks_per_head, long long num_slots,
                         const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                         uint2* __restrict__ k_cache, uint2* __restrict__ v_cache) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total_chunks;
       i += stride) {
    const long long t = i / chunks_per_token;
    const int c = (int)(i - t * chunks_per_token);
    const long long slot = slot_mapping[t];
    if (slot < 0 || slot >= num_slots) continue;
    const int h = c / chunks_per_head;
    const float ks = k_scale[h], vs = v_scale[h];
    const uint4 kv = k_new[i], vv = v_new[i];
    auto q8 = [](const uint4& v, float sc) {
      uint2 r;
      r.x = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(v.x), sc), __fdiv_rn(bf16_hi(v.x), sc)) |
            (f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(v.y), sc), __fdiv_rn(bf16_hi(v.y), sc)) << 16);
      r.y = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(v.z), sc), __fdiv_rn(bf16_hi(v.z), sc)) |
            (f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(v.w), sc), __fdiv_rn(bf16_hi(v.w), sc)) << 16);
      return r;
    };
    const long long dst = slot * chunks_per_token + c;
    k_cache[dst] = q8(kv, ks);
    v_cache[dst] = q8(vv, vs);
  }
}

pa_status check_slots(const int64_t* slot_mapping, int T, long long num_slots, cudaStream_t st) {
  std::vector<int64_t> s(T);
  if (cudaMemcpyAsync(s.data(), slot_mapping, sizeof(int64_t) * T, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return PA_ERR_CUDA;
  for (int t = 0; t < T; ++t)
    if (s[t] >= num_slots) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_kv_append(const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                                  void* v_cache, int32_t num_blocks, int32_t block_size,
                                  int32_t num_kv_heads, int32_t head_dim, void* stream) {
  using namespace pa;
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (head_dim % 8) return PA_ERR_UNSUPPORTED;  // rows move in 16-byte chunks
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  const long long num_slots = (long long)num_blocks * block_size;
  if (validating()) {
    pa_status s = check_slots(slot_mapping, num_tokens, num_slots, st);
    if (s != PA_OK) return s;
  }
  const int chunks_per_token = num_kv_heads * head_dim / 8;
  const long long total = (long long)num_tokens * chunks_per_token;
  int sms = 148;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (total + 255) / 256;
  const long long cap = (long long)sms * 8;
  const int grid = (int)(want < cap ? want : cap);
  kv_append_kernel<<<grid, 256, 0, st>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, total,
      chunks_per_token, num_slots, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache));
  return launch_status();
}

extern "C" pa_status pa_kv_append_fp8(const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping, int32_t num_tokens,
                                      void* k_cache, void* v_cache, const float* k_scale,
                                      const float* v_scale, int32_t num_blocks,
                                      int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                      void* stream) {
  using namespace pa;
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PA_ERR_INVALID_ARG;
  if (head_dim % 8) return PA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  const long long num_slots = (long long)num_blocks * block_size;
  if (validating()) {
    pa_status s = check_slots(slot_mapping, num_tokens, num_slots, st);
    if (s != PA_OK) return s;
  }
  const int chunks_per_token = num_kv_heads * head_dim / 8;
  const long long total = (long long)num_tokens * chunks_per_token;
  int sms = 148, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (total + 255) / 256;
  const long long cap = (long long)sms * 8;
  const int grid = (int)(want < cap ? want : cap);
  kv_append_fp8_kernel<<<grid, 256, 0, st>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, total,
      chunks_per_token, head_dim / 8, num_slots, k_scale, v_scale, static_cast<uint2*>(k_cache),
      static_cast<uint2*>(v_cache));
  return launch_status();
}
