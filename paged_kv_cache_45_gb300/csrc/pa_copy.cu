// pa_copy.cu -- copy-on-write of whole pool blocks (sm_103a).
//
// "Text Generation Inference: Hugging Face's production-grade LLM inference
// server", section "Under the Hood: PagedAttention" (prefix sharing): before
// a sequence writes into a block it shares, the block is copied to a fresh
// one. The prefix cache (pa_prefix.cpp) decides the (src, dst) pairs; this is
// the device side: a byte copy of block src to block dst in both caches.
//
// HBM-bound streaming copy. Thread block (x, y, z) copies 16 KB of copy z's
// block: of the K cache (y = 0) or the V cache (y = 1), chunks
// 1024 x .. 1024 x + 1023 of 16 bytes; each thread issues its four 16-byte
// loads (256 apart, so a warp's accesses stay coalesced) before its four
// stores. The pair (src, dst) is the same for the whole thread block; ids
// outside the pool are skipped. (Copies past the grid's z extent, 65535, are
// taken in turn by the same blocks.)

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "pa_host.h"
#include "pagedkv.h"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                       long long chunks_per_block, int num_copies, int num_blocks) {
  uint4* pool = blockIdx.y ? v_cache : k_cache;
  const long long off0 = (long long)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x;
  for (int c = blockIdx.z; c < num_copies; c += gridDim.z) {
    const int s = __ldg(src + c), d = __ldg(dst + c);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) continue;
    const uint4* from = pool + (long long)s * chunks_per_block;
    uint4* to = pool + (long long)d * chunks_per_block;
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const long long off = off0 + (long long)u * kCopyThreads;
      if (off < chunks_per_block) v[u] = from[off];
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const long long off = off0 + (long long)u * kCopyThreads;
      if (off < chunks_per_block) to[off] = v[u];
    }
  }
}

pa_status check_copies(const int32_t* src, const int32_t* dst, int n, int num_blocks,
                       cudaStream_t st) {
  std::vector<int32_t> s(n), d(n);
  if (cudaMemcpyAsync(s.data(), src, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(d.data(), dst, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return PA_ERR_CUDA;
  std::vector<char> is_src(num_blocks, 0), is_dst(num_blocks, 0);
  for (int i = 0; i < n; ++i) {
    if (s[i] < 0 || s[i] >= num_blocks || d[i] < 0 || d[i] >= num_blocks) return PA_ERR_INVALID_ARG;
    is_src[s[i]] = 1;
  }
  for (int i = 0; i < n; ++i) {
    if (is_dst[d[i]] || is_src[d[i]]) return PA_ERR_INVALID_ARG;
    is_dst[d[i]] = 1;
  }
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* src,
                                    const int32_t* dst, int32_t num_copies, int32_t num_blocks,
                                    int64_t block_bytes, void* stream) {
  using namespace pa;
  if (num_copies < 0 || num_blocks <= 0 || block_bytes <= 0 || block_bytes % 16)
    return PA_ERR_INVALID_ARG;
  if (num_copies == 0) return PA_OK;
  if (!k_cache || !v_cache || !src || !dst || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (validating()) {
    const pa_status s = check_copies(src, dst, num_copies, num_blocks, st);
    if (s != PA_OK) return s;
  }
  const long long cpb = block_bytes / 16;
  const long long per_cta = (long long)kCopyThreads * kCopyUnroll;
  const long long gx = (cpb + per_cta - 1) / per_cta;
  if (gx > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)gx, 2, (unsigned)(num_copies < 65535 ? num_copies : 65535));
  copy_blocks_kernel<<<grid, kCopyThreads, 0, st>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src, dst, cpb, num_copies,
      num_blocks);
  return launch_status();
}
