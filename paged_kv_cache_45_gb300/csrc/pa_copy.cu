// pa_copy.cu -- copy-on-write of whole pool blocks (sm_103a).
//
// "Text Generation Inference: Hugging Face's production-grade LLM inference
// server", section "Under the Hood: PagedAttention" (prefix sharing): before
// a sequence writes into a block it shares, the block is copied to a fresh
// one. The prefix cache (pa_prefix.cpp) decides the (src, dst) pairs; this is
// the device side: a byte copy of block src to block dst in both caches.
//
// HBM-bound streaming copy: each thread issues four 16-byte loads (strided by
// the block size so a warp's accesses stay coalesced) before its four stores,
// so a 256-thread block keeps 16 KB in flight. Ids outside the pool are
// skipped.

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
                       long long chunks_per_block, long long total, int num_blocks) {
  const long long base = (long long)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x;
  uint4 v[kCopyUnroll];
  uint4* to[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    to[u] = nullptr;
    const long long g = base + (long long)u * kCopyThreads;
    if (g >= total) continue;
    const long long per_copy = 2 * chunks_per_block;
    const long long c = g / per_copy;
    const long long r = g - c * per_copy;
    const int which = r >= chunks_per_block;  // 0: K, 1: V
    const long long off = r - which * chunks_per_block;
    const int s = __ldg(src + c), d = __ldg(dst + c);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) continue;
    uint4* pool = which ? v_cache : k_cache;
    v[u] = pool[(long long)s * chunks_per_block + off];
    to[u] = pool + (long long)d * chunks_per_block + off;
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u)
    if (to[u]) *to[u] = v[u];
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
  const long long total = 2 * cpb * (long long)num_copies;
  const long long per_cta = (long long)kCopyThreads * kCopyUnroll;
  const long long grid = (total + per_cta - 1) / per_cta;
  if (grid > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  copy_blocks_kernel<<<(unsigned)grid, kCopyThreads, 0, st>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src, dst, cpb, total,
      num_blocks);
  return launch_status();
}
