// pa_reduce.cu -- log-sum-exp merge of context-split partials (sm_103a).
//
// Each split of a long context leaves a normalised partial output O_s and the
// natural-log log-sum-exp lse_s of its scaled logits. The exact whole-context
// result is sum_s w_s O_s / sum_s w_s with w_s = exp(lse_s - max_s lse_s):
// the same rescaling by exp(old max - new max) that the streaming softmax of
// "Text Generation Inference: Hugging Face's production-grade LLM inference
// server" (section "Under the Hood: Flash Attention") applies tile by tile,
// here applied once per split.
//
// One warp per (sequence, query head): lanes own D/32 contiguous columns, so
// every partial row is read as one coalesced 512-byte (D = 128) transaction.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pa_host.h"
#include "pagedkv.h"

namespace pa {
namespace {

template <int D>
__global__ void __launch_bounds__(128)
    splitk_reduce_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                         const int32_t* __restrict__ context_lens, int num_rows, int num_q_heads,
                         int split_tokens, int max_splits, __nv_bfloat16* __restrict__ out) {
  constexpr int V = D / 32;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);  // b * Hq + h
  const int lane = threadIdx.x & 31;
  if (row >= num_rows) return;
  const int b = row / num_q_heads;
  int ctx = context_lens[b];
  ctx = ctx < 0 ? 0 : ctx;
  const int n = min((int)(((long long)ctx + split_tokens - 1) / split_tokens), max_splits);
  const size_t base = (size_t)row * max_splits;

  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, part_lse[base + s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float acc[V];
#pragma unroll
  for (int j = 0; j < V; ++j) acc[j] = 0.f;
  float W = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int s = 0; s < n; ++s) {
      const float lse = part_lse[base + s];
      const float w = expf(lse - M);  // an empty split (lse = -inf) weighs 0
      const float* src = part_out + (base + s) * D + lane * V;
      float v[V];
      if constexpr (V == 4) {
        const float4 t = *reinterpret_cast<const float4*>(src);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(src);
        v[0] = t.x; v[1] = t.y;
      }
      if (w > 0.f) {
        W += w;
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] += w * v[j];
      }
    }
  }
  __nv_bfloat16 r[V];
#pragma unroll
  for (int j = 0; j < V; ++j) r[j] = __float2bfloat16_rn(W > 0.f ? acc[j] / W : 0.f);
  __nv_bfloat16* dst = out + (size_t)row * D + lane * V;
  if constexpr (V == 4)
    *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(r);
  else
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(r);
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_splitk_reduce(const float* part_out, const float* part_lse,
                                             const int32_t* context_lens, int32_t num_seqs,
                                             int32_t num_q_heads, int32_t head_dim,
                                             int32_t split_tokens, int32_t max_splits, void* out,
                                             void* stream) {
  using namespace pa;
  if (num_seqs < 0 || num_q_heads <= 0 || split_tokens <= 0 || max_splits <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!part_out || !part_lse || !context_lens || !out) return PA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!aligned16(part_out) || !aligned16(out)) return PA_ERR_INVALID_ARG;
  const long long rows = (long long)num_seqs * num_q_heads;
  if (rows > (1ll << 31) - 1) return PA_ERR_INVALID_ARG;
  const int grid = (int)((rows + 3) / 4);
  cudaStream_t st = as_stream(stream);
  if (head_dim == 128)
    splitk_reduce_kernel<128><<<grid, 128, 0, st>>>(part_out, part_lse, context_lens, (int)rows,
                                                    num_q_heads, split_tokens, max_splits,
                                                    static_cast<__nv_bfloat16*>(out));
  else
    splitk_reduce_kernel<64><<<grid, 128, 0, st>>>(part_out, part_lse, context_lens, (int)rows,
                                                   num_q_heads, split_tokens, max_splits,
                                                   static_cast<__nv_bfloat16*>(out));
  return launch_status();
}
