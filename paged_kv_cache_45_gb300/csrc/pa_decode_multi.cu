// pa_decode_multi.cu -- paged attention for several new query tokens per
// sequence under a causal mask (sm_103a).
//
// A chunk of a prompt ("Text Generation Inference: Hugging Face's
// production-grade LLM inference server", section "Advanced Pattern: Chunked
// Prefill (TGI v3)") or the drafted tokens plus one that a speculative step
// verifies in one pass ("How to Speed Up LLM Inference: KV Cache to
// Production Serving", section "Speculative decoding: more than one token per
// weight-read") give sequence b n_b query tokens, the last n_b positions of
// its context after the append. Token i (position ctx_b - n_b + i) attends to
// positions 0 .. ctx_b - n_b + i.
//
// One thread block per (KV head, context split, sequence), as in the decode
// kernel of pa_decode.cu, but the n = 8 side of the transposed MMA now holds
// (token, head) columns: column c = i * G + g of the unit's n_b * G query rows.
// Consumer warp w owns columns 8w .. 8w + 7 and folds EVERY K/V tile of the
// split into them (a tile's stage is released when all NC consumer warps have
// read it), so each K/V byte is still read from HBM once per block while the
// tensor-core work grows with n_b. Per-column causal limits mask the scores
// (attend_tile_causal); no merge between warps is needed. Outputs go through
// shared memory so that every row is written with coalesced stores: bf16 rows
// (one split) or fp32 partials + natural-log LSEs for pa_decode_splitk_reduce,
// whose per-row context lengths this kernel writes to row_lens.

#include <math.h>

#include <cstring>
#include <vector>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_tile.cuh"
#include "pagedkv.h"

namespace pa {
namespace {

__device__ unsigned int g_multi_error;

__device__ __forceinline__ void report(unsigned int bits) { atomicOr(&g_multi_error, bits); }

constexpr int kMaxColumnWarps = 8;  // up to 64 (token, head) columns per unit
constexpr int kMultiStages = 4;

struct MultiParams {
  const __nv_bfloat16* q;      // [R, Hq, D]
  const int32_t* q_start;      // [B + 1]
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_out;             // [R, Hq, S, D]
  float* part_lse;             // [R, Hq, S]
  int32_t* row_lens;           // [R], split mode
  __nv_bfloat16* out;          // [R, Hq, D]
  TileSrc src;
  int max_blocks;
  int num_q_heads;
  int group;
  int split_tokens;
  int max_splits;
  int max_q_len;
  float scale_log2;
};

template <int D>
struct MultiSmem {
  static constexpr int kStageBytes = TileGeom<D>::kStageBytes;
  static constexpr int kRingBytes = kMultiStages * kStageBytes;
  static constexpr int kOutBytes = kMaxColumnWarps * 8 * D * 4;  // aliases the ring
  static_assert(kRingBytes >= kOutBytes, "ring too small to stage the outputs");
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kFlagOff = kBarOff + 2 * kMultiStages * 8;
  static constexpr int kAlloc = kFlagOff + 16 + 1024;
};

// Column of element d of column row j in a warp's output buffer: XOR-swizzled
// in 8-float groups so the 4 column rows one store touches use 4 bank groups.
__device__ __forceinline__ int out_col(int j, int d) { return d ^ ((j >> 1) << 3); }

template <int D, bool kTma>
__global__ void __launch_bounds__((kMaxColumnWarps + 1) * 32, 2)
    multi_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const MultiParams p) {
  using L = MultiSmem<D>;
  using Gm = TileGeom<D>;
  constexpr int STAGES = kMultiStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kFlagOff);

  const int NC = (int)(blockDim.x >> 5) - 1;  // consumer warps (column groups)
  const int kvh = blockIdx.x;
  const int split = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  const int row0 = p.q_start[b];
  const int n = p.q_start[b + 1] - row0;  // new query tokens of the sequence
  int ctx = p.context_lens[b];
  const int cap = p.max_blocks << p.src.log2_bs;
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  if (n <= 0) return;
  if (n > p.max_q_len || n * G > NC * 8) {
    if (threadIdx.x == 0) report(kErrShape);
    return;
  }
  if (p.split_tokens > 0 && kvh == 0 && split == 0) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int len = ctx - n + i + 1;
      p.row_lens[row0 + i] = len > 0 ? len : 0;
    }
  }
  int t_begin = 0, t_end = ctx;
  if (p.split_tokens > 0) {
    t_begin = split * p.split_tokens;
    t_end = min(t_begin + p.split_tokens, ctx);
  }
  if (t_begin >= t_end) {
    if (p.split_tokens == 0) {  // no context at all: zero rows
      for (int i = threadIdx.x; i < n * G * (D / 8); i += blockDim.x) {
        const int c = i / (D / 8), c8 = i % (D / 8);
        __nv_bfloat16* dst =
            p.out + ((size_t)(row0 + c / G) * p.num_q_heads + kvh * G + c % G) * D + c8 * 8;
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }
  const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], kTma ? 1 : 32);
      mbar_init(&empty[s], NC);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t ring = smem_u32(smem);

  if (warp == NC) {
    // ------------------------------------------------------------ loader warp
    if (kTma && lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const int32_t* bt = p.block_tables + (size_t)b * p.max_blocks;
    const int n_seq_blocks = (ctx + p.src.block_size - 1) >> p.src.log2_bs;
    int tc_base = -(1 << 30);
    int tc_val = -1;
    int issued = 0;
    for (int i = 0; i < n_tiles; ++i) {
      if (__any_sync(0xffffffffu, *abort_flag)) break;
      const int stage = i % STAGES;
      if (i >= STAGES &&
          !__all_sync(0xffffffffu, mbar_wait(&empty[stage], ((i / STAGES) - 1) & 1))) {
        if (lane == 0) report(kErrWaitEmpty);
        *abort_flag = 1;
        break;
      }
      const int t0 = t_begin + i * kTile;
      const int blk_first = t0 >> p.src.log2_bs;
      const int blk_last = (t0 + kTile - 1) >> p.src.log2_bs;
      if (blk_first < tc_base || blk_last >= tc_base + 32) {  // warp-uniform refill
        tc_base = blk_first;
        const int idx = tc_base + lane;
        tc_val = idx < n_seq_blocks ? bt[idx] : -1;
      }
      issue_tile<D, kTma>(ring + stage * Gm::kStageBytes, &full[stage], &tmap_k, &tmap_v, p.src,
                          kvh, t0, t_end, n_seq_blocks, tc_base, tc_val, lane);
      ++issued;
    }
    const int first = issued > STAGES ? issued - STAGES : 0;
    for (int i = first; i < issued; ++i) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[i % STAGES], (i / STAGES) & 1))) {
        if (lane == 0) report(kErrDrain);
        break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // B operand of Q^T: this lane's column is 8 * warp + lane / 4
  uint32_t qf[D / 16][2];
  {
    const int c = 8 * warp + (lane >> 2);
    const int i = c / G;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) qf[ks][0] = qf[ks][1] = 0u;
    if (i < n) {
      const unsigned int* rowp = reinterpret_cast<const unsigned int*>(
          p.q + ((size_t)(row0 + i) * p.num_q_heads + kvh * G + c % G) * D + 2 * (lane & 3));
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qf[ks][0] = __ldg(rowp + ks * 8);
        qf[ks][1] = __ldg(rowp + ks * 8 + 4);
      }
    }
  }
  // causal limits (last attended position) of this lane's two score columns
  const int tk = 2 * (lane & 3);
  const int ca = 8 * warp + tk;
  const int lim_a = ca / G < n ? ctx - n + ca / G : -1;
  const int lim_b = (ca + 1) / G < n ? ctx - n + (ca + 1) / G : -1;
  AttnState<D> st;
  st.reset();
  bool aborted = false;
  for (int i = 0; i < n_tiles; ++i) {
    if (__any_sync(0xffffffffu, *abort_flag)) {
      aborted = true;
      break;
    }
    const int stage = i % STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (i / STAGES) & 1))) {
      if (lane == 0) report(kErrWaitFull);
      *abort_flag = 1;
      aborted = true;
      break;
    }
    const uint32_t sK = ring + stage * Gm::kStageBytes;
    const int t0 = t_begin + i * kTile;
    const int valid = min(kTile, t_end - t0);
    const int va = max(0, min(valid, lim_a - t0 + 1));
    const int vb = max(0, min(valid, lim_b - t0 + 1));
    attend_tile_causal<D>(st, sK, sK + Gm::kKVBytes, qf, valid, va, vb, p.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // ---- outputs: normalise, stage through shared memory, coalesced rows -----
  st.reduce_l();
  named_barrier_sync(1, NC * 32);  // every consumer is done with the ring
  if (__any_sync(0xffffffffu, aborted) || *abort_flag) return;
  float* buf = reinterpret_cast<float*>(smem) + (size_t)warp * 8 * D;
  const float inv0 = st.l0 > 0.f ? 1.f / st.l0 : 0.f;
  const float inv1 = st.l1 > 0.f ? 1.f / st.l1 : 0.f;
  const int r0 = lane >> 2;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int d0 = mt * 16 + r0;
    buf[tk * D + out_col(tk, d0)] = st.o[mt][0] * inv0;
    buf[(tk + 1) * D + out_col(tk + 1, d0)] = st.o[mt][1] * inv1;
    buf[tk * D + out_col(tk, d0 + 8)] = st.o[mt][2] * inv0;
    buf[(tk + 1) * D + out_col(tk + 1, d0 + 8)] = st.o[mt][3] * inv1;
  }
  // log-sum-exp (natural log) of the 8 columns: lanes 0..3 hold them
  float lse_a = -INFINITY, lse_b = -INFINITY;
  if (st.l0 > 0.f) lse_a = (st.m0 + log2f(st.l0)) * 0.69314718055994530942f;
  if (st.l1 > 0.f) lse_b = (st.m1 + log2f(st.l1)) * 0.69314718055994530942f;
  __syncwarp();
  for (int j = 0; j < 8; ++j) {
    const int c = 8 * warp + j;
    const int i = c / G;
    if (i >= n) break;
    const int lim = ctx - n + i;
    const int h = kvh * G + c % G;
    const size_t r = (size_t)(row0 + i) * p.num_q_heads + h;
    if (lim < t_begin) {  // no token of this split for the row
      if (p.split_tokens == 0)  // (a row before the context's start) a zero row
        for (int d8 = lane; d8 < D / 8; d8 += 32)
          *reinterpret_cast<uint4*>(p.out + r * D + 8 * d8) = make_uint4(0, 0, 0, 0);
      continue;
    }
    if (p.split_tokens > 0) {
      float* dst = p.part_out + (r * p.max_splits + split) * D;
      for (int d4 = lane; d4 < D / 4; d4 += 32)
        *reinterpret_cast<float4*>(dst + 4 * d4) =
            *reinterpret_cast<const float4*>(buf + j * D + out_col(j, 4 * d4));
      const float la = __shfl_sync(0xffffffffu, lse_a, (j >> 1) & 3);
      const float lb = __shfl_sync(0xffffffffu, lse_b, (j >> 1) & 3);
      if (lane == 0) p.part_lse[r * p.max_splits + split] = (j & 1) ? lb : la;
    } else {
      __nv_bfloat16* dst = p.out + r * D;
      for (int d4 = lane; d4 < D / 4; d4 += 32) {
        const float4 v = *reinterpret_cast<const float4*>(buf + j * D + out_col(j, 4 * d4));
        uint2 pk;
        pk.x = pack_bf16x2(v.x, v.y);
        pk.y = pack_bf16x2(v.z, v.w);
        *reinterpret_cast<uint2*>(dst + 4 * d4) = pk;
      }
    }
  }
}

template <int D, bool kTma>
pa_status launch_multi(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& prm,
                       int nc, int B, int num_kv_heads, cudaStream_t stream) {
  using L = MultiSmem<D>;
  auto kern = multi_decode_kernel<D, kTma>;
  const int threads = (nc + 1) * 32;
  const pa_status s = prepare_kernel(reinterpret_cast<const void*>(kern), threads, L::kAlloc,
                                     nullptr);
  if (s != PA_OK) return s;
  dim3 grid(num_kv_heads, prm.split_tokens > 0 ? prm.max_splits : 1, B);
  kern<<<grid, threads, L::kAlloc, stream>>>(mk, mv, prm);
  return launch_status();
}

pa_status check_q_start(const int32_t* q_start, const int32_t* context_lens, int B, int R,
                        int max_q_len, cudaStream_t st) {
  std::vector<int32_t> qs(B + 1), cl(B);
  if (cudaMemcpyAsync(qs.data(), q_start, sizeof(int32_t) * (B + 1), cudaMemcpyDeviceToHost,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(cl.data(), context_lens, sizeof(int32_t) * B, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return PA_ERR_CUDA;
  if (qs[0] != 0 || qs[B] != R) return PA_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int n = qs[b + 1] - qs[b];
    if (n < 0 || n > max_q_len || n > cl[b]) return PA_ERR_INVALID_ARG;
  }
  return PA_OK;
}

}  // namespace

unsigned int take_multi_errors() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_multi_error, sizeof(v)) != cudaSuccess) return 0x80000000u;
  if (v) cudaMemcpyToSymbol(g_multi_error, &zero, sizeof(zero));
  return v;
}

}  // namespace pa

extern "C" pa_status pa_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, const int32_t* q_start,
                                     int32_t num_seqs, int32_t num_q_rows, int32_t max_q_len,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t block_size, int32_t num_blocks, float scale,
                                     int32_t split_tokens, int32_t max_splits, float* part_out,
                                     float* part_lse, int32_t* row_lens, void* out,
                                     void* stream) {
  using namespace pa;
  if (split_tokens < 0 || num_q_rows < 0 || max_q_len < 1) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_q_rows == 0) return PA_OK;
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale, out);
  if (s != PA_OK) return s;
  if (!q_start) return PA_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if ((long long)max_q_len * G > kMaxColumnWarps * 8) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  if (split_tokens > 0) {
    if (split_tokens % kTile) return PA_ERR_INVALID_ARG;
    if (max_splits <= 0 || max_splits > 65535) return PA_ERR_INVALID_ARG;
    if (!part_out || !part_lse || !row_lens) return PA_ERR_WORKSPACE;
    if (!aligned16(part_out)) return PA_ERR_INVALID_ARG;
  }
  cudaStream_t st = as_stream(stream);
  if (validating()) {
    s = check_tables(block_tables, max_blocks_per_seq, context_lens, num_seqs, num_blocks,
                     block_size, split_tokens, max_splits, st);
    if (s != PA_OK) return s;
    s = check_q_start(q_start, context_lens, num_seqs, num_q_rows, max_q_len, st);
    if (s != PA_OK) return s;
  }
  MultiParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.q_start = q_start;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.part_out = part_out;
  prm.part_lse = part_lse;
  prm.row_lens = row_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.src.k_cache = static_cast<const unsigned char*>(k_cache);
  prm.src.v_cache = static_cast<const unsigned char*>(v_cache);
  prm.src.num_kv_heads = num_kv_heads;
  prm.src.block_size = block_size;
  prm.src.log2_bs = ilog2(block_size);
  prm.src.num_blocks = num_blocks;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_q_heads = num_q_heads;
  prm.group = G;
  prm.split_tokens = split_tokens;
  prm.max_splits = split_tokens > 0 ? max_splits : 1;
  prm.max_q_len = max_q_len;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  const int nc = (max_q_len * G + 7) / 8;

  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  const bool tma = block_size >= 8;
  if (tma) {
    const long long rows = (long long)num_blocks * block_size;
    const int box_rows = block_size < kTile ? block_size : kTile;
    if (!make_cache_map(&mk, k_cache, num_kv_heads, head_dim, rows, box_rows) ||
        !make_cache_map(&mv, v_cache, num_kv_heads, head_dim, rows, box_rows))
      return PA_ERR_CUDA;
  }
  if (head_dim == 128)
    return tma ? launch_multi<128, true>(mk, mv, prm, nc, num_seqs, num_kv_heads, st)
               : launch_multi<128, false>(mk, mv, prm, nc, num_seqs, num_kv_heads, st);
  return tma ? launch_multi<64, true>(mk, mv, prm, nc, num_seqs, num_kv_heads, st)
             : launch_multi<64, false>(mk, mv, prm, nc, num_seqs, num_kv_heads, st);
}
