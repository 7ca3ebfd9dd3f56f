// pa_decode.cu -- paged decode attention, one thread block per (KV head,
// context split, sequence) (sm_103a).
//
// Computes, per sequence b and query head h, softmax(scale * q K^T) V over the
// logical tokens of one context split, whose K/V rows sit in the physical
// blocks named by block_tables[b] ("Text Generation Inference: Hugging Face's
// production-grade LLM inference server", section "Under the Hood:
// PagedAttention"). The tile math and layout are in pa_tile.cuh.
//
// Block shape:
//   * warp NCW is the loader: its lanes hold 32 block-table entries at a time
//     and it streams 16-token K/V tiles into a ring of STAGES shared-memory
//     stages (TMA for block sizes >= 8, a cp.async gather below), each stage
//     completing on a "full" mbarrier and released on an "empty" one;
//   * warps 0..NCW-1 consume tiles round-robin (tile i -> warp i % NCW), every
//     K/V tile serving all G = Hq/Hkv query heads of the KV head ("How to Speed
//     Up LLM Inference: KV Cache to Production Serving", section "The KV cache:
//     the memory problem that runs the show", item 3);
//   * the NCW warps' states are merged through shared memory and written as
//     bf16 (one split per sequence) or as an fp32 partial + natural-log LSE
//     for pa_decode_splitk_reduce.
// Every wait is bounded; a wait that runs out sets a bit in this file's
// device error word and the block finishes without hanging.

#include <math.h>

#include <cstring>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_tile.cuh"
#include "pagedkv.h"

namespace pa {
namespace {

__device__ unsigned int g_decode_error;

__device__ __forceinline__ void report(unsigned int bits) { atomicOr(&g_decode_error, bits); }

struct DecodeParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_out;
  float* part_lse;
  __nv_bfloat16* out;
  TileSrc src;
  int max_blocks;
  int num_q_heads;
  int group;
  int split_tokens;
  int max_splits;
  float scale_log2;
};

template <int D, int NCW, int STAGES>
struct Smem {
  static constexpr int kStageBytes = TileGeom<D>::kStageBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kCombineBytes = NCW * kMaxGroup * D * 4;  // aliases the ring
  static_assert(kRingBytes >= kCombineBytes, "ring too small to hold the merge buffer");
  static constexpr int kStatsOff = kRingBytes;                          // m, l per warp
  static constexpr int kBarOff = kStatsOff + 2 * NCW * kMaxGroup * 4;  // full, empty
  static constexpr int kFlagOff = kBarOff + 2 * STAGES * 8;
  static constexpr int kBytes = kFlagOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the ring to 1 KiB
};

template <int D, int NCW, int STAGES, bool kTma>
__global__ void __launch_bounds__((NCW + 1) * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  // Every stage must belong to one consumer warp (tile i -> warp i % NCW,
  // stage i % STAGES): a warp then polls a stage's "full" barrier only after
  // consuming that stage's previous tile, never one phase early.
  static_assert(STAGES % NCW == 0, "each ring stage must belong to one consumer warp");
  using L = Smem<D, NCW, STAGES>;
  using Gm = TileGeom<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stat_m = reinterpret_cast<float*>(smem + L::kStatsOff);
  float* stat_l = stat_m + NCW * kMaxGroup;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kFlagOff);

  const int kvh = blockIdx.x;
  const int split = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  int ctx = p.context_lens[b];
  const int cap = p.max_blocks << p.src.log2_bs;
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  int t_begin = 0, t_end = ctx;
  if (p.split_tokens > 0) {
    t_begin = split * p.split_tokens;
    t_end = min(t_begin + p.split_tokens, ctx);
  }
  if (t_begin >= t_end) {
    // No tokens: a whole empty sequence writes a zero row; an empty split
    // writes nothing (the reduce never reads splits past the context).
    if (p.split_tokens == 0) {
      for (int i = threadIdx.x; i < G * (D / 8); i += blockDim.x) {
        const int g = i / (D / 8), c = i % (D / 8);
        __nv_bfloat16* dst = p.out + ((size_t)b * p.num_q_heads + kvh * G + g) * D + c * 8;
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    return;
  }
  const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], kTma ? 1 : 32);
      mbar_init(&empty[s], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const uint32_t ring = smem_u32(smem);

  if (warp == NCW) {
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
    // Drain: the last copy issued into each stage must have landed before the
    // block may exit (its shared memory must outlive the copies).
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
  uint32_t qf[D / 16][2];
  load_q_frags<D>(qf, p.q + ((size_t)b * p.num_q_heads + kvh * G) * D, G, lane);
  AttnState<D> st;
  st.reset();

  for (int i = warp; i < n_tiles; i += NCW) {
    if (__any_sync(0xffffffffu, *abort_flag)) break;
    const int stage = i % STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (i / STAGES) & 1))) {
      if (lane == 0) report(kErrWaitFull);
      *abort_flag = 1;
      break;
    }
    const uint32_t sK = ring + stage * Gm::kStageBytes;
    const int valid = min(kTile, t_end - (t_begin + i * kTile));
    attend_tile<D>(st, sK, sK + Gm::kKVBytes, qf, valid, p.scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // ------------------------------------------------ merge the NCW warps' state
  st.reduce_l();
  const int r0 = lane >> 2;
  const int tk = 2 * (lane & 3);
  if (lane < 4) {
    stat_m[warp * kMaxGroup + tk] = st.m0;
    stat_m[warp * kMaxGroup + tk + 1] = st.m1;
    stat_l[warp * kMaxGroup + tk] = st.l0;
    stat_l[warp * kMaxGroup + tk + 1] = st.l1;
  }
  named_barrier_sync(1, NCW * 32);  // every consumer is done with the ring
  float* comb = reinterpret_cast<float*>(smem);  // [NCW][8 heads][D]
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int d0 = mt * 16 + r0;
    float* base = comb + (size_t)warp * kMaxGroup * D;
    base[tk * D + d0] = st.o[mt][0];
    base[(tk + 1) * D + d0] = st.o[mt][1];
    base[tk * D + d0 + 8] = st.o[mt][2];
    base[(tk + 1) * D + d0 + 8] = st.o[mt][3];
  }
  named_barrier_sync(1, NCW * 32);

  constexpr int kC8 = D / 8;  // 8-column chunks per head row
  for (int idx = threadIdx.x; idx < G * kC8; idx += NCW * 32) {
    const int g = idx / kC8, c8 = idx % kC8;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, stat_m[w * kMaxGroup + g]);
    float Lsum = 0.f, acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) {
      const float wt = exp2f(stat_m[w * kMaxGroup + g] - M);
      Lsum += wt * stat_l[w * kMaxGroup + g];
      const float4* src = reinterpret_cast<const float4*>(comb + ((size_t)w * kMaxGroup + g) * D + c8 * 8);
      const float4 u = src[0], v = src[1];
      acc[0] += wt * u.x; acc[1] += wt * u.y; acc[2] += wt * u.z; acc[3] += wt * u.w;
      acc[4] += wt * v.x; acc[5] += wt * v.y; acc[6] += wt * v.z; acc[7] += wt * v.w;
    }
    const int h = kvh * G + g;
    if (p.split_tokens > 0) {
      const size_t row = ((size_t)b * p.num_q_heads + h) * p.max_splits + split;
      float4* dst = reinterpret_cast<float4*>(p.part_out + row * D + c8 * 8);
      dst[0] = make_float4(acc[0] / Lsum, acc[1] / Lsum, acc[2] / Lsum, acc[3] / Lsum);
      dst[1] = make_float4(acc[4] / Lsum, acc[5] / Lsum, acc[6] / Lsum, acc[7] / Lsum);
      if (c8 == 0) p.part_lse[row] = (M + log2f(Lsum)) * 0.69314718055994530942f;
    } else {
      uint4 pk;
      pk.x = pack_bf16x2(acc[0] / Lsum, acc[1] / Lsum);
      pk.y = pack_bf16x2(acc[2] / Lsum, acc[3] / Lsum);
      pk.z = pack_bf16x2(acc[4] / Lsum, acc[5] / Lsum);
      pk.w = pack_bf16x2(acc[6] / Lsum, acc[7] / Lsum);
      *reinterpret_cast<uint4*>(p.out + ((size_t)b * p.num_q_heads + h) * D + c8 * 8) = pk;
    }
  }
}

template <int D, int NCW, int STAGES, bool kTma>
pa_status launch(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& prm, int B,
                 int num_kv_heads, cudaStream_t stream) {
  using L = Smem<D, NCW, STAGES>;
  auto kern = paged_decode_kernel<D, NCW, STAGES, kTma>;
  const pa_status s =
      prepare_kernel(reinterpret_cast<const void*>(kern), (NCW + 1) * 32, L::kAlloc, nullptr);
  if (s != PA_OK) return s;
  dim3 grid(num_kv_heads, prm.split_tokens > 0 ? prm.max_splits : 1, B);
  kern<<<grid, (NCW + 1) * 32, L::kAlloc, stream>>>(mk, mv, prm);
  return launch_status();
}

// One warp waits, bounded by limit_ns, on an mbarrier that expects one
// arrival nobody makes; the wait runs out and the warp records kErrSelfTest.
__global__ void __launch_bounds__(32) selftest_wait_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = __all_sync(0xffffffffu, mbar_wait(&bar, 0, limit_ns));
  if (!done && threadIdx.x == 0) report(kErrSelfTest);
}

}  // namespace

unsigned int take_decode_errors() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v)) != cudaSuccess) return 0x80000000u;
  if (v) cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(zero));
  return v;
}

}  // namespace pa

extern "C" pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, float scale, int32_t split_tokens,
                               int32_t max_splits, float* part_out, float* part_lse, void* out,
                               void* stream) {
  using namespace pa;
  if (split_tokens < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale, out);
  if (s != PA_OK) return s;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  if (split_tokens > 0) {
    if (split_tokens % kTile) return PA_ERR_INVALID_ARG;
    if (max_splits <= 0 || max_splits > 65535) return PA_ERR_INVALID_ARG;
    if (!part_out || !part_lse) return PA_ERR_WORKSPACE;
    if (!aligned16(part_out)) return PA_ERR_INVALID_ARG;
  }
  cudaStream_t st = as_stream(stream);
  if (validating()) {
    s = check_tables(block_tables, max_blocks_per_seq, context_lens, num_seqs, num_blocks,
                     block_size, split_tokens, max_splits, st);
    if (s != PA_OK) return s;
  }

  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.part_out = part_out;
  prm.part_lse = part_lse;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.src.k_cache = static_cast<const unsigned char*>(k_cache);
  prm.src.v_cache = static_cast<const unsigned char*>(v_cache);
  prm.src.num_kv_heads = num_kv_heads;
  prm.src.block_size = block_size;
  prm.src.log2_bs = ilog2(block_size);
  prm.src.num_blocks = num_blocks;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_q_heads = num_q_heads;
  prm.group = num_q_heads / num_kv_heads;
  prm.split_tokens = split_tokens;
  prm.max_splits = split_tokens > 0 ? max_splits : 1;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);

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
  constexpr int NCW = 4;
  if (head_dim == 128)
    return tma ? launch<128, NCW, 4, true>(mk, mv, prm, num_seqs, num_kv_heads, st)
               : launch<128, NCW, 4, false>(mk, mv, prm, num_seqs, num_kv_heads, st);
  return tma ? launch<64, NCW, 4, true>(mk, mv, prm, num_seqs, num_kv_heads, st)
             : launch<64, NCW, 4, false>(mk, mv, prm, num_seqs, num_kv_heads, st);
}

extern "C" pa_status pa_selftest_wait_timeout(int32_t limit_us, void* stream) {
  using namespace pa;
  if (limit_us <= 0 || limit_us > 2000000) return PA_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>((unsigned long long)limit_us * 1000ull);
  return launch_status();
}
