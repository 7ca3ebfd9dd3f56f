// pa_decode.cu -- paged decode attention with grouped-query heads (sm_103a).
//
// Computes, per sequence b and query head h, softmax(scale * q K^T) V over the
// first context_lens[b] logical tokens, whose K/V rows sit in physical blocks
// named by block_tables[b] ("Text Generation Inference: Hugging Face's
// production-grade LLM inference server", section "Under the Hood:
// PagedAttention"), with the running-max / running-sum recurrence of section
// "Under the Hood: Flash Attention" of the same page.
//
// Kernel shape. One thread block per (KV head, context split, sequence):
//   * warp NCW is the loader. Its lanes prefetch 32 block-table entries at a
//     time; lane 0 issues 2-D TMA tile loads (cp.async.bulk.tensor) of each
//     16-token K and V tile into a ring of STAGES shared-memory stages, each
//     completing on a "full" mbarrier. Block sizes below 8 use a per-lane
//     cp.async gather into the same layout instead (a TMA box there would be
//     smaller than one 128-byte swizzle row group).
//   * warps 0..NCW-1 consume tiles round-robin (tile i -> warp i % NCW). Every
//     K/V tile is read from HBM once and serves all G = Hq/Hkv query heads of
//     the KV head ("How to Speed Up LLM Inference: KV Cache to Production
//     Serving", section "The KV cache: the memory problem that runs the
//     show", item 3; "The inference request lifecycle", section "KV cache
//     grows with the sum of cached tokens").
//   * the G query heads are the n = 8 side of a warp MMA, in transposed form:
//       S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]   (m16n8k16, bf16 -> fp32)
//       O^T[D x 8 heads]     += V^T[D x 16] . P^T[16 x 8]
//     so a 16-token tile costs D/16 + D/16 MMAs with no padding for G = 8.
//     The score fragment becomes the B operand of the second product with one
//     movmatrix transpose per 8x8 half.
//   * online softmax in fp32, base-2 exponentials (scale * log2(e) folded into
//     one multiply), running max per head reduced with warp shuffles. The
//     running sum adds the bf16-rounded weights that the PV product uses, so
//     the output is an exactly normalised average of the V rows.
//   * at the end the NCW warps' (m, l, O) are merged through shared memory and
//     either written as bf16 (one split) or as an fp32 partial + natural-log
//     LSE for pa_decode_splitk_reduce.
// Shared-memory tiles use the 128-byte swizzle (16-byte chunk c of row r at
// chunk c ^ (r & 7)), so the ldmatrix reads of 8 rows hit 8 distinct banks.
//
// Every wait is bounded (pa_device.cuh); a wait that runs out sets a bit in
// the per-device error word and the block finishes without hanging.

#include <cudaTypedefs.h>
#include <math.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pagedkv.h"

__device__ unsigned int g_pa_error_word;

namespace pa {
namespace {

constexpr int kTile = 16;        // tokens per MMA tile (the m of S^T)
constexpr int kMaxGroup = 8;     // query heads per KV head (the n of the MMA)
constexpr int kHalfBytes = kTile * 128;  // one 64-wide column half of a tile

struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_out;
  float* part_lse;
  __nv_bfloat16* out;
  int max_blocks;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int block_size;
  int log2_bs;
  int num_blocks;
  int split_tokens;
  int max_splits;
  float scale_log2;
};

template <int D, int NCW, int STAGES>
struct Smem {
  static constexpr int kHalves = D / 64;
  static constexpr int kKVBytes = kHalves * kHalfBytes;   // one K (or V) tile
  static constexpr int kStageBytes = 2 * kKVBytes;         // K then V
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kCombineBytes = NCW * kMaxGroup * D * 4;  // aliases the ring
  static_assert(kRingBytes >= kCombineBytes, "ring too small to hold the merge buffer");
  static constexpr int kStatsOff = kRingBytes;                              // m, l per warp
  static constexpr int kBarOff = kStatsOff + 2 * NCW * kMaxGroup * 4;      // full, empty
  static constexpr int kFlagOff = kBarOff + 2 * STAGES * 8;
  static constexpr int kBytes = kFlagOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the ring to 1 KiB
};

__device__ __forceinline__ void report(unsigned int bits) { atomicOr(&g_pa_error_word, bits); }

template <int D, int NCW, int STAGES, bool kTma>
__global__ void __launch_bounds__((NCW + 1) * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
  using L = Smem<D, NCW, STAGES>;
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
  const int cap = p.max_blocks << p.log2_bs;
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
    const int n_seq_blocks = (ctx + p.block_size - 1) >> p.log2_bs;
    const int bs = p.block_size;
    const long long oob_row = (long long)p.num_blocks * bs;  // a row past the pool: TMA fills zeros
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
      const int blk_first = t0 >> p.log2_bs;
      const int blk_last = (t0 + kTile - 1) >> p.log2_bs;
      if (blk_first < tc_base || blk_last >= tc_base + 32) {  // warp-uniform refill
        tc_base = blk_first;
        const int idx = tc_base + lane;
        tc_val = idx < n_seq_blocks ? bt[idx] : -1;
      }
      const uint32_t sK = ring + stage * L::kStageBytes;
      const uint32_t sV = sK + L::kKVBytes;
      if constexpr (kTma) {
        // bs >= 8: one box of min(bs, 16) rows per 64-column half per block.
        const int box_rows = bs < kTile ? bs : kTile;
        const int nsub = kTile / box_rows;
        int rows[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int blk = blk_first + j;
          const int phys = __shfl_sync(0xffffffffu, tc_val, (blk - tc_base) & 31);
          long long row = (long long)phys * bs + (bs > kTile ? (t0 & (bs - 1)) : 0);
          if (j >= nsub || blk >= n_seq_blocks || phys < 0 || phys >= p.num_blocks) row = oob_row;
          rows[j] = (int)row;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
          for (int h = 0; h < L::kHalves; ++h) {
            const int x = kvh * D + h * 64;
            for (int j = 0; j < nsub; ++j) {
              const uint32_t off = h * kHalfBytes + j * box_rows * 128;
              tma_load_2d(sK + off, &tmap_k, x, rows[j], &full[stage]);
              tma_load_2d(sV + off, &tmap_v, x, rows[j], &full[stage]);
            }
          }
        }
      } else {
        // bs < 8: every lane copies 16-byte chunks of rows with cp.async.
        constexpr int kChunks = D / 8;  // 16-byte chunks per row
        const size_t row_elems = (size_t)p.num_kv_heads * D;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const __nv_bfloat16* cache = which == 0 ? p.k_cache : p.v_cache;
          const uint32_t dst_tile = which == 0 ? sK : sV;
#pragma unroll
          for (int k = 0; k < kTile * kChunks / 32; ++k) {
            const int idx = k * 32 + lane;
            const int r = idx / kChunks, c = idx % kChunks;
            const int t = t0 + r;
            const int blk = t >> p.log2_bs;
            const int phys = __shfl_sync(0xffffffffu, tc_val, (blk - tc_base) & 31);
            const bool ok = t < t_end && blk < n_seq_blocks && phys >= 0 && phys < p.num_blocks;
            const __nv_bfloat16* src =
                ok ? cache + ((size_t)phys * bs + (t & (bs - 1))) * row_elems + (size_t)kvh * D + c * 8
                   : cache;
            const uint32_t dst = dst_tile + (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
            cp_async_16_zfill(dst, src, ok);
          }
        }
        cp_async_arrive_noinc(&full[stage]);
      }
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
  const int gq = lane >> 2;  // query head of the group this lane feeds to the MMA
  uint32_t qf[D / 16][2];
  {
    const __nv_bfloat16* qrow = p.q + ((size_t)b * p.num_q_heads + kvh * G + gq) * D + 2 * (lane & 3);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qf[ks][0] = gq < G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16) : 0u;
      qf[ks][1] = gq < G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8) : 0u;
    }
  }
  float o[D / 16][4];
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int r0 = lane >> 2;
  const int tk = 2 * (lane & 3);

  for (int i = warp; i < n_tiles; i += NCW) {
    if (__any_sync(0xffffffffu, *abort_flag)) break;
    const int stage = i % STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (i / STAGES) & 1))) {
      if (lane == 0) report(kErrWaitFull);
      *abort_flag = 1;
      break;
    }
    const uint32_t sK = ring + stage * L::kStageBytes;
    const uint32_t sV = sK + L::kKVBytes;

    // S^T = K . Q^T  (16 tokens x 8 heads)
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int r = lane & 15;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int cg = 2 * ks + (lane >> 4);
        uint32_t a[4];
        ldsm_x4(sK + (cg >> 3) * kHalfBytes + r * 128 + (((cg & 7) ^ (r & 7)) << 4), a);
        mma_bf16_16816(s, a, qf[ks][0], qf[ks][1]);
      }
    }
    // streaming softmax over this tile (base 2)
    const int valid = min(kTile, t_end - (t_begin + i * kTile));
    const float y0 = r0 < valid ? s[0] * p.scale_log2 : -INFINITY;
    const float y1 = r0 < valid ? s[1] * p.scale_log2 : -INFINITY;
    const float y2 = r0 + 8 < valid ? s[2] * p.scale_log2 : -INFINITY;
    const float y3 = r0 + 8 < valid ? s[3] * p.scale_log2 : -INFINITY;
    float mx0 = fmaxf(y0, y2), mx1 = fmaxf(y1, y3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
    const uint32_t p01 = pack_bf16x2(exp2f(y0 - mn0), exp2f(y1 - mn1));
    const uint32_t p23 = pack_bf16x2(exp2f(y2 - mn0), exp2f(y3 - mn1));
    l0 = l0 * a0 + (bf16_lo(p01) + bf16_lo(p23));
    l1 = l1 * a1 + (bf16_hi(p01) + bf16_hi(p23));
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      o[mt][0] *= a0;
      o[mt][1] *= a1;
      o[mt][2] *= a0;
      o[mt][3] *= a1;
    }
    const uint32_t pb0 = movmatrix_trans(p01);  // P^T rows (tokens 0-7) as the MMA's B operand
    const uint32_t pb1 = movmatrix_trans(p23);  // tokens 8-15

    // O^T += V^T . P^T
    uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
    if (valid < kTile) {  // zero V rows past the end so 0 * NaN cannot appear
      vm01 = (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
      vm23 = (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
    }
    {
      const int mi = lane >> 3;
      const int r = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        const int cg = 2 * mt + (mi & 1);
        uint32_t a[4];
        ldsm_x4_trans(sV + (cg >> 3) * kHalfBytes + r * 128 + (((cg & 7) ^ (r & 7)) << 4), a);
        a[0] &= vm01;
        a[1] &= vm01;
        a[2] &= vm23;
        a[3] &= vm23;
        mma_bf16_16816(o[mt], a, pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // ------------------------------------------------ merge the NCW warps' state
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  if (lane < 4) {
    stat_m[warp * kMaxGroup + tk] = m0;
    stat_m[warp * kMaxGroup + tk + 1] = m1;
    stat_l[warp * kMaxGroup + tk] = l0;
    stat_l[warp * kMaxGroup + tk + 1] = l1;
  }
  named_barrier_sync(1, NCW * 32);  // every consumer is done with the ring
  float* comb = reinterpret_cast<float*>(smem);  // [NCW][8 heads][D]
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int d0 = mt * 16 + r0;
    float* base = comb + (size_t)warp * kMaxGroup * D;
    base[tk * D + d0] = o[mt][0];
    base[(tk + 1) * D + d0] = o[mt][1];
    base[tk * D + d0 + 8] = o[mt][2];
    base[(tk + 1) * D + d0 + 8] = o[mt][3];
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

// ------------------------------------------------------------------ host side

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

// 2-D view of a cache as [num_blocks*block_size rows, Hkv*D columns] with a
// box of 64 columns (128 bytes, the 128-byte swizzle's width) x box_rows.
bool make_cache_map(CUtensorMap* map, const void* base, int hkv, int d, long long rows,
                    int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)hkv * d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hkv * d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int NCW, int STAGES, bool kTma>
pa_status launch(const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& prm, int B,
                 cudaStream_t stream) {
  using L = Smem<D, NCW, STAGES>;
  auto kern = paged_decode_kernel<D, NCW, STAGES, kTma>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  dim3 grid(prm.num_kv_heads, prm.split_tokens > 0 ? prm.max_splits : 1, B);
  kern<<<grid, (NCW + 1) * 32, L::kAlloc, stream>>>(mk, mv, prm);
  return launch_status();
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

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, float scale, int32_t split_tokens,
                               int32_t max_splits, float* part_out, float* part_lse, void* out,
                               void* stream) {
  using namespace pa;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || split_tokens < 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if (G > kMaxGroup) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!is_pow2(block_size) || block_size > 256) return PA_ERR_UNSUPPORTED;
  if ((long long)num_blocks * block_size >= (1ll << 31)) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (!(scale == scale)) return PA_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  if (split_tokens > 0) {
    if (split_tokens % kTile) return PA_ERR_INVALID_ARG;
    if (max_splits <= 0 || max_splits > 65535) return PA_ERR_INVALID_ARG;
    if (!part_out || !part_lse) return PA_ERR_WORKSPACE;
    if (!aligned16(part_out)) return PA_ERR_INVALID_ARG;
  }
  cudaStream_t st = as_stream(stream);
  if (validating()) {
    pa_status s = check_tables(block_tables, max_blocks_per_seq, context_lens, num_seqs, num_blocks,
                               block_size, split_tokens, max_splits, st);
    if (s != PA_OK) return s;
  }

  DecodeParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  prm.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.part_out = part_out;
  prm.part_lse = part_lse;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.max_blocks = max_blocks_per_seq;
  prm.num_q_heads = num_q_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.group = G;
  prm.block_size = block_size;
  prm.log2_bs = ilog2(block_size);
  prm.num_blocks = num_blocks;
  prm.split_tokens = split_tokens;
  prm.max_splits = split_tokens > 0 ? max_splits : 1;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);

  CUtensorMap mk, mv;
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
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
    return tma ? launch<128, NCW, 4, true>(mk, mv, prm, num_seqs, st)
               : launch<128, NCW, 4, false>(mk, mv, prm, num_seqs, st);
  return tma ? launch<64, NCW, 4, true>(mk, mv, prm, num_seqs, st)
             : launch<64, NCW, 4, false>(mk, mv, prm, num_seqs, st);
}

extern "C" pa_status pa_last_device_error(int32_t* code) {
  if (!code) return PA_ERR_INVALID_ARG;
  unsigned int v = 0, zero = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(&v, g_pa_error_word, sizeof(v)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_pa_error_word, &zero, sizeof(zero)) != cudaSuccess)
    return PA_ERR_CUDA;
  *code = (int32_t)v;
  return v ? PA_ERR_DEVICE : PA_OK;
}
