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
// (attend_tile_causal_nt); no merge between warps is needed. Outputs go through
// shared memory so that every row is written with coalesced stores: bf16 rows
// (one split) or fp32 partials + natural-log LSEs for pa_decode_splitk_reduce,
// whose per-row context lengths this kernel writes to row_lens.
//
// balanced_multi_kernel runs the same column-warp tile math on the
// work-balanced persistent schedule of pa_balance.cuh (one launch, every block
// the same number of tiles, no tail): a unit is (sequence, KV head) over the
// sequence's context, each of its tiles folded by every column warp; a unit
// cut by a block range leaves per-column records that the block publishing
// the last of them merges by log-sum-exp, column warp by column warp.

#include <math.h>

#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "pa_balance.cuh"
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
  const float* k_scale;        // [Hkv], e4m3 pools only
  const float* v_scale;        // [Hkv], e4m3 pools only
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

// A 32-token e4m3 tile for query columns with their own causal limits: the
// score and PV math of attend_tile_fp8 (K and V bytes widened exactly to f16,
// Q in the e4m3 tiles' k order), with the per-column masks of
// attend_tile_causal_nt: rows >= valid_a (valid_b) are masked for this lane's
// column 2 (lane % 4) (its column + 1), V rows >= valid are zeroed, and a
// column whose every score so far is masked keeps m = -inf, l = 0, O = 0.
// score_scale_log2 = scale * k_scale * log2(e); O is in the fp8 output dim
// order (fp8_out_dim) and still to be multiplied by v_scale.
template <int D>
__device__ __forceinline__ void attend_tile_causal_fp8(AttnState<D>& st, uint32_t sK,
                                                       uint32_t sV,
                                                       const uint32_t (&qf)[D / 16][2],
                                                       int valid, int valid_a, int valid_b,
                                                       float score_scale_log2, int lane) {
  static_assert(D == 128, "e4m3 tiles are one 128-byte row per token");
  const int r = lane & 15;
  const int cadd = lane >> 4;
  float sa[4] = {0.f, 0.f, 0.f, 0.f};  // tokens 0-15
  float sb[4] = {0.f, 0.f, 0.f, 0.f};  // tokens 16-31
#pragma unroll
  for (int sidx = 0; sidx < D / 32; ++sidx) {
    const uint32_t sw = (uint32_t)(((2 * sidx + cadd) ^ (r & 7)) << 4);
    uint32_t ka[4], kb[4], a[4];
    ldsm_x4(sK + r * 128 + sw, ka);
    ldsm_x4(sK + (r + 16) * 128 + sw, kb);
    fp8_k_operand(ka, 0, a);
    mma_f16_16816(sa, a, qf[2 * sidx][0], qf[2 * sidx][1]);
    fp8_k_operand(kb, 0, a);
    mma_f16_16816(sb, a, qf[2 * sidx][0], qf[2 * sidx][1]);
    fp8_k_operand(ka, 2, a);
    mma_f16_16816(sa, a, qf[2 * sidx + 1][0], qf[2 * sidx + 1][1]);
    fp8_k_operand(kb, 2, a);
    mma_f16_16816(sb, a, qf[2 * sidx + 1][0], qf[2 * sidx + 1][1]);
  }
  const int r0 = lane >> 2;
  const int tk = 2 * (lane & 3);
  float y[8];  // tokens r0 + 8i (i = 0..3) x columns tk (even entries), tk + 1 (odd)
  const float s8[8] = {sa[0], sa[1], sa[2], sa[3], sb[0], sb[1], sb[2], sb[3]};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    y[2 * i] = r0 + 8 * i < valid_a ? s8[2 * i] * score_scale_log2 : -INFINITY;
    y[2 * i + 1] = r0 + 8 * i < valid_b ? s8[2 * i + 1] * score_scale_log2 : -INFINITY;
  }
  float mx0 = fmaxf(fmaxf(y[0], y[2]), fmaxf(y[4], y[6]));
  float mx1 = fmaxf(fmaxf(y[1], y[3]), fmaxf(y[5], y[7]));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
  const float e0 = mn0 == -INFINITY ? 0.f : mn0, e1 = mn1 == -INFINITY ? 0.f : mn1;
  const float a0 = exp2f(st.m0 - e0), a1 = exp2f(st.m1 - e1);
  uint32_t pw[4];  // f16 weights of tokens r0 + 8i, columns tk | tk + 1
#pragma unroll
  for (int i = 0; i < 4; ++i) pw[i] = pack_f16x2(exp2f(y[2 * i] - e0), exp2f(y[2 * i + 1] - e1));
  st.l0 = st.l0 * a0 + ((f16_lo(pw[0]) + f16_lo(pw[1])) + (f16_lo(pw[2]) + f16_lo(pw[3])));
  st.l1 = st.l1 * a1 + ((f16_hi(pw[0]) + f16_hi(pw[1])) + (f16_hi(pw[2]) + f16_hi(pw[3])));
  st.m0 = mn0;
  st.m1 = mn1;
  if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {  // only when a max moved
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.o[mt][0] *= a0;
      st.o[mt][1] *= a1;
      st.o[mt][2] *= a0;
      st.o[mt][3] *= a1;
    }
  }
  uint32_t pb[4];  // B fragments of P^T: tokens 0-7, 8-15, 16-23, 24-31
#pragma unroll
  for (int i = 0; i < 4; ++i) pb[i] = movmatrix_trans(pw[i]);
  uint32_t vm[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
  const bool masked = valid < kFp8Tile;
  if (masked) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      vm[i] = (tk + 8 * i < valid ? 0x0000ffffu : 0u) | (tk + 8 * i + 1 < valid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int sidx = 0; sidx < D / 32; ++sidx) {
    const uint32_t sw = (uint32_t)(((2 * sidx + cadd) ^ (r & 7)) << 4);
    uint32_t va[4], vb[4];
    ldsm_x4_trans(sV + r * 128 + sw, va);
    ldsm_x4_trans(sV + (r + 16) * 128 + sw, vb);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t x0 = byte_perm(va[2 * hf], 0u, 0x3120u);      // tokens 0-7
      uint32_t x1 = byte_perm(va[2 * hf + 1], 0u, 0x3120u);  // tokens 8-15
      uint32_t a[4];
      e4m3x4_to_f16x2x2(x0, a[0], a[1]);
      e4m3x4_to_f16x2x2(x1, a[2], a[3]);
      if (masked) {
        a[0] &= vm[0]; a[1] &= vm[0]; a[2] &= vm[1]; a[3] &= vm[1];
      }
      mma_f16_16816(st.o[2 * sidx + hf], a, pb[0], pb[1]);
      x0 = byte_perm(vb[2 * hf], 0u, 0x3120u);      // tokens 16-23
      x1 = byte_perm(vb[2 * hf + 1], 0u, 0x3120u);  // tokens 24-31
      e4m3x4_to_f16x2x2(x0, a[0], a[1]);
      e4m3x4_to_f16x2x2(x1, a[2], a[3]);
      if (masked) {
        a[0] &= vm[2]; a[1] &= vm[2]; a[2] &= vm[3]; a[3] &= vm[3];
      }
      mma_f16_16816(st.o[2 * sidx + hf], a, pb[2], pb[3]);
    }
  }
}

// Column of element d of column row j in a warp's output buffer: XOR-swizzled
// in 8-float groups so the 4 column rows one store touches use 4 bank groups.
__device__ __forceinline__ int out_col(int j, int d) { return d ^ ((j >> 1) << 3); }

template <int D, bool kTma, bool kFp8 = false>
__global__ void __launch_bounds__((kMaxColumnWarps + 1) * 32, 2)
    multi_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const MultiParams p) {
  // e4m3 pools: 32-token tiles of 128-byte rows (the same 8 KB stage)
  constexpr int EB = kFp8 ? 1 : 2;
  constexpr int TT = kFp8 ? kFp8Tile : kTile;
  using L = MultiSmem<D>;
  using Gm = TileGeom<D, EB, TT>;
  static_assert(Gm::kStageBytes == TileGeom<D>::kStageBytes, "one ring layout for both");
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
  const int n_tiles = (t_end - t_begin + TT - 1) / TT;

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
      const int t0 = t_begin + i * TT;
      const int blk_first = t0 >> p.src.log2_bs;
      const int blk_last = (t0 + TT - 1) >> p.src.log2_bs;
      if (blk_first < tc_base || blk_last >= tc_base + 32) {  // warp-uniform refill
        tc_base = blk_first;
        const int idx = tc_base + lane;
        tc_val = idx < n_seq_blocks ? bt[idx] : -1;
      }
      issue_tile<D, kTma, EB, TT>(ring + stage * Gm::kStageBytes, &full[stage], &tmap_k,
                                  &tmap_v, p.src, kvh, t0, t_end, n_seq_blocks, tc_base, tc_val,
                                  lane);
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
  uint32_t qfs[1][D / 16][2];
  auto& qf = qfs[0];
  {
    const int c = 8 * warp + (lane >> 2);
    const int i = c / G;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) qf[ks][0] = qf[ks][1] = 0u;
    if (i < n) {
      const __nv_bfloat16* qrow = p.q + ((size_t)(row0 + i) * p.num_q_heads + kvh * G + c % G) * D;
      if constexpr (kFp8) {  // f16, in the e4m3 tiles' k order (dims 4c .. 4c + 3 of a step)
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(qrow + ks * 16 + 4 * (lane & 3)));
          qf[ks][0] = pack_f16x2(bf16_lo(v.x), bf16_hi(v.x));
          qf[ks][1] = pack_f16x2(bf16_lo(v.y), bf16_hi(v.y));
        }
      } else {
        const unsigned int* rowp = reinterpret_cast<const unsigned int*>(qrow + 2 * (lane & 3));
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          qf[ks][0] = __ldg(rowp + ks * 8);
          qf[ks][1] = __ldg(rowp + ks * 8 + 4);
        }
      }
    }
  }
  const float score_scale_log2 = kFp8 ? p.scale_log2 * p.k_scale[kvh] : p.scale_log2;
  const float out_scale = kFp8 ? p.v_scale[kvh] : 1.f;
  // causal limits (last attended position) of this lane's two score columns
  const int tk = 2 * (lane & 3);
  const int ca = 8 * warp + tk;
  const int lim_a = ca / G < n ? ctx - n + ca / G : -1;
  const int lim_b = (ca + 1) / G < n ? ctx - n + (ca + 1) / G : -1;
  AttnState<D> sts[1];
  AttnState<D>& st = sts[0];
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
    const int t0 = t_begin + i * TT;
    const int valid = min(TT, t_end - t0);
    const int va[1] = {max(0, min(valid, lim_a - t0 + 1))};
    const int vb[1] = {max(0, min(valid, lim_b - t0 + 1))};
    if constexpr (kFp8)
      attend_tile_causal_fp8<D>(st, sK, sK + Gm::kKVBytes, qf, valid, va[0], vb[0],
                                score_scale_log2, lane);
    else
      attend_tile_causal_nt<D, 1>(sts, sK, sK + Gm::kKVBytes, qfs, valid, va, vb,
                                  score_scale_log2, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // ---- outputs: normalise, stage through shared memory, coalesced rows -----
  st.reduce_l();
  named_barrier_sync(1, NC * 32);  // every consumer is done with the ring
  if (__any_sync(0xffffffffu, aborted) || *abort_flag) return;
  float* buf = reinterpret_cast<float*>(smem) + (size_t)warp * 8 * D;
  const float inv0 = st.l0 > 0.f ? out_scale / st.l0 : 0.f;
  const float inv1 = st.l1 > 0.f ? out_scale / st.l1 : 0.f;
  const int r0 = lane >> 2;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    // the dims of this lane's accumulators: rows r0 and r0 + 8 of the output
    // tile (bf16 tiles) or dims 2 r0 and 2 r0 + 1 (e4m3 tiles)
    const int d0 = kFp8 ? fp8_out_dim(mt, lane, false) : mt * 16 + r0;
    const int d1 = kFp8 ? fp8_out_dim(mt, lane, true) : mt * 16 + r0 + 8;
    buf[tk * D + out_col(tk, d0)] = st.o[mt][0] * inv0;
    buf[(tk + 1) * D + out_col(tk + 1, d0)] = st.o[mt][1] * inv1;
    buf[tk * D + out_col(tk, d1)] = st.o[mt][2] * inv0;
    buf[(tk + 1) * D + out_col(tk + 1, d1)] = st.o[mt][3] * inv1;
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

template <int D, bool kTma, bool kFp8 = false>
pa_status launch_multi(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& prm,
                       int nc, int B, int num_kv_heads, cudaStream_t stream) {
  using L = MultiSmem<D>;
  auto kern = multi_decode_kernel<D, kTma, kFp8>;
  const int threads = (nc + 1) * 32;
  const pa_status s = prepare_kernel(reinterpret_cast<const void*>(kern), threads, L::kAlloc,
                                     nullptr);
  if (s != PA_OK) return s;
  dim3 grid(num_kv_heads, prm.split_tokens > 0 ? prm.max_splits : 1, B);
  kern<<<grid, threads, L::kAlloc, stream>>>(mk, mv, prm);
  return launch_status();
}

// ---------------------------------------------------------------------------
// long query chunks: row blocks in the standard MMA form
// ---------------------------------------------------------------------------
// A chunk of a long prompt brings more (token, head) rows than the n side
// holds (n_b * G > 64). Then the rows go on the MMA's m side, as in a
// FlashAttention-2 forward pass: a block takes 64 rows (the (token, head)
// pairs 64 rb .. 64 rb + 63 of one sequence and KV head, row = token * G +
// head), four warps of 16 rows; per 16-key tile each warp computes
// S[16 x 16] = Q K^T (8 k-steps x 2 key groups of m16n8k16), the online
// softmax per row, and O[16 x D] += P V with P taken straight from the score
// accumulators as the A operand. Every warp folds every tile of the block's
// key range [0, last position of its last token], read through the same TMA
// ring as the other kernels (K/V tiles are re-read from L2 by the sequence's
// other row blocks: prefill is compute-bound).

constexpr int kRowWarps = 4;   // 16 rows each
constexpr int kRowsPerBlock = 16 * kRowWarps;

template <int D>
struct RowSmem {
  static constexpr int kStageBytes = TileGeom<D>::kStageBytes;
  static constexpr int kRingBytes = kMultiStages * kStageBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kFlagOff = kBarOff + 2 * kMultiStages * 8;
  static constexpr int kAlloc = kFlagOff + 16 + 1024;
};

template <int D, bool kTma>
__global__ void __launch_bounds__((kRowWarps + 1) * 32, 2)
    rowblock_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const MultiParams p) {
  using L = RowSmem<D>;
  using Gm = TileGeom<D>;
  constexpr int STAGES = kMultiStages;
  constexpr int NW = kRowWarps;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kFlagOff);

  const int rb = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int row0 = p.q_start[b];
  const int n = p.q_start[b + 1] - row0;
  const int rows = n * G;
  if (rb * kRowsPerBlock >= rows) return;
  if (n > p.max_q_len) {
    if (threadIdx.x == 0) report(kErrShape);
    return;
  }
  int ctx = p.context_lens[b];
  const int cap = p.max_blocks << p.src.log2_bs;
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  // keys the block needs: up to the last position of its last token
  const int last_row = min(rows, (rb + 1) * kRowsPerBlock) - 1;
  const int t_end = min(ctx, ctx - n + last_row / G + 1);
  const int n_tiles = t_end > 0 ? (t_end + kTile - 1) / kTile : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], kTma ? 1 : 32);
      mbar_init(&empty[s], NW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const uint32_t ring = smem_u32(smem);

  if (warp == NW) {
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
      const int t0 = i * kTile;
      const int blk_first = t0 >> p.src.log2_bs;
      const int blk_last = (t0 + kTile - 1) >> p.src.log2_bs;
      if (blk_first < tc_base || blk_last >= tc_base + 32) {  // warp-uniform refill
        tc_base = blk_first;
        const int idx = tc_base + lane;
        tc_val = idx < n_seq_blocks ? bt[idx] : -1;
      }
      issue_tile<D, kTma>(ring + stage * Gm::kStageBytes, &full[stage], &tmap_k, &tmap_v, p.src,
                          kvh, t0, ctx, n_seq_blocks, tc_base, tc_val, lane);
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
  const int gq = lane >> 2;          // this lane's rows: gq and gq + 8 of the warp
  const int cq = lane & 3;
  const int wrow = rb * kRowsPerBlock + warp * 16;
  const int ra = wrow + gq, rbw = wrow + gq + 8;  // the lane's two rows
  // the rows' query tokens, causal limits (last attended position) and q rows
  const int lim_a = ra < rows ? ctx - n + ra / G : -1;
  const int lim_b = rbw < rows ? ctx - n + rbw / G : -1;
  // A operand of Q: rows gq / gq + 8, dims 16 ks + 2 cq (+1) and + 8
  uint32_t qa[D / 16][4];
  {
    const unsigned int* pa_row = ra < rows ? reinterpret_cast<const unsigned int*>(
        p.q + ((size_t)(row0 + ra / G) * p.num_q_heads + kvh * G + ra % G) * D + 2 * cq) : nullptr;
    const unsigned int* pb_row = rbw < rows ? reinterpret_cast<const unsigned int*>(
        p.q + ((size_t)(row0 + rbw / G) * p.num_q_heads + kvh * G + rbw % G) * D + 2 * cq) : nullptr;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = pa_row ? __ldg(pa_row + ks * 8) : 0u;
      qa[ks][1] = pb_row ? __ldg(pb_row + ks * 8) : 0u;
      qa[ks][2] = pa_row ? __ldg(pa_row + ks * 8 + 4) : 0u;
      qa[ks][3] = pb_row ? __ldg(pb_row + ks * 8 + 4) : 0u;
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int db = 0; db < D / 8; ++db) o[db][0] = o[db][1] = o[db][2] = o[db][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const int mi = lane >> 3;          // the 8x8 matrix this lane addresses for ldmatrix
  for (int i = 0; i < n_tiles; ++i) {
    if (__any_sync(0xffffffffu, *abort_flag)) break;
    const int stage = i % STAGES;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (i / STAGES) & 1))) {
      if (lane == 0) report(kErrWaitFull);
      *abort_flag = 1;
      break;
    }
    const uint32_t sK = ring + stage * Gm::kStageBytes;
    const uint32_t sV = sK + Gm::kKVBytes;
    const int t0 = i * kTile;
    // S = Q K^T: key groups 0-7 (s0) and 8-15 (s1)
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int key = 8 * (mi >> 1) + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int cg = 2 * ks + (mi & 1);
        uint32_t kb[4];  // (keys 0-7, dims lo), (keys 0-7, hi), (keys 8-15, lo), (keys 8-15, hi)
        ldsm_x4(sK + (cg >> 3) * kHalfBytes + key * 128 + (((cg & 7) ^ (key & 7)) << 4), kb);
        mma_bf16_16816(s0, qa[ks], kb[0], kb[1]);
        mma_bf16_16816(s1, qa[ks], kb[2], kb[3]);
      }
    }
    // causal + context masks: key t0 + k valid for a row if <= its limit
    const int k0 = t0 + 2 * cq;
    float y[8];  // row a: keys k0, k0+1, k0+8, k0+9; row b: the same
    y[0] = k0 <= lim_a ? s0[0] * p.scale_log2 : -INFINITY;
    y[1] = k0 + 1 <= lim_a ? s0[1] * p.scale_log2 : -INFINITY;
    y[2] = k0 + 8 <= lim_a ? s1[0] * p.scale_log2 : -INFINITY;
    y[3] = k0 + 9 <= lim_a ? s1[1] * p.scale_log2 : -INFINITY;
    y[4] = k0 <= lim_b ? s0[2] * p.scale_log2 : -INFINITY;
    y[5] = k0 + 1 <= lim_b ? s0[3] * p.scale_log2 : -INFINITY;
    y[6] = k0 + 8 <= lim_b ? s1[2] * p.scale_log2 : -INFINITY;
    y[7] = k0 + 9 <= lim_b ? s1[3] * p.scale_log2 : -INFINITY;
    float mxa = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
    float mxb = fmaxf(fmaxf(y[4], y[5]), fmaxf(y[6], y[7]));
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
    }
    const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
    const float ea = mna == -INFINITY ? 0.f : mna, eb = mnb == -INFINITY ? 0.f : mnb;
    const float aa = exp2f(m_a - ea), ab = exp2f(m_b - eb);
    // P as the A operand of P V: rows a / b, keys 2cq (+1) and + 8
    uint32_t pa4[4];
    pa4[0] = pack_bf16x2(exp2f(y[0] - ea), exp2f(y[1] - ea));
    pa4[1] = pack_bf16x2(exp2f(y[4] - eb), exp2f(y[5] - eb));
    pa4[2] = pack_bf16x2(exp2f(y[2] - ea), exp2f(y[3] - ea));
    pa4[3] = pack_bf16x2(exp2f(y[6] - eb), exp2f(y[7] - eb));
    float la = (bf16_lo(pa4[0]) + bf16_hi(pa4[0])) + (bf16_lo(pa4[2]) + bf16_hi(pa4[2]));
    float lb = (bf16_lo(pa4[1]) + bf16_hi(pa4[1])) + (bf16_lo(pa4[3]) + bf16_hi(pa4[3]));
    l_a = l_a * aa + la;
    l_b = l_b * ab + lb;
    m_a = mna;
    m_b = mnb;
    if (__any_sync(0xffffffffu, aa != 1.f || ab != 1.f)) {
#pragma unroll
      for (int db = 0; db < D / 8; ++db) {
        o[db][0] *= aa;
        o[db][1] *= aa;
        o[db][2] *= ab;
        o[db][3] *= ab;
      }
    }
    // V rows past the context are zeroed (stale or NaN slots)
    const int valid = min(kTile, ctx - t0);
    uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
    const bool masked = valid < kTile;
    if (masked) {
      const int kr = (lane & 3) * 2;  // .trans: this lane holds keys kr, kr+1 (+8)
      vm0 = (kr < valid ? 0x0000ffffu : 0u) | (kr + 1 < valid ? 0xffff0000u : 0u);
      vm1 = (kr + 8 < valid ? 0x0000ffffu : 0u) | (kr + 9 < valid ? 0xffff0000u : 0u);
    }
    {
      // O += P V: B operand of V via ldmatrix.trans, dim blocks 2 d2 and 2 d2 + 1
      const int key = 8 * (mi & 1) + (lane & 7);
#pragma unroll
      for (int d2 = 0; d2 < D / 16; ++d2) {
        const int cg = 2 * d2 + (mi >> 1);
        uint32_t vb[4];  // (keys 0-7, dims 16 d2..+7), (keys 8-15, ..), (0-7, +8..), (8-15, +8..)
        ldsm_x4_trans(sV + (cg >> 3) * kHalfBytes + key * 128 + (((cg & 7) ^ (key & 7)) << 4),
                      vb);
        if (masked) {
          vb[0] &= vm0;
          vb[1] &= vm1;
          vb[2] &= vm0;
          vb[3] &= vm1;
        }
        mma_bf16_16816(o[2 * d2], pa4, vb[0], vb[1]);
        mma_bf16_16816(o[2 * d2 + 1], pa4, vb[2], vb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
  if (__any_sync(0xffffffffu, *abort_flag)) return;

  // ---- rows out: sum the row sums over the 4 lanes of a row, normalise ------
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
  if (ra < rows) {
    __nv_bfloat16* dst =
        p.out + ((size_t)(row0 + ra / G) * p.num_q_heads + kvh * G + ra % G) * D + 2 * cq;
#pragma unroll
    for (int db = 0; db < D / 8; ++db)
      *reinterpret_cast<uint32_t*>(dst + 8 * db) = pack_bf16x2(o[db][0] * ia, o[db][1] * ia);
  }
  if (rbw < rows) {
    __nv_bfloat16* dst =
        p.out + ((size_t)(row0 + rbw / G) * p.num_q_heads + kvh * G + rbw % G) * D + 2 * cq;
#pragma unroll
    for (int db = 0; db < D / 8; ++db)
      *reinterpret_cast<uint32_t*>(dst + 8 * db) = pack_bf16x2(o[db][2] * ib, o[db][3] * ib);
  }
}

template <int D, bool kTma>
pa_status launch_rowblock(const CUtensorMap& mk, const CUtensorMap& mv, const MultiParams& prm,
                          int B, int num_kv_heads, int max_rows, cudaStream_t stream) {
  using L = RowSmem<D>;
  auto kern = rowblock_decode_kernel<D, kTma>;
  const int threads = (kRowWarps + 1) * 32;
  const pa_status s = prepare_kernel(reinterpret_cast<const void*>(kern), threads, L::kAlloc,
                                     nullptr);
  if (s != PA_OK) return s;
  const int nrb = (max_rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (nrb > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
  dim3 grid(nrb, num_kv_heads, B);
  kern<<<grid, threads, L::kAlloc, stream>>>(mk, mv, prm);
  return launch_status();
}

// ---------------------------------------------------------------------------
// the work-balanced persistent schedule
// ---------------------------------------------------------------------------

constexpr int kMaxCols = kMaxColumnWarps * 8;  // (token, head) columns of a unit
constexpr int kMultiBlocksPerSM = 4;           // the most a launch uses (workspace sizing)

struct BalMultiParams {
  const __nv_bfloat16* q;      // [R, Hq, D]
  const int32_t* q_start;      // [B + 1]
  const int32_t* block_tables;
  const int32_t* context_lens;
  __nv_bfloat16* out;          // [R, Hq, D]
  int* counters;               // [B * Hkv * kMaxColumnWarps], zero between launches
  float* rec_lse;              // [blocks][2][kMaxCols], base 2
  float* rec_o;                // [blocks][2][kMaxCols][D]
  TileSrc src;
  int max_blocks;
  int num_seqs;
  int num_q_heads;
  int group;
  float scale_log2;
};

template <int D, int NC, int NT>
struct BalMultiSmem {
  static constexpr int kStageBytes = TileGeom<D>::kStageBytes;
  static constexpr int kRingBytes = kMultiStages * kStageBytes;
  static constexpr int kOutOff = kRingBytes;                        // [NC][8 NT][D] fp32 staging
  static constexpr int kBarOff = kOutOff + NC * 8 * NT * D * 4;     // full, empty
  static constexpr int kMiscOff = kBarOff + 2 * kMultiStages * 8;   // abort flag
  static constexpr int kTotOff = kMiscOff + 16;                     // warp totals [NC + 1]
  static constexpr int kScanOff = kTotOff + ((NC + 1) * 4 + 15) / 16 * 16;  // S[B + 1]
  static constexpr int bytes(int B) { return kScanOff + (B + 1) * 4 + 1024; }
};

// NC column warps of 8 columns each. (Two groups of 8 columns a warp, the
// K/V fragments read once for both, measured slower on the speculative-verify
// batch: 0.556 against 0.542 ms; the per-warp state stays one group.)
template <int D, bool kTma, int NC, int BPS>
__global__ void __launch_bounds__((NC + 1) * 32, BPS)
    balanced_multi_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const BalMultiParams p) {
  constexpr int NT = 1;  // groups of 8 columns per warp
  using L = BalMultiSmem<D, NC, NT>;
  constexpr int CW = 8 * NT;
  using Gm = TileGeom<D>;
  constexpr int STAGES = kMultiStages;
  constexpr int kThreads = (NC + 1) * 32;
  constexpr int TT = kTile;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stage_out = reinterpret_cast<float*>(smem + L::kOutOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  int* warp_tot = reinterpret_cast<int*>(smem + L::kTotOff);
  int* S = reinterpret_cast<int*>(smem + L::kScanOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = p.num_seqs;
  const int hkv = p.src.num_kv_heads;
  const int G = p.group;
  const int cap = p.max_blocks << p.src.log2_bs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], kTma ? 1 : 32);
      mbar_init(&empty[s], NC);
    }
    *abort_flag = 0;
  }
  // a sequence with query rows holds its context's tiles; one without, none
  tile_prefix_sum_of<kThreads>(S, warp_tot, B, [&](int i) {
    return p.q_start[i + 1] > p.q_start[i] ? tiles_of<TT>(p.context_lens[i], cap) : 0;
  });
  fence_mbar_init();
  __syncthreads();

  // query rows of sequences with no context: zero rows
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (S[b + 1] != S[b]) continue;
    const int r0 = p.q_start[b], n = p.q_start[b + 1] - r0;
    uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)r0 * p.num_q_heads * D);
    for (int i = threadIdx.x; i < n * p.num_q_heads * D / 8; i += kThreads)
      dst[i] = make_uint4(0, 0, 0, 0);
  }

  const long long N = (long long)S[B] * hkv;
  const long long W = min((long long)gridDim.x, N);
  const int c = blockIdx.x;
  if (c >= W) return;
  const long long g0 = (long long)c * N / W, g1 = (long long)(c + 1) * N / W;
  const int count = (int)(g1 - g0);
  const uint32_t ring = smem_u32(smem);

  if (warp == NC) {
    // ------------------------------------------------------------ loader warp
    if (kTma && lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    Cursor ic;
    ic.seek(g0, S, B, hkv);
    int ic_ctx = 0, ic_nblk = 0, ic_b = -1;
    int tc_b = -1, tc_base = 0, tc_val = -1;
    int issued = 0;
    for (int j = 0; j < count; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag)) break;
      if (ic.b != ic_b) {
        ic_b = ic.b;
        ic_ctx = min(max(p.context_lens[ic.b], 0), cap);
        ic_nblk = (ic_ctx + p.src.block_size - 1) >> p.src.log2_bs;
      }
      const int stage = j % STAGES;
      if (j >= STAGES &&
          !__all_sync(0xffffffffu, mbar_wait(&empty[stage], ((j / STAGES) - 1) & 1))) {
        if (lane == 0) report(kErrWaitEmpty);
        *abort_flag = 1;
        break;
      }
      const int t0 = ic.t * TT;
      const int blk_first = t0 >> p.src.log2_bs;
      const int blk_last = (t0 + TT - 1) >> p.src.log2_bs;
      if (tc_b != ic.b || blk_first < tc_base || blk_last >= tc_base + 32) {  // warp-uniform
        tc_b = ic.b;
        tc_base = blk_first;
        const int idx = tc_base + lane;
        tc_val = idx < ic_nblk ? p.block_tables[(size_t)ic.b * p.max_blocks + idx] : -1;
      }
      issue_tile<D, kTma>(ring + stage * Gm::kStageBytes, &full[stage], &tmap_k, &tmap_v, p.src,
                          ic.kvh, t0, ic_ctx, ic_nblk, tc_base, tc_val, lane);
      ++issued;
      if (++ic.t == ic.n) ic.next_unit(S, B, hkv);
    }
    const int first = issued > STAGES ? issued - STAGES : 0;
    for (int j = first; j < issued; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[j % STAGES], (j / STAGES) & 1))) {
        if (lane == 0) report(kErrDrain);
        break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tk = 2 * (lane & 3);
  const int r0 = lane >> 2;
  float* buf = stage_out + (size_t)warp * CW * D;
  Cursor uc;
  uc.seek(g0, S, B, hkv);
  uint32_t qf[NT][D / 16][2];
  AttnState<D> st[NT];
  int lim_a[NT], lim_b[NT];
  int j0 = 0;
  while (j0 < count) {
    const int b = uc.b, kvh = uc.kvh;
    const int m = min(uc.n - uc.t, count - j0);  // this block's tiles of the unit
    const int ctx = min(max(__ldg(p.context_lens + b), 0), cap);
    const int row0 = __ldg(p.q_start + b);
    const int n = __ldg(p.q_start + b + 1) - row0;
    if (n * G > NC * CW && warp == 0 && lane == 0) report(kErrShape);
#pragma unroll
    for (int g8 = 0; g8 < NT; ++g8) {
      // B operand of Q^T for group g8: this lane's column is CW warp + 8 g8 + lane / 4
      const int cq = CW * warp + 8 * g8 + (lane >> 2);
      const int i = cq / G;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) qf[g8][ks][0] = qf[g8][ks][1] = 0u;
      if (i < n) {
        const unsigned int* rowp = reinterpret_cast<const unsigned int*>(
            p.q + ((size_t)(row0 + i) * p.num_q_heads + kvh * G + cq % G) * D + 2 * (lane & 3));
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          qf[g8][ks][0] = __ldg(rowp + ks * 8);
          qf[g8][ks][1] = __ldg(rowp + ks * 8 + 4);
        }
      }
      const int ca = CW * warp + 8 * g8 + tk;
      lim_a[g8] = ca / G < n ? ctx - n + ca / G : -1;
      lim_b[g8] = (ca + 1) / G < n ? ctx - n + (ca + 1) / G : -1;
      st[g8].reset();
    }
    for (int j = j0; j < j0 + m; ++j) {  // every column warp folds every tile
      if (__any_sync(0xffffffffu, *abort_flag)) break;
      const int stage = j % STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (j / STAGES) & 1))) {
        if (lane == 0) report(kErrWaitFull);
        *abort_flag = 1;
        break;
      }
      const uint32_t sK = ring + stage * Gm::kStageBytes;
      const int t0 = (uc.t + (j - j0)) * TT;
      const int valid = min(TT, ctx - t0);
      int va[NT], vb[NT];
#pragma unroll
      for (int g8 = 0; g8 < NT; ++g8) {
        va[g8] = max(0, min(valid, lim_a[g8] - t0 + 1));
        vb[g8] = max(0, min(valid, lim_b[g8] - t0 + 1));
      }
      attend_tile_causal_nt<D, NT>(st, sK, sK + Gm::kKVBytes, qf, valid, va, vb, p.scale_log2,
                                   lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (__any_sync(0xffffffffu, *abort_flag)) break;

    // ---- this warp's columns: rows, or records of a unit cut by a range -----
    const int ncols = min(CW, n * G - CW * warp);  // valid columns of this warp
    if (ncols > 0) {
      const long long U = (long long)hkv * S[b] + (long long)kvh * uc.n;
      const int c0 = owner_of(U, N, W), c1 = owner_of(U + uc.n - 1, N, W);
      const bool cut = c0 != c1;
      float la[NT], lb[NT];  // base-2 log-sum-exp of this lane's columns (-inf: no token)
#pragma unroll
      for (int g8 = 0; g8 < NT; ++g8) {
        st[g8].reduce_l();
        const float i0 = st[g8].l0 > 0.f ? 1.f / st[g8].l0 : 0.f;
        const float i1 = st[g8].l1 > 0.f ? 1.f / st[g8].l1 : 0.f;
        const int ja = 8 * g8 + tk, jb = ja + 1;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d0 = mt * 16 + r0;
          buf[ja * D + out_col(ja, d0)] = st[g8].o[mt][0] * i0;
          buf[jb * D + out_col(jb, d0)] = st[g8].o[mt][1] * i1;
          buf[ja * D + out_col(ja, d0 + 8)] = st[g8].o[mt][2] * i0;
          buf[jb * D + out_col(jb, d0 + 8)] = st[g8].o[mt][3] * i1;
        }
        la[g8] = st[g8].l0 > 0.f ? st[g8].m0 + log2f(st[g8].l0) : -INFINITY;
        lb[g8] = st[g8].l1 > 0.f ? st[g8].m1 + log2f(st[g8].l1) : -INFINITY;
      }
      __syncwarp();
      const int rec = 2 * c + (c == c0 ? 1 : 0);
      for (int jc = 0; jc < ncols; ++jc) {
        const int col = CW * warp + jc;
        const size_t r = (size_t)(row0 + col / G) * p.num_q_heads + kvh * G + col % G;
        float mine = -INFINITY;  // this lane's candidate for column jc's lse
#pragma unroll
        for (int g8 = 0; g8 < NT; ++g8)
          if ((jc >> 3) == g8) mine = (jc & 1) ? lb[g8] : la[g8];
        const float lse = __shfl_sync(0xffffffffu, mine, (jc >> 1) & 3);
        if (!cut) {
          for (int d4 = lane; d4 < D / 4; d4 += 32) {
            const float4 v = *reinterpret_cast<const float4*>(buf + jc * D + out_col(jc, 4 * d4));
            uint2 pk;
            pk.x = pack_bf16x2(v.x, v.y);
            pk.y = pack_bf16x2(v.z, v.w);
            *reinterpret_cast<uint2*>(p.out + r * D + 4 * d4) = pk;
          }
        } else {
          float* dst = p.rec_o + ((size_t)rec * kMaxCols + col) * D;
          for (int d4 = lane; d4 < D / 4; d4 += 32)
            *reinterpret_cast<float4*>(dst + 4 * d4) =
                *reinterpret_cast<const float4*>(buf + jc * D + out_col(jc, 4 * d4));
          if (lane == 0) p.rec_lse[rec * kMaxCols + col] = lse;
        }
      }
      if (cut) {
        // publish: the warp's record stores, then one lane's GPU-scope fence
        // and ticket (cumulative over what the warp wrote)
        __syncwarp();
        int ticket = 0;
        int* counter = p.counters + ((size_t)b * hkv + kvh) * kMaxColumnWarps + warp;
        if (lane == 0) {
          fence_acq_rel_gpu();
          ticket = atomicAdd(counter, 1);
          fence_acq_rel_gpu();
        }
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket == c1 - c0) {  // the last block on the unit merges the records
          for (int jc = 0; jc < ncols; ++jc) {
            const int col = CW * warp + jc;
            const size_t r = (size_t)(row0 + col / G) * p.num_q_heads + kvh * G + col % G;
            float M = -INFINITY;
            for (int cc = c0; cc <= c1; ++cc)
              M = fmaxf(M, __ldcg(p.rec_lse + (2 * cc + (cc == c0 ? 1 : 0)) * kMaxCols + col));
            for (int d4 = lane; d4 < D / 4; d4 += 32) {
              float Wsum = 0.f;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              if (M != -INFINITY) {
                for (int cc = c0; cc <= c1; ++cc) {
                  const int rr = 2 * cc + (cc == c0 ? 1 : 0);
                  const float wt = exp2f(__ldcg(p.rec_lse + rr * kMaxCols + col) - M);
                  const float4 v = __ldcg(reinterpret_cast<const float4*>(
                      p.rec_o + ((size_t)rr * kMaxCols + col) * D + 4 * d4));
                  Wsum += wt;
                  acc.x += wt * v.x; acc.y += wt * v.y; acc.z += wt * v.z; acc.w += wt * v.w;
                }
              }
              const float f = Wsum > 0.f ? 1.f / Wsum : 0.f;
              uint2 pk;
              pk.x = pack_bf16x2(acc.x * f, acc.y * f);
              pk.y = pack_bf16x2(acc.z * f, acc.w * f);
              *reinterpret_cast<uint2*>(p.out + r * D + 4 * d4) = pk;
            }
          }
          if (lane == 0) *counter = 0;
        }
      }
      __syncwarp();  // the staging buffer is read before the next unit's writes
    }
    j0 += m;
    uc.next_unit(S, B, hkv);
  }
}

struct MultiWsLayout {
  size_t counters, rec_lse, rec_o, total;
};

MultiWsLayout multi_ws_layout(int num_seqs, int num_kv_heads, int head_dim, int blocks) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  MultiWsLayout l;
  l.counters = 0;
  l.rec_lse = up((size_t)num_seqs * num_kv_heads * kMaxColumnWarps * sizeof(int));
  l.rec_o = l.rec_lse + up((size_t)blocks * 2 * kMaxCols * sizeof(float));
  l.total = l.rec_o + up((size_t)blocks * 2 * kMaxCols * head_dim * sizeof(float));
  return l;
}

template <int D, bool kTma, int NC, int BPS>
pa_status launch_bal_multi(const CUtensorMap& mk, const CUtensorMap& mv, const BalMultiParams& prm,
                           int sms, cudaStream_t stream) {
  auto kern = balanced_multi_kernel<D, kTma, NC, BPS>;
  const int smem = BalMultiSmem<D, NC, 1>::bytes(prm.num_seqs);
  if (smem > 227 * 1024) return PA_ERR_UNSUPPORTED;
  int per_sm = 0;
  const pa_status s =
      prepare_kernel(reinterpret_cast<const void*>(kern), (NC + 1) * 32, smem, &per_sm);
  if (s != PA_OK) return s;
  per_sm = per_sm > BPS ? BPS : per_sm;
  kern<<<sms * per_sm, (NC + 1) * 32, smem, stream>>>(mk, mv, prm);
  return launch_status();
}

// Column warps: the fewest of 1, 2, 4, 8 covering max_q_len * G columns.
template <int D, bool kTma>
pa_status launch_bal_multi_for(int cols, const CUtensorMap& mk, const CUtensorMap& mv,
                               const BalMultiParams& prm, int sms, cudaStream_t stream) {
  if (cols <= 8) return launch_bal_multi<D, kTma, 1, 4>(mk, mv, prm, sms, stream);
  if (cols <= 16) return launch_bal_multi<D, kTma, 2, 4>(mk, mv, prm, sms, stream);
  if (cols <= 32) return launch_bal_multi<D, kTma, 4, 4>(mk, mv, prm, sms, stream);
  return launch_bal_multi<D, kTma, 8, 2>(mk, mv, prm, sms, stream);
}

int multi_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
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

// PA_PREFILL_KERNEL=rowblock runs long chunks on the mma.sync row-block
// kernel instead of the tcgen05 one (read at every call).
bool prefill_rowblock_forced() {
  const char* v = std::getenv("PA_PREFILL_KERNEL");
  return v && std::strcmp(v, "rowblock") == 0;
}

// PA_MULTI_KERNEL=columns keeps short chunks over bf16 caches on the
// column-warp kernel instead of the tcgen05 one (read at every call).
bool columns_forced() {
  const char* v = std::getenv("PA_MULTI_KERNEL");
  return v && std::strcmp(v, "columns") == 0;
}

// The tcgen05 kernel takes a short-chunk launch (see verify_tc_supported).
bool use_verify_tc(int head_dim, int block_size, int group, int max_q_len, int split_tokens,
                   int num_q_rows, int num_q_heads) {
  return !columns_forced() && (long long)num_q_rows * num_q_heads < (1LL << 31) &&
         verify_tc_supported(head_dim, block_size, group, max_q_len, split_tokens);
}

// Device address of this unit's error word (looked up once per device).
unsigned int* multi_error_word() {
  static std::mutex mu;
  static std::map<int, unsigned int*> addr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = addr.find(dev);
  if (it != addr.end()) return it->second;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_multi_error) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  addr[dev] = static_cast<unsigned int*>(ptr);
  return static_cast<unsigned int*>(ptr);
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
  // more (token, head) rows than the n side holds: the row-block kernel
  // (no context split: its many row blocks fill the GPU)
  const bool long_chunk = (long long)max_q_len * G > kMaxColumnWarps * 8;
  if (long_chunk && split_tokens > 0) return PA_ERR_UNSUPPORTED;
  if ((long long)max_q_len * G > (1LL << 30)) return PA_ERR_UNSUPPORTED;
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
  MultiParams prm{};
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
  if (long_chunk && prefill_tc_supported(head_dim, block_size, G) && !prefill_rowblock_forced()) {
    unsigned int* err = multi_error_word();
    if (!err) return PA_ERR_CUDA;
    return launch_prefill_tc(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                             q_start, num_seqs, max_q_len, num_q_heads, num_kv_heads, head_dim,
                             block_size, num_blocks, scale, out, err, st);
  }
  if (long_chunk) {
    const int max_rows = max_q_len * G;
    if (head_dim == 128)
      return tma ? launch_rowblock<128, true>(mk, mv, prm, num_seqs, num_kv_heads, max_rows, st)
                 : launch_rowblock<128, false>(mk, mv, prm, num_seqs, num_kv_heads, max_rows, st);
    return tma ? launch_rowblock<64, true>(mk, mv, prm, num_seqs, num_kv_heads, max_rows, st)
               : launch_rowblock<64, false>(mk, mv, prm, num_seqs, num_kv_heads, max_rows, st);
  }
  if (use_verify_tc(head_dim, block_size, G, max_q_len, split_tokens, num_q_rows, num_q_heads)) {
    unsigned int* err = multi_error_word();
    if (!err) return PA_ERR_CUDA;
    return launch_verify_tc(q, k_cache, v_cache, block_tables,
                            max_blocks_per_seq, context_lens, q_start, num_seqs, max_q_len,
                            num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                            split_tokens, max_splits, part_out, part_lse, row_lens, out, err, st);
  }
  if (head_dim == 128)
    return tma ? launch_multi<128, true>(mk, mv, prm, nc, num_seqs, num_kv_heads, st)
               : launch_multi<128, false>(mk, mv, prm, nc, num_seqs, num_kv_heads, st);
  return tma ? launch_multi<64, true>(mk, mv, prm, nc, num_seqs, num_kv_heads, st)
             : launch_multi<64, false>(mk, mv, prm, nc, num_seqs, num_kv_heads, st);
}

extern "C" pa_status pa_decode_multi_fp8(
    const void* q, const void* k_codes, const void* v_codes, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, const int32_t* q_start, int32_t num_seqs, int32_t num_q_rows,
    int32_t max_q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int32_t num_blocks, float scale, int32_t split_tokens, int32_t max_splits,
    float* part_out, float* part_lse, int32_t* row_lens, void* out, void* stream) {
  using namespace pa;
  if (split_tokens < 0 || num_q_rows < 0 || max_q_len < 1) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_q_rows == 0) return PA_OK;
  pa_status s = check_decode_args(q, k_codes, v_codes, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale, out);
  if (s != PA_OK) return s;
  if (!q_start || !k_scale || !v_scale) return PA_ERR_INVALID_ARG;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;  // one 128-byte e4m3 row per token
  const int G = num_q_heads / num_kv_heads;
  // more (token, head) rows than the n side holds: the tcgen05 kernel
  // (no context split)
  const bool long_chunk = (long long)max_q_len * G > kMaxColumnWarps * 8;
  if (long_chunk && (split_tokens > 0 || !prefill_tc_supported(head_dim, block_size, G)))
    return PA_ERR_UNSUPPORTED;
  if ((long long)max_q_len * G > (1LL << 30)) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  if (split_tokens > 0) {
    if (split_tokens % kFp8Tile) return PA_ERR_INVALID_ARG;
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
  MultiParams prm{};
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.q_start = q_start;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.part_out = part_out;
  prm.part_lse = part_lse;
  prm.row_lens = row_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.src.k_cache = static_cast<const unsigned char*>(k_codes);
  prm.src.v_cache = static_cast<const unsigned char*>(v_codes);
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
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  if (long_chunk) {
    unsigned int* err = multi_error_word();
    if (!err) return PA_ERR_CUDA;
    return launch_prefill_tc_fp8(q, k_codes, v_codes, k_scale, v_scale, block_tables,
                                 max_blocks_per_seq, context_lens, q_start, num_seqs, max_q_len,
                                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                 scale, out, err, st);
  }
  const int nc = (max_q_len * G + 7) / 8;

  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  const bool tma = block_size >= 8;
  if (tma) {
    const long long rows = (long long)num_blocks * block_size;
    const int box_rows = block_size < kFp8Tile ? block_size : kFp8Tile;
    if (!make_cache_map(&mk, k_codes, num_kv_heads, head_dim, rows, box_rows, 1) ||
        !make_cache_map(&mv, v_codes, num_kv_heads, head_dim, rows, box_rows, 1))
      return PA_ERR_CUDA;
  }
  return tma ? launch_multi<128, true, true>(mk, mv, prm, nc, num_seqs, num_kv_heads, st)
             : launch_multi<128, false, true>(mk, mv, prm, nc, num_seqs, num_kv_heads, st);
}

extern "C" size_t pa_decode_multi_balanced_workspace_bytes(int32_t num_seqs,
                                                           int32_t num_kv_heads,
                                                           int32_t head_dim) {
  using namespace pa;
  const int sms = multi_sm_count();
  if (num_seqs <= 0 || num_kv_heads <= 0 || head_dim <= 0 || sms <= 0) return 0;
  return multi_ws_layout(num_seqs, num_kv_heads, head_dim, sms * kMultiBlocksPerSM).total;
}

extern "C" pa_status pa_decode_multi_balanced(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* q_start,
    int32_t num_seqs, int32_t num_q_rows, int32_t max_q_len, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
    void* workspace, size_t workspace_bytes, void* out, void* stream) {
  using namespace pa;
  if (num_q_rows < 0 || max_q_len < 1) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_q_rows == 0) return PA_OK;
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale, out);
  if (s != PA_OK) return s;
  if (!q_start) return PA_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if ((long long)max_q_len * G > kMaxCols) return PA_ERR_UNSUPPORTED;
  const int sms = multi_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const MultiWsLayout lay =
      multi_ws_layout(num_seqs, num_kv_heads, head_dim, sms * kMultiBlocksPerSM);
  if (!workspace || workspace_bytes < lay.total) return PA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (validating()) {
    s = check_tables(block_tables, max_blocks_per_seq, context_lens, num_seqs, num_blocks,
                     block_size, 0, 0, st);
    if (s != PA_OK) return s;
    s = check_q_start(q_start, context_lens, num_seqs, num_q_rows, max_q_len, st);
    if (s != PA_OK) return s;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  if (!columns_forced() &&
      verify_tc_balanced_supported(head_dim, block_size, G, max_q_len, num_seqs)) {
    unsigned int* err = multi_error_word();
    if (!err) return PA_ERR_CUDA;
    return launch_verify_tc_balanced(
        q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, q_start, num_seqs,
        max_q_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
        reinterpret_cast<int*>(ws + lay.counters), reinterpret_cast<float*>(ws + lay.rec_lse),
        reinterpret_cast<float*>(ws + lay.rec_o), kMaxCols, out, err, st);
  }
  BalMultiParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.q_start = q_start;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.counters = reinterpret_cast<int*>(ws + lay.counters);
  prm.rec_lse = reinterpret_cast<float*>(ws + lay.rec_lse);
  prm.rec_o = reinterpret_cast<float*>(ws + lay.rec_o);
  prm.src.k_cache = static_cast<const unsigned char*>(k_cache);
  prm.src.v_cache = static_cast<const unsigned char*>(v_cache);
  prm.src.num_kv_heads = num_kv_heads;
  prm.src.block_size = block_size;
  prm.src.log2_bs = ilog2(block_size);
  prm.src.num_blocks = num_blocks;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_seqs = num_seqs;
  prm.num_q_heads = num_q_heads;
  prm.group = G;
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
  const int cols = max_q_len * G;
  if (head_dim == 128)
    return tma ? launch_bal_multi_for<128, true>(cols, mk, mv, prm, sms, st)
               : launch_bal_multi_for<128, false>(cols, mk, mv, prm, sms, st);
  return tma ? launch_bal_multi_for<64, true>(cols, mk, mv, prm, sms, st)
             : launch_bal_multi_for<64, false>(cols, mk, mv, prm, sms, st);
}
