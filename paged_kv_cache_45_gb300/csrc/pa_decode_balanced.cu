// pa_decode_balanced.cu -- paged decode attention with a work-balanced,
// persistent schedule (sm_103a).
//
// Same result as pa_decode (softmax(scale * q K^T) V per query head over each
// sequence's paged context, "Text Generation Inference: Hugging Face's
// production-grade LLM inference server", sections "Under the Hood:
// PagedAttention" and "Under the Hood: Flash Attention"), scheduled for a
// continuously batched set of sequences whose lengths differ by 60x:
//
//   * the work is the list of TT-token tiles (16 for bf16, 32 for e4m3) of
//     every (sequence, KV head) unit, sequence-major; its length
//     N = Hkv * sum_b ceil(ctx_b / TT) is computed on the device by every
//     block from context_lens (a prefix sum in shared memory, pa_balance.cuh),
//     so the host needs neither the lengths nor a sync;
//   * each block of a persistent grid (kBlocksPerSM per SM) owns the
//     contiguous tile range [c N / C, (c + 1) N / C): every block streams the
//     same number of tiles (to one) whatever the length mix, and no block is
//     launched for an empty context split;
//   * inside a block, the structure of pa_decode: a loader warp streams the
//     range's K/V tiles through a ring of stages (TMA, or a cp.async gather
//     below block size 8), crossing unit boundaries without a pause, and the
//     consumer warps (four for bf16, two for e4m3) fold tiles round-robin,
//     each serving the whole GQA group;
//   * the fused step (pa_append_decode) also writes each sequence's new K/V
//     row: the warp that folds a unit's last tile stores that KV head's row
//     to the pool and patches it into the landed tile;
//   * at the end of each unit the consumer warps' states are merged through
//     shared memory. A unit inside one block's range is written as bf16. A
//     unit cut by a range boundary leaves one normalised fp32 partial + base-2
//     log-sum-exp per block; the block that arrives last on the unit's
//     counter (an atomic ticket, no waiting) merges them by log-sum-exp and
//     resets the counter to zero.
// The workspace (counters + partials) must be zero-filled before its first
// use; every call leaves the counters at zero again.

#include <math.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_balance.cuh"
#include "pa_tile.cuh"
#include "pagedkv.h"

namespace pa {
namespace {

__device__ unsigned int g_balanced_error;

__device__ __forceinline__ void report(unsigned int bits) { atomicOr(&g_balanced_error, bits); }

// Block shape: 4 consumer warps + 1 loader warp, a 4-stage ring, 4 blocks per
// SM (16 tiles in flight per SM). Chosen by measurement on the 70B-shape
// continuous batch over {4 warps x 8 stages x 2 blocks, 8 x 8 x 2}, which
// reached 71% and 66% of HBM peak against this shape's 93%.
// The ring depth must be a multiple of the consumer count: then every stage
// is always read by the same warp, which polls a stage's "full" barrier only
// after consuming that stage's previous tile, so the barrier is never more
// than one phase ahead of the parity the warp waits for.
constexpr int kConsumers = 4;
constexpr int kStages = 4;
// e4m3 tiles cost twice the math per byte: two consumer warps with two ring
// stages each overlap a warp's tile math with its next tile's load (measured
// on the 70B batch: 0.1875 ms per step against 0.2021 with 4 x 1)
constexpr int kConsumersFp8 = 2;
// (five stages, the most that fit four blocks per SM, need one more barrier
// wait per tile for a stage shared by both warps: 0.1666 against 0.1636 ms)
constexpr int kStagesFp8 = 4;
constexpr int kBlocksPerSM = 4;
constexpr int kMaxBlocksPerSM = kBlocksPerSM;
// The unit list goes KV head by KV head (PartitionT<true>): the blocks
// running together then read the heads of the same token rows together.
constexpr bool kHeadMajorLine = true;

struct BalParams {
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  __nv_bfloat16* out;
  int* counters;   // [num_seqs * Hkv]
  float* rec_lse;  // [blocks][2][8]     base-2 LSE of each partial
  float* rec_o;    // [blocks][2][8][D]  normalised partial outputs
  TileSrc src;
  int max_blocks;
  int num_seqs;
  int num_q_heads;
  int group;
  int unit_cost;  // tiles charged per unit for its merge (the Partition's K)
  float scale_log2;
  // fused append (pa_append_decode): one new K/V row per sequence
  const __nv_bfloat16* k_new;  // [num_seqs, Hkv, D]
  const __nv_bfloat16* v_new;
  const int64_t* slot_mapping;  // [num_seqs]
  unsigned char* k_dst;         // the caches, written at the slots
  unsigned char* v_dst;
  long long num_slots;
  // FP8 (e4m3) pools: per-KV-head scales, value = code * scale
  const float* k_scale;  // [Hkv]
  const float* v_scale;
};

constexpr int kMaxFp8Heads = 64;  // KV heads whose scales an FP8 block keeps in shared memory

// Tokens per K/V tile: e4m3 tiles hold 32 tokens so that a stage carries as
// many bytes (8 KB at head_dim 128) as a 16-token bf16 tile.
template <int EB>
__host__ __device__ constexpr int tile_tokens() { return EB == 1 ? kFp8Tile : kTile; }

template <int D, int NC, int STAGES, bool kMma = true, int EB = 2>
struct BalSmem {
  static constexpr int kStageBytes = TileGeom<D, EB, tile_tokens<EB>()>::kStageBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kMergeOff = kRingBytes;                                  // [NC][8][D] fp32
  static constexpr int kQOff = kMergeOff + NC * kMaxGroup * D * 4;             // [2][8][D] bf16
  static constexpr int kNewOff = kQOff + 2 * kMaxGroup * D * 2;  // [2][K,V][D] bf16 (fused append)
  static constexpr int kStatsOff = kNewOff + 2 * 2 * D * 2;                    // m, l [NC][8]
  static constexpr int kBarOff = kStatsOff + 2 * NC * kMaxGroup * 4;           // barriers
  static constexpr int kNumBars = 2 * STAGES + 4;  // full, empty, q_full[2], q_empty[2]
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // abort, ticket, stop, ctx[2]
  static constexpr int kTotOff = kMiscOff + 32;            // warp totals [NC + 1]
  // FMA ablation only: fp32 q rows [8][D] and per-warp weights [NC][8][16]
  static constexpr int kQf32Off = kTotOff + (NC + 1) * 4 + 12;
  static constexpr int kWeightsOff = kQf32Off + (kMma ? 0 : kMaxGroup * D * 4);
  static constexpr int kScaleOff = kWeightsOff + (kMma ? 0 : NC * kMaxGroup * kTile * 4);
  static constexpr int kScanOff = kScaleOff + (EB == 1 ? 2 * kMaxFp8Heads * 4 : 0);  // S[B+1]
  static constexpr int bytes(int B) { return kScanOff + (B + 1) * 4 + 1024; }
};

// Column of element d of head row h in the merge buffer: XOR-swizzled in
// groups of 8 floats so the 4 head rows one store instruction touches fall
// in 4 different bank groups (8-float groups stay contiguous for float4).
__device__ __forceinline__ int merge_col(int h, int d) { return d ^ ((h >> 1) << 3); }

// Four e4m3 codes (one u32, low byte first) of four bf16 values / scale.
__device__ __forceinline__ uint32_t quantize4_e4m3(uint2 v, float scale) {
  const float f0 = __fdiv_rn(bf16_lo(v.x), scale), f1 = __fdiv_rn(bf16_hi(v.x), scale);
  const float f2 = __fdiv_rn(bf16_lo(v.y), scale), f3 = __fdiv_rn(bf16_hi(v.y), scale);
  return f32x2_to_e4m3x2(f0, f1) | (f32x2_to_e4m3x2(f2, f3) << 16);
}

template <int D, bool kTma, int NC, int STAGES, int BPS, bool kMma, bool kAppend, bool kFp8>
__global__ void __launch_bounds__((NC + 1) * 32, BPS)
    balanced_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v, const BalParams p) {
  static_assert(STAGES % NC == 0, "each ring stage must belong to one consumer warp");
  static_assert(BPS <= kMaxBlocksPerSM, "workspace is sized for kMaxBlocksPerSM blocks per SM");
  static_assert(!kFp8 || (D == 128 && kMma), "FP8 tiles: head_dim 128, tensor-core math");
  constexpr int EB = kFp8 ? 1 : 2;  // bytes per cache element
  constexpr int TT = tile_tokens<EB>();
  using Gm = TileGeom<D, EB, TT>;
  using L = BalSmem<D, NC, STAGES, kMma, EB>;
  constexpr int kThreads = (NC + 1) * 32;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* merge = reinterpret_cast<float*>(smem + L::kMergeOff);
  __nv_bfloat16* sq = reinterpret_cast<__nv_bfloat16*>(smem + L::kQOff);
  float* stat_m = reinterpret_cast<float*>(smem + L::kStatsOff);
  float* stat_l = stat_m + NC * kMaxGroup;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + STAGES;
  uint64_t* q_full = empty + STAGES;
  uint64_t* q_empty = q_full + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  volatile int* ticket_s = abort_flag + 1;
  volatile int* stop_s = abort_flag + 2;
  volatile int* q_ctx = abort_flag + 3;  // [2]
  __nv_bfloat16* s_new = reinterpret_cast<__nv_bfloat16*>(smem + L::kNewOff);  // [2][2][D]
  int* warp_tot = reinterpret_cast<int*>(smem + L::kTotOff);
  int* S = reinterpret_cast<int*>(smem + L::kScanOff);
  float* qs32 = reinterpret_cast<float*>(smem + L::kQf32Off);     // FMA ablation only
  float* weights = reinterpret_cast<float*>(smem + L::kWeightsOff);
  float* sc_k = reinterpret_cast<float*>(smem + L::kScaleOff);  // FP8 only: [kMaxFp8Heads] x 2
  float* sc_v = sc_k + kMaxFp8Heads;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = p.num_seqs;
  const int hkv = p.src.num_kv_heads;
  const int G = p.group;
  const int cap = p.max_blocks << p.src.log2_bs;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], kTma ? 1 : 32);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], NC);
    }
    *abort_flag = 0;
  }
  if constexpr (kFp8) {
    for (int i = threadIdx.x; i < hkv; i += kThreads) {
      sc_k[i] = p.k_scale[i];
      sc_v[i] = p.v_scale[i];
    }
  }

  // ---- S[b] = tiles of the sequences before b (exclusive prefix sum) -------
  tile_prefix_sum<TT, kThreads>(S, warp_tot, p.context_lens, B, cap);
  fence_mbar_init();
  __syncthreads();

  // ---- sequences with no tokens get zero rows (and, fused, their append) ---
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (S[b + 1] != S[b]) continue;
    uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)b * p.num_q_heads * D);
    for (int i = threadIdx.x; i < p.num_q_heads * D / 8; i += kThreads)
      dst[i] = make_uint4(0, 0, 0, 0);
    if constexpr (kAppend) {
      const long long slot = p.slot_mapping[b];
      if (slot >= 0 && slot < p.num_slots) {
        if constexpr (kFp8) {  // quantize 4 values per thread
          const size_t quads = (size_t)hkv * D / 4;
          const uint2* ks = reinterpret_cast<const uint2*>(p.k_new) + (size_t)b * quads;
          const uint2* vs = reinterpret_cast<const uint2*>(p.v_new) + (size_t)b * quads;
          for (size_t i = threadIdx.x; i < quads; i += kThreads) {
            const int h = (int)(i / (D / 4));
            reinterpret_cast<uint32_t*>(p.k_dst)[slot * quads + i] = quantize4_e4m3(ks[i], sc_k[h]);
            reinterpret_cast<uint32_t*>(p.v_dst)[slot * quads + i] = quantize4_e4m3(vs[i], sc_v[h]);
          }
        } else {
          const size_t row = (size_t)hkv * D / 8;  // 16-byte chunks per pool row
          const uint4* ks = reinterpret_cast<const uint4*>(p.k_new) + (size_t)b * row;
          const uint4* vs = reinterpret_cast<const uint4*>(p.v_new) + (size_t)b * row;
          for (size_t i = threadIdx.x; i < row; i += kThreads) {
            reinterpret_cast<uint4*>(p.k_dst)[slot * row + i] = ks[i];
            reinterpret_cast<uint4*>(p.v_dst)[slot * row + i] = vs[i];
          }
        }
      }
    }
  }

  // ---- this block's tile range -----------------------------------------------
  PartitionT<kHeadMajorLine> part;
  part.init(S, B, hkv, p.unit_cost, gridDim.x);
  const int c = blockIdx.x;
  if (c >= part.W) return;
  long long g0, g1;
  part.range(c, S, B, hkv, g0, g1);
  const int count = (int)(g1 - g0);
  if (count == 0) return;
  const uint32_t ring = smem_u32(smem);
  const uint32_t q_bytes = (uint32_t)(G * D * 2);

  if (warp == NC) {
    // ------------------------------------------------------------ loader warp
    // Streams the range's K/V tiles and, ahead of each unit's first tile,
    // the unit's q rows and context length (double-buffered q slots).
    if (kTma && lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    CursorT<kHeadMajorLine> ic;
    ic.seek(g0, S, B, hkv);
    int ic_ctx = 0, ic_nblk = 0;
    int tc_b = -1, tc_base = 0, tc_val = -1;
    int issued = 0, units = 0, q_issued = 0;
    bool unit_start = true;
    for (int j = 0; j < count; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag)) break;
      if (unit_start) {
        if (ic_ctx == 0 || tc_b != ic.b) {
          ic_ctx = min(max(p.context_lens[ic.b], 0), cap);
          ic_nblk = (ic_ctx + p.src.block_size - 1) >> p.src.log2_bs;
        }
        const int slot = units & 1;
        if (units >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait(&q_empty[slot], ((units >> 1) - 1) & 1))) {
          if (lane == 0) report(kErrWaitEmpty);
          *abort_flag = 1;
          break;
        }
        if (lane == 0) {
          q_ctx[slot] = ic_ctx;
          if constexpr (kAppend) {
            // the unit's new K/V row, for the fused append
            mbar_arrive_expect_tx(&q_full[slot], q_bytes + 4 * D);
            const size_t row = ((size_t)ic.b * hkv + ic.kvh) * D;
            bulk_load(smem_u32(s_new + slot * 2 * D), p.k_new + row, 2 * D, &q_full[slot]);
            bulk_load(smem_u32(s_new + slot * 2 * D + D), p.v_new + row, 2 * D, &q_full[slot]);
          } else {
            mbar_arrive_expect_tx(&q_full[slot], q_bytes);
          }
          bulk_load(smem_u32(sq + slot * kMaxGroup * D),
                    p.q + ((size_t)ic.b * p.num_q_heads + ic.kvh * G) * D, q_bytes,
                    &q_full[slot]);
        }
        ++units;
        q_issued = units;
        unit_start = false;
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
      issue_tile<D, kTma, EB, TT>(ring + stage * Gm::kStageBytes, &full[stage], &tmap_k, &tmap_v,
                                  p.src, ic.kvh, t0, ic_ctx, ic_nblk, tc_base, tc_val, lane);
      ++issued;
      if (++ic.t == ic.n) {
        const int prev_b = ic.b;
        ic.next_unit(S, B, hkv);
        unit_start = true;
        if (ic.b != prev_b) ic_ctx = 0;  // reload for the new sequence
      }
    }
    // Drain: copies still in flight must land before the block may exit.
    const int first = issued > STAGES ? issued - STAGES : 0;
    for (int j = first; j < issued; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[j % STAGES], (j / STAGES) & 1))) {
        if (lane == 0) report(kErrDrain);
        break;
      }
    }
    for (int u = q_issued > 2 ? q_issued - 2 : 0; u < q_issued; ++u) {
      if (!__all_sync(0xffffffffu, mbar_wait(&q_full[u & 1], (u >> 1) & 1))) {
        if (lane == 0) report(kErrDrain);
        break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tid = threadIdx.x;  // 0 .. NC*32-1
  const int r0 = lane >> 2;
  const int tk = 2 * (lane & 3);
  CursorT<kHeadMajorLine> uc;
  uc.seek(g0, S, B, hkv);
  uint32_t qf[D / 16][2];
  AttnState<D> st;
  AttnStateFma<D> sf;  // the FMA ablation's state
  int j0 = 0;     // block-local index of the current unit's first tile
  int units = 0;  // units started (selects the q slot)
  while (j0 < count) {
    const int b = uc.b, kvh = uc.kvh;
    const int m = min(uc.n - uc.t, count - j0);  // this block's tiles of the unit
    const int slot = units & 1;
    int ctx = 0;
    long long new_slot = -1;
    uint2 k_piece = make_uint2(0, 0), v_piece = make_uint2(0, 0);
    if (__all_sync(0xffffffffu, mbar_wait(&q_full[slot], (units >> 1) & 1))) {
      ctx = q_ctx[slot];
      if constexpr (kAppend) {
        if (4 * lane < D) {
          k_piece = *reinterpret_cast<const uint2*>(s_new + slot * 2 * D + 4 * lane);
          v_piece = *reinterpret_cast<const uint2*>(s_new + slot * 2 * D + D + 4 * lane);
          if constexpr (kFp8) {  // quantized now: 4 codes in .x, fewer live registers
            k_piece.x = quantize4_e4m3(k_piece, sc_k[kvh]);
            v_piece.x = quantize4_e4m3(v_piece, sc_v[kvh]);
          }
        }
      }
      if constexpr (kMma) {
        if constexpr (kFp8)
          load_q_frags_fp8<D>(qf, sq + slot * kMaxGroup * D, G, lane);
        else
          load_q_frags_smem<D>(qf, sq + slot * kMaxGroup * D, G, lane);
      } else {
        const __nv_bfloat16* src = sq + slot * kMaxGroup * D;
        for (int i = tid; i < kMaxGroup * D; i += NC * 32)
          qs32[i] = i < G * D ? __bfloat162float(src[i]) : 0.f;
      }
    } else {
      if (lane == 0) report(kErrWaitFull);
      *abort_flag = 1;
    }
    if constexpr (!kMma) named_barrier_sync(1, NC * 32);  // fp32 q rows ready
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[slot]);
    ++units;
    if constexpr (kMma) st.reset(); else sf.reset();
    // Fused append: the warp that folds the unit's last tile (which holds the
    // new token, logical position ctx - 1) writes the new K/V row of this KV
    // head to the pool and patches it into that tile after the tile lands.
    // No other block reads that row in this step.
    bool owns_new = false;
    if constexpr (kAppend) {
      const int last = j0 + (uc.n - 1 - uc.t);  // block-local index of the unit's last tile
      owns_new = uc.n - uc.t <= count - j0 && last % NC == warp;
      // issued now, first used at the unit's last tile: the load overlaps the tiles
      if (owns_new) new_slot = __ldg(p.slot_mapping + b);
    }
    // tiles j0 .. j0+m-1, round-robin: tile j -> warp j % NC
    for (int j = j0 + ((warp - j0) % NC + NC) % NC; j < j0 + m; j += NC) {
      if (__any_sync(0xffffffffu, *abort_flag)) break;
      const int stage = j % STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (j / STAGES) & 1))) {
        if (lane == 0) report(kErrWaitFull);
        *abort_flag = 1;
        break;
      }
      const uint32_t sK = ring + stage * Gm::kStageBytes;
      const int t = uc.t + (j - j0);
      if constexpr (kAppend) {
        if (owns_new && t == uc.n - 1 && new_slot >= 0 && new_slot < p.num_slots) {
          if (4 * lane < D) {
            const int r = (ctx - 1) & (TT - 1);  // the new token's row in the tile
            if constexpr (kFp8) {
              // this lane's 4 dims quantized to 4 bytes: chunk lane / 4, byte 4 * (lane % 4)
              const uint32_t kq = k_piece.x, vq = v_piece.x;
              const int c = lane >> 2;
              const uint32_t off = (c >> 3) * Gm::kHalfStride + r * 128 +
                                   (((c & 7) ^ (r & 7)) << 4) + (lane & 3) * 4;
              asm volatile("st.shared.u32 [%0], %1;" ::"r"(sK + off), "r"(kq) : "memory");
              asm volatile("st.shared.u32 [%0], %1;" ::"r"(sK + Gm::kKVBytes + off), "r"(vq)
                           : "memory");
              const size_t g = ((size_t)new_slot * hkv + kvh) * D + 4 * lane;  // bytes
              *reinterpret_cast<uint32_t*>(p.k_dst + g) = kq;
              *reinterpret_cast<uint32_t*>(p.v_dst + g) = vq;
            } else {
              const int c = lane >> 1;  // 16-byte chunk of this lane's 8 bytes
              const uint32_t off = (c >> 3) * Gm::kHalfStride + r * 128 +
                                   (((c & 7) ^ (r & 7)) << 4) + (lane & 1) * 8;
              asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(sK + off), "r"(k_piece.x),
                           "r"(k_piece.y)
                           : "memory");
              asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(sK + Gm::kKVBytes + off),
                           "r"(v_piece.x), "r"(v_piece.y)
                           : "memory");
              const size_t g = (((size_t)new_slot * hkv + kvh) * D + 4 * lane) * 2;  // bytes
              *reinterpret_cast<uint2*>(p.k_dst + g) = k_piece;
              *reinterpret_cast<uint2*>(p.v_dst + g) = v_piece;
            }
          }
          __syncwarp();
        }
      }
      if constexpr (kFp8)
        attend_tile_fp8<D>(st, sK, sK + Gm::kKVBytes, qf, min(TT, ctx - t * TT),
                           p.scale_log2 * sc_k[kvh], lane);
      else if constexpr (kMma)
        attend_tile<D>(st, sK, sK + Gm::kKVBytes, qf, min(kTile, ctx - t * kTile), p.scale_log2,
                       lane);
      else
        attend_tile_fma<D>(sf, sK, sK + Gm::kKVBytes, qs32, weights + warp * kMaxGroup * kTile,
                           min(kTile, ctx - t * kTile), p.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }

    // ---- merge the NC warps' states of this unit --------------------------
    if constexpr (kMma) {
      st.reduce_l();
      if (lane < 4) {
        stat_m[warp * kMaxGroup + tk] = st.m0;
        stat_m[warp * kMaxGroup + tk + 1] = st.m1;
        stat_l[warp * kMaxGroup + tk] = st.l0;
        stat_l[warp * kMaxGroup + tk + 1] = st.l1;
      }
      float* base = merge + (size_t)warp * kMaxGroup * D;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        // output dims of this lane's two accumulator rows (FP8 tiles permute them)
        const int dA = kFp8 ? fp8_out_dim(mt, lane, false) : mt * 16 + r0;
        const int dB = kFp8 ? fp8_out_dim(mt, lane, true) : mt * 16 + r0 + 8;
        base[tk * D + merge_col(tk, dA)] = st.o[mt][0];
        base[(tk + 1) * D + merge_col(tk + 1, dA)] = st.o[mt][1];
        base[tk * D + merge_col(tk, dB)] = st.o[mt][2];
        base[(tk + 1) * D + merge_col(tk + 1, dB)] = st.o[mt][3];
      }
    } else {
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h)  // static indices keep sf in registers
        if (lane == h) {
          stat_m[warp * kMaxGroup + h] = sf.m[h];
          stat_l[warp * kMaxGroup + h] = sf.l[h];
        }
      float* base = merge + (size_t)warp * kMaxGroup * D;
      constexpr int kCols = D / 32;
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h)
#pragma unroll
        for (int jc = 0; jc < kCols; ++jc)
          base[h * D + merge_col(h, kCols * lane + jc)] = sf.o[h][jc];
    }
    named_barrier_sync(1, NC * 32);
    // one snapshot of the abort flag decides, for every consumer warp alike,
    // whether to stop after this unit (the loader may set it at any time)
    if (tid == 0) *stop_s = *abort_flag;

    const long long U = part.pos(S, hkv, b, kvh, uc.n, 0);
    const int c0 = part.owner(U), c1 = part.owner(U + uc.n - 1);
    const bool cut = c0 != c1;
    const int rec = 2 * c + (c == c0 ? 1 : 0);
    __nv_bfloat16* orow = p.out + ((size_t)b * p.num_q_heads + kvh * G) * D;
    constexpr int kC8 = D / 8;
    for (int idx = tid; idx < G * kC8; idx += NC * 32) {
      const int g = idx / kC8, c8 = idx % kC8;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, stat_m[w * kMaxGroup + g]);
      float Lsum = 0.f, acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float wt = exp2f(stat_m[w * kMaxGroup + g] - M);
        Lsum += wt * stat_l[w * kMaxGroup + g];
        const float4* src = reinterpret_cast<const float4*>(
            merge + ((size_t)w * kMaxGroup + g) * D + merge_col(g, c8 * 8));
        const float4 u = src[0], v = src[1];
        acc[0] += wt * u.x; acc[1] += wt * u.y; acc[2] += wt * u.z; acc[3] += wt * u.w;
        acc[4] += wt * v.x; acc[5] += wt * v.y; acc[6] += wt * v.z; acc[7] += wt * v.w;
      }
      // divisor of the output values: the running sum (and, FP8, over v_scale)
      const float Ld = kFp8 ? Lsum / sc_v[kvh] : Lsum;
      if (!cut) {
        uint4 pk;
        pk.x = pack_bf16x2(acc[0] / Ld, acc[1] / Ld);
        pk.y = pack_bf16x2(acc[2] / Ld, acc[3] / Ld);
        pk.z = pack_bf16x2(acc[4] / Ld, acc[5] / Ld);
        pk.w = pack_bf16x2(acc[6] / Ld, acc[7] / Ld);
        *reinterpret_cast<uint4*>(orow + (size_t)g * D + c8 * 8) = pk;
      } else {
        float4* dst = reinterpret_cast<float4*>(p.rec_o + ((size_t)rec * kMaxGroup + g) * D + c8 * 8);
        dst[0] = make_float4(acc[0] / Ld, acc[1] / Ld, acc[2] / Ld, acc[3] / Ld);
        dst[1] = make_float4(acc[4] / Ld, acc[5] / Ld, acc[6] / Ld, acc[7] / Ld);
        if (c8 == 0) p.rec_lse[rec * kMaxGroup + g] = M + log2f(Lsum);
      }
    }
    if (cut) {
      // Publish this block's partial: block barrier, then one thread's GPU-scope
      // fence + ticket (the fence is cumulative over the block's stores).
      named_barrier_sync(1, NC * 32);
      if (tid == 0) {
        fence_acq_rel_gpu();
        *ticket_s = atomicAdd(&p.counters[b * hkv + kvh], 1);
        fence_acq_rel_gpu();
      }
      named_barrier_sync(1, NC * 32);
      if (*ticket_s == c1 - c0) {
        // last block on this unit: merge every block's partial by log-sum-exp
        for (int idx = tid; idx < G * (D / 4); idx += NC * 32) {
          const int g = idx / (D / 4), c4 = idx % (D / 4);
          float M = -INFINITY;
          for (int cc = c0; cc <= c1; ++cc)
            M = fmaxf(M, __ldcg(p.rec_lse + (2 * cc + (cc == c0 ? 1 : 0)) * kMaxGroup + g));
          float Wsum = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int cc = c0; cc <= c1; ++cc) {
            const int r = 2 * cc + (cc == c0 ? 1 : 0);
            const float wt = exp2f(__ldcg(p.rec_lse + r * kMaxGroup + g) - M);
            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                p.rec_o + ((size_t)r * kMaxGroup + g) * D + c4 * 4));
            Wsum += wt;
            acc.x += wt * v.x; acc.y += wt * v.y; acc.z += wt * v.z; acc.w += wt * v.w;
          }
          uint2 pk;
          pk.x = pack_bf16x2(acc.x / Wsum, acc.y / Wsum);
          pk.y = pack_bf16x2(acc.z / Wsum, acc.w / Wsum);
          *reinterpret_cast<uint2*>(orow + (size_t)g * D + c4 * 4) = pk;
        }
        if (tid == 0) p.counters[b * hkv + kvh] = 0;
      }
    }
    named_barrier_sync(1, NC * 32);  // the merge buffer is free again
    if (*stop_s) break;
    j0 += m;
    uc.next_unit(S, B, hkv);
  }
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

struct WsLayout {
  size_t counters, rec_lse, rec_o, total;
};

WsLayout ws_layout(int num_seqs, int num_kv_heads, int head_dim, int blocks) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  WsLayout l;
  l.counters = 0;
  l.rec_lse = up((size_t)num_seqs * num_kv_heads * sizeof(int));
  l.rec_o = l.rec_lse + up((size_t)blocks * 2 * kMaxGroup * sizeof(float));
  l.total = l.rec_o + (size_t)blocks * 2 * kMaxGroup * head_dim * sizeof(float);
  return l;
}

template <int D, bool kTma, int NC, int STAGES, int BPS, bool kMma, bool kAppend,
          bool kFp8 = false>
pa_status launch_shape(const CUtensorMap& mk, const CUtensorMap& mv, const BalParams& prm, int sms,
                       cudaStream_t stream) {
  auto kern = balanced_decode_kernel<D, kTma, NC, STAGES, BPS, kMma, kAppend, kFp8>;
  const int smem = BalSmem<D, NC, STAGES, kMma, kFp8 ? 1 : 2>::bytes(prm.num_seqs);
  if (smem > 227 * 1024) return PA_ERR_UNSUPPORTED;
  int per_sm = 0;
  const pa_status s = prepare_kernel(reinterpret_cast<const void*>(kern), (NC + 1) * 32, smem,
                                     &per_sm);
  if (s != PA_OK) return s;
  per_sm = per_sm > BPS ? BPS : per_sm;
  kern<<<sms * per_sm, (NC + 1) * 32, smem, stream>>>(mk, mv, prm);
  return launch_status();
}

// Tiles charged per (sequence, KV head) unit in the block ranges, for the
// merge at the unit's end (measured on the 70B-shape continuous batch,
// head-major line, charges 0..4: bf16 0.2589 / 0.2567 / 0.2556 / 0.2554 /
// 0.2554 ms, e4m3 0.1646 / 0.1615 / 0.1589 / 0.1578 / 0.1587 ms).
// PA_BALANCE_UNIT_COST=<n> overrides it (read once), for tuning.
constexpr int kUnitCostBf16 = 2;
constexpr int kUnitCostFp8 = 3;
int unit_cost(bool fp8) {
  static const int over = [] {
    const char* v = std::getenv("PA_BALANCE_UNIT_COST");
    return v && *v ? std::atoi(v) : -1;
  }();
  if (over >= 0 && over <= 64) return over;
  return fp8 ? kUnitCostFp8 : kUnitCostBf16;
}

// PA_DECODE_MATH=fma selects the CUDA-core ablation of the tile math (kept
// to measure what the tensor-core form buys); anything else, the default.
bool fma_ablation() {
  static const bool on = [] {
    const char* v = std::getenv("PA_DECODE_MATH");
    return v && std::strcmp(v, "fma") == 0;
  }();
  return on;
}

template <int D, bool kTma>
pa_status launch_balanced(const CUtensorMap& mk, const CUtensorMap& mv, const BalParams& prm,
                          int sms, cudaStream_t stream) {
  if (prm.k_scale) {
    if constexpr (D == 128) {
      if (prm.slot_mapping)
        return launch_shape<D, kTma, kConsumersFp8, kStagesFp8, kBlocksPerSM, true, true, true>(
            mk, mv, prm, sms, stream);
      return launch_shape<D, kTma, kConsumersFp8, kStagesFp8, kBlocksPerSM, true, false, true>(
          mk, mv, prm, sms, stream);
    } else {
      return PA_ERR_UNSUPPORTED;
    }
  }
  if (prm.slot_mapping)
    return launch_shape<D, kTma, kConsumers, kStages, kBlocksPerSM, true, true>(mk, mv, prm, sms,
                                                                              stream);
  if (fma_ablation())  // its larger shared-memory footprint fits 3 blocks per SM
    return launch_shape<D, kTma, kConsumers, kStages, 3, false, false>(mk, mv, prm, sms, stream);
  return launch_shape<D, kTma, kConsumers, kStages, kBlocksPerSM, true, false>(mk, mv, prm, sms,
                                                                             stream);
}

// ---- built-in scratch for callers that cannot allocate device memory ------
// A fixed 6 MiB array that every device loading this library keeps until the
// process exits. In host code `g_static_scratch` names a host-side stand-in,
// not the device array, so its device address is looked up once per device
// (with that device current) and cached.
constexpr size_t kStaticScratchBytes = size_t(6) << 20;
constexpr int kMaxDevices = 64;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device, or nullptr.
void* static_scratch(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) {
      cudaGetLastError();  // leave no error behind for the next launch check
      return nullptr;
    }
    g_static_ptr[dev] = ptr;
  }
  return g_static_ptr[dev];
}

}  // namespace

unsigned int take_balanced_errors() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_balanced_error, sizeof(v)) != cudaSuccess) return 0x80000000u;
  if (v) cudaMemcpyToSymbol(g_balanced_error, &zero, sizeof(zero));
  return v;
}

}  // namespace pa

extern "C" size_t pa_decode_balanced_workspace_bytes(int32_t num_seqs, int32_t num_kv_heads,
                                                     int32_t head_dim) {
  using namespace pa;
  const int sms = sm_count();
  if (num_seqs <= 0 || num_kv_heads <= 0 || head_dim <= 0 || sms <= 0) return 0;
  return ws_layout(num_seqs, num_kv_heads, head_dim, sms * kMaxBlocksPerSM).total;
}

namespace pa {
namespace {

// Shared body of pa_decode_balanced and pa_append_decode (k_new == nullptr:
// no fused append).
pa_status balanced_entry(const void* q, const void* k_new, const void* v_new,
                         const int64_t* slot_mapping, void* k_cache, void* v_cache,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, float scale, void* workspace, size_t workspace_bytes,
                         void* out, void* stream, const float* k_scale = nullptr,
                         const float* v_scale = nullptr) {
  if (num_seqs == 0) return PA_OK;
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale, out);
  if (s != PA_OK) return s;
  const bool fused = k_new != nullptr;
  if (fused && (!v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)))
    return PA_ERR_INVALID_ARG;
  const bool fp8 = k_scale != nullptr;
  if (fp8) {
    if (!v_scale) return PA_ERR_INVALID_ARG;
    if (head_dim != 128 || num_kv_heads > kMaxFp8Heads) return PA_ERR_UNSUPPORTED;
  }
  const int sms = sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const WsLayout lay = ws_layout(num_seqs, num_kv_heads, head_dim, sms * kMaxBlocksPerSM);
  if (!workspace || workspace_bytes < lay.total) return PA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (validating()) {
    s = check_tables(block_tables, max_blocks_per_seq, context_lens, num_seqs, num_blocks,
                     block_size, 0, 0, st);
    if (s != PA_OK) return s;
  }

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  BalParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
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
  prm.group = num_q_heads / num_kv_heads;
  prm.unit_cost = unit_cost(fp8);
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  prm.k_new = static_cast<const __nv_bfloat16*>(k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(v_new);
  prm.slot_mapping = fused ? slot_mapping : nullptr;
  prm.k_dst = static_cast<unsigned char*>(k_cache);
  prm.v_dst = static_cast<unsigned char*>(v_cache);
  prm.num_slots = (long long)num_blocks * block_size;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;

  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  const bool tma = block_size >= 8;
  if (tma) {
    const long long rows = (long long)num_blocks * block_size;
    const int tt = fp8 ? tile_tokens<1>() : tile_tokens<2>();  // tokens per tile
    const int box_rows = block_size < tt ? block_size : tt;
    const int eb = fp8 ? 1 : 2;
    if (!make_cache_map(&mk, k_cache, num_kv_heads, head_dim, rows, box_rows, eb) ||
        !make_cache_map(&mv, v_cache, num_kv_heads, head_dim, rows, box_rows, eb))
      return PA_ERR_CUDA;
  }
  if (head_dim == 128)
    return tma ? launch_balanced<128, true>(mk, mv, prm, sms, st)
               : launch_balanced<128, false>(mk, mv, prm, sms, st);
  return tma ? launch_balanced<64, true>(mk, mv, prm, sms, st)
             : launch_balanced<64, false>(mk, mv, prm, sms, st);
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_balanced(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                        float scale, void* workspace, size_t workspace_bytes,
                                        void* out, void* stream) {
  return pa::balanced_entry(q, nullptr, nullptr, nullptr, const_cast<void*>(k_cache),
                            const_cast<void*>(v_cache), block_tables, max_blocks_per_seq,
                            context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            block_size, num_blocks, scale, workspace, workspace_bytes, out, stream);
}

extern "C" pa_status pa_append_decode(const void* q, const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                      float scale, void* workspace, size_t workspace_bytes,
                                      void* out, void* stream) {
  if (!k_new) return PA_ERR_INVALID_ARG;
  return pa::balanced_entry(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                            max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, scale, workspace, workspace_bytes,
                            out, stream);
}

extern "C" pa_status pa_decode_balanced_fp8(const void* q, const void* k_cache,
                                            const void* v_cache, const float* k_scale,
                                            const float* v_scale, const int32_t* block_tables,
                                            int32_t max_blocks_per_seq,
                                            const int32_t* context_lens, int32_t num_seqs,
                                            int32_t num_q_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t block_size,
                                            int32_t num_blocks, float scale, void* workspace,
                                            size_t workspace_bytes, void* out, void* stream) {
  if (num_seqs == 0) return PA_OK;
  if (!k_scale || !v_scale) return PA_ERR_INVALID_ARG;
  return pa::balanced_entry(q, nullptr, nullptr, nullptr, const_cast<void*>(k_cache),
                            const_cast<void*>(v_cache), block_tables, max_blocks_per_seq,
                            context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                            block_size, num_blocks, scale, workspace, workspace_bytes, out, stream,
                            k_scale, v_scale);
}

extern "C" pa_status pa_append_decode_fp8(const void* q, const void* k_new, const void* v_new,
                                          const int64_t* slot_mapping, void* k_cache,
                                          void* v_cache, const float* k_scale,
                                          const float* v_scale, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t num_seqs,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size,
                                          int32_t num_blocks, float scale, void* workspace,
                                          size_t workspace_bytes, void* out, void* stream) {
  if (num_seqs == 0) return PA_OK;
  if (!k_new || !k_scale || !v_scale) return PA_ERR_INVALID_ARG;
  return pa::balanced_entry(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                            max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, scale, workspace, workspace_bytes,
                            out, stream, k_scale, v_scale);
}

extern "C" pa_status pa_decode_balanced_static(const void* q, const void* k_cache,
                                               const void* v_cache, const int32_t* block_tables,
                                               int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, int32_t num_seqs,
                                               int32_t num_q_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t block_size,
                                               int32_t num_blocks, float scale, void* out,
                                               void* stream) {
  using namespace pa;
  if (num_seqs == 0) return PA_OK;
  pa_status s = check_decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, scale, out);
  if (s != PA_OK) return s;
  const int sms = sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const WsLayout lay = ws_layout(num_seqs, num_kv_heads, head_dim, sms * kMaxBlocksPerSM);
  if (lay.total > kStaticScratchBytes) return PA_ERR_WORKSPACE;  // beyond the built-in 6 MiB
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  unsigned char* scratch = static_cast<unsigned char*>(static_scratch(dev));
  if (!scratch) return PA_ERR_CUDA;
  // The array keeps whatever the previous call left; the per-unit counters
  // must start at zero, so clear them on this call's stream first.
  if (cudaMemsetAsync(scratch + lay.counters, 0, (size_t)num_seqs * num_kv_heads * sizeof(int),
                      as_stream(stream)) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  return pa_decode_balanced(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                            num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                            scale, scratch, kStaticScratchBytes, out, stream);
}
