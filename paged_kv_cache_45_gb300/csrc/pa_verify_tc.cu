// pa_verify_tc.cu -- a few new query tokens per sequence under the causal
// mask on the fifth-generation tensor cores of sm_103a, with the keys on the
// MMA's M side.
//
// The drafted tokens plus one that a speculative step verifies in one pass
// ("How to Speed Up LLM Inference: KV Cache to Production Serving", section
// "Speculative decoding: more than one token per weight-read"), or a short
// chunk of a prompt ("Text Generation Inference: Hugging Face's
// production-grade LLM inference server", section "Advanced Pattern: Chunked
// Prefill (TGI v3)"), give sequence b n_b query tokens, the last n_b
// positions of its context after the append; token i (position
// ctx_b - n_b + i) attends to positions 0 .. ctx_b - n_b + i through the
// sequence's block table ("Text Generation Inference ...", section
// "PagedAttention").
//
// pa_decode_multi's column-warp kernel puts the n_b * G (token, head) columns
// of a (sequence, KV head) unit on the n = 8 side of warp MMAs, so every
// column warp folds every K/V tile and re-reads the tile's fragments from
// shared memory. Here (bf16 caches; e4m3 pools keep the column-warp kernel)
// one MMA per product covers the unit, the 128 keys of a tile on M and the
// unit's columns (at most 32) on N:
//   S^T  = K_j Q^T       A = the K tile (K-major), B = Q as 32 K-major rows
//   O^T += V_j^T P_j^T   A = the V tile read M-major (its rows are keys, each
//                        holding the head dims), B = P as 32 K-major rows
// with S^T and O^T in tensor memory (32 columns each). Thread k of the softmax
// warpgroup reads key k's 32 scores; a column's maximum over the tile comes
// from a shuffle transpose-reduction in each warp (lane l ends with column l)
// and the four warps' partials in shared memory; the weights go to shared
// memory as P (2-byte stores, one per key and column); each thread keeps
// partial row sums for its key and the column sums are reduced once, at the
// end.
//
// A persistent launch, one block per SM, in two schedules. Split mode
// (pa_decode_multi): the (sequence, context split, KV head) units go round
// robin over the blocks. Balanced mode (pa_decode_multi_balanced): every
// block an equal range of the 128-key tiles of all (sequence, KV head) units,
// on a line ordered KV head by KV head (so the blocks running together read
// a token row's heads together); a unit cut by ranges leaves per-block
// records in the caller's workspace, and the epilogue warp with the last
// ticket on it merges them (log-sum-exp), so one launch needs no reduce.
// Every warp role walks the block's items in the same order with counters
// that run on across items, so the loads of the next item overlap the work
// of the current one. Warps:
//   0     loader: K_j and V_j (128 keys each) of every item in turn through a
//         ring of 32 KB operand slots (6; 5 in balanced mode, whose prefix sum
//         over the sequences takes the room of the sixth), one 4-D TMA box per paged
//         block, lane i issuing box i (the slot layout of the chunked-prefill
//         kernel);
//   1     allocates 128 TMEM columns (two S^T and two O^T buffers of 32); one
//         lane issues, for tile jg of the block, S(jg) into S^T buffer jg % 2
//         and then PV(jg - 1), so the softmax of one tile overlaps the
//         products of its neighbours; the pipe runs in issue order, so S(jg)
//         finished means PV(jg - 2) finished (P buffer jg % 2 is free);
//   2-5   the softmax warpgroup (TMEM lane quarter = warp % 4), one key of
//         the tile per thread; hands each unit's column sums and maxima on;
//   6-9   epilogue: stages Q of the items two ahead (two Q buffers), writes
//         each item's outputs from its O^T buffer (two, alternating by
//         item) or its record, zero rows and per-row context lengths.
// Arithmetic: bf16 MMA operands with fp32 accumulation, weights rounded to
// bf16 and their rounded values summed, as in the column-warp kernel; a column's
// running max moves only when a tile's max exceeds it by more than 2^8 (the
// final division uses the same max, so the result is the softmax either way).
// Outputs: bf16 rows (one split) or fp32 partials and natural-log LSEs for
// pa_decode_splitk_reduce, with the per-row context lengths in row_lens.

#include <cudaTypedefs.h>
#include <math.h>

#include <cstring>

#include "pa_balance.cuh"
#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_tc_common.cuh"
#include "pa_umma.cuh"
#include "pagedkv.h"

namespace pa {
namespace {

constexpr int kVfCols = 32;            // (token, head) columns of a unit: the MMAs' N
constexpr int kVfSoftmaxWarps = 4;     // warps 2-5
constexpr int kVfEpiWarps = 4;         // warps 6-9
constexpr int kVfFirstSoftmax = 2;
constexpr int kVfFirstEpi = kVfFirstSoftmax + kVfSoftmaxWarps;
constexpr int kVfThreads = (kVfFirstEpi + kVfEpiWarps) * 32;
constexpr float kVfRescaleLog2 = 8.0f;   // move a column's max when it grows by > 2^8
constexpr int kVfPanel = kVfCols * 128;  // Q and P: bytes of one 64-element panel
constexpr int kVfOpBytes = 2 * kVfPanel; // one Q or P buffer (two panels)
constexpr uint32_t kVfTmemCols = 4 * kVfCols;  // S^T x 2, O^T x 2

// kBal: the balanced schedule (a range of tiles per block), whose per-block
// prefix sum over the sequences takes the room of one ring slot.
template <bool kBal>
struct VfSmem {
  static constexpr int kSlots = kBal ? 5 : 6;                 // K/V operand slots of 32 KB
  static constexpr int kSlotBytes = TcShape<128>::kKvBytes;
  static constexpr int kRing = 0;
  static constexpr int kQ = kRing + kSlots * kSlotBytes;      // 2 x Q: [panel][column][128 B]
  static constexpr int kP = kQ + 2 * kVfOpBytes;              // 2 x P: [key panel][column][128 B]
  static constexpr int kRed = kP + 2 * kVfOpBytes;            // 2 x [warp][column] fp32 maxima
  static constexpr int kLm = kRed + 2 * kVfSoftmaxWarps * kVfCols * 4;  // 2 x (l [4][32], m [32])
  static constexpr int kLmFloats = (kVfSoftmaxWarps + 1) * kVfCols;
  static constexpr int kBar = kLm + 2 * kLmFloats * 4;
  // full[S], empty[S], q_ready[2], s_full[2], p_full[2], lm_full[2], o_full[2],
  // o_free[2], pv_done[2], red_full, mma_done
  static constexpr int kNumBars = 2 * kSlots + 14 + 2;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kFlag = kTmemSlot + 8;
  static constexpr int kTot = kFlag + 8;                      // balanced: warp totals of the scan
  static constexpr int kScan = kTot + 48;                     // balanced: S[B + 1]
  // the base must be 1024-byte aligned (checked)
  static constexpr int bytes(int B) { return kScan + (kBal ? (B + 1) * 4 : 0); }
};
constexpr int kVfMaxBalSeqs = 8192;  // sequences whose prefix sum fits beside the 5-slot ring
static_assert(VfSmem<false>::kQ % 1024 == 0 && VfSmem<false>::kP % 1024 == 0 &&
                  VfSmem<true>::kQ % 1024 == 0 && VfSmem<true>::kP % 1024 == 0,
              "swizzled operands start on 1024-byte boundaries");
static_assert(VfSmem<false>::bytes(0) <= 232448 && VfSmem<true>::bytes(kVfMaxBalSeqs) <= 232448,
              "over the 227 KB of shared memory per block");

struct VfParams {
  const __nv_bfloat16* q;       // [R, Hq, 128]
  const int32_t* q_start;       // [B + 1]
  const int32_t* block_tables;  // [B, max_blocks]
  const int32_t* context_lens;  // [B]
  __nv_bfloat16* out;           // [R, Hq, 128]
  float* part_out;              // [R, Hq, S, 128], split mode
  float* part_lse;              // [R, Hq, S]
  int32_t* row_lens;            // [R]
  unsigned int* err;            // device error word
  int num_seqs;
  int num_kv_heads;
  int max_blocks;
  int num_q_heads;
  int group;
  int max_q_len;
  int block_size;
  int log2_bs;
  int box_rows;                 // min(block_size, 128)
  int num_blocks;
  int split_tokens;             // 0 or a multiple of 128
  int max_splits;               // 1 when split_tokens is 0
  float scale_log2;
  // balanced schedule: the records of units cut by block ranges
  int* counters;                // [B * Hkv * 8] tickets, zero between launches
  float* rec_lse;               // [blocks][2][rec_cols], base 2
  float* rec_o;                 // [blocks][2][rec_cols][128]
  int rec_cols;
};

// A (sequence, split, KV head) unit of the launch: unit u is sequence
// u / (S Hkv), split (u / Hkv) % S, KV head u % Hkv (the KV heads of one
// sequence and split on neighbouring blocks).
struct VfUnit {
  int b, split, kvh;
  int row0, n, nG;      // query rows row0 .. row0 + n - 1; columns c = i G + g < nG
  int ctx, t_begin, t_end;
  int n_tiles;          // 128-key tiles of [t_begin, t_end); 0: nothing to attend
  bool bad;             // more tokens than the launch was sized for (skipped, reported)
  // balanced schedule: a segment of the unit (b, kvh), whose first and last
  // tiles the blocks c0 and c1 own; cut: c0 != c1, partial records merged
  bool cut;
  int c0, c1;
};

__device__ __forceinline__ VfUnit vf_unit(const VfParams& p, int u) {
  VfUnit w;
  const int per_seq = p.max_splits * p.num_kv_heads;
  w.b = u / per_seq;
  const int r = u - w.b * per_seq;
  w.split = r / p.num_kv_heads;
  w.kvh = r - w.split * p.num_kv_heads;
  w.row0 = p.q_start[w.b];
  w.n = p.q_start[w.b + 1] - w.row0;
  w.nG = w.n * p.group;
  int ctx = p.context_lens[w.b];
  const int cap = p.max_blocks << p.log2_bs;
  w.ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  w.t_begin = 0;
  w.t_end = w.ctx;
  if (p.split_tokens > 0) {
    w.t_begin = w.split * p.split_tokens;
    w.t_end = min(w.t_begin + p.split_tokens, w.ctx);
  }
  w.bad = w.n > p.max_q_len || w.nG > kVfCols;
  w.n_tiles = (w.n > 0 && !w.bad && w.t_begin < w.t_end)
                  ? (w.t_end - w.t_begin + kTcKeys - 1) / kTcKeys
                  : 0;
  w.cut = false;
  w.c0 = w.c1 = blockIdx.x;
  return w;
}

// Sequence b's tiles in the balanced schedule: none for a sequence without
// query rows or with more than the launch was sized for.
__device__ __forceinline__ int vf_seq_tiles(const VfParams& p, int b) {
  const int n = p.q_start[b + 1] - p.q_start[b];
  if (n <= 0 || n > p.max_q_len || n * p.group > kVfCols) return 0;
  return tiles_of<kTcKeys>(p.context_lens[b], p.max_blocks << p.log2_bs);
}

// A place on the balanced schedule's line of 128-key tiles, KV head by KV
// head: unit (b, h) holds the tiles h T + S[b] .. h T + S[b + 1] - 1, T =
// S[B]. (Head-major: the blocks W / Hkv apart on the line walk the same
// sequences' positions of neighbouring heads at the same time, so the heads
// of one token row are read together.)
struct VfCursor {
  int b, kvh, t, n;

  __device__ __forceinline__ void seek(long long g, const int* S, int B) {
    const long long T = S[B];
    kvh = (int)(g / T);
    const int r = (int)(g - (long long)kvh * T);
    int lo = 0, hi = B - 1;  // largest b with S[b] <= r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (S[mid] <= r) lo = mid; else hi = mid - 1;
    }
    b = lo;
    n = S[b + 1] - S[b];
    t = r - S[b];
  }

  // Move to the first tile of the next unit.
  __device__ __forceinline__ void next_unit(const int* S, int B) {
    t = 0;
    do {
      if (++b == B) {
        b = 0;
        ++kvh;
      }
    } while (S[b + 1] == S[b] && S[B] > 0);
    n = S[b + 1] - S[b];
  }

  __device__ __forceinline__ long long unit_start(const int* S, int B) const {
    return (long long)kvh * S[B] + S[b];
  }
};

// The block's work items in order. Split mode: units blockIdx.x,
// blockIdx.x + gridDim.x, ... Balanced mode: the segments of the block's
// range [c N / W, (c + 1) N / W) of the N = Hkv S[B] tiles of the line.
template <bool kBal>
struct VfWalk {
  int u;
  VfCursor cur;
  long long left, N, W;

  __device__ __forceinline__ void init(const VfParams& p, const int* S) {
    u = blockIdx.x;
    left = 0;
    if constexpr (kBal) {
      N = (long long)S[p.num_seqs] * p.num_kv_heads;
      W = min((long long)gridDim.x, N);
      if ((long long)blockIdx.x < W) {
        const long long g0 = (long long)blockIdx.x * N / W;
        left = (long long)(blockIdx.x + 1) * N / W - g0;
        if (left > 0) cur.seek(g0, S, p.num_seqs);
      }
    }
  }

  // The next item with tiles, or (split mode, all) the next unit.
  __device__ __forceinline__ bool next(const VfParams& p, const int* S, VfUnit& w, bool all) {
    if constexpr (kBal) {
      if (left <= 0) return false;
      w.b = cur.b;
      w.kvh = cur.kvh;
      w.split = 0;
      w.row0 = p.q_start[w.b];
      w.n = p.q_start[w.b + 1] - w.row0;
      w.nG = w.n * p.group;
      const int cap = p.max_blocks << p.log2_bs;
      const int ctx = p.context_lens[w.b];
      w.ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
      const int m = (int)min((long long)(cur.n - cur.t), left);
      w.t_begin = cur.t * kTcKeys;
      w.t_end = min((cur.t + m) * kTcKeys, w.ctx);
      w.n_tiles = m;
      w.bad = false;
      const long long u0 = cur.unit_start(S, p.num_seqs);
      w.c0 = owner_of(u0, N, W);
      w.c1 = owner_of(u0 + cur.n - 1, N, W);
      w.cut = w.c0 != w.c1;
      left -= m;
      if (cur.t + m == cur.n) {
        if (left > 0) cur.next_unit(S, p.num_seqs);
      } else {
        cur.t += m;
      }
      return true;
    } else {
      const int U = p.num_seqs * p.max_splits * p.num_kv_heads;
      while (u < U) {
        w = vf_unit(p, u);
        u += gridDim.x;
        if (all || w.n_tiles > 0) return true;
      }
      return false;
    }
  }
};

__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"((unsigned short)(v & 0xffffu))
               : "memory");
}

// 32 values a lane, value i for column i -> lane l returns the maximum
// (kMax) or the sum of column l over the warp's 32 lanes. Five exchange steps
// of width w = 16, 8, 4, 2, 1: a lane keeps the half of its current columns
// whose bit w matches its own lane bit and combines it with the partner's
// (lane ^ w) values of those columns.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(const float (&x)[32], int lane) {
  float v[16];
  {
    const bool up = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = up ? x[i] : x[i + 16];
      const float keep = up ? x[i + 16] : x[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, 16);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// The unit's Q as kVfCols K-major rows (zeros for padding columns) into a Q
// buffer; 128 threads (t = 0..127).
__device__ __forceinline__ void vf_stage_q(const VfParams& p, const VfUnit& w, uint32_t dst,
                                           int t) {
  constexpr int D = 128;
  constexpr int kPer = kVfCols * (D / 8) / 128;  // 16-byte chunks a thread
  uint4 v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {  // every load in flight before the stores
    const int idx = t + 128 * k;
    const int c = idx >> 4, ch = idx & 15;
    v[k] = make_uint4(0u, 0u, 0u, 0u);
    if (c < w.nG) {
      const int i = c / p.group;
      v[k] = ld_global_nc_v4(p.q + ((size_t)(w.row0 + i) * p.num_q_heads + w.kvh * p.group +
                                    (c - i * p.group)) * D + ch * 8);
    }
  }
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int idx = t + 128 * k;
    const int c = idx >> 4, ch = idx & 15;
    st_shared_v4(dst + (ch >> 3) * kVfPanel + c * 128 + (((ch & 7) ^ (c & 7)) << 4), v[k].x,
                 v[k].y, v[k].z, v[k].w);
  }
}

template <bool kBal>
__global__ void __launch_bounds__(kVfThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const VfParams p) {
  constexpr int D = 128;
  constexpr int NC = kVfCols;
  using L = VfSmem<kBal>;
  constexpr int S = L::kSlots;
  using Sh = TcShape<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrLayout);
    return;
  }

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + S;
  uint64_t* q_ready = empty + S;
  uint64_t* s_full = q_ready + 2;
  uint64_t* p_full = s_full + 2;
  uint64_t* lm_full = p_full + 2;
  uint64_t* o_full = lm_full + 2;
  uint64_t* o_free = o_full + 2;
  uint64_t* pv_done = o_free + 2;  // [jg % 2]: PV(jg) finished
  uint64_t* red_full = pv_done + 2;
  uint64_t* mma_done = red_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kFlag);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  float* lm = reinterpret_cast<float*>(smem + L::kLm);
  int* Sc = reinterpret_cast<int*>(smem + L::kScan);  // balanced: tiles before each sequence
  const uint32_t ring = smem_u32(smem + L::kRing);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sP = smem_u32(smem + L::kP);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&q_ready[k], kVfEpiWarps);
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], kVfSoftmaxWarps);
      mbar_init(&lm_full[k], kVfSoftmaxWarps);
      mbar_init(&o_full[k], 1);
      mbar_init(&o_free[k], kVfEpiWarps);
      mbar_init(&pv_done[k], 1);
    }
    mbar_init(red_full, kVfSoftmaxWarps);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kVfTmemCols);
    tmem_relinquish();
  }
  if constexpr (kBal)  // (ends with the block synchronised)
    tile_prefix_sum_of<kVfThreads>(Sc, reinterpret_cast<int*>(smem + L::kTot), p.num_seqs,
                                   [&](int i) { return vf_seq_tiles(p, i); });
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S^T buffers at columns 0, 32; O^T at 64, 96

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    // K_j, V_j of every unit in turn through the ring (load Lg of the block
    // goes to slot Lg % S). The warp holds 32 consecutive block-table entries
    // of the unit (one coalesced read per refill); lane i issues the tile's
    // box i.
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const int rb = p.box_rows;
    const int boxes = kTcKeys / rb;
    constexpr int kRowBytes = D * 2;  // one key's row of this head
    int Lg = 0;
    bool ok = true;
    VfWalk<kBal> wk;
    wk.init(p, Sc);
    VfUnit w;
    while (ok && wk.next(p, Sc, w, false)) {
      const int32_t* bt = p.block_tables + (size_t)w.b * p.max_blocks;
      const int n_entries = ((w.t_end - 1) >> p.log2_bs) + 1;
      int ent_base = -(1 << 30);
      int ent_val = -1;
      for (int Lu = 0; Lu < 2 * w.n_tiles; ++Lu, ++Lg) {
        const int slot = Lg % S;
        if (Lg >= S &&
            !__all_sync(0xffffffffu, wait_or_abort(&empty[slot], ((Lg / S) - 1) & 1, abort_flag))) {
          if (lane == 0) give_up(abort_flag, p.err, kErrWaitEmpty);
          ok = false;
          break;
        }
        const CUtensorMap* map = (Lu & 1) ? &tmap_v : &tmap_k;
        const int t0 = w.t_begin + (Lu >> 1) * kTcKeys;
        const int nbox = min(boxes, (w.t_end - 1 - t0) / rb + 1);
        const int e_first = t0 >> p.log2_bs;
        const int e_last = (t0 + nbox * rb - 1) >> p.log2_bs;
        if (e_first < ent_base || e_last >= ent_base + 32) {  // warp-uniform refill
          ent_base = e_first;
          const int idx = ent_base + lane;
          ent_val = idx < n_entries ? bt[idx] : -1;
        }
        if (lane == 0)
          mbar_arrive_expect_tx(&full[slot], (uint32_t)(nbox * rb * kRowBytes));
        const int i = lane < nbox ? lane : 0;
        const int key0 = t0 + i * rb;
        const int blk = __shfl_sync(0xffffffffu, ent_val, (key0 >> p.log2_bs) - ent_base);
        if (lane < nbox) {
          // rb rows (rb / 8 groups) of this head; a block id outside the pool
          // reads zeros (a box wholly out of range)
          const int grp = (blk >= 0 && blk < p.num_blocks)
                              ? (blk * p.block_size + (key0 & (p.block_size - 1))) >> 3
                              : -(rb >> 3);
          tma_load_4d(ring + slot * Sh::kKvBytes + (i * rb >> 3) * Sh::kKvGroup, map, 0, 0,
                      Sh::kHalves * w.kvh, grp, &full[slot]);
        }
      }
    }
    if (lane == 0) {  // every copy issued must land before the block ends
      for (int s = 0; s < S; ++s) {
        if (Lg <= s) continue;
        const int last = s + ((Lg - 1 - s) / S) * S;
        if (!mbar_wait(&full[s], (last / S) & 1)) atomicOr(p.err, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Tile jg of the block (over all its units): S(jg) into S^T buffer jg % 2,
    // then PV(jg - 1), so the softmax of tile jg runs while PV(jg - 1) and
    // S(jg + 1) are computed.
    if (lane == 0) {
      constexpr uint32_t kIdS = umma_idesc_16bit(kTcKeys, NC, false, false, false);
      constexpr uint32_t kIdO = umma_idesc_16bit(D, NC, false, true, false);
      constexpr uint64_t kSlotStep = Sh::kKvBytes >> 4;
      constexpr uint64_t kOpStep = kVfOpBytes >> 4;
      // built once; a k-step, a slot or a buffer moves only the start address
      const uint64_t d_k = umma_desc_sw128(ring, 16, Sh::kKvGroup);       // K rows, K-major
      const uint64_t d_v = umma_desc_sw128(ring, kKvHalf, Sh::kKvGroup);  // V^T, M-major
      const uint64_t d_q = umma_desc_sw128(sQ, 16, 1024);
      const uint64_t d_p = umma_desc_sw128(sP, 16, 1024);
      auto ready = [&](int Lg) { return wait_or_abort(&full[Lg % S], (Lg / S) & 1, abort_flag); };
      struct Pending {
        int jg, ug;
        bool first, last;
      };
      auto issue_pv = [&](const Pending& q) -> bool {
        const int LV = 2 * q.jg + 1;
        if (!wait_or_abort(&p_full[q.jg & 1], (q.jg >> 1) & 1, abort_flag) || !ready(LV))
          return false;
        // the O^T buffer's previous unit (ug - 2) has been read out
        if (q.first && q.ug >= 2 &&
            !wait_or_abort(&o_free[q.ug & 1], ((q.ug >> 1) - 1) & 1, abort_flag))
          return false;
        tc_fence_after();
        const uint64_t vd = d_v + (uint64_t)(LV % S) * kSlotStep;
        const uint64_t pd = d_p + (uint64_t)(q.jg & 1) * kOpStep;
        const uint32_t t_o = tmem + 2 * NC + (q.ug & 1) * NC;
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk) {
          const uint64_t voff = (uint64_t)((kk * 2 * Sh::kKvGroup) >> 4);
          const uint64_t poff = (uint64_t)(((kk >> 2) * kVfPanel + (kk & 3) * 32) >> 4);
          umma_bf16_ss(t_o, vd + voff, pd + poff, kIdO, (!q.first || kk > 0) ? 1u : 0u);
        }
        umma_commit(&empty[LV % S]);
        umma_commit(&pv_done[q.jg & 1]);
        if (q.last) umma_commit(&o_full[q.ug & 1]);
        return true;
      };
      bool ok = true, pending = false;
      Pending pend{0, 0, false, false};
      int jg = 0, ug = 0;
      VfWalk<kBal> wk;
      wk.init(p, Sc);
      VfUnit w;
      while (ok && wk.next(p, Sc, w, false)) {
        if (!(ok = wait_or_abort(&q_ready[ug & 1], (ug >> 1) & 1, abort_flag))) break;
        const uint64_t qd = d_q + (uint64_t)(ug & 1) * kOpStep;
        for (int j = 0; j < w.n_tiles; ++j, ++jg) {
          const int LK = 2 * jg;
          if (!(ok = ready(LK))) break;
          tc_fence_after();
          const uint64_t kd = d_k + (uint64_t)(LK % S) * kSlotStep;
          const uint32_t t_s = tmem + (jg & 1) * NC;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t koff = (uint64_t)(((kk >> 2) * kKvHalf + (kk & 3) * 32) >> 4);
            const uint64_t qoff = (uint64_t)(((kk >> 2) * kVfPanel + (kk & 3) * 32) >> 4);
            umma_bf16_ss(t_s, kd + koff, qd + qoff, kIdS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[jg & 1]);
          umma_commit(&empty[LK % S]);
          if (pending && !(ok = issue_pv(pend))) break;
          pend = Pending{jg, ug, j == 0, j == w.n_tiles - 1};
          pending = true;
        }
        ++ug;
      }
      if (ok && pending) ok = issue_pv(pend);
      if (!ok) give_up(abort_flag, p.err, kErrWaitFull);
      umma_commit(mma_done);  // every MMA issued is done: TMEM free to go
      if (!mbar_wait(mma_done, 0)) atomicOr(p.err, kErrDrain);
    }
  } else if (warp >= kVfFirstSoftmax && warp < kVfFirstEpi) {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;                    // TMEM lanes 32 quad .. 32 quad + 31
    const int key = quad * 32 + lane;             // this thread's key of a tile (S^T row)
    const int sw = warp - kVfFirstSoftmax;        // 0..3
    const int st = sw * 32 + lane;                // 0..127
    const uint32_t lanes = tmem + ((uint32_t)(quad * 32) << 16);
    // P element (key, column c) of buffer 0 at pb[c % 8] + 128 c: [key / 64]
    // [c][128 B], 16-byte chunk (key % 64) / 8 swizzled with c % 8
    uint32_t pb[8];
#pragma unroll
    for (int m = 0; m < 8; ++m)
      pb[m] = sP + (key >> 6) * kVfPanel + ((((key & 63) >> 3) ^ m) << 4) + (key & 7) * 2;
    bool ok = true;
    int jg = 0, ug = 0;
    VfWalk<kBal> wk;
    wk.init(p, Sc);
    VfUnit w;
    while (ok && wk.next(p, Sc, w, false)) {
      const float sl2 = p.scale_log2;
      const int pos0 = w.ctx - w.n;  // column c (token c / G) sees positions <= pos0 + c / G
      const uint32_t t_o = lanes + 2 * NC + (ug & 1) * NC;
      float m_run = -INFINITY;  // column `lane`: running max (log2 units, the one P and O use)
      float l_part[NC];         // this thread's key's share of each column's running sum
#pragma unroll
      for (int c = 0; c < NC; ++c) l_part[c] = 0.f;
      for (int j = 0; j < w.n_tiles; ++j, ++jg) {
        // S(jg) done also means PV(jg - 2) done (issued before it): P buffer
        // jg % 2 is free
        ok = __all_sync(0xffffffffu, wait_or_abort(&s_full[jg & 1], (jg >> 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        float y[NC];
        tmem_ld32_sync(lanes + (jg & 1) * NC, y);
        const int t0 = w.t_begin + j * kTcKeys;
        if (t0 + kTcKeys - 1 <= pos0 && t0 + kTcKeys <= w.t_end && w.nG == NC) {
#pragma unroll
          for (int c = 0; c < NC; ++c) y[c] *= sl2;  // every key visible in every column
        } else {
          // column c sees key t when t < t_end and t <= pos0 + c / G, i.e.
          // c >= G (t - pos0)
          const int t = t0 + key;
          const int cmin = t < w.t_end ? max(0, G * (t - pos0)) : NC;
#pragma unroll
          for (int c = 0; c < NC; ++c) y[c] = (c >= cmin && c < w.nG) ? y[c] * sl2 : -INFINITY;
        }
        // column maxima: this warp's keys, then the four warps' (buffer jg % 2:
        // a warp may run one tile ahead of the others, not two)
        float* rb = red + (jg & 1) * (kVfSoftmaxWarps * NC);
        rb[sw * NC + lane] = warp_transpose_reduce<true>(y, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full);
        ok = __all_sync(0xffffffffu, wait_or_abort(red_full, jg & 1, abort_flag));
        if (!ok) break;
        const float tm = max3(rb[lane], rb[NC + lane], fmaxf(rb[2 * NC + lane], rb[3 * NC + lane]));
        const bool grow = tm > m_run + kVfRescaleLog2;  // also the first finite max
        const float m_use = grow ? tm : m_run;
        const float alpha = grow ? ex2_approx(m_run - m_use) : 1.f;  // 0 when m_run = -inf
        m_run = m_use;
        const float msub = m_use == -INFINITY ? 0.f : m_use;
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // rescale the columns whose max moved: the partial sums and O^T
          // (after PV(jg - 1) has added to it)
          ok = __all_sync(0xffffffffu, wait_or_abort(&pv_done[(jg - 1) & 1], ((jg - 1) >> 1) & 1,
                                                      abort_flag));
          if (!ok) break;
          tc_fence_after();
          float o[NC];
          tmem_ld32_sync(t_o, o);
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const float ac = __shfl_sync(0xffffffffu, alpha, c);
            l_part[c] *= ac;
            o[c] *= ac;
          }
          tmem_st32_sync(t_o, o);
        }
        const uint32_t pbuf = (jg & 1) * kVfOpBytes;
#pragma unroll
        for (int c = 0; c < NC; c += 2) {
          const float m0 = __shfl_sync(0xffffffffu, msub, c);
          const float m1 = __shfl_sync(0xffffffffu, msub, c + 1);
          const float e0 = ex2_approx(y[c] - m0), e1 = ex2_approx(y[c + 1] - m1);
          // the partial sums add the rounded weights that multiply V
          const uint32_t pr = pack_bf16x2(e0, e1);
          add_halves<false>(l_part[c], l_part[c + 1], pr);
          st_shared_b16(pb[c & 7] + pbuf + c * 128, pr);
          st_shared_b16(pb[(c + 1) & 7] + pbuf + (c + 1) * 128, pr >> 16);
        }
        if (w.t_end - t0 < kTcKeys) {
          // the unit's last V tile: zero its rows past t_end (unwritten
          // slots, or another sequence's keys, may hold anything)
          const int LV = 2 * jg + 1;
          ok = __all_sync(0xffffffffu, wait_or_abort(&full[LV % S], (LV / S) & 1, abort_flag));
          if (ok) {
            const int first = w.t_end - t0;
            const uint32_t vt = ring + (LV % S) * Sh::kKvBytes;
            for (int i = st; i < (kTcKeys - first) * (D / 8); i += 4 * 32) {
              const int row = first + i / (D / 8), c = i % (D / 8);
              st_shared_v4(vt + (row >> 3) * Sh::kKvGroup + (c >> 3) * kKvHalf + (row & 7) * 128 +
                               (c & 7) * 16,
                           0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();  // P (and zeroed V rows) for the tensor cores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[jg & 1]);
        if (!ok) break;
      }
      if (!ok) break;
      // the unit's column sums and maxima for the epilogue warps (their
      // buffer ug % 2 is free once unit ug - 2 has been written out)
      if (ug >= 2) {
        ok = __all_sync(0xffffffffu, wait_or_abort(&o_free[ug & 1], ((ug >> 1) - 1) & 1, abort_flag));
        if (!ok) break;
      }
      float* lmb = lm + (ug & 1) * L::kLmFloats;
      lmb[sw * NC + lane] = warp_transpose_reduce<false>(l_part, lane);
      if (sw == 0) lmb[kVfSoftmaxWarps * NC + lane] = m_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&lm_full[ug & 1]);
      ++ug;
    }
    if (!ok) give_up(abort_flag, p.err, kErrWaitFull);
  } else if (warp >= kVfFirstEpi) {
    // ------------------------------------------------------------ epilogue
    // Stages Q of the items two ahead, writes each item's outputs from its
    // O^T buffer (balanced mode: a cut unit's partial record, merged by the
    // warp that arrives last on it), and handles the units with nothing to
    // attend (zero rows, reported shapes) and the per-row context lengths of
    // split mode.
    const int quad = warp & 3;
    const int dim = quad * 32 + lane;             // O^T row: this thread's head dim
    const int et = (warp - kVfFirstEpi) * 32 + lane;  // 0..127
    const uint32_t lanes = tmem + ((uint32_t)(quad * 32) << 16);
    VfWalk<kBal> qw;  // the next item whose Q is to be staged
    qw.init(p, Sc);
    int qn = 0;       // items staged so far
    auto stage_next = [&]() {
      VfUnit w;
      if (!qw.next(p, Sc, w, false)) return;
      vf_stage_q(p, w, sQ + (qn & 1) * kVfOpBytes, et);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_ready[qn & 1]);
      ++qn;
    };
    stage_next();
    stage_next();
    if constexpr (kBal) {
      // sequences without tiles: zero rows (no context), or reported shapes
      for (int b = blockIdx.x; b < p.num_seqs; b += gridDim.x) {
        const int row0 = p.q_start[b], n = p.q_start[b + 1] - row0;
        if (n <= 0 || Sc[b + 1] != Sc[b]) continue;
        if (n > p.max_q_len || n * G > NC) {
          if (et == 0) atomicOr(p.err, kErrShape);
          continue;
        }
        uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)row0 * p.num_q_heads * D);
        for (int i = et; i < n * p.num_q_heads * (D / 8); i += 128) dst[i] = make_uint4(0, 0, 0, 0);
      }
    }
    bool ok = true;
    int ug = 0;
    VfWalk<kBal> wk;
    wk.init(p, Sc);
    VfUnit w;
    while (ok && wk.next(p, Sc, w, !kBal)) {
      if (w.n <= 0) continue;
      if (w.bad) {
        if (et == 0 && w.kvh == 0 && w.split == 0) atomicOr(p.err, kErrShape);
        continue;
      }
      if (p.split_tokens > 0 && w.kvh == 0 && w.split == 0) {
        for (int i = et; i < w.n; i += 128) {
          const int len = w.ctx - w.n + i + 1;
          p.row_lens[w.row0 + i] = len > 0 ? len : 0;
        }
      }
      if (w.n_tiles == 0) {
        if (p.split_tokens == 0) {  // no context at all: zero rows
          for (int i = et; i < w.nG * (D / 8); i += 128) {
            const int c = i / (D / 8), c8 = i % (D / 8);
            __nv_bfloat16* dst = p.out + ((size_t)(w.row0 + c / G) * p.num_q_heads +
                                          w.kvh * G + c % G) * D + c8 * 8;
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      ok = __all_sync(0xffffffffu, wait_or_abort(&o_full[ug & 1], (ug >> 1) & 1, abort_flag)) &&
           __all_sync(0xffffffffu, wait_or_abort(&lm_full[ug & 1], (ug >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      // every S of this item is done: its Q buffer takes the item two ahead
      stage_next();
      const float* lmb = lm + (ug & 1) * L::kLmFloats;
      const float lsum = (lmb[lane] + lmb[NC + lane]) + (lmb[2 * NC + lane] + lmb[3 * NC + lane]);
      const float m_fin = lmb[kVfSoftmaxWarps * NC + lane];
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      // column `lane`: its output row, and whether this item holds a key of it
      const int ti = min(lane, w.nG - 1) / G;
      const int pos0 = w.ctx - w.n;
      const int r_lane = (w.row0 + ti) * p.num_q_heads + w.kvh * G + (lane - ti * G);
      const bool seen = lane < w.nG && pos0 + ti >= w.t_begin;
      if (p.split_tokens > 0 && quad == 0 && seen)
        p.part_lse[(size_t)r_lane * p.max_splits + w.split] =
            (m_fin + log2f(lsum)) * 0.69314718055994530942f;
      float o[NC];
      tmem_ld32_sync(lanes + 2 * NC + (ug & 1) * NC, o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ug & 1]);  // O^T and l/m of buffer ug % 2 read
      if (kBal && w.cut) {
        // a unit cut by block ranges: this block's part as a record (the
        // normalised output and the base-2 log-sum-exp of each column), then
        // this quarter's ticket; the warp with the last ticket merges the
        // unit's records for its 32 head dims
        const int rec = 2 * (int)blockIdx.x + ((int)blockIdx.x == w.c0 ? 1 : 0);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float ic = __shfl_sync(0xffffffffu, inv, c);
          if (c < w.nG) p.rec_o[((size_t)rec * p.rec_cols + c) * D + dim] = o[c] * ic;
        }
        if (lane < w.nG)
          p.rec_lse[rec * p.rec_cols + lane] = seen && lsum > 0.f ? m_fin + log2f(lsum) : -INFINITY;
        __syncwarp();
        int* counter = p.counters + ((size_t)w.b * p.num_kv_heads + w.kvh) * 8 + quad;
        int ticket = 0;
        if (lane == 0) {
          fence_acq_rel_gpu();
          ticket = atomicAdd(counter, 1);
          fence_acq_rel_gpu();
        }
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket == w.c1 - w.c0) {
          // lane c: column c's base-2 maximum and weight sum over the parts;
          // every thread: its head dim of every column, a part at a time
          float mc = -INFINITY;
          for (int cc = w.c0; cc <= w.c1; ++cc) {
            const int rr = 2 * cc + (cc == w.c0 ? 1 : 0);
            if (lane < w.nG) mc = fmaxf(mc, __ldcg(p.rec_lse + rr * p.rec_cols + lane));
          }
          float acc[NC];
#pragma unroll
          for (int c = 0; c < NC; ++c) acc[c] = 0.f;
          float wsum = 0.f;
          for (int cc = w.c0; cc <= w.c1; ++cc) {
            const int rr = 2 * cc + (cc == w.c0 ? 1 : 0);
            const float lk = lane < w.nG ? __ldcg(p.rec_lse + rr * p.rec_cols + lane) : -INFINITY;
            const float wk = mc == -INFINITY ? 0.f : exp2f(lk - mc);
            wsum += wk;
            const float* src = p.rec_o + (size_t)rr * p.rec_cols * D + dim;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
              const float wc = __shfl_sync(0xffffffffu, wk, c);
              if (c < w.nG) acc[c] += wc * __ldcg(src + (size_t)c * D);
            }
          }
          const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const float f = __shfl_sync(0xffffffffu, winv, c);
            const int r = __shfl_sync(0xffffffffu, r_lane, c);
            if (c < w.nG) p.out[(size_t)r * D + dim] = __float2bfloat16_rn(acc[c] * f);
          }
          if (lane == 0) *counter = 0;
        }
      } else {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float ic = __shfl_sync(0xffffffffu, inv, c);
          const int r = __shfl_sync(0xffffffffu, r_lane, c);
          const bool sc = __shfl_sync(0xffffffffu, seen, c);
          if (c < w.nG) {
            if (!sc) {  // no key of this item for the row
              if (p.split_tokens == 0) p.out[(size_t)r * D + dim] = __float2bfloat16_rn(0.f);
            } else if (p.split_tokens > 0) {
              p.part_out[((size_t)r * p.max_splits + w.split) * D + dim] = o[c] * ic;
            } else {
              p.out[(size_t)r * D + dim] = __float2bfloat16_rn(o[c] * ic);
            }
          }
        }
      }
      ++ug;
    }
    if (!ok) give_up(abort_flag, p.err, kErrWaitFull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kVfTmemCols);
  }
}

template <bool kBal>
pa_status launch_verify_as(const CUtensorMap& mk, const CUtensorMap& mv, const VfParams& prm,
                           cudaStream_t stream) {
  auto kern = verify_tc_kernel<kBal>;
  const int smem = VfSmem<kBal>::bytes(prm.num_seqs);
  const pa_status s =
      prepare_kernel(reinterpret_cast<const void*>(kern), kVfThreads, smem, nullptr);
  if (s != PA_OK) return s;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return PA_ERR_CUDA;
  // persistent: one block per SM (split mode: no more blocks than units)
  const long long units = (long long)prm.num_seqs * prm.max_splits * prm.num_kv_heads;
  const int grid = kBal ? sms : (int)(units < sms ? units : sms);
  kern<<<grid, kVfThreads, smem, stream>>>(mk, mv, prm);
  return launch_status();
}

}  // namespace

bool verify_tc_supported(int head_dim, int block_size, int group, int max_q_len,
                         int split_tokens) {
  return head_dim == 128 && block_size >= 8 && group >= 1 &&
         (long long)max_q_len * group <= kVfCols && split_tokens >= 0 &&
         split_tokens % kTcKeys == 0;
}

bool verify_tc_balanced_supported(int head_dim, int block_size, int group, int max_q_len,
                                  int num_seqs) {
  return verify_tc_supported(head_dim, block_size, group, max_q_len, 0) &&
         num_seqs <= kVfMaxBalSeqs;
}

namespace {

// Parameters and tensor maps both schedules share.
pa_status verify_params(VfParams& prm, CUtensorMap& mk, CUtensorMap& mv, const void* q,
                        const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        int max_blocks, const int32_t* context_lens, const int32_t* q_start,
                        int num_seqs, int max_q_len, int num_q_heads, int num_kv_heads,
                        int block_size, int num_blocks, float scale, void* out,
                        unsigned int* err) {
  if (num_kv_heads > 65535 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  std::memset(&prm, 0, sizeof(prm));
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.q_start = q_start;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.err = err;
  prm.num_seqs = num_seqs;
  prm.num_kv_heads = num_kv_heads;
  prm.max_blocks = max_blocks;
  prm.num_q_heads = num_q_heads;
  prm.group = num_q_heads / num_kv_heads;
  prm.max_q_len = max_q_len;
  prm.block_size = block_size;
  prm.log2_bs = ilog2(block_size);
  prm.box_rows = block_size < kTcKeys ? block_size : kTcKeys;
  prm.num_blocks = num_blocks;
  prm.max_splits = 1;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  const long long rows = (long long)num_blocks * block_size;
  if (!make_tc_map<128>(&mk, k_cache, num_kv_heads, rows, prm.box_rows) ||
      !make_tc_map<128>(&mv, v_cache, num_kv_heads, rows, prm.box_rows))
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

pa_status launch_verify_tc(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                           int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int num_blocks, float scale, int split_tokens,
                           int max_splits, float* part_out, float* part_lse, int32_t* row_lens,
                           void* out, unsigned int* err, cudaStream_t stream) {
  const int G = num_q_heads / num_kv_heads;
  if (!verify_tc_supported(head_dim, block_size, G, max_q_len, split_tokens))
    return PA_ERR_UNSUPPORTED;
  if ((long long)num_seqs * (split_tokens > 0 ? max_splits : 1) * num_kv_heads >= (1LL << 31))
    return PA_ERR_UNSUPPORTED;
  VfParams prm;
  CUtensorMap mk, mv;
  const pa_status s =
      verify_params(prm, mk, mv, q, k_cache, v_cache, block_tables, max_blocks, context_lens,
                    q_start, num_seqs, max_q_len, num_q_heads, num_kv_heads, block_size,
                    num_blocks, scale, out, err);
  if (s != PA_OK) return s;
  prm.part_out = part_out;
  prm.part_lse = part_lse;
  prm.row_lens = row_lens;
  prm.split_tokens = split_tokens;
  prm.max_splits = split_tokens > 0 ? max_splits : 1;
  return launch_verify_as<false>(mk, mv, prm, stream);
}

pa_status launch_verify_tc_balanced(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int max_blocks,
                                    const int32_t* context_lens, const int32_t* q_start,
                                    int num_seqs, int max_q_len, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, float scale, int* counters, float* rec_lse,
                                    float* rec_o, int rec_cols, void* out, unsigned int* err,
                                    cudaStream_t stream) {
  const int G = num_q_heads / num_kv_heads;
  if (!verify_tc_balanced_supported(head_dim, block_size, G, max_q_len, num_seqs) ||
      rec_cols < kVfCols)
    return PA_ERR_UNSUPPORTED;
  VfParams prm;
  CUtensorMap mk, mv;
  const pa_status s =
      verify_params(prm, mk, mv, q, k_cache, v_cache, block_tables, max_blocks, context_lens,
                    q_start, num_seqs, max_q_len, num_q_heads, num_kv_heads, block_size,
                    num_blocks, scale, out, err);
  if (s != PA_OK) return s;
  prm.counters = counters;
  prm.rec_lse = rec_lse;
  prm.rec_o = rec_o;
  prm.rec_cols = rec_cols;
  return launch_verify_as<true>(mk, mv, prm, stream);
}

}  // namespace pa
