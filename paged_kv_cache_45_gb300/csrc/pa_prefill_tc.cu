// pa_prefill_tc.cu -- long query chunks (chunked prefill) on the fifth-
// generation tensor cores of sm_103a.
//
// A chunk of a prompt ("Text Generation Inference: Hugging Face's
// production-grade LLM inference server", section "Advanced Pattern: Chunked
// Prefill (TGI v3)") brings n_b new tokens whose K/V rows are already in the
// paged pool; token i (position ctx_b - n_b + i) attends to positions
// 0 .. ctx_b - n_b + i through the sequence's block table ("Text Generation
// Inference ...", section "PagedAttention": the block table maps a logical
// token to a physical block). With n_b * G query rows per KV head the scores
// are a dense contraction, so they run on tcgen05.mma with the accumulators
// in tensor memory.
//
// One thread block per (row tile counted from the chunk's end, KV head,
// sequence), 256 query rows = two M = 128 tiles (row = token * G + head; a
// block covers floor(256 / G) tokens), 10 warps:
//   warp 0     loader: K_j and V_j tiles of 128 keys through a 160 KB ring
//              (5 slots at head_dim 128, 10 at 64); a paged block's rows of
//              one head land with ONE 4-D TMA box (64 columns x 8 rows x the
//              head's 128-byte panels x block_size / 8 row groups, 128-byte
//              swizzle), lane i issuing box i so that the boxes' issue costs
//              overlap;
//   warp 1     allocates 512 TMEM columns (S_0, S_1 scores, O_0, O_1 outputs)
//              and one lane issues every MMA, descriptors built once:
//                S_w = Q_w K_j^T  (SS: M 128, N 128 keys, K = head_dim)
//                O_w += P_w V_j   (TS: P_w from TMEM, M 128, N head_dim,
//                                  K 128 keys)
//              in the order P_0 V_j, S_0(j+1), P_1 V_j, S_1(j+1), ... so the
//              tensor cores work on one tile's products while the other
//              tile's softmax runs;
//   warps 2-9  two softmax warpgroups, one per Q tile, one thread per row:
//              read the row's 128 scores from TMEM, apply the causal limit,
//              take the online softmax in base 2 (the running output is
//              rescaled only when the running max grew by more than 2^8 --
//              exact, as the final division uses the same stale max), write
//              P as bf16 pairs into the first 64 columns of S_w (the next
//              S_w is issued after P_w V_j, and the pipe runs in order), and
//              after the last tile divide O by the row sum and store bf16.
// The key range of a block is [0, last position of its last token]; blocks
// of one sequence and head fold its tiles in rotated orders. Keys past a
// row's own position are masked, and V rows past the block's last position
// are zeroed before their P.V (they may be unwritten slots).
//
// e4m3 pools (head_dim 128): the same block with two more warps. The loader
// lands each paged block's e4m3 rows (128 bytes a token and head) in the
// upper half of the tile's operand slot; warps 10-11 widen them in place,
// exactly, to f16 (every e4m3 value is an f16 value) in the layout the bf16
// path's TMA writes, zeroing V rows past the block's last position on the
// way. The MMAs then run kind::f16 on f16 Q (q is
// converted once: exact for 2^-14 <= |q| <= 65504), f16 K/V and f16 P; the
// per-head scales go into the score factor (k_scale) and the final division
// (v_scale).

#include <cudaTypedefs.h>
#include <math.h>

#include <cstring>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_tc_common.cuh"
#include "pa_umma.cuh"
#include "pagedkv.h"

namespace pa {
namespace {

constexpr int kTcQTiles = 2;                       // Q tiles per block
constexpr int kTcPanel = kTcRows * 128;            // Q: one 64-column panel, 16 KB
constexpr int kTcSoftmaxWarps = 4 * kTcQTiles;
constexpr int kTcThreads = (2 + kTcSoftmaxWarps) * 32;
constexpr uint32_t kTcCols = 512;                  // TMEM columns
constexpr float kRescaleLog2 = 8.0f;               // rescale O when the max grows by > 2^8

template <bool kFp8>
constexpr int tc_threads() { return kTcThreads + (kFp8 ? kTcConvWarps * 32 : 0); }

template <int D, bool kFp8 = false>
struct TcSmem {
  using S = TcShape<D, kFp8>;
  static constexpr int kQ = 0;                                   // Q_0, Q_1
  static constexpr int kRing = kQ + kTcQTiles * S::kQBytes;      // K/V slots
  static constexpr int kBar = kRing + S::kSlots * S::kKvBytes;
  // barriers: full[kSlots], empty[kSlots], s_full[2], p_full[2], q_ready,
  // o_final; e4m3: landed[kSlots] (the codes are in; full = widened)
  static constexpr int kNumBars = 2 * S::kSlots + 2 * kTcQTiles + 2 + (kFp8 ? S::kSlots : 0);
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kFlag = kTmemSlot + 8;
  static constexpr int kAlloc = kFlag + 8 + 1024;                // + 1024-byte alignment
};
static_assert(TcSmem<128>::kAlloc <= 232448, "over the 227 KB of shared memory per block");
static_assert(TcSmem<64>::kAlloc <= 232448, "over the 227 KB of shared memory per block");
static_assert(TcSmem<128, true>::kAlloc <= 232448, "over the 227 KB of shared memory per block");

struct TcParams {
  const __nv_bfloat16* q;       // [R, Hq, D]
  const int32_t* q_start;       // [B + 1]
  const int32_t* block_tables;  // [B, max_blocks]
  const int32_t* context_lens;  // [B]
  __nv_bfloat16* out;           // [R, Hq, D]
  unsigned int* err;            // device error word
  int max_blocks;
  int num_q_heads;
  int group;
  int tokens_per_block;         // floor(256 / G)
  int max_q_len;
  int block_size;
  int log2_bs;
  int box_rows;                 // min(block_size, 128)
  int num_blocks;
  float scale_log2;
  const float* k_scale;         // [Hkv], e4m3 pools only
  const float* v_scale;
  const void* k_src;            // the caches, for the gather path (block sizes < 8)
  const void* v_src;
  int num_kv_heads;
};

// Byte offset of 16-byte chunk c (0..15) of row r in a two-panel swizzled tile.
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) {
  return (uint32_t)((c >> 3) * kTcPanel + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Ring position of K_i and V_i: K0 V0 K1 V1 ..., the order the MMAs consume them in.
__device__ __forceinline__ int k_seq(int i) { return 2 * i; }
__device__ __forceinline__ int v_seq(int i) { return 2 * i + 1; }

// kGather: block sizes below 8, where a paged block holds less than one
// 8-row group of a TMA box: the loader warp gathers the tile's rows with
// 16-byte cp.async copies into the same slot layout instead.
template <int D, bool kFp8, bool kGather>
__global__ void __launch_bounds__(tc_threads<kFp8>(), 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const TcParams p) {
  static_assert(!kFp8 || D == 128, "e4m3 pools: one 128-byte row per token and head");
  using Sh = TcShape<D, kFp8>;
  using L = TcSmem<D, kFp8>;
  constexpr int kSlots = Sh::kSlots;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // blockIdx.x counts row tiles from the chunk's end (longest key range
  // first); a sequence's row tiles are neighbours in launch order, so the
  // blocks running together share its K/V in L2.
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int TPB = p.tokens_per_block;
  const int row0 = p.q_start[b];
  const int n = p.q_start[b + 1] - row0;
  const int tok_hi = n - (int)blockIdx.x * TPB;  // this block: chunk tokens [tok_lo, tok_hi)
  if (tok_hi <= 0) return;
  if (n > p.max_q_len) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.err, kErrShape);
    return;
  }
  const int tok_lo = tok_hi - TPB > 0 ? tok_hi - TPB : 0;
  int ctx = p.context_lens[b];
  const int cap = p.max_blocks << p.log2_bs;
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  const int pos_base = ctx - n;                 // position of the chunk's token 0
  const int pos_last = pos_base + tok_hi - 1;   // the block's last attended position
  const int n_tiles = pos_last >= 0 ? pos_last / kTcKeys + 1 : 0;
  // Iteration i folds key tile (i + rot) mod n_tiles: the blocks of one
  // sequence and KV head run together, and a rotation of their order keeps
  // them from all reading the same tile (the same L2 lines) at the same time.
  const int rot = n_tiles > 0 ? (int)((blockIdx.x * 7u) % (unsigned)n_tiles) : 0;
  auto tile_of = [&](int i) { return i + rot < n_tiles ? i + rot : i + rot - n_tiles; };

  // softmax thread -> (Q tile, row); rows past the block's tokens are padding
  const int sw = warp - 2;                      // softmax warp 0..7
  const int qt = sw >> 2;                       // Q tile
  const int quarter = warp & 3;                 // TMEM lanes 32 * quarter ..
  const int r = quarter * 32 + lane;            // row within the Q tile
  const int R = qt * kTcRows + r;               // row within the block
  const bool row_valid = sw >= 0 && sw < kTcSoftmaxWarps && R / G < tok_hi - tok_lo;
  const int tok = tok_lo + R / G;
  const int pos = row_valid ? pos_base + tok : -1;
  const size_t out_off =
      ((size_t)(row0 + tok) * p.num_q_heads + (size_t)kvh * G + (R % G)) * D;

  if (n_tiles == 0) {  // no position to attend: zero rows, nothing else
    if (row_valid) {
      uint4* o = reinterpret_cast<uint4*>(p.out + out_off);
      for (int c = 0; c < D / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty = full + kSlots;
  uint64_t* s_full = empty + kSlots;
  uint64_t* p_full = s_full + kTcQTiles;
  uint64_t* q_ready = p_full + kTcQTiles;
  uint64_t* o_final = q_ready + 1;
  uint64_t* landed = o_final + 1;       // e4m3: a slot's codes landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kFlag);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t ring = smem_u32(smem + L::kRing);

  if (threadIdx.x == 0) {
    // the loads complete on `landed` (e4m3) or `full` (bf16): one arrival
    // with the byte count for a TMA tile, one per loader lane for a gathered one
    constexpr int kLoadArrivals = kGather ? 32 : 1;
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], kFp8 ? kTcConvWarps : kLoadArrivals);  // e4m3: one per converter
      mbar_init(&empty[s], 1);
    }
    if constexpr (kFp8) {
      for (int s = 0; s < kSlots; ++s) mbar_init(&landed[s], kLoadArrivals);
    }
    for (int w = 0; w < kTcQTiles; ++w) {
      mbar_init(&s_full[w], 1);
      mbar_init(&p_full[w], kTcRows / 32);  // one arrival per softmax warp
    }
    mbar_init(q_ready, kTcSoftmaxWarps);
    mbar_init(o_final, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTcCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    // The whole warp holds 32 consecutive block-table entries (one coalesced
    // read per refill, bt[ent_base + lane]); lane i issues the tile's box i.
    if (!kGather && lane == 0) {  // (the gather path has no tensor maps)
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const int32_t* bt = p.block_tables + (size_t)b * p.max_blocks;
    const int rb = p.box_rows;
    const int boxes = kTcKeys / rb;
    const int n_entries = (pos_last >> p.log2_bs) + 1;      // entries the block reads
    int ent_base = -(1 << 30);
    int ent_val = -1;
    // e4m3 pools: the codes land in the slot's upper half and complete on
    // `landed` (the converter warps then widen them and arrive on `full`)
    constexpr int kDst = kSlots;
    uint64_t* landed_bar = kFp8 ? landed : full;
    uint64_t* free_bar = empty;
    int L = 0;
    for (; L < 2 * n_tiles; ++L) {
      const int slot = L % kDst;
      if (L >= kDst &&
          !__all_sync(0xffffffffu, wait_or_abort(&free_bar[slot], ((L / kDst) - 1) & 1,
                                                 abort_flag))) {
        if (lane == 0) give_up(abort_flag, p.err, kErrWaitEmpty);
        break;
      }
      const bool is_v = (L & 1) != 0;  // L = 2 j: K_j, L = 2 j + 1: V_j
      const int j = tile_of(L >> 1);
      if constexpr (kGather) {
        // rows j*128 .. pos_last (at most 128) of this head, 16 bytes a copy;
        // each lane reads its rows' table entries itself (a block holds at
        // most 4 rows here). Ids outside the pool give zeros. (Reading the
        // tile's entries once and passing them by shuffles measured slower:
        // 27.3 against 19.7 ms for the 8 x 2048-token chunk step at block
        // size 4.)
        constexpr int kRowBytes = kFp8 ? 128 : D * 2;
        constexpr int kCpr = kRowBytes / 16;  // 16-byte chunks per row
        const unsigned char* cache = static_cast<const unsigned char*>(is_v ? p.v_src : p.k_src);
        const int n_rows = min(kTcKeys, pos_last - j * kTcKeys + 1);
        const uint32_t dst = ring + (L % kDst) * Sh::kKvBytes;
        for (int idx = lane; idx < n_rows * kCpr; idx += 32) {
          const int r = idx / kCpr, c = idx % kCpr;
          const int key = j * kTcKeys + r;
          const int blk = __ldg(bt + (key >> p.log2_bs));
          const bool ok = blk >= 0 && blk < p.num_blocks;
          const unsigned char* src =
              ok ? cache + ((size_t)(blk * p.block_size + (key & (p.block_size - 1))) *
                                p.num_kv_heads + kvh) * kRowBytes + c * 16
                 : cache;
          cp_async_16_zfill(dst + kv_chunk_offset<D, kFp8>(r, c), src, ok);
        }
        cp_async_arrive_noinc(&landed_bar[L % kDst]);
        continue;
      }
      const CUtensorMap* map = is_v ? &tmap_v : &tmap_k;
      const int nbox = min(boxes, (pos_last - j * kTcKeys) / rb + 1);
      const int e_first = (j * kTcKeys) >> p.log2_bs;
      const int e_last = (j * kTcKeys + nbox * rb - 1) >> p.log2_bs;
      if (e_first < ent_base || e_last >= ent_base + 32) {  // warp-uniform refill
        ent_base = e_first;
        const int idx = ent_base + lane;
        ent_val = idx < n_entries ? bt[idx] : -1;
      }
      constexpr int kRowBytes = kFp8 ? 128 : D * 2;  // one key's row of this head
      if (lane == 0) mbar_arrive_expect_tx(&landed_bar[slot], (uint32_t)(nbox * rb * kRowBytes));
      // one box per lane, issued together: a TMA instruction costs a lane a
      // few hundred cycles, and lanes overlap them
      const uint32_t dst = ring + slot * Sh::kKvBytes;
      const int i = lane < nbox ? lane : 0;
      const int key0 = j * kTcKeys + i * rb;
      const int blk = __shfl_sync(0xffffffffu, ent_val, (key0 >> p.log2_bs) - ent_base);
      if (lane < nbox) {
        // rb rows (rb / 8 groups) x all panels of this head; a block id
        // outside the pool reads zeros (a box wholly out of range)
        const int grp = (blk >= 0 && blk < p.num_blocks)
                            ? (blk * p.block_size + (key0 & (p.block_size - 1))) >> 3
                            : -(rb >> 3);
        // e4m3: 1 KB a code group (8 rows of 128 codes), placed by kCodePos
        // (a box holds at most 4 groups, which stay contiguous there)
        const uint32_t at = kFp8 ? kCodeHalf + kCodePos(i * rb >> 3) * 1024
                                 : (uint32_t)((i * rb >> 3) * Sh::kKvGroup);
        tma_load_4d(dst + at, map, 0, 0, (kFp8 ? 1 : Sh::kHalves) * kvh, grp, &landed_bar[slot]);
      }
    }
    // every copy issued must land before the block ends
    if (lane == 0) {
      for (int s = 0; s < kDst; ++s) {
        if (L <= s) continue;
        const int last = s + ((L - 1 - s) / kDst) * kDst;
        if (!mbar_wait(&landed_bar[s], (last / kDst) & 1)) atomicOr(p.err, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS =
          kFp8 ? umma_idesc_f16(kTcRows, kTcKeys, false) : umma_idesc_bf16(kTcRows, kTcKeys, false);
      constexpr uint32_t kIdO =
          kFp8 ? umma_idesc_f16(kTcRows, D, true) : umma_idesc_bf16(kTcRows, D, true);
      // Descriptors are built once; a k-step or a slot moves only the start
      // address (bits 0-13, address >> 4), so each MMA costs one 64-bit add.
      // (Building them per MMA made the issuing thread, not the tensor pipe,
      // the bottleneck.)
      constexpr uint64_t kQStep = Sh::kQBytes >> 4;
      constexpr uint64_t kSlotStep = Sh::kKvBytes >> 4;
      const uint64_t d_q = umma_desc_sw128(sQ, 16, 1024);             // Q_0, K-major
      const uint64_t d_k = umma_desc_sw128(ring, 16, Sh::kKvGroup);          // slot 0, K-major
      const uint64_t d_v = umma_desc_sw128(ring, kKvHalf, Sh::kKvGroup);     // slot 0, MN-major
      auto issue_s = [&](int w, int L) {  // S_w = Q_w K^T, K in slot L % kSlots
        const uint64_t qd = d_q + (uint64_t)w * kQStep;
        const uint64_t kd = d_k + (uint64_t)(L % kSlots) * kSlotStep;
        const uint32_t dst = tmem + w * kTcKeys;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t qoff = (uint64_t)(((kk >> 2) * kTcPanel + (kk & 3) * 32) >> 4);
          const uint64_t koff = (uint64_t)(((kk >> 2) * kKvHalf + (kk & 3) * 32) >> 4);
          umma_bf16_ss(dst, qd + qoff, kd + koff, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int w, int L, int j) {  // O_w += P_w V; P_w in TMEM, V in a slot
        const uint64_t vd = d_v + (uint64_t)(L % kSlots) * kSlotStep;
        const uint32_t dst = tmem + 2 * kTcKeys + w * D;
        const uint32_t pa_ = tmem + w * kTcKeys;
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk)
          umma_bf16_ts(dst, pa_ + kk * 8, vd + (uint64_t)(kk * ((2 * Sh::kKvGroup) >> 4)), kIdO,
                       (j > 0 || kk > 0) ? 1u : 0u);
      };
      auto landed = [&](int L) {
        return wait_or_abort(&full[L % kSlots], (L / kSlots) & 1, abort_flag);
      };
      // Tensor-pipe order: P_0 V_j, S_0(j+1), P_1 V_j, S_1(j+1), ...: while
      // one warpgroup's softmax runs, the other's products are computed. P_w
      // lives in S_w's columns, so S_w(j+1) follows P_w V_j (the pipe runs
      // in issue order).
      bool ok = wait_or_abort(q_ready, 0, abort_flag) && landed(k_seq(0));
      if (ok) {
        tc_fence_after();
        issue_s(0, k_seq(0));
        umma_commit(&s_full[0]);
        issue_s(1, k_seq(0));
        umma_commit(&s_full[1]);
        umma_commit(&empty[k_seq(0) % kSlots]);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const bool more = j + 1 < n_tiles;
        const int LV = v_seq(j), LK = k_seq(j + 1);
        if (!(ok = landed(LV))) break;
        for (int w = 0; w < kTcQTiles; ++w) {
          if (!(ok = wait_or_abort(&p_full[w], j & 1, abort_flag))) break;
          tc_fence_after();
          issue_pv(w, LV, j);
          if (w == kTcQTiles - 1) umma_commit(&empty[LV % kSlots]);
          if (more) {
            if (w == 0 && !(ok = landed(LK))) break;
            issue_s(w, LK);
            umma_commit(&s_full[w]);
            if (w == kTcQTiles - 1) umma_commit(&empty[LK % kSlots]);
          }
        }
      }
      if (!ok) give_up(abort_flag, p.err, kErrWaitFull);
      umma_commit(o_final);  // every MMA issued is done: outputs final, TMEM free to go
      if (!mbar_wait(o_final, 0)) atomicOr(p.err, kErrDrain);
    }
  } else if (kFp8 && warp >= 2 + kTcSoftmaxWarps) {
    // ------------------------------------------------------------ e4m3 widening
    // Tile L (K_j or V_j of 128 keys) of slot L % kSlots, widened in place.
    const int cw = warp - (2 + kTcSoftmaxWarps);  // converter warp 0 or 1
    bool ok = true;
    for (int L = 0; ok && L < 2 * n_tiles; ++L) {
      const int slot = L % kSlots;
      ok = __all_sync(0xffffffffu, wait_or_abort(&landed[slot], (L / kSlots) & 1, abort_flag));
      if (!ok) {
        if (lane == 0) give_up(abort_flag, p.err, kErrWaitFull);
        break;
      }
      const bool is_v = (L & 1) != 0;
      const int j = tile_of(L >> 1);
      const int rb = p.box_rows;
      const int loaded = min(kTcKeys / rb, (pos_last - j * kTcKeys) / rb + 1) * rb;
      // V rows past the block's last position become zeros (they may be
      // unwritten slots); K rows there are masked by every row's limit
      const int keep = is_v ? min(loaded, pos_last - j * kTcKeys + 1) : loaded;
      const uint32_t base = ring + slot * Sh::kKvBytes;
      widen_e4m3_slot(base, cw, lane, keep, is_v);
      // the f16 writes become visible to the tensor cores
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[slot]);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lanes = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t t_s = lanes + qt * kTcKeys;               // S of this tile; P in its first half
    const uint32_t t_o = lanes + 2 * kTcKeys + qt * D;       // O of this tile
    const uint32_t my_q = sQ + qt * Sh::kQBytes;
    {  // this row of Q into the K-major swizzled tile (zeros for padding rows)
      const __nv_bfloat16* src = p.q + out_off;
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        uint4 v = row_valid ? ld_global_nc_v4(src + 8 * c) : make_uint4(0, 0, 0, 0);
        if constexpr (kFp8) {  // the f16 MMA takes f16 q
          v = make_uint4(pack_f16x2(bf16_lo(v.x), bf16_hi(v.x)), pack_f16x2(bf16_lo(v.y), bf16_hi(v.y)),
                         pack_f16x2(bf16_lo(v.z), bf16_hi(v.z)), pack_f16x2(bf16_lo(v.w), bf16_hi(v.w)));
        }
        st_shared_v4(my_q + sw_chunk(r, c), v.x, v.y, v.z, v.w);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const float sl2 = kFp8 ? p.scale_log2 * __ldg(p.k_scale + kvh) : p.scale_log2;
    float m_run = -INFINITY;  // running max, log2 units (the one P and O use)
    float l_run = 0.f;        // running row sum of P
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      // S_w(j) done implies P_w V_{j-1} done (issued before it): O is current
      // and S's columns may take P
      ok = __all_sync(0xffffffffu, wait_or_abort(&s_full[qt], j & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float s[kTcKeys];
      tmem_ld128_sync(t_s, s);
      const int tile = tile_of(j);
      const int lim = pos - tile * kTcKeys;  // keys 0 .. lim of the tile are visible
      if (lim < kTcKeys - 1) {
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) s[c] = c <= lim ? s[c] : -INFINITY;
      }
      float mx8[8];  // 8 independent chains of three-input maxes
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
      for (int c = 16; c < kTcKeys; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = max3(mx8[i], s[c + i], s[c + 8 + i]);
      const float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]),
                            fmaxf(mx8[6], mx8[7]));
      const float m_tile = mx * sl2;
      const bool grow = m_tile > m_run + kRescaleLog2;  // also the first finite max
      const float m_use = grow ? m_tile : m_run;
      const float alpha = grow ? ex2_approx(m_run - m_use) : 1.f;  // 0 when m_run = -inf
      const float ms = m_use == -INFINITY ? 0.f : m_use;
      uint32_t pk[kTcKeys / 2];  // P row as bf16 pairs
      float sum8[8];             // 4 packed (even, odd) running sums
#pragma unroll
      for (int i = 0; i < 8; ++i) sum8[i] = 0.f;
      const uint64_t sl2x2 = splat2(sl2), negms2 = splat2(-ms);
#pragma unroll
      for (int c = 0; c < kTcKeys; c += 2) {
        float x0, x1;
        fma2(x0, x1, s[c], s[c + 1], sl2x2, negms2);
        const float e0 = ex2_approx(x0);
        const float e1 = ex2_approx(x1);
        const int a = (c >> 1) & 3;
        // the running sum adds the rounded weights that multiply V (bf16; f16
        // for e4m3 pools), each half straight from the packed pair by a
        // mixed-precision add
        const uint32_t pr = kFp8 ? pack_f16x2(e0, e1) : pack_bf16x2(e0, e1);
        pk[c >> 1] = pr;
        add_halves<kFp8>(sum8[2 * a], sum8[2 * a + 1], pr);
      }
      tmem_st64_sync(t_s, pk);
      const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                        ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l_run = l_run * alpha + sum;
      m_run = m_use;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {  // rescale the running output
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32_sync(t_o + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32_sync(t_o + c, o);
        }
      }
      if (!kFp8 && qt == 0 && tile == n_tiles - 1) {  // (e4m3: the converters zero them)
        // the last V tile: zero its rows past the block's last position
        const int first = pos_last - tile * kTcKeys + 1;
        if (first < kTcKeys) {
          const int LV = v_seq(j);
          ok = __all_sync(0xffffffffu, wait_or_abort(&full[LV % kSlots],
                                                      (LV / kSlots) & 1, abort_flag));
          if (ok) {
            const uint32_t vt = ring + (LV % kSlots) * Sh::kKvBytes;
            for (int i = r; i < (kTcKeys - first) * (D / 8); i += kTcRows) {
              const int row = first + i / (D / 8), c = i % (D / 8);
              st_shared_v4(vt + (row >> 3) * Sh::kKvGroup + (c >> 3) * kKvHalf + (row & 7) * 128 +
                               (c & 7) * 16,
                           0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[qt]);
      if (!ok) break;
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(o_final, 0, abort_flag));
    if (!ok) {
      give_up(abort_flag, p.err, kErrWaitFull);
    } else {
      tc_fence_after();
      const float inv = l_run > 0.f ? (kFp8 ? __ldg(p.v_scale + kvh) : 1.f) / l_run : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.out + out_off);
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float o[32];
        tmem_ld32_sync(t_o + c, o);
        if (row_valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[c / 8 + i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                        pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                        pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                        pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
  }
}

template <int D, bool kFp8, bool kGather>
pa_status launch_tc_as(const CUtensorMap& mk, const CUtensorMap& mv, const TcParams& prm,
                       long long tiles, int num_kv_heads, int num_seqs, cudaStream_t stream) {
  using L = TcSmem<D, kFp8>;
  constexpr int kThreads = tc_threads<kFp8>();
  auto kern = prefill_tc_kernel<D, kFp8, kGather>;
  const pa_status s =
      prepare_kernel(reinterpret_cast<const void*>(kern), kThreads, L::kAlloc, nullptr);
  if (s != PA_OK) return s;
  const dim3 grid((unsigned)tiles, num_kv_heads, num_seqs);
  kern<<<grid, kThreads, L::kAlloc, stream>>>(mk, mv, prm);
  return launch_status();
}

// TMA boxes for block sizes >= 8, the cp.async gather below.
template <int D, bool kFp8 = false>
pa_status launch_tc(const CUtensorMap& mk, const CUtensorMap& mv, const TcParams& prm,
                    long long tiles, int num_kv_heads, int num_seqs, cudaStream_t stream) {
  if (prm.block_size < 8)
    return launch_tc_as<D, kFp8, true>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream);
  return launch_tc_as<D, kFp8, false>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream);
}

// Parameters shared by the bf16 and e4m3 launches.
TcParams tc_params(const void* q, const int32_t* block_tables, int max_blocks,
                   const int32_t* context_lens, const int32_t* q_start, int max_q_len,
                   int num_q_heads, int num_kv_heads, int block_size, int num_blocks, float scale,
                   void* out, unsigned int* err) {
  TcParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.q_start = q_start;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.err = err;
  prm.max_blocks = max_blocks;
  prm.num_q_heads = num_q_heads;
  prm.group = num_q_heads / num_kv_heads;
  prm.tokens_per_block = kTcQTiles * kTcRows / prm.group;
  prm.max_q_len = max_q_len;
  prm.block_size = block_size;
  prm.log2_bs = ilog2(block_size);
  prm.box_rows = block_size < kTcKeys ? block_size : kTcKeys;
  prm.num_blocks = num_blocks;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  prm.k_scale = nullptr;
  prm.v_scale = nullptr;
  prm.k_src = nullptr;
  prm.v_src = nullptr;
  prm.num_kv_heads = num_kv_heads;
  return prm;
}

}  // namespace

bool prefill_tc_supported(int head_dim, int block_size, int group) {
  return (head_dim == 64 || head_dim == 128) && block_size >= 1 && group >= 1 &&
         group <= kTcQTiles * kTcRows;
}

pa_status launch_prefill_tc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks,
                            const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                            int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, float scale, void* out,
                            unsigned int* err, cudaStream_t stream) {
  const int G = num_q_heads / num_kv_heads;
  if (!prefill_tc_supported(head_dim, block_size, G)) return PA_ERR_UNSUPPORTED;
  TcParams prm = tc_params(q, block_tables, max_blocks, context_lens, q_start, max_q_len,
                           num_q_heads, num_kv_heads, block_size, num_blocks, scale, out, err);
  prm.k_src = k_cache;
  prm.v_src = v_cache;
  const long long tiles = ((long long)max_q_len + prm.tokens_per_block - 1) / prm.tokens_per_block;
  if (tiles > 0x7fffffffLL || num_kv_heads > 65535 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  const long long rows = (long long)num_blocks * block_size;
  if (block_size < 8) {  // the cp.async gather: no tensor maps
    return head_dim == 128 ? launch_tc<128>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream)
                           : launch_tc<64>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream);
  }
  if (head_dim == 128) {
    if (!make_tc_map<128>(&mk, k_cache, num_kv_heads, rows, prm.box_rows) ||
        !make_tc_map<128>(&mv, v_cache, num_kv_heads, rows, prm.box_rows))
      return PA_ERR_CUDA;
    return launch_tc<128>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream);
  }
  if (!make_tc_map<64>(&mk, k_cache, num_kv_heads, rows, prm.box_rows) ||
      !make_tc_map<64>(&mv, v_cache, num_kv_heads, rows, prm.box_rows))
    return PA_ERR_CUDA;
  return launch_tc<64>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream);
}

}  // namespace pa

namespace pa {

pa_status launch_prefill_tc_fp8(const void* q, const void* k_codes, const void* v_codes,
                                const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, int max_blocks,
                                const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                                int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, float scale, void* out,
                                unsigned int* err, cudaStream_t stream) {
  const int G = num_q_heads / num_kv_heads;
  if (head_dim != 128 || !prefill_tc_supported(head_dim, block_size, G)) return PA_ERR_UNSUPPORTED;
  TcParams prm = tc_params(q, block_tables, max_blocks, context_lens, q_start, max_q_len,
                           num_q_heads, num_kv_heads, block_size, num_blocks, scale, out, err);
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.k_src = k_codes;
  prm.v_src = v_codes;
  prm.box_rows = block_size < 32 ? block_size : 32;  // at most 4 code groups a box (kCodePos)
  const long long tiles = ((long long)max_q_len + prm.tokens_per_block - 1) / prm.tokens_per_block;
  if (tiles > 0x7fffffffLL || num_kv_heads > 65535 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  const long long rows = (long long)num_blocks * block_size;
  if (block_size < 8)  // the cp.async gather: no tensor maps
    return launch_tc<128, true>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream);
  if (!make_tc_map_fp8(&mk, k_codes, num_kv_heads, rows, prm.box_rows) ||
      !make_tc_map_fp8(&mv, v_codes, num_kv_heads, rows, prm.box_rows))
    return PA_ERR_CUDA;
  return launch_tc<128, true>(mk, mv, prm, tiles, num_kv_heads, num_seqs, stream);
}

}  // namespace pa
