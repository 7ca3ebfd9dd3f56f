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
// One thread block per (KV head, sequence, row tile counted from the chunk's
// end), 256 query rows = two M = 128 tiles (row = token * G + head; a tile
// covers floor(256 / G) tokens), 10 warps:
//   warp 0     loader: K and V tiles of 128 keys through one 3-slot ring (K_j
//              then V_j), each block's rows fetched by two TMA boxes {64
//              columns, rows} with the 128-byte swizzle, i.e. the K-major
//              layout the MMA reads for K and the MN-major one for V;
//   warp 1     allocates 512 TMEM columns (S_0, S_1 scores, O_0, O_1 outputs)
//              and one lane issues every MMA:
//                S_w = Q_w K_j^T  (M 128, N 128 keys, K 128 = head_dim)
//                O_w += P_w V_j   (M 128, N 128 = head_dim, K 128 keys)
//              in the order S_0(j), S_1(j), PV_0(j), S_0(j+1), PV_1(j),
//              S_1(j+1), ... so that the tensor cores work on one tile's
//              products while the other tile's softmax runs;
//   warps 2-9  two softmax warpgroups, one per Q tile, one thread per row:
//              read the row's 128 scores from TMEM, apply the causal limit,
//              take the online softmax in base 2 (the running output is
//              rescaled only when the running max grew by more than 2^8 --
//              exact, as the final division uses the same stale max), write
//              P as bf16 into shared memory in the K-major swizzled layout,
//              and after the last tile divide O by the row sum and store bf16.
// The key range of a block is [0, last position of its last token]; the
// rows past a row's own position in the diagonal tiles are masked, and V
// rows past the block's last position are zeroed before the last P.V (they
// may be unwritten slots).

#include <cudaTypedefs.h>
#include <math.h>

#include <cstring>
#include <mutex>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_umma.cuh"
#include "pagedkv.h"

namespace pa {
namespace {

constexpr int kTcD = 128;                          // head_dim
constexpr int kTcRows = 128;                       // rows per Q tile (MMA M)
constexpr int kTcQTiles = 2;                       // Q tiles per block
constexpr int kTcKeys = 128;                       // keys per K/V tile
constexpr int kTcSlots = 3;                        // K/V ring slots
constexpr int kTcPanel = kTcRows * 128;            // one 64-column panel: 16 KB
constexpr int kTcTileBytes = 2 * kTcPanel;         // 128 rows x 256 B: 32 KB
constexpr int kTcSoftmaxWarps = 4 * kTcQTiles;
constexpr int kTcThreads = (2 + kTcSoftmaxWarps) * 32;
constexpr uint32_t kTcCols = 512;                  // TMEM columns
constexpr float kRescaleLog2 = 8.0f;               // rescale O when the max grows by > 2^8

struct TcSmem {
  static constexpr int kQ = 0;                                   // Q_0, Q_1
  static constexpr int kP = kQ + kTcQTiles * kTcTileBytes;       // P_0, P_1
  static constexpr int kRing = kP + kTcQTiles * kTcTileBytes;    // 3 K/V slots
  static constexpr int kBar = kRing + kTcSlots * kTcTileBytes;
  // barriers: full[3], empty[3], s_full[2], p_full[2], o_done[2], q_ready, drain
  static constexpr int kNumBars = 2 * kTcSlots + 3 * kTcQTiles + 2;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kFlag = kTmemSlot + 8;
  static constexpr int kAlloc = kFlag + 8 + 1024;                // + 1024-byte alignment
};
static_assert(TcSmem::kAlloc <= 232448, "over the 227 KB of shared memory per block");

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
};

// Waits for the phase of `bar` with the given parity; false once the block
// is aborting (flag set) or after kWaitLimitNs.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Records a lost wait (unless the block is already aborting) and aborts.
__device__ __forceinline__ void give_up(volatile int* abort_flag, unsigned int* err,
                                        unsigned int bit) {
  if (!*abort_flag) atomicOr(err, bit);
  *abort_flag = 1;
}

// Byte offset of 16-byte chunk c (0..15) of row r in a two-panel swizzled tile.
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) {
  return (uint32_t)((c >> 3) * kTcPanel + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kvh = blockIdx.x;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int TPB = p.tokens_per_block;
  const int row0 = p.q_start[b];
  const int n = p.q_start[b + 1] - row0;
  const int tok_hi = n - (int)blockIdx.z * TPB;  // this block: chunk tokens [tok_lo, tok_hi)
  if (tok_hi <= 0) return;
  if (n > p.max_q_len) {
    if (threadIdx.x == 0 && blockIdx.z == 0) atomicOr(p.err, kErrShape);
    return;
  }
  const int tok_lo = tok_hi - TPB > 0 ? tok_hi - TPB : 0;
  int ctx = p.context_lens[b];
  const int cap = p.max_blocks << p.log2_bs;
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  const int pos_base = ctx - n;                 // position of the chunk's token 0
  const int pos_last = pos_base + tok_hi - 1;   // the block's last attended position
  const int n_tiles = pos_last >= 0 ? pos_last / kTcKeys + 1 : 0;

  // softmax thread -> (Q tile, row); rows past the block's tokens are padding
  const int sw = warp - 2;                      // softmax warp 0..7
  const int qt = sw >> 2;                       // Q tile
  const int quarter = warp & 3;                 // TMEM lanes 32 * quarter ..
  const int r = quarter * 32 + lane;            // row within the Q tile
  const int R = qt * kTcRows + r;               // row within the block
  const bool row_valid = sw >= 0 && R / G < tok_hi - tok_lo;
  const int tok = tok_lo + R / G;
  const int pos = row_valid ? pos_base + tok : -1;
  const size_t out_off =
      ((size_t)(row0 + tok) * p.num_q_heads + (size_t)kvh * G + (R % G)) * kTcD;

  if (n_tiles == 0) {  // no position to attend: zero rows, nothing else
    if (row_valid) {
      uint4* o = reinterpret_cast<uint4*>(p.out + out_off);
      for (int c = 0; c < kTcD / 8; ++c) o[c] = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TcSmem::kBar);
  uint64_t* empty = full + kTcSlots;
  uint64_t* s_full = empty + kTcSlots;
  uint64_t* p_full = s_full + kTcQTiles;
  uint64_t* o_done = p_full + kTcQTiles;
  uint64_t* q_ready = o_done + kTcQTiles;
  uint64_t* drain = q_ready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + TcSmem::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + TcSmem::kFlag);
  const uint32_t sQ = smem_u32(smem + TcSmem::kQ);
  const uint32_t sP = smem_u32(smem + TcSmem::kP);
  const uint32_t ring = smem_u32(smem + TcSmem::kRing);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int w = 0; w < kTcQTiles; ++w) {
      mbar_init(&s_full[w], 1);
      mbar_init(&p_full[w], kTcRows);
      mbar_init(&o_done[w], 1);
    }
    mbar_init(q_ready, kTcQTiles * kTcRows);
    mbar_init(drain, 1);
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
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
      const int32_t* bt = p.block_tables + (size_t)b * p.max_blocks;
      const int rb = p.box_rows;
      const int boxes = kTcKeys / rb;
      int L = 0;
      for (; L < 2 * n_tiles; ++L) {
        const int slot = L % kTcSlots;
        if (L >= kTcSlots &&
            !wait_or_abort(&empty[slot], ((L / kTcSlots) - 1) & 1, abort_flag)) {
          give_up(abort_flag, p.err, kErrWaitEmpty);
          break;
        }
        const int j = L >> 1;
        const CUtensorMap* map = (L & 1) ? &tmap_v : &tmap_k;
        const int nbox = min(boxes, (pos_last - j * kTcKeys) / rb + 1);
        mbar_arrive_expect_tx(&full[slot], (uint32_t)(nbox * rb * 256));
        const uint32_t dst = ring + slot * kTcTileBytes;
        for (int i = 0; i < nbox; ++i) {
          const int key0 = j * kTcKeys + i * rb;
          const int blk = bt[key0 >> p.log2_bs];
          // a block id outside the pool reads zeros (a box wholly out of range)
          const int y = (blk >= 0 && blk < p.num_blocks)
                            ? blk * p.block_size + (key0 & (p.block_size - 1))
                            : -rb;
          tma_load_2d(dst + i * rb * 128, map, kvh * kTcD, y, &full[slot]);
          tma_load_2d(dst + kTcPanel + i * rb * 128, map, kvh * kTcD + 64, y, &full[slot]);
        }
      }
      // every copy issued must land before the block ends
      for (int s = 0; s < kTcSlots; ++s) {
        if (L <= s) continue;
        const int last = s + ((L - 1 - s) / kTcSlots) * kTcSlots;
        if (!mbar_wait(&full[s], (last / kTcSlots) & 1)) atomicOr(p.err, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = umma_idesc_bf16(kTcRows, kTcKeys, false);
      constexpr uint32_t kIdO = umma_idesc_bf16(kTcRows, kTcD, true);
      auto issue_s = [&](int w, int L) {  // S_w = Q_w K^T, K in slot L % 3
        const uint32_t qa = sQ + w * kTcTileBytes;
        const uint32_t kb = ring + (L % kTcSlots) * kTcTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTcD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTcPanel + (kk & 3) * 32;
          umma_bf16_ss(tmem + w * kTcKeys, umma_desc_sw128(qa + off, 16, 1024),
                       umma_desc_sw128(kb + off, 16, 1024), kIdS, kk > 0);
        }
      };
      auto issue_pv = [&](int w, int L, int j) {  // O_w += P_w V, V in slot L % 3
        const uint32_t pa_ = sP + w * kTcTileBytes;
        const uint32_t vb = ring + (L % kTcSlots) * kTcTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTcPanel + (kk & 3) * 32;
          umma_bf16_ss(tmem + 2 * kTcKeys + w * kTcD, umma_desc_sw128(pa_ + off, 16, 1024),
                       umma_desc_sw128(vb + kk * 2048, kTcPanel, 1024), kIdO,
                       (j > 0 || kk > 0) ? 1u : 0u);
        }
      };
      auto landed = [&](int L) {
        return wait_or_abort(&full[L % kTcSlots], (L / kTcSlots) & 1, abort_flag);
      };
      bool ok = wait_or_abort(q_ready, 0, abort_flag) && landed(0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        umma_commit(&s_full[0]);
        issue_s(1, 0);
        umma_commit(&s_full[1]);
        umma_commit(&empty[0]);
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int LV = 2 * j + 1, LK1 = 2 * j + 2;
        const bool more = j + 1 < n_tiles;
        if (!(ok = landed(LV) && wait_or_abort(&p_full[0], j & 1, abort_flag))) break;
        tc_fence_after();
        issue_pv(0, LV, j);
        umma_commit(&o_done[0]);
        if (more) {
          if (!(ok = landed(LK1))) break;
          issue_s(0, LK1);
          umma_commit(&s_full[0]);
        }
        if (!(ok = wait_or_abort(&p_full[1], j & 1, abort_flag))) break;
        tc_fence_after();
        issue_pv(1, LV, j);
        umma_commit(&o_done[1]);
        umma_commit(&empty[LV % kTcSlots]);
        if (more) {
          issue_s(1, LK1);
          umma_commit(&s_full[1]);
          umma_commit(&empty[LK1 % kTcSlots]);
        }
      }
      if (!ok) give_up(abort_flag, p.err, kErrWaitFull);
      umma_commit(drain);  // every MMA issued is done before TMEM is freed
      if (!mbar_wait(drain, 0)) atomicOr(p.err, kErrDrain);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lanes = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t t_s = lanes + qt * kTcKeys;               // S of this tile
    const uint32_t t_o = lanes + 2 * kTcKeys + qt * kTcD;    // O of this tile
    const uint32_t my_q = sQ + qt * kTcTileBytes;
    const uint32_t my_p = sP + qt * kTcTileBytes;
    {  // this row of Q into the K-major swizzled tile (zeros for padding rows)
      const __nv_bfloat16* src = p.q + out_off;
#pragma unroll 4
      for (int c = 0; c < kTcD / 8; ++c) {
        const uint4 v = row_valid ? ld_global_nc_v4(src + 8 * c) : make_uint4(0, 0, 0, 0);
        st_shared_v4(my_q + sw_chunk(r, c), v.x, v.y, v.z, v.w);
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;  // running max, log2 units (the one P and O use)
    float l_run = 0.f;        // running row sum of P
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = __all_sync(0xffffffffu, wait_or_abort(&s_full[qt], j & 1, abort_flag));
      if (ok && j > 0)  // PV of tile j-1 is done: its P buffer is free, O is current
        ok = __all_sync(0xffffffffu, wait_or_abort(&o_done[qt], (j - 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float s[kTcKeys];
      tmem_ld64_sync(t_s, *reinterpret_cast<float(*)[64]>(&s[0]));
      tmem_ld64_sync(t_s + 64, *reinterpret_cast<float(*)[64]>(&s[64]));
      const int lim = pos - j * kTcKeys;  // keys 0 .. lim of the tile are visible
      if (lim < kTcKeys - 1) {
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) s[c] = c <= lim ? s[c] : -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTcKeys; ++c) mx = fmaxf(mx, s[c]);
      const float m_tile = mx * sl2;
      const bool grow = m_tile > m_run + kRescaleLog2;  // also the first finite max
      const float m_use = grow ? m_tile : m_run;
      const float alpha = grow ? ex2_approx(m_run - m_use) : 1.f;  // 0 when m_run = -inf
      const float ms = m_use == -INFINITY ? 0.f : m_use;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < kTcKeys / 8; ++c) {
        uint32_t w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float e0 = ex2_approx(fmaf(s[8 * c + 2 * i], sl2, -ms));
          const float e1 = ex2_approx(fmaf(s[8 * c + 2 * i + 1], sl2, -ms));
          sum += e0 + e1;
          w4[i] = pack_bf16x2(e0, e1);
        }
        st_shared_v4(my_p + sw_chunk(r, c), w4[0], w4[1], w4[2], w4[3]);
      }
      l_run = l_run * alpha + sum;
      m_run = m_use;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {  // rescale the running output
#pragma unroll 1
        for (int c = 0; c < kTcD; c += 32) {
          float o[32];
          tmem_ld32_sync(t_o + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32_sync(t_o + c, o);
        }
      }
      if (qt == 0 && j == n_tiles - 1) {
        // the last V tile: zero its rows past the block's last position
        const int first = pos_last - j * kTcKeys + 1;
        if (first < kTcKeys) {
          const int LV = 2 * j + 1;
          ok = __all_sync(0xffffffffu, wait_or_abort(&full[LV % kTcSlots],
                                                      (LV / kTcSlots) & 1, abort_flag));
          if (ok) {
            const uint32_t vt = ring + (LV % kTcSlots) * kTcTileBytes;
            for (int i = r; i < (kTcKeys - first) * 16; i += kTcRows) {
              const int row = first + (i >> 4), c = i & 15;
              st_shared_v4(vt + (c >> 3) * kTcPanel + row * 128 + (c & 7) * 16, 0, 0, 0, 0);
            }
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[qt]);
      if (!ok) break;
    }
    if (ok)
      ok = __all_sync(0xffffffffu,
                      wait_or_abort(&o_done[qt], (n_tiles - 1) & 1, abort_flag));
    if (!ok) {
      give_up(abort_flag, p.err, kErrWaitFull);
    } else {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.out + out_off);
#pragma unroll 1
      for (int c = 0; c < kTcD; c += 32) {
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

// cuTensorMapEncodeTiled through the runtime's driver entry point.
PFN_cuTensorMapEncodeTiled_v12000 tc_map_encoder() {
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

// 2-D map over a bf16 cache as [num_blocks * block_size rows, Hkv * 128
// columns], box {64 columns, box_rows rows}, 128-byte swizzle.
bool make_tc_map(CUtensorMap* map, const void* base, int hkv, long long rows, int box_rows) {
  auto enc = tc_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)hkv * kTcD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)hkv * kTcD * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(int head_dim, int block_size, int group) {
  return head_dim == kTcD && block_size >= 8 && group >= 1 && group <= kTcQTiles * kTcRows;
}

pa_status launch_prefill_tc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks,
                            const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                            int max_q_len, int num_q_heads, int num_kv_heads, int block_size,
                            int num_blocks, float scale, void* out, unsigned int* err,
                            cudaStream_t stream) {
  const int G = num_q_heads / num_kv_heads;
  if (!prefill_tc_supported(kTcD, block_size, G)) return PA_ERR_UNSUPPORTED;
  TcParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.q_start = q_start;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.err = err;
  prm.max_blocks = max_blocks;
  prm.num_q_heads = num_q_heads;
  prm.group = G;
  prm.tokens_per_block = kTcQTiles * kTcRows / G;
  prm.max_q_len = max_q_len;
  prm.block_size = block_size;
  prm.log2_bs = ilog2(block_size);
  prm.box_rows = block_size < kTcKeys ? block_size : kTcKeys;
  prm.num_blocks = num_blocks;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  const long long tiles = ((long long)max_q_len + prm.tokens_per_block - 1) / prm.tokens_per_block;
  if (tiles > 65535 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  const long long rows = (long long)num_blocks * block_size;
  if (!make_tc_map(&mk, k_cache, num_kv_heads, rows, prm.box_rows) ||
      !make_tc_map(&mv, v_cache, num_kv_heads, rows, prm.box_rows))
    return PA_ERR_CUDA;
  const pa_status s = prepare_kernel(reinterpret_cast<const void*>(prefill_tc_kernel),
                                     kTcThreads, TcSmem::kAlloc, nullptr);
  if (s != PA_OK) return s;
  const dim3 grid(num_kv_heads, num_seqs, (unsigned)tiles);
  prefill_tc_kernel<<<grid, kTcThreads, TcSmem::kAlloc, stream>>>(mk, mv, prm);
  return launch_status();
}

}  // namespace pa
