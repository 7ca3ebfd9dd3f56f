// pa_tc_common.cuh -- pieces the tcgen05 attention kernels share: the K/V
// operand-slot layout that one 4-D TMA box per paged block writes (bf16 rows,
// or e4m3 codes that converter warps widen in place), bounded mbarrier waits
// with a block-wide abort flag, shared-memory vector moves, packed fp32
// arithmetic, and the host-side tensor maps over the caches.
#pragma once

#include <cudaTypedefs.h>
#include <math.h>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_umma.cuh"

namespace pa {
namespace {

constexpr int kTcRows = 128;                       // rows per Q tile (MMA M)
constexpr int kTcKeys = 128;                       // keys per K/V tile
constexpr int kKvHalf = 1024;                      // 8 rows of one 64-column panel
constexpr int kRingBudget = 5 * 32768;             // shared memory of the K/V ring
constexpr int kTcConvWarps = 2;                    // e4m3: warps widening the codes
constexpr int kCodeHalf = kTcKeys * 128;           // e4m3: codes land in a slot's upper 16 KB

// e4m3 tiles are widened in place: code group k (8 keys x 128 codes, 1 KB)
// lands at kCodeHalf + kCodePos(k) KB of its slot, and f16 group g is written
// at g * 2 KB. Converter warp 0 widens groups 0-3 and 8-11, warp 1 groups 4-7
// and 12-15, reading all of its eight groups' codes before writing any;
// kCodePos puts each warp's codes under the f16 groups the same warp
// writes later (f16 groups 8-11 cover code positions 0-7, 12-15 cover 8-15),
// so no warp writes over codes the other has yet to read.
__host__ __device__ constexpr int kCodePos(int k) {
  return (k >= 4 && k < 8) ? k + 4 : ((k >= 8 && k < 12) ? k - 4 : k);
}

// Sizes that follow head_dim (64 or 128): a row is D / 64 panels of 64
// columns (128 bytes). K/V slots hold 8-row groups of all panels: group g,
// panel h at g * kKvGroup + h * kKvHalf (each 1 KB = 8 rows of 128 bytes,
// swizzled), the layout one 4-D TMA box per paged block writes.
template <int D, bool kFp8 = false>
struct TcShape {
  static constexpr int kHalves = D / 64;
  static constexpr int kQBytes = kTcRows * D * 2;     // one Q tile
  static constexpr int kKvBytes = kTcKeys * D * 2;    // one K or V tile: a ring slot
  static constexpr int kKvGroup = kHalves * kKvHalf;
  static constexpr int kSlots = kRingBudget / kKvBytes;  // 5 at D 128, 10 at D 64
};
// Shared-memory offset, within an operand slot, of 16-byte chunk c of key row
// `key` of a bf16 K/V tile ([group][panel][row], 128-byte swizzle), or of a
// code row of an e4m3 tile (the slot's upper half, group k at kCodePos(k)).
template <int D, bool kFp8>
__device__ __forceinline__ uint32_t kv_chunk_offset(int key, int c) {
  const int g = key >> 3, r = key & 7;
  if constexpr (kFp8)
    return (uint32_t)(kCodeHalf + kCodePos(g) * 1024 + r * 128 + ((c ^ r) << 4));
  else
    return (uint32_t)(g * (D / 64) * kKvHalf + (c >> 3) * kKvHalf + r * 128 +
                      (((c & 7) ^ r) << 4));
}

static_assert(kCodeHalf == TcShape<128>::kKvBytes / 2, "e4m3 codes fill a 128-dim slot's upper half");

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

// 4-D TMA tile load (coordinates innermost first), completion on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (v, v) as one 64-bit register pair.
__device__ __forceinline__ uint64_t splat2(float v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
  return r;
}

// (d0, d1) = (a0, a1) * b2 + c2 (b2, c2 packed pairs), one packed instruction.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, uint64_t b2,
                                     uint64_t c2) {
  asm("{\n\t.reg .b64 x, w;\n\tmov.b64 x, {%2, %3};\n\t"
      "fma.rn.f32x2 w, x, %4, %5;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "l"(b2), "l"(c2));
}

// (s0, s1) += (a0, a1), one packed instruction.
__device__ __forceinline__ void add2(float& s0, float& s1, float a0, float a1) {
  asm("{\n\t.reg .b64 x, y, w;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 w, x, y;\n\tmov.b64 {%0, %1}, w;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

// (s0, s1) += the two 16-bit halves of `pr` (f16 or bf16, low half to s0),
// each added to fp32 by one mixed-precision add.
template <bool kF16>
__device__ __forceinline__ void add_halves(float& s0, float& s1, uint32_t pr) {
  if constexpr (kF16)
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.f16 %0, l, %0;\n\tadd.rn.f32.f16 %1, h, %1;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "r"(pr));
  else
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(s0), "+f"(s1)
        : "r"(pr));
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// An e4m3 tile in an operand slot of head_dim 128 (K_j or V_j of 128 keys),
// widened in place by converter warp cw (0 or 1): code group k (8 rows x 128
// codes, 128-byte swizzle) at kCodeHalf + kCodePos(k) KB -> f16 group k at
// k * 2 KB ([panel][row], 64 f16 columns a panel, the same swizzle). Warp w
// takes groups 4w..4w+3 and 8+4w..: a lane first reads its sixteen 16-byte
// code chunks of the eight groups, the warp syncs, then it writes their
// 16-byte f16 chunks. Chunk u of lane l (t = 32 u + l): row 2 (t / 16) + r
// and chunk 4 (r ^ p) + t % 4, with r = t / 4 % 2, p = t / 8 % 2, so that each
// 8-thread access phase reads and writes 8 distinct bank quads. Rows >= keep:
// V rows become zeros (they may be unwritten slots), K rows are left as they
// are (every score of theirs is masked).
__device__ __forceinline__ void widen_e4m3_slot(uint32_t base, int cw, int lane, int keep,
                                                bool is_v) {
  constexpr int kGroupBytes = TcShape<128, true>::kKvGroup;  // 8 f16 rows of both panels
  // all eight of this warp's groups (4cw..4cw+3 and 8+4cw..): every code is
  // read before any f16 write
  uint4 v[8][2];
  int row[2], c[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int t = 32 * u + lane;
    const int rp = (t >> 2) & 1;
    row[u] = 2 * (t >> 4) + rp;                       // row within a group
    c[u] = ((rp ^ ((t >> 3) & 1)) << 2) | (t & 3);    // codes 16c .. 16c + 15
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int g = 4 * cw + 8 * (k >> 2) + (k & 3);
#pragma unroll
    for (int u = 0; u < 2; ++u)
      v[k][u] = 8 * g + row[u] < keep
                    ? ld_shared_v4(base + kCodeHalf + kCodePos(g) * 1024 + row[u] * 128 +
                                   ((c[u] ^ row[u]) << 4))
                    : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncwarp();  // every code of the eight groups is read before their f16 writes
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int g = 4 * cw + 8 * (k >> 2) + (k & 3);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!is_v && 8 * g + row[u] >= keep) continue;  // masked K rows: left as they are
      const uint32_t d = base + g * kGroupBytes + (c[u] >> 2) * kKvHalf + row[u] * 128;
      uint32_t h[8];
      e4m3x4_to_f16x2x2(v[k][u].x, h[0], h[1]);
      e4m3x4_to_f16x2x2(v[k][u].y, h[2], h[3]);
      e4m3x4_to_f16x2x2(v[k][u].z, h[4], h[5]);
      e4m3x4_to_f16x2x2(v[k][u].w, h[6], h[7]);
      st_shared_v4(d + ((((2 * c[u]) & 7) ^ row[u]) << 4), h[0], h[1], h[2], h[3]);
      st_shared_v4(d + ((((2 * c[u] + 1) & 7) ^ row[u]) << 4), h[4], h[5], h[6], h[7]);
    }
  }
}

// ---------------------------------------------------------------- host

// 4-D map over a bf16 cache [rows = num_blocks * block_size, Hkv, D]:
// (64 columns, 8 rows of a group, the 128-byte column panels of all heads,
// 8-row groups), box {64, 8, D / 64, box_rows / 8}: one box lands box_rows rows
// of one head, all its panels, as [group][panel][row] 1 KB swizzled atoms.
// (The panels' stride, 128 B, is below the rows'.)
template <int D>
bool make_tc_map(CUtensorMap* map, const void* base, int hkv, long long rows, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || rows % 8 != 0 || box_rows % 8 != 0) return false;
  const cuuint64_t row_bytes = (cuuint64_t)hkv * D * 2;
  cuuint64_t dims[4] = {64, 8, (cuuint64_t)hkv * TcShape<D>::kHalves, (cuuint64_t)(rows / 8)};
  cuuint64_t strides[3] = {row_bytes, 128, 8 * row_bytes};
  cuuint32_t box[4] = {64, 8, (cuuint32_t)TcShape<D>::kHalves, (cuuint32_t)(box_rows / 8)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// The same view of an e4m3 cache [rows, Hkv, 128] (uint8): (128 columns,
// 8 rows, Hkv panels, 8-row groups), box {128, 8, 1, box_rows / 8}: one box
// lands box_rows codes rows of one head as [group][row][128 B] 1 KB swizzled
// atoms. L2 promotion follows the 128-byte row.
bool make_tc_map_fp8(CUtensorMap* map, const void* base, int hkv, long long rows, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || rows % 8 != 0 || box_rows % 8 != 0) return false;
  const cuuint64_t row_bytes = (cuuint64_t)hkv * 128;
  cuuint64_t dims[4] = {128, 8, (cuuint64_t)hkv, (cuuint64_t)(rows / 8)};
  cuuint64_t strides[3] = {row_bytes, 128, 8 * row_bytes};
  cuuint32_t box[4] = {128, 8, 1, (cuuint32_t)(box_rows / 8)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa
