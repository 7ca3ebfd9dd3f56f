// pa_tile.cuh -- the K/V tile shared by the decode kernels (16 tokens of
// bf16, 32 tokens of e4m3): how a tile is fetched into shared memory and how
// one warp folds it into its running attention state for the GQA group of one
// KV head (or, for several query tokens, for 8 (token, head) columns).
//
// The tile math is the streaming softmax of "Text Generation Inference:
// Hugging Face's production-grade LLM inference server" (section "Under the
// Hood: Flash Attention"): per tile, the new running max m' per query head,
// P = exp(S - m'), l = exp(m - m') l + sum P, O = exp(m - m') O + P V. It runs
// in base 2 (scale * log2(e) folded into one multiply) and in transposed MMA
// form so that the GQA group (up to 8 query heads) is the n = 8 side:
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]    (m16n8k16, bf16 -> fp32)
//   O^T[D x 8 heads]     += V^T[D x 16] . P^T[16 x 8]
// The score accumulator becomes the B operand of the second product through a
// movmatrix transpose of each 8x8 half.
//
// Shared-memory tile layout: K then V; each is D/64 column halves of 16 rows x
// 128 bytes with the 128-byte swizzle (16-byte chunk c of row r stored at
// chunk c ^ (r & 7)), the layout TMA boxes {64 columns, 16 rows} -- or one
// 3-D box {64 columns, 16 rows, 2 halves} -- with CU_TENSOR_MAP_SWIZZLE_128B
// write. ldmatrix reads of 8 rows then hit 8 distinct bank groups.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kTile = 16;                // tokens per tile (the m of S^T)
constexpr int kMaxGroup = 8;             // query heads per KV head (the n of the MMA)
constexpr int kHalfBytes = kTile * 128;  // one 64-column half of a tile

// EB: bytes per cache element (2 = bf16, 1 = e4m3); TT: tokens per tile (16
// for bf16, 32 for e4m3, so both stages hold 8 KB). A tile row is D * EB
// bytes, stored as D * EB / 128 column "halves" of TT rows x 128 bytes.
template <int D, int EB = 2, int TT = kTile>
struct TileGeom {
  static constexpr int kRowBytes = D * EB;
  static constexpr int kHalves = kRowBytes / 128;
  static_assert(kHalves >= 1 && kRowBytes % 128 == 0, "tile rows must be multiples of 128 bytes");
  static constexpr int kBoxCols = 128 / EB;               // TMA box width in elements
  static constexpr int kHalfStride = TT * 128;            // bytes of one column half
  static constexpr int kKVBytes = kHalves * kHalfStride;  // one K (or V) tile
  static constexpr int kStageBytes = 2 * kKVBytes;        // K then V
};

// Running state of one warp for the GQA group of one KV head.
template <int D>
struct AttnState {
  float o[D / 16][4];  // O^T fragments: dims (mt*16 + lane/4 [+8]) x heads (2*(lane%4) [+1])
  float m0, m1;        // running max (base 2) of heads 2*(lane%4), 2*(lane%4)+1
  float l0, l1;        // this lane's part of the running sums of those heads

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
  }

  // Sum the running sums over the 8 lanes that share a head pair.
  __device__ __forceinline__ void reduce_l() {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }
};

// B-operand fragments of Q^T for query heads [0, G) of a group; `qg` points
// at head 0 of the group. Heads >= G are zero.
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[D / 16][2], const __nv_bfloat16* qg,
                                             int G, int lane) {
  const int g = lane >> 2;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) qf[ks][0] = qf[ks][1] = 0u;
  if (g < G) {
    const unsigned int* row =
        reinterpret_cast<const unsigned int*>(qg + (size_t)g * D + 2 * (lane & 3));
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qf[ks][0] = __ldg(row + ks * 8);
      qf[ks][1] = __ldg(row + ks * 8 + 4);
    }
  }
}

// The same fragments from a shared-memory copy of the group's q rows
// (bf16 [G][D]).
template <int D>
__device__ __forceinline__ void load_q_frags_smem(uint32_t (&qf)[D / 16][2],
                                                  const __nv_bfloat16* sq, int G, int lane) {
  const int g = lane >> 2;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) qf[ks][0] = qf[ks][1] = 0u;
  if (g < G) {
    const unsigned int* row = reinterpret_cast<const unsigned int*>(sq + g * D + 2 * (lane & 3));
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qf[ks][0] = row[ks * 8];
      qf[ks][1] = row[ks * 8 + 4];
    }
  }
}

// Fold one tile (shared-memory K at sK, V at sV) into `st`. Rows >= valid are
// masked: their scores become -inf and their V rows are zeroed in registers,
// so stale or NaN slots past the end of a sequence cannot leak into O.
template <int D>
__device__ __forceinline__ void attend_tile(AttnState<D>& st, uint32_t sK, uint32_t sV,
                                            const uint32_t (&qf)[D / 16][2], int valid,
                                            float scale_log2, int lane) {
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
  const int r0 = lane >> 2;
  const int tk = 2 * (lane & 3);
  const float y0 = r0 < valid ? s[0] * scale_log2 : -INFINITY;
  const float y1 = r0 < valid ? s[1] * scale_log2 : -INFINITY;
  const float y2 = r0 + 8 < valid ? s[2] * scale_log2 : -INFINITY;
  const float y3 = r0 + 8 < valid ? s[3] * scale_log2 : -INFINITY;
  float mx0 = fmaxf(y0, y2), mx1 = fmaxf(y1, y3);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
  const float a0 = exp2f(st.m0 - mn0), a1 = exp2f(st.m1 - mn1);
  const uint32_t p01 = pack_bf16x2(exp2f(y0 - mn0), exp2f(y1 - mn1));
  const uint32_t p23 = pack_bf16x2(exp2f(y2 - mn0), exp2f(y3 - mn1));
  // the running sum adds the same bf16-rounded weights the PV product uses
  st.l0 = st.l0 * a0 + (bf16_lo(p01) + bf16_lo(p23));
  st.l1 = st.l1 * a1 + (bf16_hi(p01) + bf16_hi(p23));
  st.m0 = mn0;
  st.m1 = mn1;
  // O is rescaled only when some running max moved (a factor of exactly 1
  // leaves it unchanged, and after the first tiles the max rarely moves)
  if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      st.o[mt][0] *= a0;
      st.o[mt][1] *= a1;
      st.o[mt][2] *= a0;
      st.o[mt][3] *= a1;
    }
  }
  const uint32_t pb0 = movmatrix_trans(p01);  // P^T tokens 0-7 as the MMA's B operand
  const uint32_t pb1 = movmatrix_trans(p23);  // tokens 8-15

  // O^T += V^T . P^T (the V masks only on a partial tile)
  uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
  const bool masked = valid < kTile;
  if (masked) {
    vm01 = (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
    vm23 = (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
  }
  const int mi = lane >> 3;
  const int r = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int cg = 2 * mt + (mi & 1);
    uint32_t a[4];
    ldsm_x4_trans(sV + (cg >> 3) * kHalfBytes + r * 128 + (((cg & 7) ^ (r & 7)) << 4), a);
    if (masked) {
      a[0] &= vm01;
      a[1] &= vm01;
      a[2] &= vm23;
      a[3] &= vm23;
    }
    mma_bf16_16816(st.o[mt], a, pb0, pb1);
  }
}

// attend_tile for query columns with their own causal limits (several new
// tokens of one sequence side by side on the n = 8 side), NT groups of 8
// columns at once (the K and V fragments are read once for all groups;
// st[i], qf[i], valid_a[i], valid_b[i] belong to group i): rows >= valid_a
// (>= valid_b) are masked for this lane's column 2 (lane % 4) (its column
// + 1); V rows >= valid (the tile's end, >= both) are zeroed. A column whose
// every score so far is masked keeps m = -inf, l = 0, O = 0 (the exponents
// use 0 in place of a -inf maximum, so no NaN appears).
template <int D, int NT>
__device__ __forceinline__ void attend_tile_causal_nt(AttnState<D> (&st)[NT], uint32_t sK,
                                                      uint32_t sV,
                                                      const uint32_t (&qf)[NT][D / 16][2],
                                                      int valid, const int (&valid_a)[NT],
                                                      const int (&valid_b)[NT], float scale_log2,
                                                      int lane) {
  float s[NT][4];
#pragma unroll
  for (int i = 0; i < NT; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
  {
    const int r = lane & 15;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int cg = 2 * ks + (lane >> 4);
      uint32_t a[4];
      ldsm_x4(sK + (cg >> 3) * kHalfBytes + r * 128 + (((cg & 7) ^ (r & 7)) << 4), a);
#pragma unroll
      for (int i = 0; i < NT; ++i) mma_bf16_16816(s[i], a, qf[i][ks][0], qf[i][ks][1]);
    }
  }
  const int r0 = lane >> 2;
  const int tk = 2 * (lane & 3);
  uint32_t pb0[NT], pb1[NT];
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const float y0 = r0 < valid_a[i] ? s[i][0] * scale_log2 : -INFINITY;
    const float y1 = r0 < valid_b[i] ? s[i][1] * scale_log2 : -INFINITY;
    const float y2 = r0 + 8 < valid_a[i] ? s[i][2] * scale_log2 : -INFINITY;
    const float y3 = r0 + 8 < valid_b[i] ? s[i][3] * scale_log2 : -INFINITY;
    float mx0 = fmaxf(y0, y2), mx1 = fmaxf(y1, y3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st[i].m0, mx0), mn1 = fmaxf(st[i].m1, mx1);
    const float e0 = mn0 == -INFINITY ? 0.f : mn0, e1 = mn1 == -INFINITY ? 0.f : mn1;
    const float a0 = exp2f(st[i].m0 - e0), a1 = exp2f(st[i].m1 - e1);
    const uint32_t p01 = pack_bf16x2(exp2f(y0 - e0), exp2f(y1 - e1));
    const uint32_t p23 = pack_bf16x2(exp2f(y2 - e0), exp2f(y3 - e1));
    st[i].l0 = st[i].l0 * a0 + (bf16_lo(p01) + bf16_lo(p23));
    st[i].l1 = st[i].l1 * a1 + (bf16_hi(p01) + bf16_hi(p23));
    st[i].m0 = mn0;
    st[i].m1 = mn1;
    if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {  // only when a max moved
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        st[i].o[mt][0] *= a0;
        st[i].o[mt][1] *= a1;
        st[i].o[mt][2] *= a0;
        st[i].o[mt][3] *= a1;
      }
    }
    pb0[i] = movmatrix_trans(p01);
    pb1[i] = movmatrix_trans(p23);
  }
  uint32_t vm01 = 0xffffffffu, vm23 = 0xffffffffu;
  const bool masked = valid < kTile;
  if (masked) {
    vm01 = (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
    vm23 = (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
  }
  const int mi = lane >> 3;
  const int r = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int cg = 2 * mt + (mi & 1);
    uint32_t a[4];
    ldsm_x4_trans(sV + (cg >> 3) * kHalfBytes + r * 128 + (((cg & 7) ^ (r & 7)) << 4), a);
    if (masked) {
      a[0] &= vm01;
      a[1] &= vm01;
      a[2] &= vm23;
      a[3] &= vm23;
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) mma_bf16_16816(st[i].o[mt], a, pb0[i], pb1[i]);
  }
}

// ---------------------------------------------------------------------------
// FP8 (e4m3) tiles: a tile row is D bytes, 32 rows per tile. K and V bytes are read with
// ldmatrix, byte pairs standing in for b16 elements, and widened exactly to f16
// (cvt.rn.f16x2.e4m3x2) for an f16 MMA. Within a 16-dim chunk, lane l's A
// registers then hold dims 4c..4c+3 (c = l % 4) where the bf16 layout has
// dims 2c, 2c+1, 2c+8, 2c+9; Q takes the same k order (load_q_frags_fp8), which
// the dot product does not see. V comes through ldmatrix.trans: rows 0-7 of a
// 16-dim output tile hold the even dims of the chunk and rows 8-15 the odd
// ones (fp8_out_dim). The per-head scales are applied outside: the score
// factor includes k_scale, the output is multiplied by v_scale.

// Output dim of accumulator element (mt, upper rows?) of this lane.
__device__ __forceinline__ int fp8_out_dim(int mt, int lane, bool upper) {
  return mt * 16 + 2 * (lane >> 2) + (upper ? 1 : 0);
}

// Q^T B fragments (f16) in the fp8 tile's k order, from the group's bf16 q
// rows in shared memory; heads >= G are zero.
template <int D>
__device__ __forceinline__ void load_q_frags_fp8(uint32_t (&qf)[D / 16][2],
                                                 const __nv_bfloat16* sq, int G, int lane) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) qf[ks][0] = qf[ks][1] = 0u;
  if (g < G) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint2 v = *reinterpret_cast<const uint2*>(sq + g * D + ks * 16 + 4 * c);
      qf[ks][0] = pack_f16x2(bf16_lo(v.x), bf16_hi(v.x));
      qf[ks][1] = pack_f16x2(bf16_lo(v.y), bf16_hi(v.y));
    }
  }
}

// attend_tile for a 32-token e4m3 tile (head_dim 128: one 128-byte row per
// token, kFp8Tile rows per K or V half); score_scale_log2 = scale * k_scale *
// log2(e). Tokens 0-15 and 16-31 form two independent MMA chains; one
// softmax update covers all 32.
constexpr int kFp8Tile = 32;

// A operand (16 tokens x 16 k) of one e4m3 K ldmatrix result: k[i] holds 4
// codes (dims 4c..4c+3 of the k step) of token r0 (i even) or r0 + 8 (i odd),
// widened by e4m3x4_to_f16x2x2.
__device__ __forceinline__ void fp8_k_operand(const uint32_t (&k)[4], int i0, uint32_t (&a)[4]) {
  e4m3x4_to_f16x2x2(k[i0], a[0], a[2]);
  e4m3x4_to_f16x2x2(k[i0 + 1], a[1], a[3]);
}

template <int D>
__device__ __forceinline__ void attend_tile_fp8(AttnState<D>& st, uint32_t sK, uint32_t sV,
                                                const uint32_t (&qf)[D / 16][2], int valid,
                                                float score_scale_log2, int lane) {
  static_assert(D == 128, "e4m3 tiles are one 128-byte row per token");
  const int r = lane & 15;     // the row whose address this lane gives ldmatrix
  const int cadd = lane >> 4;  // chunk 2s (lanes 0-15) or 2s + 1 (lanes 16-31)
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
  float y[8];  // tokens r0, r0 + 8, r0 + 16, r0 + 24 x heads tk, tk + 1
  y[0] = r0 < valid ? sa[0] * score_scale_log2 : -INFINITY;
  y[1] = r0 < valid ? sa[1] * score_scale_log2 : -INFINITY;
  y[2] = r0 + 8 < valid ? sa[2] * score_scale_log2 : -INFINITY;
  y[3] = r0 + 8 < valid ? sa[3] * score_scale_log2 : -INFINITY;
  y[4] = r0 + 16 < valid ? sb[0] * score_scale_log2 : -INFINITY;
  y[5] = r0 + 16 < valid ? sb[1] * score_scale_log2 : -INFINITY;
  y[6] = r0 + 24 < valid ? sb[2] * score_scale_log2 : -INFINITY;
  y[7] = r0 + 24 < valid ? sb[3] * score_scale_log2 : -INFINITY;
  float mx0 = fmaxf(fmaxf(y[0], y[2]), fmaxf(y[4], y[6]));
  float mx1 = fmaxf(fmaxf(y[1], y[3]), fmaxf(y[5], y[7]));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
  const float a0 = exp2f(st.m0 - mn0), a1 = exp2f(st.m1 - mn1);
  uint32_t pw[4];  // f16 weights of tokens r0 + 8i, heads tk | tk + 1
#pragma unroll
  for (int i = 0; i < 4; ++i) pw[i] = pack_f16x2(exp2f(y[2 * i] - mn0), exp2f(y[2 * i + 1] - mn1));
  st.l0 = st.l0 * a0 + ((f16_lo(pw[0]) + f16_lo(pw[1])) + (f16_lo(pw[2]) + f16_lo(pw[3])));
  st.l1 = st.l1 * a1 + ((f16_hi(pw[0]) + f16_hi(pw[1])) + (f16_hi(pw[2]) + f16_hi(pw[3])));
  st.m0 = mn0;
  st.m1 = mn1;
  // O is rescaled only when some running max moved (a factor of exactly 1
  // leaves it unchanged, and after the first tiles the max rarely moves)
  if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
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
  // the V rows this lane's A fragments hold: tokens tk + 8i and tk + 8i + 1
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
    for (int half = 0; half < 2; ++half) {
      // bytes: (token 2c: dim 2j, 2j+1), (token 2c+1: dim 2j, 2j+1) -> even | odd pairs
      uint32_t e0 = byte_perm(va[2 * half], 0u, 0x3120u);      // tokens 0-7
      uint32_t e1 = byte_perm(va[2 * half + 1], 0u, 0x3120u);  // tokens 8-15
      uint32_t a[4];
      e4m3x4_to_f16x2x2(e0, a[0], a[1]);
      e4m3x4_to_f16x2x2(e1, a[2], a[3]);
      if (masked) {
        a[0] &= vm[0]; a[1] &= vm[0]; a[2] &= vm[1]; a[3] &= vm[1];
      }
      mma_f16_16816(st.o[2 * sidx + half], a, pb[0], pb[1]);
      e0 = byte_perm(vb[2 * half], 0u, 0x3120u);      // tokens 16-23
      e1 = byte_perm(vb[2 * half + 1], 0u, 0x3120u);  // tokens 24-31
      e4m3x4_to_f16x2x2(e0, a[0], a[1]);
      e4m3x4_to_f16x2x2(e1, a[2], a[3]);
      if (masked) {
        a[0] &= vm[2]; a[1] &= vm[2]; a[2] &= vm[3]; a[3] &= vm[3];
      }
      mma_f16_16816(st.o[2 * sidx + half], a, pb[2], pb[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// CUDA-core ablation of attend_tile: the same streaming-softmax math on FP32
// FMAs, kept to measure what the tensor-core form buys. A lane computes the
// 4 scores (token lane % 16, heads 4 * (lane / 16) ..+3) from shared memory
// (K tile, the group's q rows converted to fp32 once per unit), the weights
// go through a per-warp shared buffer, and a lane accumulates O for its D/32
// columns of all 8 heads.
template <int D>
struct AttnStateFma {
  static constexpr int kCols = D / 32;  // output columns per lane
  float o[kMaxGroup][kCols];
  float m[kMaxGroup];  // running max (base 2), the same in every lane
  float l[kMaxGroup];  // running sum, the same in every lane

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
#pragma unroll
      for (int j = 0; j < kCols; ++j) o[h][j] = 0.f;
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
  }
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// qs: fp32 [8][D] q rows of the group (rows >= G zero); sp: this warp's
// fp32 [8][16] weight buffer.
template <int D>
__device__ __forceinline__ void attend_tile_fma(AttnStateFma<D>& st, uint32_t sK, uint32_t sV,
                                                const float* qs, float* sp, int valid,
                                                float scale_log2, int lane) {
  constexpr int kCols = D / 32;
  const int t = lane & 15;
  const int hq = (lane >> 4) * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    uint4 kv;
    const uint32_t addr = sK + (c >> 3) * kHalfBytes + t * 128 + (((c & 7) ^ (t & 7)) << 4);
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(kv.x), "=r"(kv.y), "=r"(kv.z), "=r"(kv.w)
                 : "r"(addr));
    float k8[8];
    bf16x8_to_f32(kv, k8);
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      const float4 qa = *reinterpret_cast<const float4*>(qs + (hq + hh) * D + c * 8);
      const float4 qb = *reinterpret_cast<const float4*>(qs + (hq + hh) * D + c * 8 + 4);
      acc[hh] = fmaf(k8[0], qa.x, acc[hh]); acc[hh] = fmaf(k8[1], qa.y, acc[hh]);
      acc[hh] = fmaf(k8[2], qa.z, acc[hh]); acc[hh] = fmaf(k8[3], qa.w, acc[hh]);
      acc[hh] = fmaf(k8[4], qb.x, acc[hh]); acc[hh] = fmaf(k8[5], qb.y, acc[hh]);
      acc[hh] = fmaf(k8[6], qb.z, acc[hh]); acc[hh] = fmaf(k8[7], qb.w, acc[hh]);
    }
  }
  // per head: tile max over the 16 tokens (lanes with the same lane / 16)
  float y[4], mx[4];
#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    y[hh] = t < valid ? acc[hh] * scale_log2 : -INFINITY;
    mx[hh] = y[hh];
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
      mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], off));
  }
  // every lane needs the new max of all 8 heads (the other half via xor 16)
  float mn[kMaxGroup], alpha[kMaxGroup];
#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    const float other = __shfl_xor_sync(0xffffffffu, mx[hh], 16);
    const float lo = lane < 16 ? mx[hh] : other;   // heads 0..3
    const float hi = lane < 16 ? other : mx[hh];   // heads 4..7
    mn[hh] = fmaxf(st.m[hh], lo);
    mn[hh + 4] = fmaxf(st.m[hh + 4], hi);
  }
  float psum[4];
#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    const float mine = lane < 16 ? mn[hh] : mn[hh + 4];  // the new max of head hq + hh
    const float pv = exp2f(y[hh] - mine);
    sp[(hq + hh) * kTile + t] = pv;
    psum[hh] = pv;
#pragma unroll
    for (int off = 1; off < 16; off <<= 1)
      psum[hh] += __shfl_xor_sync(0xffffffffu, psum[hh], off);
  }
#pragma unroll
  for (int hh = 0; hh < 4; ++hh) {
    const float other = __shfl_xor_sync(0xffffffffu, psum[hh], 16);
    const float lo = lane < 16 ? psum[hh] : other;
    const float hi = lane < 16 ? other : psum[hh];
    alpha[hh] = exp2f(st.m[hh] - mn[hh]);
    alpha[hh + 4] = exp2f(st.m[hh + 4] - mn[hh + 4]);
    st.l[hh] = st.l[hh] * alpha[hh] + lo;
    st.l[hh + 4] = st.l[hh + 4] * alpha[hh + 4] + hi;
  }
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    st.m[h] = mn[h];
#pragma unroll
    for (int j = 0; j < kCols; ++j) st.o[h][j] *= alpha[h];
  }
  __syncwarp();
  // O[h][cols] += sum_t p[h][t] V[t][cols]; this lane's columns kCols*lane..
  const int col = kCols * lane;
  const int c = col >> 3;  // 16-byte chunk holding the columns
  for (int tt = 0; tt < valid; ++tt) {
    const uint32_t addr =
        sV + (c >> 3) * kHalfBytes + tt * 128 + (((c & 7) ^ (tt & 7)) << 4) + (col & 7) * 2;
    float v[kCols];
    if constexpr (kCols == 4) {
      uint32_t a, b2;
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b2) : "r"(addr));
      v[0] = bf16_lo(a); v[1] = bf16_hi(a); v[2] = bf16_lo(b2); v[3] = bf16_hi(b2);
    } else {
      uint32_t a;
      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(a) : "r"(addr));
      v[0] = bf16_lo(a); v[1] = bf16_hi(a);
    }
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      const float pw = sp[h * kTile + tt];
#pragma unroll
      for (int j = 0; j < kCols; ++j) st.o[h][j] = fmaf(pw, v[j], st.o[h][j]);
    }
  }
  __syncwarp();
}

// Where a tile's K/V rows come from.
struct TileSrc {
  const unsigned char* k_cache;  // for the cp.async gather (block sizes < 8)
  const unsigned char* v_cache;
  int num_kv_heads;
  int block_size;
  int log2_bs;
  int num_blocks;
};

// Issue the copies of the tile starting at logical token t0 of one sequence
// (KV head kvh) into the stage at sK (V follows at sK + kKVBytes), completing
// on `full`. Warp-collective. The sequence's block-table entries
// [tc_base, tc_base + 32) are held one per lane in tc_val (-1 past the
// sequence's n_seq_blocks blocks); the tile's blocks must lie in that window.
// TMA path (block_size >= 8): lane 0 issues min(bs,16)-row boxes per column
// half; rows of blocks past the sequence or of out-of-range ids are fetched
// from a coordinate past the pool, which TMA fills with zeros. Gather path:
// every lane copies 16-byte chunks; tokens >= t_end and invalid blocks are
// zero-filled without a read.
template <int D, bool kTma, int EB = 2, int TT = kTile>
__device__ __forceinline__ void issue_tile(uint32_t sK, uint64_t* full, const CUtensorMap* tmap_k,
                                           const CUtensorMap* tmap_v, const TileSrc& src, int kvh,
                                           int t0, int t_end, int n_seq_blocks, int tc_base,
                                           int tc_val, int lane) {
  using Gm = TileGeom<D, EB, TT>;
  const int bs = src.block_size;
  const int blk_first = t0 >> src.log2_bs;
  const uint32_t sV = sK + Gm::kKVBytes;
  if constexpr (kTma) {
    // Boxes of min(bs, TT) rows. The loader issues every tile of the block,
    // so this stays straight-line for the common shapes: one box per column
    // half when a block holds the whole tile, two when it holds half of it.
    const int oob_row = src.num_blocks * bs;  // < 2^31 (checked on the host)
    auto row_of = [&](int j, unsigned off) {
      const int phys = __shfl_sync(0xffffffffu, tc_val, (blk_first + j - tc_base) & 31);
      const bool ok = blk_first + j < n_seq_blocks && phys >= 0 && phys < src.num_blocks;
      return ok ? (int)((unsigned)phys * (unsigned)bs + off) : oob_row;
    };
    if (bs >= TT) {
      const int row = row_of(0, (unsigned)(t0 & (bs - 1)));
      if (lane == 0) {
        mbar_arrive_expect_tx(full, Gm::kStageBytes);
        if constexpr (Gm::kHalves == 2) {
          // 256-byte rows: the map is 3-D (64 columns, rows, column halves),
          // one box carries both halves of the tile
          tma_load_3d(sK, tmap_k, 0, row, 2 * kvh, full);
          tma_load_3d(sV, tmap_v, 0, row, 2 * kvh, full);
        } else {
#pragma unroll
          for (int h = 0; h < Gm::kHalves; ++h) {
            const int x = kvh * D + h * Gm::kBoxCols;
            tma_load_2d(sK + h * Gm::kHalfStride, tmap_k, x, row, full);
            tma_load_2d(sV + h * Gm::kHalfStride, tmap_v, x, row, full);
          }
        }
      }
    } else if (2 * bs == TT) {
      const int row0 = row_of(0, 0u), row1 = row_of(1, 0u);
      if (lane == 0) {
        mbar_arrive_expect_tx(full, Gm::kStageBytes);
#pragma unroll
        for (int h = 0; h < Gm::kHalves; ++h) {
          const int x = kvh * D + h * Gm::kBoxCols;
          const uint32_t off = h * Gm::kHalfStride;
          tma_load_2d(sK + off, tmap_k, x, row0, full);
          tma_load_2d(sV + off, tmap_v, x, row0, full);
          tma_load_2d(sK + off + bs * 128, tmap_k, x, row1, full);
          tma_load_2d(sV + off + bs * 128, tmap_v, x, row1, full);
        }
      }
    } else {  // 8 <= bs < TT / 2: TT / bs boxes
      constexpr int kMaxSub = TT / 8;
      const int nsub = TT / bs;
      int rows[kMaxSub];
#pragma unroll
      for (int j = 0; j < kMaxSub; ++j) rows[j] = row_of(j, 0u);
      if (lane == 0) {
        mbar_arrive_expect_tx(full, Gm::kStageBytes);
#pragma unroll
        for (int h = 0; h < Gm::kHalves; ++h) {
          const int x = kvh * D + h * Gm::kBoxCols;
          const uint32_t off = h * Gm::kHalfStride;
#pragma unroll
          for (int j = 0; j < kMaxSub; ++j) {
            if (j < nsub) {
              tma_load_2d(sK + off + j * bs * 128, tmap_k, x, rows[j], full);
              tma_load_2d(sV + off + j * bs * 128, tmap_v, x, rows[j], full);
            }
          }
        }
      }
    }
  } else {
    constexpr int kChunks = Gm::kRowBytes / 16;  // 16-byte chunks per row
    const size_t row_bytes = (size_t)src.num_kv_heads * Gm::kRowBytes;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const unsigned char* cache = which == 0 ? src.k_cache : src.v_cache;
      const uint32_t dst_tile = which == 0 ? sK : sV;
#pragma unroll
      for (int k = 0; k < TT * kChunks / 32; ++k) {
        const int idx = k * 32 + lane;
        const int r = idx / kChunks, c = idx % kChunks;
        const int t = t0 + r;
        const int blk = t >> src.log2_bs;
        const int phys = __shfl_sync(0xffffffffu, tc_val, (blk - tc_base) & 31);
        const bool ok = t < t_end && blk < n_seq_blocks && phys >= 0 && phys < src.num_blocks;
        const unsigned char* p =
            ok ? cache + ((size_t)phys * bs + (t & (bs - 1))) * row_bytes +
                     (size_t)kvh * Gm::kRowBytes + c * 16
               : cache;
        const uint32_t dst =
            dst_tile + (c >> 3) * Gm::kHalfStride + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        cp_async_16_zfill(dst, p, ok);
      }
    }
    cp_async_arrive_noinc(full);
  }
}

}  // namespace pa
