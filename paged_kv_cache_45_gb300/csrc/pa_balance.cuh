// pa_balance.cuh -- the work-balanced persistent schedule shared by the
// decode kernel (pa_decode_balanced.cu) and the multi-token kernel
// (pa_decode_multi.cu).
//
// Work is a list of units, one per (sequence, KV head), sequence-major; a unit
// holds the TT-token tiles of its sequence's context. S[b] counts the tiles of
// the sequences before b, so unit (b, h) starts at global tile
// Hkv * S[b] + h * n_b. Block c of W owns a contiguous range of that list:
// the multi-token kernel splits it into equal tile counts
// [c N / W, (c + 1) N / W); the decode kernel charges each unit a fixed
// number of extra positions for its end-of-unit merge (Partition). A unit cut
// by a range boundary is merged across blocks by log-sum-exp.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int TT>
__device__ __forceinline__ int tiles_of(int ctx, int cap) {
  ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
  return (ctx + TT - 1) / TT;
}

// Largest worker whose range [w N / W, (w + 1) N / W) starts at or before tile g.
__device__ __forceinline__ int owner_of(long long g, long long N, long long W) {
  return (int)(((g + 1) * W - 1) / N);
}

// The block ranges with a fixed charge per unit. A unit's tiles are not all
// the work it costs: at its end the consumer warps merge their states (and a
// cut unit publishes a partial), which stalls the block's pipeline for about
// as long as K tiles take to stream. Unit (b, h) with n_b tiles therefore
// occupies n_b + K positions on a weighted line, its tiles first:
//   start(b, h) = Hkv * (S[b] + K b) + h (n_b + K),
// and block c of W owns the tiles whose positions fall in
// [c Nw / W, (c + 1) Nw / W), Nw = Hkv (S[B] + K B). (Every sequence is
// charged K per head, also an empty one: padding rows cost a few idle
// positions and keep the start a closed form of S.) K = 0 gives equal tile
// counts. Ownership stays contiguous in the unit list, so a cut unit is still
// merged by the blocks c0..c1 that own its first and last tiles.
//
// kHM (head-major): the units go KV head by KV head instead, unit (b, h) at
//   start(b, h) = h (S[B] + K B) + S[b] + K b,
// tile t of it being global tile h S[B] + S[b] + t of the unit list. The
// blocks Nw / Hkv positions apart then stream the same sequences' rows at
// the same time, one KV head each, so the heads of a token row (one
// Hkv * head_dim row of the pool) are read together.
template <bool kHM = false>
struct PartitionT {
  long long N;   // tiles (Hkv * S[B])
  long long Nw;  // weighted positions
  long long W;   // blocks that own a range
  int K;         // charge per unit, in tiles
  long long T;   // tiles of one KV head (S[B])
  long long Tw;  // weighted positions of one KV head

  __device__ __forceinline__ void init(const int* S, int B, int hkv, int unit_cost, int grid) {
    K = unit_cost;
    T = S[B];
    Tw = (long long)S[B] + (long long)K * B;
    N = (long long)hkv * T;
    Nw = (long long)hkv * Tw;
    W = N == 0 ? 0 : min((long long)grid, Nw);
  }
  __device__ __forceinline__ long long start(const int* S, int hkv, int b) const {
    return (long long)hkv * ((long long)S[b] + (long long)K * b);
  }
  // weighted position of tile t of unit (b, h), n = the unit's tiles
  __device__ __forceinline__ long long pos(const int* S, int hkv, int b, int h, int n,
                                           int t) const {
    if constexpr (kHM) return (long long)h * Tw + S[b] + (long long)K * b + t;
    return start(S, hkv, b) + (long long)h * (n + K) + t;
  }
  __device__ __forceinline__ int owner(long long x) const { return owner_of(x, Nw, W); }
  // global tiles (unit-list order) at weighted positions < x
  __device__ __forceinline__ long long tiles_before(long long x, const int* S, int B,
                                                    int hkv) const {
    if (x >= Nw) return N;
    if constexpr (kHM) {
      const long long h = x / Tw;
      const long long r = x - h * Tw;
      int lo = 0, hi = B - 1;  // largest b with S[b] + K b <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)S[mid] + (long long)K * mid <= r) lo = mid; else hi = mid - 1;
      }
      const long long n = S[lo + 1] - S[lo];
      const long long t = r - ((long long)S[lo] + (long long)K * lo);
      return h * T + S[lo] + (t < n ? t : n);
    }
    int lo = 0, hi = B - 1;  // largest b with start(b) <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (start(S, hkv, mid) <= x) lo = mid; else hi = mid - 1;
    }
    const long long n = S[lo + 1] - S[lo];
    const long long r = x - start(S, hkv, lo);
    const long long w = n + K;  // > 0: an empty last sequence with K = 0 has x >= Nw
    const long long h = r / w;
    const long long t = r - h * w;
    return (long long)hkv * S[lo] + h * n + (t < n ? t : n);
  }
  // block c's tiles: global indices [g0, g1)
  __device__ __forceinline__ void range(int c, const int* S, int B, int hkv, long long& g0,
                                        long long& g1) const {
    g0 = tiles_before((long long)c * Nw / W, S, B, hkv);
    g1 = tiles_before((long long)(c + 1) * Nw / W, S, B, hkv);
  }
};
using Partition = PartitionT<false>;

// Position (sequence, KV head, tile) in the unit list (kHM: head-major, as
// PartitionT<true> orders it).
template <bool kHM = false>
struct CursorT {
  int b, kvh, t, n;

  // Place the cursor on global tile g (g < N).
  __device__ __forceinline__ void seek(long long g, const int* S, int B, int hkv) {
    if constexpr (kHM) {
      const long long T = S[B];
      kvh = (int)(g / T);
      const int r = (int)(g - (long long)kvh * T);
      int lo = 0, hi = B - 1;  // largest b with S[b] <= r: a sequence with tiles
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S[mid] <= r) lo = mid; else hi = mid - 1;
      }
      b = lo;
      n = S[b + 1] - S[b];
      t = r - S[b];
      return;
    }
    int lo = 0, hi = B - 1;  // largest b with hkv * S[b] <= g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)hkv * S[mid] <= g) lo = mid; else hi = mid - 1;
    }
    b = lo;
    n = S[b + 1] - S[b];
    const long long r = g - (long long)hkv * S[b];
    kvh = (int)(r / n);
    t = (int)(r - (long long)kvh * n);
  }

  // Move to the first tile of the next unit (past the last unit: n = 0).
  __device__ __forceinline__ void next_unit(const int* S, int B, int hkv) {
    t = 0;
    if constexpr (kHM) {
      do {
        if (++b == B) {
          b = 0;
          if (++kvh == hkv) {
            n = 0;
            return;
          }
        }
      } while (S[b + 1] == S[b]);
      n = S[b + 1] - S[b];
      return;
    }
    if (++kvh == hkv) {
      kvh = 0;
      do { ++b; } while (b < B && S[b + 1] == S[b]);
      n = b < B ? S[b + 1] - S[b] : 0;
    }
  }
};
using Cursor = CursorT<false>;

// S[b] = tiles of the sequences before b (exclusive prefix sum), S[B] = all
// of them, where sequence i holds tiles(i) tiles; kThreads threads of the
// block take part, warp_tot holds one int per warp. Ends with the block
// synchronised.
template <int kThreads, typename Tiles>
__device__ __forceinline__ void tile_prefix_sum_of(int* S, int* warp_tot, int B, Tiles tiles) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = (B + kThreads - 1) / kThreads;
  const int lo = min(tid * seg, B), hi = min(lo + seg, B);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += tiles(i);
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  int run = base + incl - sum;
  for (int i = lo; i < hi; ++i) {
    S[i] = run;
    run += tiles(i);
  }
  if (tid == kThreads - 1) S[B] = base + incl;
  __syncthreads();
}

// The decode schedule: sequence i holds its context's TT-token tiles.
template <int TT, int kThreads>
__device__ __forceinline__ void tile_prefix_sum(int* S, int* warp_tot, const int32_t* context_lens,
                                                int B, int cap) {
  tile_prefix_sum_of<kThreads>(S, warp_tot, B,
                               [&](int i) { return tiles_of<TT>(context_lens[i], cap); });
}


}  // namespace pa
