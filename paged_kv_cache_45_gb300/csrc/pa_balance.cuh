// pa_balance.cuh -- the work-balanced persistent schedule shared by the
// decode kernel (pa_decode_balanced.cu) and the multi-token kernel
// (pa_decode_multi.cu).
//
// Work is a list of units, one per (sequence, KV head), sequence-major; a unit
// holds the TT-token tiles of its sequence's context. S[b] counts the tiles of
// the sequences before b, so unit (b, h) starts at global tile
// Hkv * S[b] + h * n_b. Block c of W owns the global tiles
// [c N / W, (c + 1) N / W): every block gets the same number of tiles, and a
// unit cut by a range boundary is merged across blocks by log-sum-exp.
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

// Position (sequence, KV head, tile) in the unit list.
struct Cursor {
  int b, kvh, t, n;

  // Place the cursor on global tile g (g < N).
  __device__ __forceinline__ void seek(long long g, const int* S, int B, int hkv) {
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

  // Move to the first tile of the next unit.
  __device__ __forceinline__ void next_unit(const int* S, int B, int hkv) {
    t = 0;
    if (++kvh == hkv) {
      kvh = 0;
      do { ++b; } while (b < B && S[b + 1] == S[b]);
      n = b < B ? S[b + 1] - S[b] : 0;
    }
  }
};

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
