// pa_host.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pa {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

inline int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// True when the environment asks for validating mode (PA_VALIDATE=1).
bool validating();

// Maps the last launch error to a status, clearing it.
pa_status launch_status();

// cuTensorMapEncodeTiled through the runtime's driver entry point (looked up
// once); null when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Tensor map over a cache viewed as [rows = num_blocks*block_size,
// cols = num_kv_heads*head_dim] elements of elem_bytes (2: bf16, 1: e4m3
// bytes), 128-byte swizzle, zero fill out of bounds. 2-D with box {128 bytes
// of columns, box_rows rows}; for 256-byte head rows and box_rows >= 16, 3-D
// (128-byte columns, rows, column halves) with box {128 bytes, box_rows, 2},
// which issue_tile loads with one instruction per K or V tile.
bool make_cache_map(CUtensorMap* map, const void* base, int num_kv_heads, int head_dim,
                    long long rows, int box_rows, int elem_bytes = 2);

// Validating mode: copies context_lens / block_tables to the host (stream
// synchronised) and range-checks them. split_tokens > 0 also bounds contexts
// by max_splits * split_tokens.
pa_status check_tables(const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                       int num_seqs, int num_blocks, int block_size, int split_tokens,
                       int max_splits, cudaStream_t stream);

// The shape checks every decode entry point shares; PA_OK when supported.
pa_status check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, float scale, const void* out);

// Prepares a kernel for a launch with `smem_bytes` of dynamic shared memory on
// the current device and returns its resident blocks per SM (>= 1) in
// *blocks_per_sm (may be null). The attribute call and the occupancy query
// run once per (kernel, device, size); later calls only read a cache, so a
// warmed-up entry point issues nothing but its launch (safe inside stream
// capture).
pa_status prepare_kernel(const void* func, int threads, int smem_bytes, int* blocks_per_sm);

// Long query chunks on the tcgen05 tensor cores (pa_prefill_tc.cu): supported
// for head_dim 64 or 128, any block size (TMA boxes from 8 rows, cp.async
// copies below) and a query group of at most 256 heads. Runs pa_decode_multi's unsplit causal attention with the same
// arguments; device errors are ORed into *err.
bool prefill_tc_supported(int head_dim, int block_size, int group);
pa_status launch_prefill_tc(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks,
                            const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                            int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, float scale, void* out,
                            unsigned int* err, cudaStream_t stream);
// The same over an e4m3 pool (uint8 codes, per-KV-head fp32 scales on the
// device); head_dim 128 only.
pa_status launch_prefill_tc_fp8(const void* q, const void* k_codes, const void* v_codes,
                                const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, int max_blocks,
                                const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                                int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, float scale, void* out,
                                unsigned int* err, cudaStream_t stream);

// A few query tokens per sequence on the tcgen05 tensor cores with the keys
// on the MMA's M side (pa_verify_tc.cu), bf16 caches: head_dim 128, block
// sizes >= 8, at most 32 (token, head) columns per KV head (max_q_len *
// group), split_tokens 0 or a multiple of 128, fewer than 2^31 units
// (sequences * splits * KV heads). Runs pa_decode_multi with the same
// arguments as a persistent launch (one block per SM); device errors are ORed
// into *err.
bool verify_tc_supported(int head_dim, int block_size, int group, int max_q_len,
                         int split_tokens);
pa_status launch_verify_tc(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks,
                           const int32_t* context_lens, const int32_t* q_start, int num_seqs,
                           int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int num_blocks, float scale, int split_tokens,
                           int max_splits, float* part_out, float* part_lse, int32_t* row_lens,
                           void* out, unsigned int* err, cudaStream_t stream);
// The same kernel on pa_decode_multi_balanced's schedule: every block an
// equal range of the 128-key tiles of all (sequence, KV head) units; a unit
// cut by ranges leaves records (normalised partial outputs and base-2
// log-sum-exps, record 2 c + (c is the unit's first block) of block c) that
// the last block to finish it merges, tickets in counters [B * Hkv * 8]
// (zero between launches, left zero). Up to 8192 sequences; rec_cols >= 32.
bool verify_tc_balanced_supported(int head_dim, int block_size, int group, int max_q_len,
                                  int num_seqs);
pa_status launch_verify_tc_balanced(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int max_blocks,
                                    const int32_t* context_lens, const int32_t* q_start,
                                    int num_seqs, int max_q_len, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int num_blocks, float scale, int* counters, float* rec_lse,
                                    float* rec_o, int rec_cols, void* out, unsigned int* err,
                                    cudaStream_t stream);

// Reads and clears a translation unit's device error word (synchronous).
unsigned int take_decode_errors();
unsigned int take_balanced_errors();
unsigned int take_multi_errors();

}  // namespace pa
