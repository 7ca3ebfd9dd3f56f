/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged-KV decode-attention library.
 *
 * The operation: one decode step of attention for a continuously batched set
 * of variable-length sequences whose K/V rows live in a shared pool of
 * fixed-size physical blocks, reached through per-sequence block tables, with
 * grouped-query heads (several query heads share one KV head).
 *
 * Sources, by page and section:
 *   [TGI-PA]  "Text Generation Inference: Hugging Face's production-grade LLM
 *             inference server", section "Under the Hood: PagedAttention"
 *             (block table, shared pool, append into the current block, the
 *             simplified paged forward pass).
 *   [TGI-FA]  same page, section "Under the Hood: Flash Attention" (running
 *             max / running sum / rescaled accumulator over K/V tiles).
 *   [TGI-KV]  same page, section "Production Pattern: KV Cache Math".
 *   [SPEED]   "How to Speed Up LLM Inference: KV Cache to Production Serving",
 *             sections "The physics: why generating tokens is slow" (decode is
 *             bandwidth-bound) and "The KV cache: the memory problem that runs
 *             the show" (paging, GQA).
 *   [LIFE]    "The inference request lifecycle", section "KV cache grows with
 *             the sum of cached tokens" (GQA: fewer KV heads, same query heads).
 *   [PYS-RADIX] pyshine "text-generation-inference", section "The radix
 *             prefix cache"; [PYS-BATCH] same page, "Inside the batching task".
 *
 * Conventions for every entry point:
 *   - bf16 means IEEE bfloat16 (2 bytes). All tensors are dense, row-major,
 *     in the shapes given, and DEVICE memory owned by the caller, except where
 *     a parameter says "host".
 *   - The library allocates no device memory, keeps no state between calls
 *     (apart from one 4-byte device error word per device, see
 *     pa_last_device_error, and the host-side prefix cache objects the caller
 *     creates and destroys, see pa_prefix_cache_create)
 *     and launches only on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). Calls return as soon as the kernels are queued; they do not
 *     synchronise, except in validating mode (environment PA_VALIDATE=1),
 *     where the small index tables are copied to the host and range-checked
 *     before launching.
 *   - Errors are returned, never raised on the device: bad arguments give
 *     PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED without launching anything, a
 *     failed launch gives PA_ERR_CUDA. Device code contains no traps or
 *     asserts; out-of-range block ids or slots read zeros / are skipped.
 *   - Layouts:
 *       k_cache, v_cache : bf16 [num_blocks, block_size, num_kv_heads, head_dim]
 *                          ([TGI-PA] stores K and V interleaved per token; here
 *                          they are two pools with the same per-token layout)
 *       block_tables     : int32 [num_seqs, max_blocks_per_seq]; entry [b][i] is
 *                          the physical block holding logical tokens
 *                          i*block_size .. i*block_size+block_size-1 of sequence b
 *       context_lens     : int32 [num_seqs]; tokens attended over (after append)
 *       q, out           : bf16 [num_seqs, num_q_heads, head_dim]
 *     Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - Supported: head_dim 64 or 128; num_q_heads / num_kv_heads in 1..8;
 *     block_size a power of two in 1..256; num_blocks*block_size < 2^31.
 *     q, out and both caches 16-byte aligned.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1, /* null pointer, bad size, misalignment, table out of range */
  PA_ERR_UNSUPPORTED = -2, /* valid but not built: head_dim, group size, block size  */
  PA_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed                    */
  PA_ERR_WORKSPACE = -4,   /* split mode without partial buffers                      */
  PA_ERR_DEVICE = -5,      /* a kernel's bounded wait ran out (see pa_last_device_error) */
  PA_ERR_CAPACITY = -6     /* prefix cache: not enough free or evictable blocks          */
} pa_status;

/*
 * pa_kv_append -- scatter the new tokens' K and V rows into their slots.
 * [TGI-PA]: a new token's KV pair is appended into the sequence's current
 * block (a fresh physical block when the current one is full; choosing it is
 * the host allocator's job and arrives here as `slot_mapping`).
 *
 *   k_new, v_new  bf16 [num_tokens, num_kv_heads, head_dim]
 *   slot_mapping  int64 [num_tokens]; token t goes to block slot/block_size,
 *                 offset slot%block_size. slot < 0 marks a padded row: skipped.
 *                 slot >= num_blocks*block_size is skipped too (and reported as
 *                 PA_ERR_INVALID_ARG in validating mode).
 *   k_cache, v_cache  written in place; bytes are copied unchanged.
 * Rows of two tokens mapped to the same slot race; the caller must not do so.
 */
pa_status pa_kv_append(const void* k_new, const void* v_new,
                       const int64_t* slot_mapping, int32_t num_tokens,
                       void* k_cache, void* v_cache,
                       int32_t num_blocks, int32_t block_size,
                       int32_t num_kv_heads, int32_t head_dim, void* stream);

/*
 * pa_decode -- paged decode attention, out = softmax(scale * q K^T) V per query
 * head over the first context_lens[b] logical tokens of sequence b, K/V rows
 * gathered through block_tables[b] ([TGI-PA]), computed with the streaming
 * softmax of [TGI-FA] in fp32 and rounded to bf16 (round to nearest even).
 * One thread block serves one (sequence, KV head, context split) and every
 * query head of that KV head's group ([SPEED], [LIFE]).
 *
 *   scale         the logit scale (1/sqrt(head_dim) in the pages).
 *   split_tokens  0: one split per sequence, `out` written directly.
 *                 > 0 (a multiple of 16): split s covers logical tokens
 *                 [s*split_tokens, min((s+1)*split_tokens, ctx)); each split
 *                 writes a partial to part_out/part_lse and `out` is NOT
 *                 written -- call pa_decode_splitk_reduce next.
 *   max_splits    splits per sequence in the partial buffers; must cover the
 *                 longest context (ctx <= max_splits*split_tokens). Ignored
 *                 when split_tokens == 0.
 *   part_out      fp32 [num_seqs, num_q_heads, max_splits, head_dim]: the split's
 *                 attention output over its own tokens, normalised.
 *   part_lse      fp32 [num_seqs, num_q_heads, max_splits]: natural-log
 *                 log-sum-exp of the split's scaled logits. Splits past the end
 *                 of a sequence are not written.
 *   context_lens[b] == 0 gives a zero output row (never NaN).
 *   Contexts longer than max_blocks_per_seq*block_size are clamped to it.
 */
pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t num_seqs,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t num_blocks, float scale,
                    int32_t split_tokens, int32_t max_splits,
                    float* part_out, float* part_lse,
                    void* out, void* stream);

/*
 * pa_decode_splitk_reduce -- merge split partials by log-sum-exp: per
 * (sequence, query head) over the splits s < ceil(ctx/split_tokens):
 * M = max lse_s, w_s = exp(lse_s - M), out = sum w_s O_s / sum w_s, rounded to
 * bf16. This rescaling is the same algebra as the running-max correction of
 * [TGI-FA]; the pages do not describe context splitting itself. A sequence
 * with no tokens gets a zero row.
 */
pa_status pa_decode_splitk_reduce(const float* part_out, const float* part_lse,
                                  const int32_t* context_lens, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t head_dim,
                                  int32_t split_tokens, int32_t max_splits,
                                  void* out, void* stream);

/*
 * pa_decode_balanced -- the same attention as pa_decode, in one launch,
 * scheduled for a continuously batched mix of lengths: the 16-token tiles of
 * all (sequence, KV head) pairs are divided into contiguous ranges, one per
 * thread block of a persistent grid (four blocks per SM; inside a block a
 * loader warp streams the range and the consumer warps fold its tiles
 * round-robin). The ranges are equal in tiles plus a fixed charge per pair
 * for its end-of-pair merge, so every block does the same work whatever the
 * lengths. A (sequence, KV head) pair cut by a range boundary is merged by
 * log-sum-exp (the running-max rescale of [TGI-FA]) by the last block to
 * finish its part; no separate reduce call is needed. Layouts, supported shapes and error
 * behaviour are those of pa_decode; context_lens stay on the device (the
 * schedule is computed there).
 *
 *   workspace        device memory of at least
 *                    pa_decode_balanced_workspace_bytes(num_seqs, num_kv_heads,
 *                    head_dim) bytes, 256-byte aligned, ZERO-FILLED before its
 *                    first use; every call leaves it reusable (its counters are
 *                    back at zero). Calls that share a workspace must not run
 *                    concurrently.
 *   workspace_bytes  its size; too small gives PA_ERR_WORKSPACE.
 */
pa_status pa_decode_balanced(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t num_seqs,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, float scale,
                             void* workspace, size_t workspace_bytes,
                             void* out, void* stream);

/*
 * pa_append_decode -- one decode step in one launch: pa_kv_append of one new
 * token per sequence followed by pa_decode_balanced over the contexts that
 * include it ([TGI-PA]: the new KV pair is appended to the current block, then
 * attention runs over the block table; fusing the bookkeeping into the
 * attention launch follows the kernel-fusion pattern of [TGI], section
 * "Advanced Pattern: Kernel Fusion").
 *
 *   k_new, v_new  bf16 [num_seqs, num_kv_heads, head_dim]: the new token of
 *                 each sequence.
 *   slot_mapping  int64 [num_seqs]: its slot, which must be the slot of logical
 *                 token context_lens[b] - 1 of sequence b in block_tables[b];
 *                 slot < 0 skips the write (the step then reads whatever that
 *                 slot holds, as append-then-decode would).
 *   k_cache, v_cache  written at the slots, read for attention.
 * Everything else as pa_decode_balanced (same workspace). The result equals
 * pa_kv_append followed by pa_decode_balanced.
 */
pa_status pa_append_decode(const void* q, const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, void* k_cache, void* v_cache,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale,
                           void* workspace, size_t workspace_bytes,
                           void* out, void* stream);

/*
 * FP8 KV cache. [SPEED] ("The KV cache: the memory problem that runs the
 * show": quantizing the cache to FP8 halves the 320 KB/token) and the FP8 row
 * of [TGI-KV] (163,840 B/token for the 70B class) fix the byte count; the
 * format and scaling are this library's reading:
 *   k_cache, v_cache  uint8 [num_blocks, block_size, num_kv_heads, head_dim],
 *                     OCP e4m3 codes (bias 7, no infinities, largest 448).
 *   k_scale, v_scale  fp32 [num_kv_heads], device: a code c of head h stands
 *                     for value(c) * scale[h].
 * Quantization (the appends): code = e4m3 round-to-nearest-even of
 * x / scale[h] computed in fp32 (round to nearest), saturated to +-448.
 * Supported: head_dim 128, at most 64 KV heads; otherwise PA_ERR_UNSUPPORTED.
 */

/* pa_kv_append for an FP8 pool: each new bf16 K/V row is quantized to codes. */
pa_status pa_kv_append_fp8(const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, int32_t num_tokens,
                           void* k_cache, void* v_cache,
                           const float* k_scale, const float* v_scale,
                           int32_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim, void* stream);

/* pa_decode_balanced over an FP8 pool: codes are read back as value * scale
 * (the scales folded into the score factor and the output), the tile math runs
 * on f16 MMAs (every e4m3 value is exact in f16). Same workspace. */
pa_status pa_decode_balanced_fp8(const void* q, const void* k_cache, const void* v_cache,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, int32_t num_seqs,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int32_t num_blocks, float scale,
                                 void* workspace, size_t workspace_bytes,
                                 void* out, void* stream);

/* pa_append_decode over an FP8 pool: the new rows are quantized at their slots
 * and decoded in the same launch. Equals pa_kv_append_fp8 followed by
 * pa_decode_balanced_fp8. */
pa_status pa_append_decode_fp8(const void* q, const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, void* k_cache, void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t num_blocks, float scale,
                               void* workspace, size_t workspace_bytes,
                               void* out, void* stream);

/* Workspace bytes pa_decode_balanced needs on the current device (its size
 * depends on the device's SM count); 0 for invalid sizes. */
size_t pa_decode_balanced_workspace_bytes(int32_t num_seqs, int32_t num_kv_heads,
                                          int32_t head_dim);

/*
 * pa_decode_balanced_static -- pa_decode_balanced without a workspace argument:
 * it allocates nothing and takes no scratch from the caller. (The source pages
 * have no counterpart to this entry point; it exists for callers of this
 * library.)
 *
 * Who needs it: callers that cannot allocate device memory at the call site.
 * A serving engine typically reserves nearly all free HBM for its KV block
 * pool at start-up, so a per-call cudaMalloc has nothing left to take (and
 * cudaMalloc may synchronise the device, which a per-token decode loop cannot
 * afford); a plug-in called from a host framework that owns all device memory
 * may have no allocator to ask at all.
 *
 * Instead, the library keeps one 6 MiB scratch array in device memory
 * (a file-scope __device__ array: every GPU that loads the library holds it
 * until the process exits). Inputs, output, layouts and supported shapes are
 * those of pa_decode_balanced; the output is the same.
 *
 *   - Shapes whose scratch exceeds 6 MiB return PA_ERR_WORKSPACE without
 *     launching or writing anything. The test a caller can make beforehand:
 *     pa_decode_balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim)
 *     <= 6,291,456. On a 152-SM GB300 that admits up to 317,952
 *     (sequence, KV head) pairs at head_dim 128 and 940,544 at head_dim 64.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture on the device.
 *   - Every call on a device shares the one array: calls whose kernels may
 *     overlap on the GPU (different streams without ordering between them)
 *     race on it and must not be issued. Each call clears the part that must
 *     start at zero (a memset on `stream`) before its kernel.
 */
pa_status pa_decode_balanced_static(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t num_seqs,
                                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t num_blocks, float scale,
                                    void* out, void* stream);

/* Splits needed for contexts up to max_context tokens (0 if split_tokens <= 0). */
int32_t pa_decode_num_splits(int32_t max_context, int32_t split_tokens);

/* Bytes of part_out plus part_lse for the given shape (the caller may carve
 * both from one buffer: part_lse starts at the 256-byte-aligned end of part_out). */
size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                 int32_t head_dim, int32_t max_splits);

/* KV bytes one token occupies over the whole model, 2*layers*kv_heads*head_dim*
 * bytes_per_value ([TGI-KV]; [SPEED]; [LIFE]). */
int64_t pa_kv_bytes_per_token(int32_t num_layers, int32_t num_kv_heads,
                              int32_t head_dim, int32_t bytes_per_value);

/* Reads and clears the calling device's error word (synchronises the device).
 * *code (host) receives 0 if no kernel's bounded wait has run out since the
 * last call, else a nonzero bit set. Returns PA_ERR_DEVICE when nonzero. */
pa_status pa_last_device_error(int32_t* code);

/* Failure-detection self-test. Launches one warp that waits, for at most
 * limit_us microseconds (1..2,000,000), on an mbarrier whose phase nothing
 * completes -- the same bounded wait every decode kernel uses for its K/V
 * tiles. The wait runs out, the kernel sets bit 8 of the device error word and
 * returns; pa_last_device_error then reports PA_ERR_DEVICE with that bit and
 * the context stays usable. No counterpart on the pages (they describe the
 * serving system's failure handling, not kernels'). */
pa_status pa_selftest_wait_timeout(int32_t limit_us, void* stream);

/* Attention for several new query tokens per sequence under a causal mask:
 * a chunk of a prompt ([TGI], section "Advanced Pattern: Chunked Prefill
 * (TGI v3)") or the drafted tokens plus one of a speculative step ([SPEED],
 * section "Speculative decoding: more than one token per weight-read").
 *   q          bf16 [num_q_rows, num_q_heads, head_dim]: packed query rows;
 *              sequence b owns rows q_start[b] .. q_start[b+1]-1 (its n_b new
 *              tokens in order, already appended to the caches, e.g. by
 *              pa_kv_append), so row q_start[b] + i is position
 *              context_lens[b] - n_b + i and attends to positions 0 .. that
 *              position (a row before position 0 gives zeros).
 *   q_start    int32 [num_seqs + 1], q_start[0] = 0, q_start[num_seqs] =
 *              num_q_rows, non-decreasing.
 *   max_q_len  an upper bound of every n_b. With max_q_len * (num_q_heads /
 *              num_kv_heads) <= 64 (drafted tokens, short chunks) a
 *              sequence's whole query group for one KV head is one unit: at
 *              most 32 (token, head) columns, head_dim 128, block_size >= 8
 *              and split_tokens 0 or a multiple of 128 run on the tcgen05
 *              tensor cores (keys on the MMA's M side, a persistent launch
 *              of one block per SM walking the (sequence, split, KV head)
 *              units), other short chunks, or all of them when the
 *              environment sets PA_MULTI_KERNEL=columns, on warp MMAs (one
 *              block per unit); above
 *              that (long prompt chunks) the rows are tiled, unsplit, each
 *              tile with a causal key range of its own: 256 (token, head)
 *              rows a block on the tcgen05 tensor cores (scores and outputs
 *              in tensor memory; K/V rows by TMA for block_size >= 8, by
 *              16-byte cp.async copies below), or, when the environment sets
 *              PA_PREFILL_KERNEL=rowblock, 64 rows a block on warp MMAs;
 *              split_tokens must then be 0,
 *              else PA_ERR_UNSUPPORTED. A sequence with more rows than
 *              max_q_len is skipped and sets bit 16 of the device error word
 *              (rejected in validating mode).
 *   split_tokens / max_splits / part_out / part_lse: as in pa_decode, with
 *              rows in place of sequences (part_out [num_q_rows, num_q_heads,
 *              max_splits, head_dim]); split mode also writes each row's
 *              attended length to row_lens (int32 [num_q_rows]), then
 *              pa_decode_splitk_reduce(part_out, part_lse, row_lens,
 *              num_q_rows, ...) writes out.
 *   out        bf16 [num_q_rows, num_q_heads, head_dim] (one split).
 * Other arguments, layouts and errors as pa_decode. */
pa_status pa_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, const int32_t* q_start, int32_t num_seqs,
                          int32_t num_q_rows, int32_t max_q_len, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, float scale, int32_t split_tokens,
                          int32_t max_splits, float* part_out, float* part_lse,
                          int32_t* row_lens, void* out, void* stream);

/* pa_decode_multi on the work-balanced persistent schedule of
 * pa_decode_balanced: one launch, every block the same number of K/V tiles,
 * units cut by a block's range merged in the kernel by log-sum-exp (no
 * reduce launch). workspace: caller-owned device memory of at least
 * pa_decode_multi_balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim)
 * bytes, 256-byte aligned, zero-filled before its first use and left reusable
 * (too small: PA_ERR_WORKSPACE); calls sharing a workspace must not overlap.
 * max_q_len * (num_q_heads / num_kv_heads) must be <= 64, else
 * PA_ERR_UNSUPPORTED. Other arguments, limits and errors as pa_decode_multi. */
pa_status pa_decode_multi_balanced(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* q_start,
                                   int32_t num_seqs, int32_t num_q_rows, int32_t max_q_len,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks, float scale,
                                   void* workspace, size_t workspace_bytes, void* out,
                                   void* stream);

/* pa_decode_multi over an FP8 (e4m3) pool: several new query tokens per
 * sequence under the causal mask ([SPEED], section "Speculative decoding: more
 * than one token per weight-read"; [TGI], "Advanced Pattern: Chunked Prefill
 * (TGI v3)") with the K/V codes read back as value(code) * scale of their KV
 * head ([SPEED], "The KV cache: the memory problem that runs the show"), as in
 * pa_decode_balanced_fp8: 32-token e4m3 tiles widened exactly to f16 for f16
 * MMAs, k_scale folded into the score factor and v_scale into the output.
 *   k_codes, v_codes  uint8 [num_blocks, block_size, num_kv_heads, 128]
 *              (written by pa_kv_append_fp8); k_scale, v_scale float
 *              [num_kv_heads], device.
 *   split_tokens  0, or a multiple of 32 (then part_out / part_lse /
 *              row_lens and pa_decode_splitk_reduce as in pa_decode_multi).
 * Long chunks (max_q_len * (num_q_heads / num_kv_heads) > 64 rows per KV head,
 * chunked prefill, [TGI] "Advanced Pattern: Chunked Prefill (TGI v3)") run
 * on the tcgen05 tensor cores: the e4m3 rows are widened exactly to f16 in
 * shared memory and the MMAs take f16 q (exact for 2^-14 <= |q| <= 65504)
 * and f16 weights; unsplit (split_tokens must be 0).
 * Supported: head_dim 128; otherwise, and for long chunks with a split,
 * PA_ERR_UNSUPPORTED. Other arguments, layouts and errors as
 * pa_decode_multi. */
pa_status pa_decode_multi_fp8(const void* q, const void* k_codes, const void* v_codes,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, const int32_t* q_start,
                              int32_t num_seqs, int32_t num_q_rows, int32_t max_q_len,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t num_blocks, float scale,
                              int32_t split_tokens, int32_t max_splits, float* part_out,
                              float* part_lse, int32_t* row_lens, void* out, void* stream);

/* Workspace bytes pa_decode_multi_balanced needs on the current device. */
size_t pa_decode_multi_balanced_workspace_bytes(int32_t num_seqs, int32_t num_kv_heads,
                                                int32_t head_dim);

/* ------------------------------------------------------------------------
 * Prefix cache with copy-on-write (host side) and the block copy (device).
 *
 * [TGI-PA] prefix sharing: requests with the same system prompt point their
 * tables at the same physical blocks; a write into a shared block first
 * copies it to a fresh block and repoints the writer's table.
 * [PYS-RADIX] pyshine "text-generation-inference", section "The radix prefix
 * cache": block 0 reserved, a free list plus a compressed prefix tree keyed
 * by token ids at block granularity, references on the match before any
 * eviction, least-recently-used eviction of unreferenced prefixes when the
 * free list is empty, node splits on partial overlap, double-cached blocks
 * back to the free list on release. [PYS-BATCH] same page, section "Inside
 * the batching task": a fully cached prompt gives one token back.
 *
 * A pa_prefix_cache is a host object managing block ids 1..num_blocks-1 of a
 * pool and the block tables of live sequences; it touches no device memory.
 * Its rules:
 *   - only full blocks are cached, each keyed by the whole token prefix it
 *     ends; fresh blocks are taken lowest id first;
 *   - every mutating call advances a tick; a match, an insertion and the
 *     touch on release stamp the blocks on the request's path with it;
 *     eviction frees one block at a time, the unreferenced leaf with the
 *     oldest (tick, block id);
 *   - a write into a block that is cached or shared by another sequence is
 *     a copy-on-write: the call returns the (src, dst) block pairs, which the
 *     caller copies on the device (pa_copy_blocks) before writing K/V rows;
 *   - a call that needs more fresh blocks than the free blocks plus the
 *     blocks eviction could free returns PA_ERR_CAPACITY and changes nothing
 *     (pa_prefix_append_tokens: nothing for the sequence that failed).
 * Not thread-safe: one caller at a time per object. Sequence ids are > 0.
 * ---------------------------------------------------------------------- */
typedef struct pa_prefix_cache pa_prefix_cache;

/* New empty cache for a pool of num_blocks (>= 2) blocks of block_size
 * tokens. *out receives the object (host memory owned by the library until
 * pa_prefix_cache_destroy). */
pa_status pa_prefix_cache_create(int32_t num_blocks, int32_t block_size, pa_prefix_cache** out);
void pa_prefix_cache_destroy(pa_prefix_cache* cache);

/* Admit a request with prompt tokens[0, num_tokens) (host, num_tokens >= 1):
 * match the longest cached block prefix, reference it, and give the new
 * sequence fresh blocks for the rest of the prompt. *seq_id receives the
 * sequence, *cached_tokens how many leading positions already hold their
 * K/V (the match, minus one when it covers the whole prompt). The caller
 * then writes positions [*cached_tokens, num_tokens) via
 * pa_prefix_write_slots. */
pa_status pa_prefix_admit(pa_prefix_cache* cache, const int32_t* tokens, int32_t num_tokens,
                          int64_t* seq_id, int32_t* cached_tokens);

/* Slots (host int64 [pos_end - pos_begin], block * block_size + offset) for
 * writing positions [pos_begin, pos_end) of a sequence; pos_begin must not
 * exceed its current length, which grows to pos_end. Blocks that must be
 * copied first come back as copy_src[i] -> copy_dst[i] (host int32,
 * capacity max_copies; too small gives PA_ERR_INVALID_ARG before any change),
 * *num_copies of them. */
pa_status pa_prefix_write_slots(pa_prefix_cache* cache, int64_t seq_id, int32_t pos_begin,
                                int32_t pos_end, int64_t* slots, int32_t* copy_src,
                                int32_t* copy_dst, int32_t max_copies, int32_t* num_copies);

/* One decode position for each of seq_ids[0, num_seqs) in order (the slot of
 * each sequence's next token into slots[i]: the step's slot_mapping), with
 * the copies they need (max_copies >= num_seqs). On PA_ERR_CAPACITY,
 * *num_done sequences were extended and their copies are returned. */
pa_status pa_prefix_append_tokens(pa_prefix_cache* cache, const int64_t* seq_ids,
                                  int32_t num_seqs, int64_t* slots, int32_t* copy_src,
                                  int32_t* copy_dst, int32_t max_copies, int32_t* num_copies,
                                  int32_t* num_done);

/* A new sequence sharing every block of seq_id (parallel sampling); the
 * first write of either into a shared block copies it. */
pa_status pa_prefix_fork(pa_prefix_cache* cache, int64_t seq_id, int64_t* child_id);

/* pa_prefix_fork for each of seq_ids[0, num_seqs) in order; child_ids (host
 * int64 [num_seqs]) receives the new sequences. Unknown ids: nothing done. */
pa_status pa_prefix_fork_batch(pa_prefix_cache* cache, const int64_t* seq_ids, int32_t num_seqs,
                               int64_t* child_ids);

/* End sequences without caching anything (pa_prefix_release with no
 * tokens: an aborted request, a discarded sample). Unknown ids: nothing
 * done. */
pa_status pa_prefix_discard(pa_prefix_cache* cache, const int64_t* seq_ids, int32_t num_seqs);

/* End a sequence whose positions [0, num_tokens) hold the K/V of tokens
 * (host): its full blocks along that path enter the cache unless the prefix
 * is cached already (then they return to the free list with the rest of its
 * unreferenced blocks). */
pa_status pa_prefix_release(pa_prefix_cache* cache, int64_t seq_id, const int32_t* tokens,
                            int32_t num_tokens);

/* A sequence's block table (host int32, capacity max_blocks), *num_blocks
 * entries, and its length in *num_tokens (may be NULL). */
pa_status pa_prefix_table(pa_prefix_cache* cache, int64_t seq_id, int32_t* table,
                          int32_t max_blocks, int32_t* num_blocks, int32_t* num_tokens);

/* Block tables of seq_ids[0, num_seqs) as rows of a host int32
 * [num_seqs, max_blocks] array (unused entries 0) and their lengths in
 * context_lens (host int32 [num_seqs]): the decode step's inputs. */
pa_status pa_prefix_tables(pa_prefix_cache* cache, const int64_t* seq_ids, int32_t num_seqs,
                           int32_t* tables, int32_t max_blocks, int32_t* context_lens);

/* Free blocks, cached blocks, and blocks referenced by live sequences (each
 * pointer may be NULL). */
pa_status pa_prefix_stats(const pa_prefix_cache* cache, int32_t* free_blocks,
                          int32_t* cached_blocks, int32_t* used_blocks);

/* Blocks that eviction could free right now: cached, referenced by no live
 * sequence, with no referenced block after them on their prefix's path (in
 * their tree node or below it). A call succeeds when the fresh blocks it
 * needs are at most free_blocks + this count ([PYS] "The radix prefix
 * cache": least recently used unreferenced prefixes are evicted when the
 * free list is empty). Kept up to date on every change: O(1). */
pa_status pa_prefix_evictable(const pa_prefix_cache* cache, int32_t* evictable_blocks);

/* Copy-on-write on the device: for i < num_copies, block dst[i] of both
 * caches becomes a byte copy of block src[i]. src, dst: device int32
 * [num_copies]; a block is block_bytes bytes (block_size * num_kv_heads *
 * head_dim * bytes per value; a multiple of 16; caches 16-byte aligned).
 * dst ids must be distinct and none may appear in src (the copies then run
 * in parallel). Ids outside [0, num_blocks) are skipped by the kernel and,
 * in validating mode, rejected with PA_ERR_INVALID_ARG along with overlaps. */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst,
                         int32_t num_copies, int32_t num_blocks, int64_t block_bytes,
                         void* stream);

/* Human-readable name of a status. Never NULL. */
const char* pa_status_str(pa_status status);

/* Library version string, e.g. "pagedkv 0.1.0 sm_103a". Never NULL. */
const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
