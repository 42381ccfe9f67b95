/*
 * pagedattn.h -- C ABI of libpagedattn: paged-KV-cache attention kernels for
 * NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers to contiguous row-major arrays
 *    owned by the caller; the library never frees or keeps them past the call.
 *  - dtype is PA_F16 (IEEE binary16) or PA_BF16 (bfloat16); q, key, value,
 *    caches and out all share it.  Arithmetic is fp32 inside the kernels.
 *  - The paged cache layout is k_cache, v_cache: [num_blocks, block_size,
 *    n_kv_heads, head_dim] (MiniLLM Runtime, "CUDA PagedAttention scope" and
 *    mini_engine, "Custom CUDA kernels": fixed-size KV blocks, per-request block
 *    tables).  Token t of a sequence lives at physical block
 *    block_tables[seq][t / block_size], offset t % block_size (MiniLLM Runtime,
 *    "Core class relationships": logical token -> logical block + offset ->
 *    block_table -> physical address).
 *  - Supported shapes: block_size 8, 16, 32, 64 or 128; head_dim 64, 96, 128 or 256 (96 runs in
 *    the 128-column kernels with the extra columns zero; 256 with group size 1, 2 or 4); n_q_heads a multiple
 *    of n_kv_heads with group size G = n_q_heads / n_kv_heads in {1, 2, 4, 8};
 *    query head h reads KV head h / G.
 *  - stream is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    validate on the host and enqueue kernels; they return before the GPU work
 *    finishes.  A non-zero return means nothing was launched.
 *  - Device pointers must be 16-byte aligned (PA_ERR_ALIGN otherwise).
 *  - Values the host cannot see (slots, block ids, lengths) are checked in the
 *    kernels: an out-of-range one is skipped (its reads return zeros, its write
 *    is dropped) and a bit is set in the per-device error word read by
 *    pa_device_errors().  No kernel traps or faults on bad indices.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes */
#define PA_F16 0
#define PA_BF16 1

/* status codes returned by every entry point */
#define PA_OK 0
#define PA_ERR_NULL (-1)        /* a required pointer is NULL */
#define PA_ERR_SHAPE (-2)       /* inconsistent sizes (e.g. n_q_heads % n_kv_heads != 0, negative counts) */
#define PA_ERR_UNSUPPORTED (-3) /* a valid but unsupported shape or dtype */
#define PA_ERR_CUDA (-4)        /* a CUDA runtime / driver call failed (launch, tensor-map encode) */
#define PA_ERR_BOUNDS (-5)      /* host-visible sizes out of range (e.g. max_context_len > table capacity) */
#define PA_ERR_ALIGN (-6)       /* a pointer is not 16-byte aligned */
#define PA_ERR_WORKSPACE (-7)   /* split-K workspace missing or smaller than pa_decode_workspace_size() */

/* bits of the per-device error word (pa_device_errors) */
#define PA_DEVERR_SLOT 1u    /* a slot_mapping entry outside [0, num_blocks*block_size) and not -1; for
                                pa_decode_write on the persistent and dynamic grids also one that is not
                                the slot of its sequence's last context token */
#define PA_DEVERR_BLOCK 2u   /* a block-table entry outside [0, num_blocks) was needed */
#define PA_DEVERR_LENGTH 4u  /* a context / kv length outside its allowed range */
#define PA_DEVERR_TIMEOUT 8u /* a pipeline wait in a kernel exceeded its time limit; the kernel gave up */
#define PA_DEVERR_POSITION 16u /* a rotary-embedding position outside [0, max_position) */

/* split-K piece length the pages use (mini_engine, "Custom CUDA kernels", v2) */
#define PA_DEFAULT_PARTITION_TOKENS 256

/*
 * pa_reshape_and_cache -- KV-cache write.
 * Source: mini_engine, "Custom CUDA kernels" (the KV-cache write kernel: each new
 * K/V row goes to its slot of the pool, padded rows are left out); miniserve, "Engine"
 * (slot = block_id * block_size + offset).
 *
 *  key, value      [num_tokens, n_kv_heads, head_dim]            read
 *  k_cache, v_cache [num_blocks, block_size, n_kv_heads, head_dim] written at the slots
 *  slot_mapping    [num_tokens] int64; row i is copied to flat slot slot_mapping[i]
 *                  of the cache viewed as [num_blocks*block_size, n_kv_heads, head_dim];
 *                  -1 marks a padded row, which is skipped.  Slots must be distinct.
 *  Any n_kv_heads x head_dim whose row (n_kv_heads * head_dim * 2 bytes) is a whole number of
 *  16-byte chunks (PA_ERR_UNSUPPORTED otherwise); no upper limit on the row width.
 *  The copy is bit-exact.  num_tokens == 0 launches nothing and returns PA_OK.
 */
int pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int n_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, int dtype, void* stream);

/*
 * pa_rope_table -- the cos / sin table pa_rope_reshape_and_cache reads (HOST function, no GPU).
 * Source: mini_engine, "Features" (the Qwen3 decoder uses rotary position embedding) and
 * "Roadmap" (the rotary embedding applied inside the KV-cache write).  Dimension pair i < head_dim / 2
 * of a token at position m turns by the angle m * f_i, f_i = theta^(-2 i / head_dim).
 *
 *  out   HOST buffer of max_position * head_dim floats, written: row m holds
 *        cos(m f_i) for i < head_dim / 2, then sin(m f_i) for i < head_dim / 2; angles and
 *        functions in double, stored rounded to float.  The caller copies it to the device
 *        once (it depends only on max_position, head_dim and theta).
 *  Returns PA_ERR_NULL for out == NULL; PA_ERR_SHAPE for max_position <= 0, head_dim <= 0 or
 *  odd, or theta <= 0.
 */
int pa_rope_table(float* out, int64_t max_position, int head_dim, double theta);

/*
 * pa_rope_reshape_and_cache -- KV-cache write with rotary position embedding fused in: the
 * key rows are rotated on their way into k_cache, the query rows are rotated in place.
 * Source: mini_engine, "Roadmap" (the rotary embedding applied inside the KV-cache write) and "Features"
 * (Qwen3: GQA, RoPE); miniserve, "Engine" (per forward: qkv projection, RoPE, then the KV
 * write at slot = block_id * block_size + offset).
 *
 * With c_i, s_i the table row of the token's position and half = head_dim / 2, a row x
 * becomes, for i < half (the rotate-half pairing),
 *     x'[i] = x[i] c_i - x[i + half] s_i,     x'[i + half] = x[i + half] c_i + x[i] s_i,
 * computed in fp32 and rounded to dtype (nearest even); values are copied unchanged.
 *
 *  q            [num_tokens, n_q_heads, head_dim] rotated in place (every head of every row
 *               with a valid position), or NULL to rotate keys only
 *  key, value   [num_tokens, n_kv_heads, head_dim] read
 *  k_cache, v_cache [num_blocks, block_size, n_kv_heads, head_dim]: at slot_mapping[i],
 *               k_cache gets the rotated key row and v_cache the value row
 *  slot_mapping [num_tokens] int64 as for pa_reshape_and_cache; -1: nothing is written for
 *               the row (its q is still rotated)
 *  positions    [num_tokens] int64 in [0, max_position); a row outside is left untouched (q
 *               and cache) and sets PA_DEVERR_POSITION
 *  cos_sin      [max_position, head_dim] float32, device copy of pa_rope_table's output
 *  head_dim 64, 96, 128 or 256; n_q_heads >= 0 (ignored when q is NULL).  num_tokens == 0 launches
 *  nothing and returns PA_OK.
 */
int pa_rope_reshape_and_cache(void* q, const void* key, const void* value, void* k_cache, void* v_cache,
                              const int64_t* slot_mapping, const int64_t* positions, const float* cos_sin,
                              int64_t num_tokens, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, int64_t max_position, int dtype, void* stream);

/*
 * Split-K workspace size in bytes for pa_decode / pa_decode_splitk with these
 * sizes (partition_tokens <= 0 means PA_DEFAULT_PARTITION_TOKENS): 0 when
 * ceil(max_context_len / partition_tokens) <= 1 (one piece per sequence, written directly).
 * Otherwise, each region starting on a 256-byte boundary, P = ceil(max_context_len /
 * partition_tokens) + 3: the dynamic split-K grid (group size 1 or 2, batches of up to 256
 * sequences) cuts the last partition_tokens of every context into pieces of a quarter of that
 * (at most three pieces more); a workspace sized for P = ceil(max_context_len /
 * partition_tokens) only is still accepted and runs uniform pieces:
 *   256 bytes of control, at the start whatever the sizes: bytes 0-3 the int32 counter from
 *       which the dynamic split-K grid's CTAs take their pieces, bytes 8-15 a tag
 *       (0x7FC0A5177FC02C32) meaning "the counter is at zero"
 *   m [num_seqs, n_q_heads, P] float  -- per-piece max of scale*q.K (natural-log units)
 *   l [num_seqs, n_q_heads, P] float  -- per-piece sum of exp(s - m)
 *   o [num_seqs, n_q_heads, P, head_dim] float -- per-piece normalised output
 * The caller owns it; nothing in it needs to start at zero.  A call that runs the dynamic grid
 * (group size 1 or 2, more pieces than resident CTAs) zeroes nothing before its launch: its merge
 * kernel leaves the counter at 0 and the tag set, for the next call on the workspace.  A call
 * that finds another tag (a fresh workspace, or one used for something else in between) hands
 * the pieces out in a fixed order instead (CTA b takes pieces b, b + grid, ...), with the same
 * results bit for bit, and leaves the tag set.  So a caller who writes into the workspace
 * between calls must not write the tag with the counter off zero; pa_decode_shared_prefix
 * clears the tag when it uses the counter.
 */
size_t pa_decode_workspace_size(int num_seqs, int n_q_heads, int head_dim, int max_context_len,
                                int partition_tokens);

/*
 * pa_decode -- decode attention over the paged cache, one query token per
 * sequence, with the dispatcher choosing between the one-pass kernel
 * (pa_decode_v1) and split-K (pa_decode_splitk).
 * Source: mini_engine, "Custom CUDA kernels" (paged decode attention v1 / v2 and
 * the dispatcher that takes v2 when few sequences or long contexts cannot fill
 * the GPU); MiniLLM Runtime, "Core class relationships" (direct reads through
 * the block table, no materialisation).
 *
 *  out   [num_seqs, n_q_heads, head_dim]   written
 *  q     [num_seqs, n_q_heads, head_dim]   read
 *  block_tables [num_seqs, max_blocks_per_seq] int32 physical block ids; entries
 *                past ceil(context_lens[s]/block_size) are never used (they may hold
 *                anything; the first 32 entries of a row may be loaded before the context
 *                length is known, and the table lines prefetched into L2)
 *  context_lens [num_seqs] int32, tokens in the cache for each sequence (including
 *                the one just written); 0 gives an all-zero output row
 *  max_context_len  host-side upper bound of context_lens (sizes the split-K grid);
 *                must be <= max_blocks_per_seq * block_size
 *  scale       multiplier of q.K before the softmax (1/sqrt(head_dim) usually)
 *  workspace   device scratch of at least pa_decode_workspace_size(num_seqs,
 *              n_q_heads, head_dim, max_context_len, 0) bytes (may be NULL only
 *              when the dispatcher picks the one-pass kernel; see pa_decode_plan)
 *  out[s, h] = sum_t softmax_t(scale * q[s,h].K_t) V_t over t < context_lens[s],
 *  K_t / V_t read from KV head h / G.  Stored as dtype, rounded to nearest even.
 */
int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
              int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
              int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_write -- one decode step's KV write and decode in one call: row s of key / value
 * (the step's new token of sequence s, [num_seqs, n_kv_heads, head_dim]) is written into slot
 * slot_mapping[s] of k_cache / v_cache (-1: no row), then every sequence is decoded over its
 * context_lens[s] tokens, that row included.  Results (cache and out) are those of
 * pa_reshape_and_cache(key, value, ..., slot_mapping, num_seqs, ...) followed by pa_decode.
 * Source: mini_engine, "Custom CUDA kernels" (the KV-cache write and the paged decode of a step)
 * and "Roadmap" (folding small per-step kernels together); miniserve, "Engine" (slot mapping).
 *
 *  Arguments as pa_decode, plus key, value ([num_seqs, n_kv_heads, head_dim], dtype, 16-byte
 *  aligned) and slot_mapping ([num_seqs] int64 on the device, -1 = none).  slot_mapping[s], when
 *  not -1, must be the slot of token context_lens[s] - 1 of sequence s (block_tables[s][(L - 1) /
 *  block_size] * block_size + (L - 1) % block_size): on the persistent one-pass grid (batches of
 *  two waves and more at group size 1 or 2) and on the dynamic split-K grid (group size 1 or 2,
 *  more pieces than resident CTAs) the CTA that loads the 16-token chunk holding that token of
 *  (s, g) writes head g's part of the row itself just before, so no separate write launch
 *  precedes the decode; a slot elsewhere, or outside [0, num_blocks * block_size), sets
 *  PA_DEVERR_SLOT (an outside slot writes nothing).  The other grids launch the KV-write kernel
 *  first.  Returns as pa_decode, plus PA_ERR_NULL / PA_ERR_ALIGN for key, value or slot_mapping.
 */
int pa_decode_write(void* out, const void* q, void* k_cache, void* v_cache, const int32_t* block_tables,
                    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
                    int n_q_heads, int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale,
                    int dtype, const void* key, const void* value, const int64_t* slot_mapping, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * The dispatcher's decision for these sizes on the current device, without
 * launching: returns 1 for the one-pass kernel, 2 for split-K, or a negative
 * status (PA_ERR_SHAPE / PA_ERR_UNSUPPORTED as pa_decode, PA_ERR_CUDA).
 * *partition_tokens (if not NULL) receives the split-K piece length: a
 * multiple of block_size and of 16, at least PA_DEFAULT_PARTITION_TOKENS: a
 * quarter of max_context_len when the (sequence, KV head) units fill between one
 * and two waves of the CTAs resident on the device's SMs, else the length whose
 * grid fills whole waves.  The first
 * call for a (dtype, head_dim, group) on a device queries the kernel's
 * occupancy; later calls make no CUDA call (safe inside a stream capture).
 */
int pa_decode_plan(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim, int block_size, int max_context_len,
                   int dtype, int* partition_tokens);

/*
 * pa_decode_v1 -- the one-pass decode kernel: each (sequence, KV head) unit is
 * streamed whole by one CTA, all G query heads of the group sharing each K/V
 * load (mini_engine, "Custom CUDA kernels", v1).  When the units outnumber the
 * CTAs resident on the device, the CTAs take the longest sequences first, and
 * from two waves on (G <= 2) one CTA per resident slot runs a list of units.
 * Arguments as pa_decode; no workspace.
 */
int pa_decode_v1(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int n_q_heads,
                 int n_kv_heads, int head_dim, int block_size, int64_t num_blocks, float scale, int dtype,
                 void* stream);

/*
 * pa_decode_splitk -- split-K decode (mini_engine, "Custom CUDA kernels", v2):
 * the context is cut into pieces of partition_tokens tokens (a multiple of
 * block_size and of 16; <= 0 means 256), each piece's max, exp-sum and normalised output
 * written to the workspace; a reduce kernel merges them with weights l_p * exp(m_p - max m).
 * Sequences with one piece are written directly.  When some sequence has several pieces, one
 * CTA per resident slot takes pieces, highest piece index first, from a counter in the
 * workspace (so that the SMs that stream faster take more of them).  Arguments as pa_decode.
 */
int pa_decode_splitk(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                     int max_context_len, int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                     int block_size, int64_t num_blocks, float scale, int dtype, int partition_tokens,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_splitk_static -- pa_decode_splitk without a caller-provided workspace.
 * The pages have no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory themselves: code running inside a framework that owns every
 * device allocation (a stray cudaMalloc would bypass its pool and its accounting), code on
 * a latency-critical path that cannot afford an allocation's implicit synchronisation, and
 * code running under a stream-capture mode in which cudaMalloc is not permitted.
 *
 *  The split-K partials go to a fixed scratch array of PA_STATIC_SCRATCH_BYTES inside the
 *  library's device image; every GPU that loads the library keeps that memory until the
 *  process exits.  Arguments and results are those of pa_decode_splitk, minus the workspace.
 *  Returns PA_ERR_WORKSPACE, launching nothing, when these sizes need more partials than the
 *  array holds (pa_decode_workspace_size(num_seqs, n_q_heads, head_dim, max_context_len,
 *  partition_tokens) > PA_STATIC_SCRATCH_BYTES).
 *  The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *  with that device current; make that first call before any stream capture.
 *  All calls share the one array and it keeps whatever the last call wrote (nothing in it
 *  needs to start at zero): calls that can run at the same time on the GPU -- on different
 *  streams, or from different threads -- race on it and must be serialised by the caller.
 *  No cudaMalloc, cudaFree or other allocating call is made.
 */
#define PA_STATIC_SCRATCH_BYTES (16u << 20)

int pa_decode_splitk_static(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                            int max_context_len, int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale, int dtype, int partition_tokens,
                            void* stream);

/*
 * pa_decode_shared_prefix -- decode attention for a batch whose sequences share a prefix: the
 * same physical blocks hold the first prefix_tokens tokens of every sequence.
 * Source: mini_engine, "Features" (hash-based prefix caching: requests with a common prompt
 * prefix share its KV blocks) and "Custom CUDA kernels" (paged decode attention; the kernels
 * read K/V straight from the pool, prefix hits included).  The result is that of pa_decode on
 * the same inputs (out[s, h] = softmax-weighted sum over every token t < context_lens[s]); only
 * the order of the arithmetic differs.
 *
 * The prefix part is one dense contraction per KV head -- rows: the sequences' query heads of
 * the group; keys: the prefix tokens -- run once on the tcgen05 tensor cores (the prefill
 * kernel's tiles, in pieces of prefix_piece_tokens), which leaves per-row partials (max,
 * exp-sum, normalised output) in the workspace; the tokens past the prefix are streamed per
 * sequence by the decode kernels (pa_decode's dispatcher picks one-pass or split-K for them),
 * which fold the partials into their final merge.  The decode is launched as a programmatic
 * dependent of the prefix pass, so the two overlap.
 *
 *  Arguments as pa_decode, plus:
 *  prefix_tokens  tokens every sequence shares: table entries [0, ceil(prefix_tokens /
 *                 block_size)) are the same blocks in every row the prefix reaches, and the
 *                 prefix pass reads them from row 0 (which must hold them).  Only whole 16-token
 *                 chunks of min(prefix_tokens, max_context_len) go through the prefix pass; the
 *                 remainder is streamed per sequence.  A sequence shorter than the prefix
 *                 attends to its own context_lens[s] tokens only.  0 (or fewer than 16 shared
 *                 tokens) runs plain pa_decode.  Must be <= max_blocks_per_seq * block_size.
 *  prefix_piece_tokens  keys per CTA of the prefix pass, a multiple of 128; 0 = the library's
 *                 choice (about a quarter of the SMs busy with the prefix pass; a sixteenth when
 *                 the suffix runs on the dynamic grid: one-pass suffixes at group size 1 or 2,
 *                 up to 256 sequences, more (sequence, KV head) units than its resident CTAs).
 *                 That grid's piece counter is the workspace's first 4 bytes (the control
 *                 region pa_decode uses); it is zeroed on the stream, with the tag beside it
 *                 (a 16-byte cudaMemsetAsync), before the prefix pass.  A split-K suffix has
 *                 its own counter, at the start of the suffix's part of the workspace, zeroed
 *                 on the stream (4 bytes) before its launch.
 *  workspace  at least pa_decode_shared_prefix_workspace_size(...) bytes, caller-owned.
 *  Returns PA_ERR_BOUNDS for max_context_len or prefix_tokens beyond the table's capacity,
 *  PA_ERR_UNSUPPORTED for a piece that is not a multiple of 128, PA_ERR_WORKSPACE for a missing
 *  or small workspace; otherwise as pa_decode.
 */
size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int n_q_heads, int head_dim, int max_context_len,
                                              int prefix_tokens);

int pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                            int max_context_len, int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale, int dtype, int prefix_tokens,
                            int prefix_piece_tokens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill_chunk -- attention for ragged prefill chunks that attend to their
 * earlier cached context, on the tcgen05 tensor cores (head_dim 64, 96, 128 or 256).
 * Source: mini_engine, "Custom CUDA kernels" (paged prefill attention: tiled,
 * online softmax, K/V read from the paged pool itself, ragged batches, prefix
 * hits and chunks over earlier chunks in one launch); miniserve, "Engine"
 * (query_start_loc / block_table metadata, bottom-right causal mask).
 *
 *  out, q [total_q, n_q_heads, head_dim]; chunk c owns rows
 *         [query_start_loc[c], query_start_loc[c+1])
 *  query_start_loc [num_chunks+1] int32, seq_lens [num_chunks] int32 (kv length
 *         = cached context + the chunk's own tokens, whose K/V must already be in
 *         the cache, e.g. by pa_reshape_and_cache)
 *  block_tables [num_chunks, max_blocks_per_seq] int32
 *  max_q_len  host-side upper bound of the chunks' query lengths (sizes the grid)
 *  Row j of chunk c attends to keys t <= seq_lens[c] - q_len_c + j.
 */
int pa_prefill_chunk(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start_loc,
                     const int32_t* seq_lens, int num_chunks, int max_q_len, int n_q_heads, int n_kv_heads,
                     int head_dim, int block_size, int64_t num_blocks, float scale, int dtype, void* stream);

/*
 * pa_prefill_chunk_small_m -- pa_prefill_chunk with small-M tiles: a (chunk, KV head) unit
 * whose rows (query tokens x the group's heads) fit in 64 runs its tile as M = 64 tensor-core
 * MMAs instead of M = 128.  Meant for the unified launch, where every decode sequence is a
 * one-row chunk (G valid rows of a tile).  Source: mini_engine, "Custom CUDA kernels" (the
 * unified attention mode kept for comparison) and "Results" (unified mode is slower because a
 * decode query is a single row that wastes almost all of a prefill tile).  Same arguments,
 * result (up to the order of the arithmetic) and errors as pa_prefill_chunk.
 */
int pa_prefill_chunk_small_m(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks_per_seq, const int32_t* query_start_loc,
                             const int32_t* seq_lens, int num_chunks, int max_q_len, int n_q_heads, int n_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, float scale, int dtype, void* stream);

/*
 * Reads (and with clear != 0, resets) the error word of the current device.
 * Synchronises the device first.  Returns the PA_DEVERR_* bits, or a negative
 * status if the CUDA calls fail.
 */
int pa_device_errors(int clear);

/* Human-readable name of a status code. */
const char* pa_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDATTN_H */
