/*
 * pagedkv.h -- C ABI of the paged KV-cache attention library (libpagedkv.so).
 *
 * The library implements the hot path of attention over a paged (blocked) KV
 * cache on one GB300 (sm_103a): a host block pool with reference-counted,
 * copy-on-write blocks; a slot-mapped K/V append; exact decode attention over
 * non-contiguous blocks; and a ragged mixed batch in which prefill chunks
 * attend causally to their cached prefix alongside decode tokens.
 *
 * Pages this follows (cited by title and section):
 *   [Deploy]  "大模型部署.md" (AIGC-Interview-Book), §2.1 vLLM 框架技术详解:
 *             3. 调度策略与显存块管理 (can_allocate, _allocate_sequence,
 *             append_slots with copy-on-write), 4. PageAttention 内存管理技术详解;
 *             §2.5 LMDeploy 2. TurboMind (split-K decoding);
 *             §4.1 注意力机制计算优化 (1. FlashAttention, 4. MQA 与 GQA)
 *   [Infra]   "【自用】AI infra相关", 一、推理两阶段 (decode appends K_t,V_t then
 *             attends), 二、vLLM (block table, copy-on-write, free block list)
 *   [FastGen] "DeepSpeed-FastGen 深度解析", §3.2 动态分割融合 (token budget)
 *   [Ch15]    "第 15 章：推理引擎与部署", §15.1 算法详解 (online softmax),
 *             §15.6 PagedAttention：分页 KV Cache, 两阶段与 Chunked Prefill
 *
 * Conventions for every function:
 *   - Return an int status: PKV_OK (0) or a negative PKV_ERR_* code.  No
 *     function aborts the process or throws across the ABI.
 *   - Pointers documented "device" must point to memory of the current CUDA
 *     device; pointers documented "host" to ordinary host memory.  The caller
 *     owns all memory; no entry point allocates device memory.
 *   - Device entry points only enqueue work on `stream` (a cudaStream_t passed
 *     as void*, NULL = legacy default stream) and return without waiting.
 *     Stream order holds in full: the kernels of one call are chained with
 *     programmatic dependent launch, but each waits for the work ahead of it
 *     on the stream before it reads any input or plan.
 *     Arguments that can be checked on the host are checked before anything
 *     is launched (PKV_ERR_INVALID / PKV_ERR_UNSUPPORTED, nothing enqueued).
 *     Values that live in device memory (block ids, slots, lengths) are
 *     checked by the kernels: an offending access is skipped and a code is
 *     recorded in the device error word (read it with pkv_device_error).
 *   - Cache layout (fixed): K and V are separate pools, each
 *     [num_blocks][num_kv_heads][block_size][head_dim], row-major, in the
 *     cache dtype.  One (block, kv head) tile is contiguous.  The 8-bit cache
 *     (PKV_INT8) is one pool instead, laid out with the *_int8 entry points.
 *   - Query head h uses KV head h / (num_q_heads / num_kv_heads).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define PKV_OK               0
#define PKV_ERR_INVALID     -1  /* bad argument: null pointer, bad size, unknown sequence */
#define PKV_ERR_NO_BLOCKS   -2  /* pool cannot serve the request now (LATER) */
#define PKV_ERR_NEVER       -3  /* pool can never serve the request (NEVER) */
#define PKV_ERR_UNSUPPORTED -4  /* shape / dtype the kernels do not implement */
#define PKV_ERR_CUDA        -5  /* a CUDA runtime call or launch failed */
#define PKV_ERR_WORKSPACE   -6  /* workspace null, misaligned or too small */
#define PKV_ERR_HOST        -7  /* host memory allocation failed */

/* ---- device error word codes (pkv_device_error) ------------------------ */
#define PKV_DEV_OK               0
#define PKV_DEV_BAD_BLOCK_ID     1  /* block table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_CONTEXT_LEN  2  /* context length < 1, > max_context_len, or < query length */
#define PKV_DEV_BAD_SLOT         3  /* slot >= num_blocks * block_size */
#define PKV_DEV_BAD_COPY_PAIR    4  /* copy pair block id outside the pool */
#define PKV_DEV_BAD_QUERY_LAYOUT 5  /* query_start_loc not non-decreasing from 0 to num_query_tokens */
#define PKV_DEV_WAIT_TIMEOUT     6  /* a pipeline wait exceeded its limit (internal fault) */
#define PKV_DEV_TABLE_TOO_NARROW 7  /* context needs more blocks than max_blocks_per_seq */
#define PKV_DEV_BAD_POSITION     8  /* rotary position outside [0, max_position) */

/* ---- data types -------------------------------------------------------- */
#define PKV_F32  0
#define PKV_BF16 1
#define PKV_INT8 2   /* 8-bit codes + fp32 scales in the cache; q, k, v, out bf16 */

typedef struct pkv_cache_desc {
    int32_t dtype;        /* PKV_F32 or PKV_BF16: cache, q, k, v and out share it;
                             PKV_INT8: only the *_int8 entry points take it */
    int32_t num_blocks;   /* physical blocks in each of the K and V pools (in the
                             one pool of an 8-bit cache) */
    int32_t block_size;   /* tokens per block (the kernels implement 16) */
    int32_t num_kv_heads;
    int32_t num_q_heads;  /* multiple of num_kv_heads; group size 1, 2, 4 or 8 */
    int32_t head_dim;     /* 64 or 128 */
} pkv_cache_desc;

/* ======================================================================== *
 * Host block pool (metadata only; never touches device memory).
 *
 * Follows [Deploy §2.1 3.] and [Infra 二]: fixed-size physical blocks, a free
 * block list, one block table per sequence, reference counts shared by forked
 * sequences, copy-on-write of a shared last block, and admission with a
 * watermark.  Readings where the pages are silent: the free list is a stack
 * (the block freed last is handed out first); `free_order` lists the initial
 * stack from the top; a sequence's blocks are released in table order.
 * A pool object is not thread-safe.
 * ======================================================================== */
typedef struct pkv_pool pkv_pool;

/* Create a pool of `num_blocks` blocks of `block_size` tokens.  `free_order`
 * (host, optional, [num_blocks]) is a permutation of 0..num_blocks-1 whose
 * first entry is handed out first; NULL means 0, 1, 2, ...  On success *out
 * owns the pool (release with pkv_pool_destroy). */
PKV_API int pkv_pool_create(int32_t num_blocks, int32_t block_size, int32_t watermark_blocks,
                    const int32_t* free_order, pkv_pool** out);
PKV_API int pkv_pool_destroy(pkv_pool* pool);

/* Pool variants [Deploy §2.1 BlockSpaceManager(sliding_window, enable_caching);
 * the pages refuse the two together, and so does this call with
 * PKV_ERR_UNSUPPORTED].
 *
 * PKV_POOL_PREFIX_CACHING [Deploy §2.1 CachedBlockAllocator, LRUEvictor]:
 *   - Full blocks are shared by a hash of the whole token prefix.  The hash
 *     of logical block j is FNV-1a 64 over the previous block's hash (0 for
 *     block 0; 8 bytes little-endian) followed by the block's token ids
 *     (4 bytes little-endian each).  A block holding that hash, in use or
 *     parked, is reused (reference count + 1); the partial last block of a
 *     prompt is never shared.
 *   - A hashed block whose last reference goes away is parked in the evictor,
 *     not freed.
 *   - New blocks come from the free list, else from the evictor: least
 *     recently accessed first, then the one whose hash covers the most tokens,
 *     then the one parked first.
 *   - Access times come from pkv_pool_set_clock.
 *   - Sequences are added with pkv_seq_add_tokens and grown with
 *     pkv_seq_append_token; the count-only calls return PKV_ERR_UNSUPPORTED.
 *   - When a token fills its block, the block's hash is looked up: if it is
 *     found, the sequence switches to that block (the filled block is freed
 *     and any copy pair of that call is cancelled); otherwise the block is
 *     registered under the hash.
 *   - Free counts and admission include parked blocks.
 *
 * sliding_window > 0 (a multiple of block_size; W_b = window / block_size)
 * [Deploy §2.1 block_sliding_window]:
 *   - A table is a ring of W_b blocks: logical block j >= W_b reuses entry
 *     j % W_b.  Admission counts min(blocks, W_b).
 *   - A prompt token whose slot a later token of the same prompt takes gets
 *     slot -1 (skip it when appending).
 *   - A shared ring block is copied before it is written.
 *   - pkv_block_tables exports the ring entries of the last W_b logical
 *     blocks in logical order, with context min(len, window): exactly the
 *     last `window` tokens, for decode.
 * flags = 0 and sliding_window = 0 is pkv_pool_create. */
#define PKV_POOL_PREFIX_CACHING 1
PKV_API int pkv_pool_create_ex(int32_t num_blocks, int32_t block_size, int32_t watermark_blocks,
                               const int32_t* free_order, int32_t flags, int32_t sliding_window,
                               pkv_pool** out);

/* Sliding-window pool that also serves prefill chunks [Deploy §2.1
 * block_sliding_window; the pages leave the attention mask open, and the
 * reading taken is that a query at position p sees keys max(0, p - W + 1) .. p,
 * W = sliding_window].  A chunk of C queries needs its C + W - 1 most recent
 * keys at once, more than a ring of W_b = W / block_size blocks holds, so the
 * ring here has W_b + ceil((max_chunk - 1) / block_size) blocks and holds the
 * last ring * block_size tokens; max_chunk = 1 is the pool of
 * pkv_pool_create_ex.  Everything else is as there: admission counts
 * min(blocks, ring); a prompt token whose slot a later token of the same
 * prompt takes gets slot -1; a shared ring block is copied before a write.
 * Chunked prompts are added with their first chunk (pkv_seq_add) and grown
 * chunk by chunk (pkv_seq_append_slot per token); attention takes tables from
 * pkv_window_tables and the window from paged_attention_varlen_window.
 * sliding_window: a positive multiple of block_size; max_chunk >= 1. */
PKV_API int pkv_pool_create_window(int32_t num_blocks, int32_t block_size,
                                   int32_t watermark_blocks, const int32_t* free_order,
                                   int32_t sliding_window, int32_t max_chunk, pkv_pool** out);
/* Free blocks, parked (evictable) blocks included. */
PKV_API int pkv_pool_num_free(const pkv_pool* pool, int32_t* out);
/* Parked blocks of a prefix-caching pool (0 otherwise). */
PKV_API int pkv_pool_num_evictable(const pkv_pool* pool, int32_t* out);
/* The access clock stamped on blocks handed out or parked from now on. */
PKV_API int pkv_pool_set_clock(pkv_pool* pool, int64_t now);

/* Admission of a new sequence of `num_tokens` tokens [Deploy §2.1 can_allocate]:
 * PKV_ERR_NEVER if num_blocks - need < watermark, PKV_OK if
 * free - need >= watermark, PKV_ERR_NO_BLOCKS (LATER) otherwise. */
PKV_API int pkv_pool_can_allocate(const pkv_pool* pool, int32_t num_tokens);

/* Add sequence `seq_id` with `num_tokens` prompt tokens: applies the admission
 * rule above, then takes ceil(num_tokens / block_size) blocks with reference
 * count 1.  `slots_out` (host, optional, [num_tokens]) receives the physical
 * slot block * block_size + row of every token in order.  On any error the
 * pool is unchanged. */
PKV_API int pkv_seq_add(pkv_pool* pool, int64_t seq_id, int32_t num_tokens, int64_t* slots_out);

/* Add a sequence from its token ids (host, [num_tokens]).  Prefix caching:
 * full blocks are shared as described at pkv_pool_create_ex and
 * *num_cached_tokens_out (optional) = block_size * the number of leading
 * blocks that were found, whose K/V the caller need not write again.  Other
 * pools: as pkv_seq_add, with *num_cached_tokens_out = 0. */
PKV_API int pkv_seq_add_tokens(pkv_pool* pool, int64_t seq_id, const int32_t* token_ids,
                               int32_t num_tokens, int64_t* slots_out,
                               int32_t* num_cached_tokens_out);

/* New sequence `child` shares every block of `parent` (reference count + 1 each). */
PKV_API int pkv_seq_fork(pkv_pool* pool, int64_t parent, int64_t child);

/* Grow `seq_id` by one token [Deploy §2.1 append_slots].  A new block is taken
 * only when the last block is full.  If the last block is shared (reference
 * count > 1) a fresh block replaces it in this sequence's table and the pair
 * (*cow_src, *cow_dst) tells the caller which whole block to copy (with
 * pkv_copy_blocks) before writing the token; otherwise both are set to -1.
 * *slot_out receives the token's slot.  PKV_ERR_NO_BLOCKS (pool unchanged)
 * when a block is needed and none is free. */
PKV_API int pkv_seq_append_slot(pkv_pool* pool, int64_t seq_id, int64_t* slot_out,
                        int32_t* cow_src, int32_t* cow_dst);

/* pkv_seq_append_slot for a token whose id is known; a prefix-caching pool
 * needs it to hash the block the token fills (see pkv_pool_create_ex). */
PKV_API int pkv_seq_append_token(pkv_pool* pool, int64_t seq_id, int32_t token_id,
                                 int64_t* slot_out, int32_t* cow_src, int32_t* cow_dst);

/* Drop one reference on each block of the sequence (table order); blocks that
 * reach zero return to the free list (hashed blocks of a prefix-caching pool:
 * to the evictor). */
PKV_API int pkv_seq_free(pkv_pool* pool, int64_t seq_id);

PKV_API int pkv_seq_len(const pkv_pool* pool, int64_t seq_id, int32_t* len_out);
PKV_API int pkv_block_ref_count(const pkv_pool* pool, int32_t block, int32_t* out);
/* The hash a prefix-caching pool has registered for `block`: *hashed_out = 1
 * and *hash_out = the hash, or 0 and 0. */
PKV_API int pkv_block_hash(const pkv_pool* pool, int32_t block, uint64_t* hash_out,
                           int32_t* hashed_out);

/* Export block tables and context lengths of `n` sequences (host buffers):
 * tables_out [n][max_blocks] padded with -1, ctx_lens_out [n] (optional).
 * PKV_ERR_INVALID if a table needs more than max_blocks entries.  A window
 * pool whose ring has room for chunks (pkv_pool_create_window, max_chunk > 1)
 * has no exact-window export: PKV_ERR_UNSUPPORTED (use pkv_window_tables). */
PKV_API int pkv_block_tables(const pkv_pool* pool, const int64_t* seq_ids, int32_t n,
                     int32_t max_blocks, int32_t* tables_out, int32_t* ctx_lens_out);

/* Tables of a sliding-window pool for paged_attention_varlen_window (host
 * buffers).  For sequence i of length L whose last query_lens[i] = q tokens
 * are this step's queries, the first key any of them attends is
 * f = max(0, L - q - W + 1); the row lists the ring entries of logical blocks
 * f / block_size .. ceil(L / block_size) - 1 in logical order (the first and
 * the last entry may be the same physical block) and ctx_lens_out[i] =
 * L - (f / block_size) * block_size, so table index t is position
 * (f / block_size) * block_size + t.  Rows are padded with -1 to max_blocks.
 * PKV_ERR_INVALID (nothing written) for an unknown sequence, q outside
 * [1, L], q + W - 1 above the ring's tokens, or a row wider than max_blocks;
 * PKV_ERR_UNSUPPORTED for a pool without a window. */
PKV_API int pkv_window_tables(const pkv_pool* pool, const int64_t* seq_ids,
                              const int32_t* query_lens, int32_t n, int32_t max_blocks,
                              int32_t* tables_out, int32_t* ctx_lens_out);

/* Compose one forward pass of a mixed batch under a token budget [FastGen
 * §3.2 动态分割融合: split long prompts, fuse short ones, keep every pass the
 * same size; Ch15 §15.6 两阶段与 Chunked Prefill: sum(prefill chunk tokens) +
 * decode sequences <= budget, decodes first].  `num_decode` running sequences
 * each want one token; `prompt_remaining` (host, [num_prompts]) are the
 * unprocessed prompt tokens of waiting requests in arrival order.
 * *decode_admitted = min(num_decode, budget); then chunk_out[i] (host,
 * [num_prompts]) = min(prompt_remaining[i], budget left), in order, so only
 * the last prompt served is split.  *tokens_used (optional) = tokens placed.
 * Pure host code. */
PKV_API int pkv_splitfuse_compose(int32_t token_budget, int32_t num_decode, int32_t num_prompts,
                                  const int32_t* prompt_remaining, int32_t* chunk_out,
                                  int32_t* decode_admitted, int32_t* tokens_used);

/* ======================================================================== *
 * Device entry points.
 * ======================================================================== */

/* Copy-on-write block copies [Deploy §2.1 append_slots (the new block gets the
 * shared block's tokens); Infra 二 copy-on-write]: for each pair i, K and V
 * block pairs[2i+1] become byte-for-byte copies of block pairs[2i] (all heads,
 * all rows).
 * block_pairs: device int32 [num_pairs][2] (src, dst).  Destinations must be
 * distinct and no destination may also be a source (pairs run in parallel).
 * num_pairs == 0 is a no-op. */
PKV_API int pkv_copy_blocks(const int32_t* block_pairs, int32_t num_pairs, void* k_cache, void* v_cache,
                    const pkv_cache_desc* desc, void* stream);

/* Append [Infra 一、2 解码 (K_t, V_t written into the cache); Deploy §2.1 (the
 * block manager plans slots, the cache engine writes them)]:
 *   cache[slot / block_size][h][slot % block_size][:] = x[t][h][:]
 * for K and V and every kv head h.  k, v: device [num_tokens][num_kv_heads]
 * [head_dim] in the cache dtype (a bit copy: no conversion).  slot_mapping:
 * device int64 [num_tokens]; a negative slot skips that token (padding); slots
 * must be distinct.  num_tokens == 0 is a no-op. */
PKV_API int paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                    void* k_cache, void* v_cache, const pkv_cache_desc* desc, void* stream);

/* Append with rotary position embedding fused in [Ch15 §15.3 RoPE 与 Flash
 * Attention 的融合: rotate in registers rather than in a separate pass through
 * HBM; FastGen §6 (rotary fused with the blocked-KV write)].  Rotate-half form
 * (the pages defer RoPE's formula; this is the reading taken): for token t at
 * position p = positions[t] and i < head_dim/2, with c = cos_sin[p][i] and
 * s = cos_sin[p][head_dim/2 + i],
 *   x'[i] = x[i] c - x[i + D/2] s,   x'[i + D/2] = x[i] s + x[i + D/2] c,
 * each product and sum rounded in fp32 on its own (no fused multiply-add),
 * then rounded to the cache dtype (bf16: nearest-even).  K is rotated and
 * written with V through slot_mapping as paged_kv_append does; V is copied
 * unrotated; q (device [T][Hq][D], optional) is rotated into q_out (may alias
 * q; both NULL to skip).  cos_sin: device fp32 [max_position][head_dim],
 * 16-byte aligned.  positions: device int32 [T]; a position outside
 * [0, max_position) sets PKV_DEV_BAD_POSITION and that row is skipped.
 * head_dim 64 or 128. */
PKV_API int paged_kv_append_rope(const void* q, void* q_out, const void* k, const void* v,
                                 const int64_t* slot_mapping, const int32_t* positions,
                                 const float* cos_sin, int32_t max_position, int32_t num_tokens,
                                 void* k_cache, void* v_cache, const pkv_cache_desc* desc,
                                 void* stream);

/* Bytes of workspace paged_attention_decode needs for `num_seqs` sequences
 * whose context lengths are at most `max_context_len` (0 on bad arguments). */
PKV_API size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs,
                                  int32_t max_context_len);

/* Decode attention, one query token per sequence [Ch15 §15.1 (exact softmax
 * computed with the online m / l / alpha recurrence); Ch15 §15.6 (block table
 * lookup); Deploy §4.1 4. (GQA: a KV head is read once for its whole query
 * group); Deploy §2.5 (split-K decoding)]:
 *   out[s][h] = softmax(q[s][h] . K_s^T * scale) V_s
 * over keys 0 .. context_lens[s]-1 of sequence s, where K_s/V_s are gathered
 * through block_tables[s].  context_lens counts the query's own token, which
 * must already be appended.
 *   out, q:        device [num_seqs][num_q_heads][head_dim] (cache dtype)
 *   block_tables:  device int32 [num_seqs][max_blocks_per_seq]
 *   context_lens:  device int32 [num_seqs], each in [1, max_context_len]
 *   scale:         usually 1/sqrt(head_dim)
 *   workspace:     device, >= pkv_decode_workspace_bytes(...), 256-byte aligned;
 *                  holds split partials; must not be shared by concurrent calls.
 * Long contexts are split into fixed spans of 512 tokens whose partial
 * (max, sum, output) states are merged in a second kernel; the split depends
 * only on the context length, so a sequence's result does not depend on the
 * rest of the batch, with one exception: for groups of 8 query heads, a
 * complete split whose 32 block ids a sequence shares with its neighbours in
 * the batch (parallel-sampling branches of one prompt [Deploy §2.1 4.
 * PageAttention: shared blocks]) is computed once for up to 8 of them, each
 * tile read once per KV head, and rounds differently (within the same error
 * bound) from the same split computed alone.  num_seqs == 0 is a no-op: the descriptor and the sizes
 * are checked, the pointers are not (zero-sized tensors may be null). */
PKV_API int paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const pkv_cache_desc* desc, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t max_context_len, float scale,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Decode attention for callers that cannot allocate device memory (no
 * counterpart on the pages; it exists for library users).  Callers such as a
 * plugin inside an engine that owns all device memory and offers no scratch
 * allocator, or a server whose KV pool already took the rest of HBM, have no
 * way to provide the workspace paged_attention_decode needs.  This entry point
 * computes exactly what paged_attention_decode computes, with the same
 * arguments minus the workspace, using a fixed scratch array of
 * PKV_NOALLOC_SCRATCH_BYTES that the library holds in the device memory of
 * every GPU that loads it until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - PKV_ERR_WORKSPACE (nothing enqueued) when the batch's split partials
 *     (pkv_decode_workspace_bytes) exceed PKV_NOALLOC_SCRATCH_BYTES.
 *   - The first call on a device looks up the array's device address with that
 *     device current; make that first call before any stream capture.  The
 *     address is kept for the life of the device's primary context: after a
 *     cudaDeviceReset (or any reset of that context) the library's device
 *     state is gone, and no entry point may be called on that device again in
 *     this process.
 *   - All calls share the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls that overlap on the GPU
 *     (other streams, other threads) race on it and corrupt each other's
 *     results; serialize them. */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
PKV_API int paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const pkv_cache_desc* desc,
                                           const int32_t* block_tables,
                                           int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, int32_t num_seqs,
                                           int32_t max_context_len, float scale, void* stream);

/* Bytes of workspace paged_attention_varlen needs. */
PKV_API size_t pkv_varlen_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs,
                                  int32_t num_query_tokens, int32_t max_query_len,
                                  int32_t max_context_len);

/* Ragged mixed batch [FastGen §3.2 动态分割融合; Ch15 §15.6 两阶段与 Chunked
 * Prefill]: sequence s owns query rows query_start_loc[s] .. query_start_loc[s+1]-1
 * (qlen_s rows, possibly 0).  Those rows are the sequence's last qlen_s
 * positions, whose K/V must already be appended; row i attends causally to
 * keys 0 .. context_lens[s] - qlen_s + i.  Rows with qlen_s == 1 take the
 * decode path; longer spans (prefill chunks over a cached prefix) take the
 * tensor-core prefill path.
 *   out, q:           device [num_query_tokens][num_q_heads][head_dim]
 *   query_start_loc:  device int32 [num_seqs + 1], 0 .. num_query_tokens
 *   context_lens:     device int32 [num_seqs], >= qlen_s, <= max_context_len
 *   max_query_len:    host upper bound of qlen_s
 * num_seqs == 0 or num_query_tokens == 0 is a no-op (pointers unchecked).
 * Other arguments as for paged_attention_decode. */
PKV_API int paged_attention_varlen(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const pkv_cache_desc* desc, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* query_start_loc,
                           const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_query_tokens, int32_t max_query_len,
                           int32_t max_context_len, float scale, void* workspace,
                           size_t workspace_bytes, void* stream);

/* paged_attention_varlen under a sliding window of `window` keys [Deploy §2.1
 * block_sliding_window keeps a ring of blocks per sequence; the pages leave the
 * mask open, and the reading taken is that a query sees its `window` most
 * recent keys, its own included]: row i of sequence s attends table indices
 *   max(0, a - window + 1) .. a,   a = context_lens[s] - qlen_s + i,
 * where the table lists the sequence's blocks in logical order from any block
 * (table index = position - the table's first position): the layout
 * pkv_window_tables exports, whose context_lens count from that first block.
 * Keys below a row's window are masked; decode rows (qlen 1) skip the blocks
 * and 512-token splits below their window, and the split of a sequence
 * depends only on its context length and the window, so results do not depend
 * on the batch.  window = 0 is paged_attention_varlen; window < 0 is
 * PKV_ERR_INVALID.  Other arguments, workspace and errors as for
 * paged_attention_varlen. */
PKV_API int paged_attention_varlen_window(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const pkv_cache_desc* desc,
                                          const int32_t* block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t* query_start_loc,
                                          const int32_t* context_lens, int32_t num_seqs,
                                          int32_t num_query_tokens, int32_t max_query_len,
                                          int32_t max_context_len, int32_t window, float scale,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* 8-bit KV cache [Deploy §2.5 LMDeploy, 2. TurboMind 推理引擎解析 (the KV cache
 * kept in 8 bits, halving the bytes decode reads)].  The pages give no format;
 * the one implemented is symmetric int8 with one fp32 scale per (token, kv head):
 *   amax = max_d |x[d]|,  scale = amax / 127,
 *   code[d] = clamp(rint(x[d] / scale), -127, 127)     (code = 0 when amax = 0)
 * with both divisions rounded once in fp32 (ties to even), so the stored codes
 * and scales are reproducible bit for bit.  A value reads back as code * scale.
 * Pool (desc->dtype = PKV_INT8; block_size 16; head_dim 64 or 128):
 *   kv_pool: device bytes, 16-byte aligned, owned by the caller, ordered
 *            [num_blocks][num_kv_heads][2][PKV_INT8_TILE_BYTES(head_dim)]:
 *            per (block, kv head) its K tile and then its V tile, each of
 *            PKV_INT8_TILE_BYTES(head_dim) = 16 * head_dim + 64 bytes
 *            (PKV_INT8_POOL_BYTES(num_blocks, num_kv_heads, head_dim) in all)
 * A tile holds the codes of its 16 token rows (bytes 0 .. 16 * head_dim - 1)
 * and then their 16 fp32 scales (scale of row r at byte 16 * head_dim + 4 r),
 * so the decode reads a (block, kv head)'s K and V in one contiguous run of
 * 2 * PKV_INT8_TILE_BYTES(head_dim) bytes.  Inside the
 * codes, the code of token row r (slot % 16) and dimension d is stored at
 *   K: r * head_dim + 16 * ((d / 16) ^ sw(r)) + d % 16,
 *      sw(r) = r & 7 (head_dim 128) or (r >> 1) & 3 (head_dim 64)
 *   V: d * 16 + r
 * (layouts the decode kernel reads without shared-memory bank conflicts).
 * Whole tiles can be moved as bytes: the layout depends only on r.
 *
 * Append: k, v device bf16 [num_tokens][num_kv_heads][head_dim], quantised and
 * written through slot_mapping as paged_kv_append writes (negative slot skips;
 * slot >= num_blocks * block_size sets PKV_DEV_BAD_SLOT and is skipped). */
#define PKV_INT8_TILE_BYTES(head_dim) (16 * (head_dim) + 64)
#define PKV_INT8_POOL_BYTES(num_blocks, num_kv_heads, head_dim) \
    ((size_t)(num_blocks) * (size_t)(num_kv_heads) * 2u * (size_t)PKV_INT8_TILE_BYTES(head_dim))

PKV_API int paged_kv_append_int8(const void* k, const void* v, const int64_t* slot_mapping,
                                 int32_t num_tokens, void* kv_pool, const pkv_cache_desc* desc,
                                 void* stream);

/* Copy-on-write for an 8-bit cache: for each (src, dst) pair, the tiles of
 * block src (every kv head's K and V tiles, codes and scales: one contiguous
 * run per block) are copied to block dst, as pkv_copy_blocks does for the
 * other caches.  block_pairs: device int32
 * [num_pairs][2]; an id outside [0, num_blocks) sets PKV_DEV_BAD_COPY_PAIR and
 * that pair is skipped.  desc->block_size must be 16 (the tile has 16 rows;
 * PKV_ERR_UNSUPPORTED otherwise). */
PKV_API int pkv_copy_blocks_int8(const int32_t* block_pairs, int32_t num_pairs, void* kv_pool,
                                 const pkv_cache_desc* desc, void* stream);

/* Decode attention over the 8-bit cache: exactly the attention of
 * paged_attention_decode over the dequantised keys and values (code * scale),
 * computed with the same splits and merge.  q, out: device bf16
 * [num_seqs][num_q_heads][head_dim].  workspace: >= pkv_decode_workspace_bytes
 * of the same desc.  Other arguments and errors as for paged_attention_decode. */
PKV_API int paged_attention_decode_int8(void* out, const void* q, const void* kv_pool,
                                        const pkv_cache_desc* desc,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t num_seqs,
                                        int32_t max_context_len, float scale, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Read the current device's error word into *code_out (PKV_DEV_* code of the
 * first fault recorded since the last clear) and, if `clear` is non-zero,
 * reset it.  Synchronizes the device.  The word's device address is looked up
 * once per device and kept for the life of its primary context (see
 * paged_attention_decode_noalloc on device resets). */
PKV_API int pkv_device_error(int32_t* code_out, int32_t clear);

/* Static description of a status code (never NULL). */
PKV_API const char* pkv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
