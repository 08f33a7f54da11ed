// Decode attention over a paged KV cache: planner, split kernel and merge.
//
// What is computed: for one query token per sequence, exact
// softmax(q K^T * scale) V over the sequence's keys, reached through its block
// table ("第 15 章：推理引擎与部署" §15.6 PagedAttention：分页 KV Cache).  The
// softmax is accumulated block by block with the online recurrence of §15.1
// 算法详解 (running max m, running sum l, rescale alpha = exp(m_old - m_new)),
// here in base 2: scores are pre-multiplied by scale * log2(e) and exp2 is used,
// which is the same function.  The KV tile of one block (B_c = 16 keys) is the
// recurrence's column block.
//
// GB300 design:
//  * HBM-bound: each (block, kv head) K and V tile is one contiguous 16 x D run
//    (4 KiB for bf16, D = 128), fetched by the TMA engine with cp.async.bulk
//    into a shared-memory ring guarded by mbarriers; a producer warp keeps up
//    to kStages tiles in flight per CTA.
//  * GQA packing ("大模型部署.md" §4.1 4. MQA 与 GQA): one CTA owns one KV head
//    and all G query heads that read it, so each KV byte is read once.
//  * Split-K over the context ("大模型部署.md" §2.5 TurboMind split-K
//    decoding): a sequence's context is cut into fixed 512-token splits; each
//    (split, kv head) is one work unit; partial (m, l, O) states are merged by
//    a second kernel with the same alpha rescaling.  The split depends only on
//    the context length, so results do not depend on the batch (except where
//    the planner groups sequences that read the same blocks, below).
//  * Shared prompt blocks ("大模型部署.md" §2.1 4. PageAttention: parallel
//    sampling shares a prompt's blocks by reference count): for groups of 8
//    query heads, consecutive sequences whose complete split reads the same
//    32 blocks get one work unit, so each shared tile is read once per KV head.
//  * Persistent grid (a multiple of the SM count) over a work list that a
//    one-CTA planner kernel builds on the device, so no host round trip.
//  * Sliding window of W keys ("大模型部署.md" §2.1 block_sliding_window, with
//    the reading that a query sees its W most recent keys): a decode row
//    attends keys max(0, ctx - W) .. ctx - 1 of a logically ordered table; the
//    planner starts its splits at the one holding the window's first key, a
//    split skips the blocks below it and masks the keys below it in its block,
//    and the merge starts at that split.
#include <algorithm>
#include <atomic>
#include <cfloat>
#include <cuda_runtime.h>

#include "decode_common.cuh"
#include "launch_cache.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Planner: one CTA scans the batch, validates lengths and writes the work list.
// ---------------------------------------------------------------------------
struct PlanParams {
    const int32_t* context_lens;
    const int32_t* query_start_loc;  // nullptr: decode-only batch
    int32_t num_seqs;
    int32_t num_query_tokens;
    int32_t max_context_len;
    int32_t table_stride;
    int32_t tokens_per_tile;          // prefill tile height in tokens
    int32_t num_sms;
    int32_t window;                   // sliding window in keys (0: none)
    int32_t group;                    // group sequences that share complete splits
    const int32_t* block_tables;      // read only when grouping
    float ns_per_token;               // decode: K + V bytes of a token (all KV heads) at the planning rate
    float ns_per_pair;                // prefill: QK^T + PV flops of a (query, key) pair (all
                                      // query heads) at the planning rate
    Workspace ws;
    int* err;
};

constexpr int kGroupSeqs = 4096;    // batches up to this size are grouped (shared memory)
constexpr int kSortItems = 2048;    // prefill items reordered longest first (at most)
constexpr int kSortBuckets = 256;   // key-tile counts (larger counts share the last bucket)

// Complete 512-token splits of a decode row over `ctx` keys, or 0 when the row
// fails the planner's checks (it is then flagged and gets no work).
__device__ __forceinline__ int complete_splits(const PlanParams& p, int ctx) {
    const bool valid = ctx >= 1 && ctx <= p.max_context_len &&
                       (ctx + kBlockTokens - 1) / kBlockTokens <= p.table_stride;
    return valid ? ctx / kSplitTokens : 0;
}

// Decode items of sequence s when sequences that share complete splits are
// grouped (paged_attention_decode, groups of 8 query heads, no window).
// sh[s] = n means s reads the same 32 blocks as sequence s - 1 in each of its
// first n splits (s "follows" s - 1 there).  For each split j a run of
// sequences reads the same blocks: one that does not follow, then the
// followers after it.  A run is cut into chunks at batch positions that are
// multiples of kMaxGroup; each chunk is one item, owned by its first sequence
// (a grouped item when the chunk holds two or more sequences, else a plain
// one).  So s owns split j when it starts a run there, or follows and sits at
// a multiple of kMaxGroup.  Writes s's items when `out` is given; returns
// their number.
__device__ __forceinline__ int grouped_items(const PlanParams& p, const int* sh, int s, int ctx,
                                             int2* out) {
    const int nsplit = (ctx - 1) / kSplitTokens + 1;
    const int own = sh[s];
    // how far the chunk may reach: up to the next multiple of kMaxGroup
    const int cap = min(kMaxGroup - s % kMaxGroup, p.num_seqs - s);
    int f[kMaxGroup - 1];                     // shares of the sequences after s in the chunk
#pragma unroll
    for (int k = 0; k < kMaxGroup - 1; ++k) f[k] = k + 1 < cap ? sh[s + 1 + k] : 0;
    if (own == 0 && f[0] == 0) {
        // shares nothing with its neighbours: one item per split
        if (out)
            for (int j = 0; j < nsplit; ++j) out[j] = make_int2(s, j);
        return nsplit;
    }
    const bool aligned = s % kMaxGroup == 0;
    int n = 0;
    for (int j = 0; j < nsplit; ++j) {
        if (j < own && !aligned) continue;    // inside a chunk another sequence owns
        int m = 1;                            // sequences s .. s + m - 1 read split j
#pragma unroll
        for (int k = 0; k < kMaxGroup - 1; ++k)
            if (m == k + 1 && f[k] > j) m = k + 2;
        if (out) out[n] = make_int2(s, j | (m >= 2 ? m << kItemSplitBits : 0));
        ++n;
    }
    return n;
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanParams p) {
    __shared__ int warp_d[32], warp_p[32];
    __shared__ int carry_d, carry_p;
    __shared__ unsigned long long warp_tok[32], warp_pairs[32];
    // prefill items and their sort buckets, recorded during the pass (when they
    // fit) so the longest-first reorder needs no second round of global loads
    __shared__ int2 s_item[kSortItems];
    __shared__ int s_bucket[kSortItems];
    __shared__ int hist[kSortBuckets], cursor[kSortBuckets];
    __shared__ int s_shared[kGroupSeqs];   // shared_splits of each sequence (grouped
                                           // decode batches) or the prefill rows' first
                                           // items, lengths and contexts (one_pass)
    const bool group = p.group && p.num_seqs <= kGroupSeqs;
    const bool one_pass = !group && p.num_seqs <= 1024;
    static_assert(kGroupSeqs >= 3 * 1024, "three per-row arrays for one_pass");
    unsigned long long my_tok = 0, my_pairs = 0;   // this thread's work estimate
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sortable = min(kSortItems, p.ws.max_prefill_items);
    // launched programmatically behind the previous kernel (the step's append,
    // or the previous call's merge): the lengths and the workspace are read and
    // written only after it completes.  The kernels that consume the plan may
    // launch now; each waits for this grid to complete before it reads the plan.
    pdl_wait_prerequisites();
    pdl_launch_dependents();
    // the two ends of the query layout, loaded now and checked after the pass
    // (a bad layout empties the plan), so their latency overlaps the pass
    int q_first = 0, q_last = 0;
    if (tid == 0 && p.query_start_loc) {
        q_first = p.query_start_loc[0];
        q_last = p.query_start_loc[p.num_seqs];
    }
    if (tid == 0) {
        carry_d = 0;
        carry_p = 0;
    }
    for (int i = tid; i < kSortBuckets; i += 1024) hist[i] = 0;
    if (group) {
        // How many leading complete splits each sequence shares, block for
        // block, with the one before it.  First every thread checks its
        // sequences' first block ids (one round of loads for the batch); then a
        // warp per remaining candidate compares the ids of up to 8 splits at a
        // time, a lane per block.
        constexpr int kPer = kSplitTokens / kBlockTokens;
        constexpr int kBatch = 8;
        static_assert(kPer == 32, "one block id per lane");
        for (int s = tid; s < p.num_seqs; s += 1024) {
            int cand = 0;                        // -(splits to compare) for a candidate
            if (s > 0) {
                const int c1 = p.context_lens[s], c0 = p.context_lens[s - 1];
                const int32_t* t1 = p.block_tables + size_t(s) * p.table_stride;
                const int32_t f1 = t1[0], f0 = t1[-p.table_stride];
                const int n = min(complete_splits(p, c1), complete_splits(p, c0));
                if (n > 0 && f1 == f0) cand = -n;
            }
            s_shared[s] = cand;
        }
        __syncthreads();
        for (int s = warp; s < p.num_seqs; s += 32) {
            const int n = -s_shared[s];
            if (n <= 0) continue;
            const int32_t* t1 = p.block_tables + size_t(s) * p.table_stride + lane;
            const int32_t* t0 = t1 - p.table_stride;
            int shared = 0;
            for (int j0 = 0; j0 < n && shared == j0; j0 += kBatch) {
                int a[kBatch], b[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    a[u] = j0 + u < n ? t1[(j0 + u) * kPer] : 0;
                    b[u] = j0 + u < n ? t0[(j0 + u) * kPer] : 1;
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (shared == j0 + u && __all_sync(kFull, a[u] == b[u])) shared = j0 + u + 1;
            }
            __syncwarp();
            if (lane == 0) s_shared[s] = shared;
        }
    }
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += 1024) {
        const int s = base + tid;
        int nd = 0, np = 0, first_split = 0, ctx = 0, qlen = 0;
        if (s < p.num_seqs) {
            ctx = p.context_lens[s];
            qlen = 1;
            if (p.query_start_loc) qlen = p.query_start_loc[s + 1] - p.query_start_loc[s];
            if (qlen < 0 || qlen > p.num_query_tokens) {
                flag_error(p.err, PKV_DEV_BAD_QUERY_LAYOUT);
            } else if (qlen > 0) {
                if (ctx < 1 || ctx > p.max_context_len || ctx < qlen) {
                    flag_error(p.err, PKV_DEV_BAD_CONTEXT_LEN);
                } else if ((ctx + kBlockTokens - 1) / kBlockTokens > p.table_stride) {
                    flag_error(p.err, PKV_DEV_TABLE_TOO_NARROW);
                } else if (qlen == 1) {
                    // the splits from the one holding the window's first key
                    const int lo = window_first_key(ctx - 1, p.window);
                    first_split = lo / kSplitTokens;
                    nd = group ? grouped_items(p, s_shared, s, ctx, nullptr)
                               : (ctx - 1) / kSplitTokens - first_split + 1;
                    my_tok += (unsigned long long)(ctx - lo);
                } else {
                    np = (qlen + p.tokens_per_tile - 1) / p.tokens_per_tile;
                    // causal (query, key) pairs of the chunk; with a window W, row i
                    // sees min(ctx - qlen + 1 + i, W) keys
                    const unsigned long long q = qlen, c = ctx;
                    if (p.window > 0) {
                        const long long c0 = ctx - qlen + 1;
                        const long long n1 = max(0LL, min((long long)qlen, p.window - c0));
                        my_pairs += (unsigned long long)(n1 * c0 + n1 * (n1 - 1) / 2 +
                                                         (qlen - n1) * (long long)p.window);
                    } else {
                        my_pairs += q * (c - q) + q * (q + 1) / 2;
                    }
                }
            }
        }
        // block-wide exclusive scan of nd and np
        int xd = nd, xp = np;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int yd = __shfl_up_sync(kFull, xd, off);
            const int yp = __shfl_up_sync(kFull, xp, off);
            if (lane >= off) {
                xd += yd;
                xp += yp;
            }
        }
        if (lane == 31) {
            warp_d[warp] = xd;
            warp_p[warp] = xp;
        }
        __syncthreads();
        if (warp == 0) {
            int wd = warp_d[lane], wp = warp_p[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int yd = __shfl_up_sync(kFull, wd, off);
                const int yp = __shfl_up_sync(kFull, wp, off);
                if (lane >= off) {
                    wd += yd;
                    wp += yp;
                }
            }
            warp_d[lane] = wd;  // inclusive prefix over warps
            warp_p[lane] = wp;
        }
        __syncthreads();
        const int before_d = carry_d + (warp ? warp_d[warp - 1] : 0) + xd - nd;
        const int before_p = carry_p + (warp ? warp_p[warp - 1] : 0) + xp - np;
        if (group) {
            if (nd) grouped_items(p, s_shared, s, ctx, p.ws.items + before_d);
        } else {
            for (int k = 0; k < nd; ++k) p.ws.items[before_d + k] = make_int2(s, first_split + k);
        }
        // Prefill item k of sequence s: recorded for the longest-first reorder
        // (its bucket: the item's key tiles, from the tile of its first token's
        // first key to its last token's key) and written in batch order.
        auto prefill_item = [&](int idx, int s_, int k, int qlen_, int ctx_) {
            if (idx < p.ws.max_prefill_items) p.ws.prefill_items[idx] = make_int2(s_, k);
            if (idx < sortable) {
                const int t0 = k * p.tokens_per_tile;
                const int nt = min(p.tokens_per_tile, qlen_ - t0);
                const int n_keys = ctx_ - qlen_ + t0 + nt;
                const int key0 =
                    window_first_key(ctx_ - qlen_ + t0, p.window) / kPrefillKeys * kPrefillKeys;
                const int tiles = (n_keys - key0 + kPrefillKeys - 1) / kPrefillKeys;
                const int b = kSortBuckets - 1 - min(tiles, kSortBuckets - 1);   // descending
                s_item[idx] = make_int2(s_, k);
                s_bucket[idx] = b;
                atomicAdd(&hist[b], 1);
            }
        };
        if (one_pass) {
            // a batch of up to 1024 rows: the items are spread over all threads
            // (a chunk's items would otherwise be one thread's serial loop); the
            // owner of item idx is the last row whose first item is <= idx
            int* s_first = s_shared;                  // free: no grouping with prefill rows
            int* s_qlen = s_shared + 1024;
            int* s_ctx = s_shared + 2048;
            if (s < p.num_seqs) {
                s_first[s] = before_p;
                s_qlen[s] = qlen;
                s_ctx[s] = ctx;
            }
            __syncthreads();
            const int total_p = warp_p[31];
            for (int idx = tid; idx < total_p; idx += 1024) {
                int lo = 0, hi = p.num_seqs - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_first[mid] <= idx) lo = mid;
                    else hi = mid - 1;
                }
                prefill_item(idx, lo, idx - s_first[lo], s_qlen[lo], s_ctx[lo]);
            }
        } else {
            for (int k = 0; k < np; ++k) prefill_item(before_p + k, s, k, qlen, ctx);
        }
        __syncthreads();
        if (tid == 0) {
            carry_d += warp_d[31];
            carry_p += warp_p[31];
        }
        __syncthreads();
    }
    // block-wide sums of the work estimates
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        my_tok += __shfl_xor_sync(kFull, my_tok, off);
        my_pairs += __shfl_xor_sync(kFull, my_pairs, off);
    }
    if (lane == 0) {
        warp_tok[warp] = my_tok;
        warp_pairs[warp] = my_pairs;
    }
    __syncthreads();
    if (warp == 0) {
        unsigned long long dec_tokens = warp_tok[lane], pre_pairs = warp_pairs[lane];
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            dec_tokens += __shfl_xor_sync(kFull, dec_tokens, off);
            pre_pairs += __shfl_xor_sync(kFull, pre_pairs, off);
        }
        if (lane == 0) {
            if (p.query_start_loc && (q_first != 0 || q_last != p.num_query_tokens)) {
                flag_error(p.err, PKV_DEV_BAD_QUERY_LAYOUT);
                carry_d = 0;
                carry_p = 0;
            }
            p.ws.counters[0] = carry_d;
            p.ws.counters[1] = min(carry_p, p.ws.max_prefill_items);
            // SMs for the prefill chunks: their share of the estimated time, so
            // that tensor-bound chunks and HBM-bound decode rows finish together
            // (an estimate: single precision is plenty, and double precision
            // arithmetic is slow on this GPU)
            int sms_prefill = 0;
            if (pre_pairs && carry_p) {
                const float t_pre = float(pre_pairs) * p.ns_per_pair;
                const float t_dec = float(dec_tokens) * p.ns_per_token;
                sms_prefill = int(ceilf(float(p.num_sms) * (t_pre / (t_pre + t_dec))));
                sms_prefill = max(1, min(p.num_sms, sms_prefill));
            }
            p.ws.counters[2] = sms_prefill;
            p.ws.counters[3] = 0;  // decode unit ticket
            p.ws.counters[4] = 0;  // prefill unit ticket
        }
    }
    // Longest first: prefill units are taken from a ticket in item order, so the
    // items are reordered by descending key-tile count (a counting sort of the
    // items recorded in shared memory; items with equal counts in any order).
    // Lists longer than the recorded ones keep their order.
    __syncthreads();
    const int n_pre = min(carry_p, p.ws.max_prefill_items);
    if (n_pre < 2 || n_pre > sortable) return;
    if (warp == 0) {
        // exclusive scan of the histogram, kSortBuckets / 32 buckets per lane
        constexpr int kPer = kSortBuckets / 32;
        int run = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) run += hist[lane * kPer + i];
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += y;
        }
        int acc = incl - run;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int h = hist[lane * kPer + i];
            cursor[lane * kPer + i] = acc;
            acc += h;
        }
    }
    __syncthreads();
    for (int i = tid; i < n_pre; i += 1024)
        p.ws.prefill_items[atomicAdd(&cursor[s_bucket[i]], 1)] = s_item[i];
}

int launch_plan(const AttnArgs& a) {
    PlanParams p;
    p.context_lens = a.context_lens;
    p.query_start_loc = a.query_start_loc;
    p.num_seqs = a.num_seqs;
    p.num_query_tokens = a.num_query_tokens;
    p.max_context_len = a.max_context_len;
    p.table_stride = a.table_stride;
    p.tokens_per_tile = kPrefillRows / (a.desc->num_q_heads / a.desc->num_kv_heads);
    p.num_sms = num_sms();
    p.window = a.window;
    // grouped items are read only by the tensor-core kernel for groups of 8
    p.group = a.group_splits && a.window == 0 && !a.query_start_loc &&
              decode_mma_eligible(a.desc) && a.desc->num_q_heads == 8 * a.desc->num_kv_heads;
    p.block_tables = a.block_tables;
    p.ns_per_token = float(2.0 * a.desc->num_kv_heads * a.desc->head_dim *
                           double(elem_bytes(a.desc->dtype)) / kDecodeBytesPerNs);
    p.ns_per_pair = float(4.0 * a.desc->head_dim * a.desc->num_q_heads / kPrefillFlopsPerNs);
    p.ws = a.ws;
    p.err = a.err;
    return cuda_status(launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, a.stream, p));
}

// ---------------------------------------------------------------------------
// Split kernel
// ---------------------------------------------------------------------------
struct SplitParams {
    const void* q;
    void* out;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start_loc;
    const int2* items;
    const int32_t* n_items;
    int32_t* ticket;
    float2* part_ml;
    float* part_o;
    int32_t table_stride;
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t max_splits;
    int32_t wait_plan;   // launched right behind the planner: wait for its work list
    int32_t window;      // sliding window in keys (0: none)
    float scale_log2;
    int* err;
};

constexpr size_t align_up_c(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <typename T, int D, int G>
struct SplitCfg {
    static constexpr int kWarps = 4;                        // consumer warps
    static constexpr int kThreads = (kWarps + 1) * 32;      // + one producer warp
    static constexpr int kDPL = D / 32;                     // head dims per lane
    static constexpr int kTileBytes = kBlockTokens * D * int(sizeof(T));
    static constexpr int kStageBytes = 2 * kTileBytes;      // K tile + V tile
    static constexpr int kStages = kStageBytes <= 8192 ? 8 : 4;
    static constexpr int kTC = G == 1 ? 16 : 32 / G;        // tokens per reduction chunk
    static constexpr int kNV = kTC * G;                     // values per reduction (16 or 32)
    static constexpr int kNC = kBlockTokens / kTC;          // chunks per block
    static constexpr int kPBuf = G * kBlockTokens + G;      // p values + alphas per warp
    static constexpr int kComb = G * (D + 2);               // per-warp combine record
    static constexpr size_t kRingOff = 0;
    static constexpr size_t kPBufOff = size_t(kStages) * kStageBytes;
    static constexpr size_t kCombOff = kPBufOff + size_t(kWarps) * kPBuf * 4;
    static constexpr size_t kBarOff = align_up_c(kCombOff + size_t(kWarps) * kComb * 4, 16);
    static constexpr size_t kQueueOff = kBarOff + 2 * kStages * 8;
    static constexpr size_t kSmem = kQueueOff + sizeof(UnitQueue);
    static_assert(kDPL == 2 || kDPL == 4, "head_dim 64 or 128");
    // a consumer warp waits on a stage by parity: its previous use must be the
    // same warp's own tile (tiles of a unit go to warps round-robin)
    static_assert(kStages % kWarps == 0, "stage ring must be a multiple of the consumer warps");
    static_assert(kNV == 16 || kNV == 32, "group size 1, 2, 4 or 8");
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(SplitCfg<T, D, G>::kThreads)
    decode_split_kernel(SplitParams p) {
    using C = SplitCfg<T, D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem + C::kRingOff;
    float* pbuf_all = reinterpret_cast<float*>(smem + C::kPBufOff);
    float* comb = reinterpret_cast<float*>(smem + C::kCombOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* empty = full + C::kStages;
    UnitQueue* uq = reinterpret_cast<UnitQueue*>(smem + C::kQueueOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        uq_init(uq);
        fence_mbar_init();
    }
    __syncthreads();
    // behind the planner (programmatic launch): its work list must be complete
    // before anything below reads it; the merge kernel may launch now
    if (p.wait_plan) pdl_wait_prerequisites();
    pdl_launch_dependents();

    const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
    const int n_units = p.n_items[0] * Hkv;

    if (warp == C::kWarps) {
        // ---------------- producer warp: keeps the ring full ----------------
        uint32_t it = 0;
        bool ok = true;
        const unsigned char* kb = static_cast<const unsigned char*>(p.k_cache);
        const unsigned char* vb = static_cast<const unsigned char*>(p.v_cache);
        int next = uq_first_ticket(p.ticket, lane);
        for (uint32_t k = 0;; ++k) {
            const int u = uq_produce(uq, k, next, p.ticket, n_units, lane, p.err, ok);
            if (u < 0) break;
            const int2 item = p.items[u / Hkv];
            const int kvh = u % Hkv;
            const SplitSpan sp = split_span(p.context_lens[item.x], item.y, p.window);
            const int b0 = sp.begin;
            const int nb = max(0, sp.end - b0);
            int my_blk = 0;
            if (lane < nb) my_blk = p.block_tables[size_t(item.x) * p.table_stride + b0 + lane];
            for (int j = 0; j < nb; ++j, ++it) {
                const int blk = __shfl_sync(kFull, my_blk, j);
                const int st = it % C::kStages;
                const uint32_t par = (it / C::kStages) & 1;
                ok = __all_sync(kFull, mbar_wait(&empty[st], par ^ 1, p.err));
                if (!ok) break;
#ifdef PKV_TEST_SKIP_TILE
                // wait-timeout test build only: this tile is never copied and its
                // stage never marked full, so the consumer's bounded wait on it
                // runs out (no copy is in flight for it at any time)
                if (it == uint32_t(PKV_TEST_SKIP_TILE)) continue;
#endif
                if (lane == 0) {
                    if (blk < 0 || blk >= p.num_blocks) {
                        flag_error(p.err, PKV_DEV_BAD_BLOCK_ID);
                        mbar_arrive(&full[st]);  // no data: consumers read a stale tile
                    } else {
                        mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                        const size_t off = (size_t(blk) * Hkv + kvh) * C::kTileBytes;
                        unsigned char* dst = ring + size_t(st) * C::kStageBytes;
                        bulk_g2s(dst, kb + off, C::kTileBytes, &full[st]);
                        bulk_g2s(dst + C::kTileBytes, vb + off, C::kTileBytes, &full[st]);
                    }
                }
                __syncwarp();
            }
        }
        // never leave with bulk copies in flight: wait for the last fill of each stage
        if (lane == 0) {
            for (int k = 0; k < C::kStages && uint32_t(k) < it; ++k) {
                const uint32_t last = it - 1 - k;
                mbar_wait(&full[last % C::kStages], (last / C::kStages) & 1, p.err);
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------
    constexpr int DPL = C::kDPL, TC = C::kTC, NV = C::kNV, NC = C::kNC;
    const int my_head = G == 1 ? 0 : lane / TC;          // query head (within group) this lane scores
    const int my_tok = G == 1 ? (lane >> 1) : lane % TC; // token (within chunk) this lane scores
    float* pbuf = pbuf_all + warp * C::kPBuf;
    const T* qbase = static_cast<const T*>(p.q);
    uint32_t it_base = 0;
    bool ok = true;

    for (uint32_t k = 0;; ++k) {
        const int u = uq_consume(uq, k, C::kWarps * 32, p.err, ok);
        if (u < 0) break;
        const int2 item = p.items[u / Hkv];
        const int seq = item.x, split = item.y;
        const int kvh = u % Hkv;
        const int ctx = p.context_lens[seq];
        const SplitSpan sp = split_span(ctx, split, p.window);
        const int b0 = sp.begin;
        const int nb = max(0, sp.end - b0);
        const int qrow = p.query_start_loc ? p.query_start_loc[seq] : seq;

        float qr[G][DPL];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float t[DPL];
            Elem<T>::template load<DPL>(qbase + (size_t(qrow) * Hq + kvh * G + j) * D + lane * DPL, t);
#pragma unroll
            for (int d = 0; d < DPL; ++d) qr[j][d] = t[d] * p.scale_log2;
        }
        float m = -INFINITY, l = 0.f;
        float o[G][DPL];
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[j][d] = 0.f;

        for (int jb = warp; jb < nb; jb += C::kWarps) {
            const uint32_t it = it_base + jb;
            const int st = it % C::kStages;
            if (ok) ok = __all_sync(kFull, mbar_wait(&full[st], (it / C::kStages) & 1, p.err));
            if (!ok) continue;
            const T* kt = reinterpret_cast<const T*>(ring + size_t(st) * C::kStageBytes);
            const T* vt = kt + kBlockTokens * D;
            const int nvalid = min(kBlockTokens, ctx - (b0 + jb) * kBlockTokens);
            // keys below the window's first key (its block only) are masked
            const int fvalid = b0 + jb == sp.lo / kBlockTokens ? sp.lo % kBlockTokens : 0;

            // scores s = q . k for this lane's (head, token) in each chunk
            float s[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float part[NV];
#pragma unroll
                for (int tt = 0; tt < TC; ++tt) {
                    float kf[DPL];
                    Elem<T>::template load<DPL>(kt + (c * TC + tt) * D + lane * DPL, kf);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        float acc = qr[j][0] * kf[0];
#pragma unroll
                        for (int d = 1; d < DPL; ++d) acc = fmaf(qr[j][d], kf[d], acc);
                        part[j * TC + tt] = acc;
                    }
                }
                s[c] = reduce_scatter<NV>(part, lane);
                if (c * TC + my_tok >= nvalid || c * TC + my_tok < fvalid) s[c] = -INFINITY;
            }
            // online softmax update over this block (column block of 16 keys)
            float mx = s[0];
#pragma unroll
            for (int c = 1; c < NC; ++c) mx = fmaxf(mx, s[c]);
            mx = group_max<G, TC>(mx);
            const float m_new = fmaxf(m, mx);
            const float alpha = exp2f(m - m_new);
            float psum = 0.f;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const float pc = exp2f(s[c] - m_new);
                psum += pc;
                pbuf[my_head * kBlockTokens + c * TC + my_tok] = pc;
            }
            psum = group_sum<G, TC>(psum);
            l = l * alpha + psum;
            m = m_new;
            if (my_tok == 0) pbuf[G * kBlockTokens + my_head] = alpha;
            __syncwarp();
            // O = diag(alpha) O + P V
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float a = pbuf[G * kBlockTokens + j];
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[j][d] *= a;
            }
            for (int t = fvalid; t < nvalid; ++t) {
                float vf[DPL];
                Elem<T>::template load<DPL>(vt + t * D + lane * DPL, vf);
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float pj = pbuf[j * kBlockTokens + t];
#pragma unroll
                    for (int d = 0; d < DPL; ++d) o[j][d] = fmaf(pj, vf[d], o[j][d]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        it_base += nb;

        // ---- combine the consumer warps' states ----
        float* rec = comb + warp * C::kComb;
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int d = 0; d < DPL; ++d) rec[j * D + lane * DPL + d] = o[j][d];
        if (my_tok == 0) {
            rec[G * D + my_head] = m;
            rec[G * D + G + my_head] = l;
        }
        consumer_sync(C::kWarps * 32);
        const int nsplit = sp.nsplit;
        for (int idx = threadIdx.x; idx < G * D; idx += C::kWarps * 32) {
            const int j = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, comb[w * C::kComb + G * D + j]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) {
                const float* r = comb + w * C::kComb;
                const float sc = exp2f(r[G * D + j] - M);
                L = fmaf(r[G * D + G + j], sc, L);
                O = fmaf(r[j * D + d], sc, O);
            }
            const int h = kvh * G + j;
            if (nsplit == 1) {
                static_cast<T*>(p.out)[(size_t(qrow) * Hq + h) * D + d] = Elem<T>::store_val(O / L);
            } else {
                const size_t slot = (size_t(seq) * Hq + h) * p.max_splits + split;
                const uint64_t keep = l2_evict_last_policy();
                st_keep(p.part_o + slot * D + d, O, keep);
                if (d == 0) st_keep(p.part_ml + slot, make_float2(M, L), keep);
            }
        }
        consumer_sync(C::kWarps * 32);
    }
    // a preceding prefill kernel overlapped this grid: finish only after it has
    if (threadIdx.x == 0) pdl_wait_prerequisites();
}

// ---------------------------------------------------------------------------
// Merge kernel: one warp per (sequence, query head) whose row has more than
// one split:
//   M = max_k m_k,  L = sum_k l_k 2^(m_k - M),  out = sum_k O_k 2^(m_k - M) / L
// It is launched behind the split kernel with programmatic dependent launch,
// so it is resident when the split kernel ends and only waits for it.  Lane k
// holds the (m, l) of split k (32 splits per pass); the O rows of eight splits
// are requested before any is used, so their latencies overlap, and they are
// summed in split index order.  (One warp per KV-head group, with one split's
// G rows in flight at a time, took 49 us on 64-split rows at G = 8: the
// longest row's serial latency chain.)
// ---------------------------------------------------------------------------
struct MergeParams {
    void* out;
    const int32_t* context_lens;
    const int32_t* query_start_loc;
    const float2* part_ml;
    const float* part_o;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t max_splits;
    int32_t max_context_len;
    int32_t window;
};

template <typename T, int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(MergeParams p) {
    pdl_wait_prerequisites();   // the split kernel's partials
    pdl_launch_dependents();    // the next call's first kernel may become resident
    constexpr int DPL = D / 32;
    // splits whose O rows are requested together (16 and 32 measured no faster
    // overall: the registers they take cost the short rows' occupancy)
    constexpr int kBatch = 8;
    const int lane = threadIdx.x & 31;
    const int wid = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int Hq = p.num_q_heads;
    if (wid >= p.num_seqs * Hq) return;
    const int seq = wid / Hq, h = wid % Hq;
    int qrow = seq;
    if (p.query_start_loc) {
        qrow = p.query_start_loc[seq];
        if (p.query_start_loc[seq + 1] - qrow != 1) return;  // not a decode row
    }
    const int ctx = p.context_lens[seq];
    if (ctx < 1 || ctx > p.max_context_len) return;          // flagged by the planner
    // splits first .. first + n - 1 (first > 0 when a window starts past split 0)
    const int first = window_first_key(ctx - 1, p.window) / kSplitTokens;
    const int n = (ctx - 1) / kSplitTokens - first + 1;
    if (n <= 1) return;                                     // written by the split kernel
    // slot of split first + k: base + k
    const size_t base = (size_t(seq) * Hq + h) * p.max_splits + first;
    // (m, l) of splits lane and lane + 32 stay in registers for the second pass
    const float2 none = make_float2(-INFINITY, 0.f);
    const float2 ml_a = lane < n ? p.part_ml[base + lane] : none;
    const float2 ml_b = lane + 32 < n ? p.part_ml[base + lane + 32] : none;
    float M = fmaxf(ml_a.x, ml_b.x);
    for (int k = lane + 64; k < n; k += 32) M = fmaxf(M, p.part_ml[base + k].x);
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float L = 0.f, acc[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
    for (int k0 = 0; k0 < n; k0 += 32) {
        float w = 0.f;
        if (k0 + lane < n) {
            const float2 ml = k0 == 0 ? ml_a : k0 == 32 ? ml_b : __ldcs(p.part_ml + base + k0 + lane);
            w = exp2f(ml.x - M);
            L = fmaf(ml.y, w, L);
        }
        const int cnt = min(32, n - k0);                    // the same in every lane
        const float* src = p.part_o + (base + k0) * D + lane * DPL;
        // the rows of a batch of splits are requested together; the next
        // batch's requests go out before this one is summed (in split order)
        float ov[2][kBatch][DPL];
        auto fetch = [&](float(&dst)[kBatch][DPL], int i) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (i + u < cnt) {
                    // read once: let the kept lines go
                    const float* r = src + size_t(i + u) * D;
                    if constexpr (DPL == 4) {
                        const float4 v = __ldcs(reinterpret_cast<const float4*>(r));
                        dst[u][0] = v.x; dst[u][1] = v.y; dst[u][2] = v.z; dst[u][3] = v.w;
                    } else {
                        const float2 v = __ldcs(reinterpret_cast<const float2*>(r));
                        dst[u][0] = v.x; dst[u][1] = v.y;
                    }
                }
            }
        };
        auto sum = [&](const float(&rows)[kBatch][DPL], int i) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (i + u < cnt) {
                    const float wi = __shfl_sync(kFull, w, i + u);
#pragma unroll
                    for (int d = 0; d < DPL; ++d) acc[d] = fmaf(wi, rows[u][d], acc[d]);
                }
            }
        };
        fetch(ov[0], 0);
        for (int i = 0; i < cnt; i += 2 * kBatch) {
            if (i + kBatch < cnt) fetch(ov[1], i + kBatch);
            sum(ov[0], i);
            if (i + kBatch < cnt) {
                if (i + 2 * kBatch < cnt) fetch(ov[0], i + 2 * kBatch);
                sum(ov[1], i + kBatch);
            }
        }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
    const float inv = 1.f / L;
    T* o = static_cast<T*>(p.out) + (size_t(qrow) * Hq + h) * D + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] = Elem<T>::store_val(acc[d] * inv);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
int num_sms() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

template <typename T, int D, int G>
int launch_split_t(const AttnArgs& a) {
    using C = SplitCfg<T, D, G>;
    auto kern = decode_split_kernel<T, D, G>;
    const int per_sm = kernel_occupancy<decode_split_kernel<T, D, G>>(C::kThreads, int(C::kSmem));
    if (per_sm < 1) return PKV_ERR_CUDA;
    const int64_t bound_units =
        int64_t(a.num_seqs) * a.ws.max_splits * a.desc->num_kv_heads;  // upper bound
    const int64_t grid = std::min<int64_t>(int64_t(num_sms()) * per_sm, bound_units);
    if (grid < 1) return PKV_OK;
    SplitParams p;
    p.q = a.q;
    p.out = a.out;
    p.k_cache = a.k_cache;
    p.v_cache = a.v_cache;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.query_start_loc = a.query_start_loc;
    p.items = a.ws.items;
    p.n_items = a.ws.counters;
    p.ticket = a.ws.counters + 3;
    p.part_ml = a.ws.part_ml;
    p.part_o = a.ws.part_o;
    p.table_stride = a.table_stride;
    p.num_blocks = a.desc->num_blocks;
    p.num_kv_heads = a.desc->num_kv_heads;
    p.num_q_heads = a.desc->num_q_heads;
    p.max_splits = a.ws.max_splits;
    p.wait_plan = a.pdl ? 0 : 1;   // behind a prefill kernel, the plan is complete
    p.window = a.window;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, p));
}

template <typename T, int D>
int launch_split_d(const AttnArgs& a, int g) {
    switch (g) {
        case 1: return launch_split_t<T, D, 1>(a);
        case 2: return launch_split_t<T, D, 2>(a);
        case 4: return launch_split_t<T, D, 4>(a);
        case 8: return launch_split_t<T, D, 8>(a);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

template <typename T, int D>
int launch_merge_d(const AttnArgs& a) {
    MergeParams p;
    p.out = a.out;
    p.context_lens = a.context_lens;
    p.query_start_loc = a.query_start_loc;
    p.part_ml = a.ws.part_ml;
    p.part_o = a.ws.part_o;
    p.num_seqs = a.num_seqs;
    p.num_q_heads = a.desc->num_q_heads;
    p.max_splits = a.ws.max_splits;
    p.max_context_len = a.max_context_len;
    p.window = a.window;
    const int64_t warps = int64_t(a.num_seqs) * a.desc->num_q_heads;   // one per (seq, head)
    const int64_t blocks = (warps + 3) / 4;
    if (blocks < 1) return PKV_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(128);
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, D>, p));
}

}  // namespace

int launch_decode_split(const AttnArgs& a) {
    if (decode_mma_eligible(a.desc)) return launch_decode_split_mma(a);
    const int g = a.desc->num_q_heads / a.desc->num_kv_heads;
    const bool bf = a.desc->dtype == PKV_BF16;
    if (a.desc->head_dim == 128)
        return bf ? launch_split_d<__nv_bfloat16, 128>(a, g) : launch_split_d<float, 128>(a, g);
    if (a.desc->head_dim == 64)
        return bf ? launch_split_d<__nv_bfloat16, 64>(a, g) : launch_split_d<float, 64>(a, g);
    return PKV_ERR_UNSUPPORTED;
}

int launch_decode_merge(const AttnArgs& a) {
    // a single split is finished by the split kernel itself
    if (a.ws.max_splits <= 1) return PKV_OK;
    const bool bf = a.desc->dtype == PKV_BF16;
    if (a.desc->head_dim == 128)
        return bf ? launch_merge_d<__nv_bfloat16, 128>(a) : launch_merge_d<float, 128>(a);
    if (a.desc->head_dim == 64)
        return bf ? launch_merge_d<__nv_bfloat16, 64>(a) : launch_merge_d<float, 64>(a);
    return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
