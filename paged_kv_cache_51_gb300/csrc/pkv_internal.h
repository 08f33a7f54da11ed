// Host-side internals shared by the translation units of libpagedkv.so.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "pagedkv.h"

namespace pkv {

constexpr int kSplitTokens = 512;       // context span of one decode split
constexpr int kPrefillRows = 128;       // query rows (tokens x group heads) per prefill tile
constexpr int kPrefillKeys = 128;       // keys per prefill key tile

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int ceil_div(int64_t a, int64_t b) { return int((a + b - 1) / b); }

inline size_t elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }

// Validates a cache descriptor; `attention` additionally checks the head
// grouping and head_dim the attention kernels implement.
int check_desc(const pkv_cache_desc* d, bool attention);

// Address of this device's error word (looked up once per device).
int* device_error_ptr(int* status);

// Status for a CUDA error (clears sticky-free errors from the runtime's slot).
inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// Workspace carve-up shared by decode and varlen.
struct Workspace {
    int32_t* counters;   // [0] decode items, [1] prefill items, [2] SMs for prefill,
                         // [3] decode unit ticket, [4] prefill unit ticket
    int2* items;         // decode items (seq, split)
    int2* prefill_items; // prefill items (seq, row tile)
    float2* part_ml;     // [num_seqs][num_q_heads][max_splits] (max, sum), log2 domain
    float* part_o;       // [num_seqs][num_q_heads][max_splits][head_dim]
    int32_t max_splits;
    int32_t max_prefill_items;
};

size_t workspace_layout(const pkv_cache_desc* d, int32_t num_seqs, int32_t max_context_len,
                        int32_t num_prefill_items, void* base, Workspace* ws);

struct AttnArgs {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const pkv_cache_desc* desc;
    const int32_t* block_tables;
    int32_t table_stride;
    const int32_t* query_start_loc;  // nullptr: one query per sequence
    const int32_t* context_lens;
    int32_t num_seqs;
    int32_t num_query_tokens;
    int32_t max_query_len;
    int32_t max_context_len;
    float scale;
    Workspace ws;
    cudaStream_t stream;
    int* err;
    bool pdl;            // decode kernels may start while the preceding prefill kernel runs
    int32_t window;      // sliding window in keys (0: none); tables in logical order
    bool group_splits;   // decode call: group sequences that share a complete split
};

// Decode work items are int2 (seq, split word).  The split word holds the split
// index in its low kItemSplitBits bits and, for a grouped item, the number of
// consecutive sequences from `seq` (2 .. kMaxGroup) that read the split's 32
// blocks block for block, above them (0: the item is one sequence's split).
constexpr int kItemSplitBits = 26;
constexpr int kItemSplitMask = (1 << kItemSplitBits) - 1;
constexpr int kMaxGroup = 8;

// Planning rates for the split of SMs between prefill chunks and decode rows
// of one mixed batch (what this library's kernels sustain on GB300).
constexpr double kDecodeBytesPerNs = 6400.0;     // decode streams KV at ~6.4 TB/s
constexpr double kPrefillFlopsPerNs = 450000.0;  // prefill kernel ~450 TFLOP/s over causal pairs

int num_sms();

// tmap.cpp: tensor map of a bf16 cache viewed as 2-D [num_blocks * Hkv * bs rows][head_dim],
// box = one block of one head (bs rows) x 64 dims, 128-byte swizzled in shared memory.
bool make_cache_tensor_map(struct CUtensorMap_st* map, const void* cache, const pkv_cache_desc* d);
// tmap.cpp: queries [tokens][Hq][128] bf16; box = one 64-dim half of a 128-row prefill Q tile
bool make_query_tensor_map(struct CUtensorMap_st* map, const void* q, int32_t num_tokens,
                           int32_t num_q_heads, int32_t group);

// decode_mma.cu: tensor-core split kernel for bf16 GQA groups of 2, 4 or 8
bool decode_mma_eligible(const pkv_cache_desc* d);
int launch_decode_split_mma(const AttnArgs& a);
// decode.cu
int launch_plan(const AttnArgs& a);
int launch_decode_split(const AttnArgs& a);
int launch_decode_merge(const AttnArgs& a);
// prefill_tc.cu
int prefill_supported(const pkv_cache_desc* d);
int launch_prefill(const AttnArgs& a);
int prefill_item_bound(int32_t num_seqs, int32_t num_query_tokens, int32_t group);

}  // namespace pkv
