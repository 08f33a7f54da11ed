// C ABI entry points for attention, argument validation, workspace layout and
// the device error word.
#include <cmath>
#include <cuda_runtime.h>
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"

// One error word per device that loads the library (first fault wins).
__device__ int g_pkv_error_word;

namespace pkv {

int check_desc(const pkv_cache_desc* d, bool attention) {
    if (!d) return PKV_ERR_INVALID;
    if (d->dtype != PKV_F32 && d->dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
    if (d->num_blocks < 1 || d->block_size < 1 || d->num_kv_heads < 1 || d->num_q_heads < 1 ||
        d->head_dim < 1)
        return PKV_ERR_INVALID;
    if (d->num_q_heads % d->num_kv_heads) return PKV_ERR_INVALID;
    if (attention) {
        const int g = d->num_q_heads / d->num_kv_heads;
        if (d->block_size != kBlockTokens) return PKV_ERR_UNSUPPORTED;
        if (d->head_dim != 64 && d->head_dim != 128) return PKV_ERR_UNSUPPORTED;
        if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_UNSUPPORTED;
    }
    return PKV_OK;
}

int* device_error_ptr(int* status) {
    static std::mutex mu;
    static int* addr[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
        *status = PKV_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pkv_error_word) != cudaSuccess) {
            *status = PKV_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = static_cast<int*>(p);
    }
    *status = PKV_OK;
    return addr[dev];
}

size_t workspace_layout(const pkv_cache_desc* d, int32_t num_seqs, int32_t max_context_len,
                        int32_t num_prefill_items, void* base, Workspace* ws) {
    const int32_t max_splits = ceil_div(max_context_len, kSplitTokens);
    const size_t n_part = max_splits > 1 ? size_t(num_seqs) * d->num_q_heads * max_splits : 0;
    size_t off = 0;
    const size_t o_counters = off;
    off += 256;
    const size_t o_items = off;
    off = align_up(off + size_t(num_seqs) * max_splits * sizeof(int2), 256);
    const size_t o_pitems = off;
    off = align_up(off + size_t(num_prefill_items) * sizeof(int2), 256);
    const size_t o_ml = off;
    off = align_up(off + n_part * sizeof(float2), 256);
    const size_t o_o = off;
    off = align_up(off + n_part * d->head_dim * sizeof(float), 256);
    if (ws) {
        char* b = static_cast<char*>(base);
        ws->counters = reinterpret_cast<int32_t*>(b + o_counters);
        ws->items = reinterpret_cast<int2*>(b + o_items);
        ws->prefill_items = reinterpret_cast<int2*>(b + o_pitems);
        ws->part_ml = reinterpret_cast<float2*>(b + o_ml);
        ws->part_o = reinterpret_cast<float*>(b + o_o);
        ws->max_splits = max_splits;
        ws->max_prefill_items = num_prefill_items;
    }
    return off;
}

}  // namespace pkv

using namespace pkv;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Checks that do not look at the pointers (run first: an empty batch is a
// no-op whatever its pointers hold, as zero-sized tensors often give null).
int check_attention_scalars(const pkv_cache_desc* desc, int32_t max_blocks_per_seq,
                            int32_t max_context_len, float scale) {
    int st = check_desc(desc, true);
    if (st != PKV_OK) return st;
    if (max_blocks_per_seq < 1 || max_context_len < 1) return PKV_ERR_INVALID;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID;
    return PKV_OK;
}

int check_attention_pointers(void* out, const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens) {
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKV_ERR_INVALID;
    return PKV_OK;
}

}  // namespace

extern "C" size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs,
                                             int32_t max_context_len) {
    if (!desc) return 0;
    pkv_cache_desc d = *desc;
    if (d.dtype == PKV_INT8) d.dtype = PKV_BF16;  // the partials do not depend on the cache type
    if (check_desc(&d, false) != PKV_OK || num_seqs < 0 || max_context_len < 1) return 0;
    return workspace_layout(&d, num_seqs, max_context_len, 0, nullptr, nullptr);
}

extern "C" size_t pkv_varlen_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs,
                                             int32_t num_query_tokens, int32_t max_query_len,
                                             int32_t max_context_len) {
    if (check_desc(desc, false) != PKV_OK || num_seqs < 0 || num_query_tokens < 0 ||
        max_query_len < 0 || max_context_len < 1)
        return 0;
    const int g = desc->num_q_heads / desc->num_kv_heads;
    const int32_t np = max_query_len > 1 ? prefill_item_bound(num_seqs, num_query_tokens, g) : 0;
    return workspace_layout(desc, num_seqs, max_context_len, np, nullptr, nullptr);
}

extern "C" int paged_attention_decode(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const pkv_cache_desc* desc,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t max_context_len, float scale, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    if (num_seqs < 0) return PKV_ERR_INVALID;
    int st = check_attention_scalars(desc, max_blocks_per_seq, max_context_len, scale);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    st = check_attention_pointers(out, q, k_cache, v_cache, block_tables, context_lens);
    if (st != PKV_OK) return st;
    const size_t need = pkv_decode_workspace_bytes(desc, num_seqs, max_context_len);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    AttnArgs a{};
    workspace_layout(desc, num_seqs, max_context_len, 0, workspace, &a.ws);
    a.err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.desc = desc;
    a.block_tables = block_tables;
    a.table_stride = max_blocks_per_seq;
    a.query_start_loc = nullptr;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_query_tokens = num_seqs;
    a.max_query_len = 1;
    a.max_context_len = max_context_len;
    a.scale = scale;
    a.stream = static_cast<cudaStream_t>(stream);
    a.group_splits = true;
    if ((st = launch_plan(a)) != PKV_OK) return st;
    if ((st = launch_decode_split(a)) != PKV_OK) return st;
    return launch_decode_merge(a);
}

static int varlen_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const pkv_cache_desc* desc, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* query_start_loc,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_query_tokens,
                       int32_t max_query_len, int32_t max_context_len, int32_t window,
                       float scale, void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs < 0 || num_query_tokens < 0 || max_query_len < 0 || window < 0)
        return PKV_ERR_INVALID;
    int st = check_attention_scalars(desc, max_blocks_per_seq, max_context_len, scale);
    if (st != PKV_OK) return st;
    if (num_seqs == 0 || num_query_tokens == 0) return PKV_OK;
    st = check_attention_pointers(out, q, k_cache, v_cache, block_tables, context_lens);
    if (st != PKV_OK) return st;
    if (!query_start_loc || !aligned(query_start_loc, 4)) return PKV_ERR_INVALID;
    if (max_query_len > max_context_len) return PKV_ERR_INVALID;
    if (max_query_len > 1 && !prefill_supported(desc)) return PKV_ERR_UNSUPPORTED;
    const size_t need = pkv_varlen_workspace_bytes(desc, num_seqs, num_query_tokens,
                                                   max_query_len, max_context_len);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    const int g = desc->num_q_heads / desc->num_kv_heads;
    const int32_t np = max_query_len > 1 ? prefill_item_bound(num_seqs, num_query_tokens, g) : 0;
    AttnArgs a{};
    workspace_layout(desc, num_seqs, max_context_len, np, workspace, &a.ws);
    a.err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.desc = desc;
    a.block_tables = block_tables;
    a.table_stride = max_blocks_per_seq;
    a.query_start_loc = query_start_loc;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_query_tokens = num_query_tokens;
    a.max_query_len = max_query_len;
    a.max_context_len = max_context_len;
    a.window = window;
    a.scale = scale;
    a.stream = static_cast<cudaStream_t>(stream);
    if ((st = launch_plan(a)) != PKV_OK) return st;
    if (max_query_len > 1) {
        // prefill chunks first, on the SMs the planner gives them; the decode
        // kernel may start beside it on the rest (programmatic dependent launch)
        if ((st = launch_prefill(a)) != PKV_OK) return st;
        a.pdl = true;
    }
    if ((st = launch_decode_split(a)) != PKV_OK) return st;
    return launch_decode_merge(a);
}

extern "C" int paged_attention_varlen(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const pkv_cache_desc* desc,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* query_start_loc, const int32_t* context_lens,
                                      int32_t num_seqs, int32_t num_query_tokens,
                                      int32_t max_query_len, int32_t max_context_len, float scale,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    return varlen_impl(out, q, k_cache, v_cache, desc, block_tables, max_blocks_per_seq,
                       query_start_loc, context_lens, num_seqs, num_query_tokens, max_query_len,
                       max_context_len, 0, scale, workspace, workspace_bytes, stream);
}

extern "C" int paged_attention_varlen_window(void* out, const void* q, const void* k_cache,
                                             const void* v_cache, const pkv_cache_desc* desc,
                                             const int32_t* block_tables,
                                             int32_t max_blocks_per_seq,
                                             const int32_t* query_start_loc,
                                             const int32_t* context_lens, int32_t num_seqs,
                                             int32_t num_query_tokens, int32_t max_query_len,
                                             int32_t max_context_len, int32_t window, float scale,
                                             void* workspace, size_t workspace_bytes,
                                             void* stream) {
    return varlen_impl(out, q, k_cache, v_cache, desc, block_tables, max_blocks_per_seq,
                       query_start_loc, context_lens, num_seqs, num_query_tokens, max_query_len,
                       max_context_len, window, scale, workspace, workspace_bytes, stream);
}

extern "C" int pkv_device_error(int32_t* code_out, int32_t clear) {
    if (!code_out) return PKV_ERR_INVALID;
    int st = PKV_OK;
    int* p = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    (void)p;
    if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pkv_error_word, sizeof(int)) != cudaSuccess) return PKV_ERR_CUDA;
    *code_out = v;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_pkv_error_word, &zero, sizeof(int)) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID: return "invalid argument";
        case PKV_ERR_NO_BLOCKS: return "no free block now (LATER)";
        case PKV_ERR_NEVER: return "request can never be served by this pool (NEVER)";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_WORKSPACE: return "workspace null, misaligned or too small";
        case PKV_ERR_HOST: return "host allocation failed";
        default: return "unknown status";
    }
}
