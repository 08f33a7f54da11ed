// Slot-mapped KV append and copy-on-write block copies.
//
// Append ("【自用】AI infra相关" 一、推理两阶段 2、解码: each step's K_t, V_t are
// written into the cache; "大模型部署.md" §2.1: the block manager plans the
// physical slot, the cache engine writes it):
//     cache[slot / bs][h][slot % bs][:] = x[t][h][:]      for K and V.
// Copy-on-write ("大模型部署.md" §2.1 append_slots, "Allocate a new block and
// copy the tokens"): a whole block (all heads, all rows) of K and V.
//
// Both are pure byte movement, bound by HBM bandwidth: every thread moves one
// 16-byte vector with a coalesced load and store; source rows are read once,
// with the non-coherent (read-only) path, and nothing is converted, so the
// cache bytes equal the input bytes exactly.
#include <cuda_runtime.h>

#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

struct AppendParams {
    const uint4* k;
    const uint4* v;
    const int64_t* slots;
    uint4* k_cache;
    uint4* v_cache;
    int64_t num_tokens;
    int32_t vec_per_row;      // 16-byte vectors per head row (head_dim * elem / 16)
    int32_t num_kv_heads;
    int32_t block_size;
    int64_t num_slots;        // num_blocks * block_size
    int* err;
};

// grid-stride over (token, kv head, vector); K and V handled by the same thread
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
    const int64_t per_tok = int64_t(p.num_kv_heads) * p.vec_per_row;
    const int64_t total = p.num_tokens * per_tok;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = i / per_tok;
        const int64_t r = i - t * per_tok;            // (head, vector) within the token
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;                       // padding token
        if (slot >= p.num_slots) {
            flag_error(p.err, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const int64_t row = slot - blk * p.block_size;
        const int64_t h = r / p.vec_per_row;
        const int64_t c = r - h * p.vec_per_row;
        const int64_t dst = ((blk * p.num_kv_heads + h) * p.block_size + row) * p.vec_per_row + c;
        const uint4 kv = __ldg(p.k + i);
        const uint4 vv = __ldg(p.v + i);
        p.k_cache[dst] = kv;
        p.v_cache[dst] = vv;
    }
}

struct CopyParams {
    const int32_t* pairs;
    uint4* k_cache;
    uint4* v_cache;
    int64_t vec_per_block;    // 16-byte vectors per physical block (all heads)
    int32_t num_blocks;
    int* err;
};

// blockIdx.y = pair; blockIdx.x strides over the block's vectors
__global__ void __launch_bounds__(256) copy_blocks_kernel(CopyParams p) {
    const int pair = blockIdx.y;
    const int src = __ldg(p.pairs + 2 * pair), dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(p.err, PKV_DEV_BAD_COPY_PAIR);
        return;
    }
    const uint4* ks = p.k_cache + int64_t(src) * p.vec_per_block;
    const uint4* vs = p.v_cache + int64_t(src) * p.vec_per_block;
    uint4* kd = p.k_cache + int64_t(dst) * p.vec_per_block;
    uint4* vd = p.v_cache + int64_t(dst) * p.vec_per_block;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < p.vec_per_block;
         i += int64_t(gridDim.x) * blockDim.x) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}
}  // namespace

}  // namespace pkv

using namespace pkv;

extern "C" int paged_kv_append(const void* k, const void* v, const int64_t* slot_mapping,
                               int32_t num_tokens, void* k_cache, void* v_cache,
                               const pkv_cache_desc* desc, void* stream) {
    int st = check_desc(desc, false);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID;
    const int64_t row_bytes = int64_t(desc->head_dim) * int64_t(elem_bytes(desc->dtype));
    if (row_bytes % 16) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    AppendParams p;
    p.k = static_cast<const uint4*>(k);
    p.v = static_cast<const uint4*>(v);
    p.slots = slot_mapping;
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.num_tokens = num_tokens;
    p.vec_per_row = int32_t(row_bytes / 16);
    p.num_kv_heads = desc->num_kv_heads;
    p.block_size = desc->block_size;
    p.num_slots = int64_t(desc->num_blocks) * desc->block_size;
    p.err = err;
    const int64_t total = int64_t(num_tokens) * desc->num_kv_heads * p.vec_per_row;
    const int64_t cap = int64_t(std::max(sm_count(), 1)) * 8;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, cap);
    append_kernel<<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cuda_status(cudaGetLastError());
}

extern "C" int pkv_copy_blocks(const int32_t* block_pairs, int32_t num_pairs, void* k_cache,
                               void* v_cache, const pkv_cache_desc* desc, void* stream) {
    int st = check_desc(desc, false);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!block_pairs || !k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_pairs) & 3u))
        return PKV_ERR_INVALID;
    const int64_t block_bytes = int64_t(desc->num_kv_heads) * desc->block_size * desc->head_dim *
                                int64_t(elem_bytes(desc->dtype));
    if (block_bytes % 16) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    CopyParams p;
    p.pairs = block_pairs;
    p.k_cache = static_cast<uint4*>(k_cache);
    p.v_cache = static_cast<uint4*>(v_cache);
    p.vec_per_block = block_bytes / 16;
    p.num_blocks = desc->num_blocks;
    p.err = err;
    const unsigned gx = unsigned(std::min<int64_t>((p.vec_per_block + 255) / 256, 64));
    copy_blocks_kernel<<<dim3(gx, unsigned(num_pairs)), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cuda_status(cudaGetLastError());
}
