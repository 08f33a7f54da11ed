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

// grid-stride over (token, kv head, vector); K and V handled by the same thread.
// Idx is the type of the flat index: 32-bit unsigned whenever the launch's
// element count fits (its divisions are a few instructions, where 64-bit ones
// by a run-time divisor are a long emulated sequence per 16-byte vector), else
// 64-bit.  Cache offsets are always 64-bit.
template <typename Idx>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
    const Idx per_tok = Idx(p.num_kv_heads) * Idx(p.vec_per_row);
    const Idx total = Idx(p.num_tokens) * per_tok;
    const Idx vec = Idx(p.vec_per_row);
    for (Idx i = Idx(blockIdx.x) * Idx(blockDim.x) + Idx(threadIdx.x); i < total;
         i += Idx(gridDim.x) * Idx(blockDim.x)) {
        const Idx t = i / per_tok;
        const Idx r = i - t * per_tok;                // (head, vector) within the token
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;                       // padding token
        if (slot >= p.num_slots) {
            flag_error(p.err, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const int64_t row = slot - blk * p.block_size;
        const Idx h = r / vec;
        const Idx c = r - h * vec;
        const int64_t dst =
            ((blk * p.num_kv_heads + int64_t(h)) * p.block_size + row) * p.vec_per_row + int64_t(c);
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


// ---------------------------------------------------------------------------
// Rotary position embedding fused with the append ("第 15 章：推理引擎与部署"
// §15.3 RoPE 与 Flash Attention 的融合: rotate in registers instead of a separate
// pass through HBM; "DeepSpeed-FastGen 深度解析" §6 linear_blocked_kv_rotary:
// rotary fused with the blocked-KV write).  Rotate-half form: for i < D/2,
//   x'[i] = x[i] c - x[i+D/2] s,   x'[i+D/2] = x[i] s + x[i+D/2] c,
// with (c, s) from the caller's table at the token's position.  Each product
// and sum is rounded on its own (no fused multiply-add), then the result is
// rounded to the cache dtype, so the stored bytes are reproducible exactly.
// Values are copied unrotated.
// ---------------------------------------------------------------------------
struct RopeParams {
    const void* q;
    void* q_out;
    const void* k;
    const void* v;
    const int64_t* slots;
    const int32_t* positions;
    const float* cos_sin;     // [max_position][D]: cos of the D/2 angles, then their sin
    void* k_cache;
    void* v_cache;
    int64_t num_tokens;
    int32_t num_q_rows;       // Hq, or 0 when q is not rotated
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t max_position;
    int64_t num_slots;
    int* err;
};

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&x)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&x)[8]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&x)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// One thread per (token, 8-pair chunk): it loads the chunk's cos and sin once
// and applies them to every rotated row of the token (its q heads, then its K
// heads), then copies the chunk of its V heads.  Eight consecutive threads
// cover a 256-byte row, so loads and stores stay coalesced.  (Idx as for
// append_kernel.)
template <typename T, int D, typename Idx>
__global__ void __launch_bounds__(256) append_rope_kernel(RopeParams p) {
    constexpr int kChunks = D / 16;           // 8-pair chunks per head row
    const Idx total = Idx(p.num_tokens) * Idx(kChunks);
    for (Idx i = Idx(blockIdx.x) * Idx(blockDim.x) + Idx(threadIdx.x); i < total;
         i += Idx(gridDim.x) * Idx(blockDim.x)) {
        const int64_t t = int64_t(i / Idx(kChunks));
        const int c = int(i % Idx(kChunks));
        const int pos = __ldg(p.positions + t);
        const bool pos_ok = pos >= 0 && pos < p.max_position;
        const int64_t slot = __ldg(p.slots + t);
        // a bad position matters to the rows that rotate: q heads, and K heads
        // whose slot is in range (a padding or out-of-range slot skips K and V)
        if (!pos_ok && c == 0 && (p.num_q_rows > 0 || (slot >= 0 && slot < p.num_slots)))
            flag_error(p.err, PKV_DEV_BAD_POSITION);
        float co[8], si[8];
        if (pos_ok) {
            const float* cs = p.cos_sin + int64_t(pos) * D;
            load8<float>(cs + 8 * c, co);
            load8<float>(cs + D / 2 + 8 * c, si);
        }
        auto rotate = [&](float (&x1)[8], float (&x2)[8]) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float a = __fmul_rn(x1[j], co[j]), b = __fmul_rn(x2[j], si[j]);
                const float e = __fmul_rn(x1[j], si[j]), f = __fmul_rn(x2[j], co[j]);
                x1[j] = __fsub_rn(a, b);
                x2[j] = __fadd_rn(e, f);
            }
        };
        // q heads: rotated into q_out (no slot involved)
        if (pos_ok) {
            const T* qs = static_cast<const T*>(p.q) + t * p.num_q_rows * D + 8 * c;
            T* qd = static_cast<T*>(p.q_out) + t * p.num_q_rows * D + 8 * c;
#pragma unroll 4
            for (int h = 0; h < p.num_q_rows; ++h) {
                float x1[8], x2[8];
                load8<T>(qs + h * D, x1);
                load8<T>(qs + h * D + D / 2, x2);
                rotate(x1, x2);
                store8<T>(qd + h * D, x1);
                store8<T>(qd + h * D + D / 2, x2);
            }
        }
        // K (rotated) and V (copied) heads into the token's slot
        if (slot < 0) continue;                                        // padding token
        if (slot >= p.num_slots) {
            if (c == 0) flag_error(p.err, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / p.block_size;
        const int64_t row0 = blk * p.num_kv_heads * p.block_size + (slot - blk * p.block_size);
        const T* ks = static_cast<const T*>(p.k) + t * p.num_kv_heads * D + 8 * c;
        const T* vs = static_cast<const T*>(p.v) + t * p.num_kv_heads * D + 8 * c;
        T* kd = static_cast<T*>(p.k_cache) + 8 * c;
        T* vd = static_cast<T*>(p.v_cache) + 8 * c;
#pragma unroll 4
        for (int h = 0; h < p.num_kv_heads; ++h) {
            const int64_t dst = (row0 + int64_t(h) * p.block_size) * D;
            float x1[8], x2[8];
            load8<T>(vs + h * D, x1);
            load8<T>(vs + h * D + D / 2, x2);
            store8<T>(vd + dst, x1);
            store8<T>(vd + dst + D / 2, x2);
            if (pos_ok) {
                load8<T>(ks + h * D, x1);
                load8<T>(ks + h * D + D / 2, x2);
                rotate(x1, x2);
                store8<T>(kd + dst, x1);
                store8<T>(kd + dst + D / 2, x2);
            }
        }
    }
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

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
    const int64_t cap = int64_t(std::max(num_sms(), 1)) * 8;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, cap);
    if (total < (int64_t(1) << 31))
        append_kernel<uint32_t><<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    else
        append_kernel<int64_t><<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
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

extern "C" int pkv_copy_blocks_int8(const int32_t* block_pairs, int32_t num_pairs,
                                    void* k_codes, void* v_codes, float* k_scales,
                                    float* v_scales, const pkv_cache_desc* desc, void* stream) {
    if (!desc) return PKV_ERR_INVALID;
    if (desc->dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
    pkv_cache_desc bd = *desc;
    bd.dtype = PKV_BF16;
    int st = check_desc(&bd, false);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!block_pairs || !k_codes || !v_codes || !k_scales || !v_scales || !aligned16(k_codes) ||
        !aligned16(v_codes) || !aligned16(k_scales) || !aligned16(v_scales) ||
        (reinterpret_cast<uintptr_t>(block_pairs) & 3u))
        return PKV_ERR_INVALID;
    const int64_t rows = int64_t(desc->num_kv_heads) * desc->block_size;   // per block
    const int64_t code_bytes = rows * desc->head_dim, scale_bytes = rows * 4;
    if (code_bytes % 16 || scale_bytes % 16) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // whole blocks as bytes: codes, then scales (the tile layout depends only on the row)
    const int64_t bytes[2] = {code_bytes, scale_bytes};
    void* kp[2] = {k_codes, k_scales};
    void* vp[2] = {v_codes, v_scales};
    for (int i = 0; i < 2; ++i) {
        CopyParams p;
        p.pairs = block_pairs;
        p.k_cache = static_cast<uint4*>(kp[i]);
        p.v_cache = static_cast<uint4*>(vp[i]);
        p.vec_per_block = bytes[i] / 16;
        p.num_blocks = desc->num_blocks;
        p.err = err;
        const unsigned gx = unsigned(std::min<int64_t>((p.vec_per_block + 255) / 256, 64));
        copy_blocks_kernel<<<dim3(gx, unsigned(num_pairs)), 256, 0, s>>>(p);
        if ((st = cuda_status(cudaGetLastError())) != PKV_OK) return st;
    }
    return PKV_OK;
}

extern "C" int paged_kv_append_rope(const void* q, void* q_out, const void* k, const void* v,
                                    const int64_t* slot_mapping, const int32_t* positions,
                                    const float* cos_sin, int32_t max_position,
                                    int32_t num_tokens, void* k_cache, void* v_cache,
                                    const pkv_cache_desc* desc, void* stream) {
    int st = check_desc(desc, false);
    if (st != PKV_OK) return st;
    if (num_tokens < 0 || max_position < 1) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (!k || !v || !slot_mapping || !positions || !cos_sin || !k_cache || !v_cache ||
        (q && !q_out) || (!q && q_out))
        return PKV_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(cos_sin) || (q && (!aligned16(q) || !aligned16(q_out))) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
        (reinterpret_cast<uintptr_t>(positions) & 3u))
        return PKV_ERR_INVALID;
    int* err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    RopeParams p;
    p.q = q;
    p.q_out = q_out;
    p.k = k;
    p.v = v;
    p.slots = slot_mapping;
    p.positions = positions;
    p.cos_sin = cos_sin;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.num_tokens = num_tokens;
    p.num_q_rows = q ? desc->num_q_heads : 0;
    p.num_kv_heads = desc->num_kv_heads;
    p.block_size = desc->block_size;
    p.max_position = max_position;
    p.num_slots = int64_t(desc->num_blocks) * desc->block_size;
    p.err = err;
    const int64_t total = int64_t(num_tokens) * (desc->head_dim / 16);   // (token, chunk) pairs
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, int64_t(std::max(num_sms(), 1)) * 8);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bf = desc->dtype == PKV_BF16;
    const bool narrow = total < (int64_t(1) << 31);
    if (desc->head_dim == 128) {
        if (bf) {
            if (narrow) append_rope_kernel<__nv_bfloat16, 128, uint32_t><<<unsigned(blocks), 256, 0, s>>>(p);
            else append_rope_kernel<__nv_bfloat16, 128, int64_t><<<unsigned(blocks), 256, 0, s>>>(p);
        } else {
            if (narrow) append_rope_kernel<float, 128, uint32_t><<<unsigned(blocks), 256, 0, s>>>(p);
            else append_rope_kernel<float, 128, int64_t><<<unsigned(blocks), 256, 0, s>>>(p);
        }
    } else {
        if (bf) {
            if (narrow) append_rope_kernel<__nv_bfloat16, 64, uint32_t><<<unsigned(blocks), 256, 0, s>>>(p);
            else append_rope_kernel<__nv_bfloat16, 64, int64_t><<<unsigned(blocks), 256, 0, s>>>(p);
        } else {
            if (narrow) append_rope_kernel<float, 64, uint32_t><<<unsigned(blocks), 256, 0, s>>>(p);
            else append_rope_kernel<float, 64, int64_t><<<unsigned(blocks), 256, 0, s>>>(p);
        }
    }
    return cuda_status(cudaGetLastError());
}
