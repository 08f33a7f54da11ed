// Slot-mapped KV append and copy-on-write block copies.
//
// Append ("【自用】AI infra相关" 一、推理两阶段 2、解码: each step's K_t, V_t are
// written into the cache; "大模型部署.md" §2.1: the block manager plans the
// physical slot, the cache engine writes it):
//     cache[slot / bs][h][slot % bs][:] = x[t][h][:]      for K and V.
// Copy-on-write ("大模型部署.md" §2.1 append_slots: a shared last block gets a
// private copy before the write): a whole block (all heads, all rows) of K and V.
//
// Both are pure byte movement, bound by HBM bandwidth: every thread moves one
// 16-byte vector with a coalesced load and store; source rows are read once,
// with the non-coherent (read-only) path, and nothing is converted, so the
// cache bytes equal the input bytes exactly.
#include <cuda_runtime.h>

#include <algorithm>

#include "launch_cache.h"
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

// grid-stride over (token, kv head, vector); K and V handled by the same thread,
// kAppendUnroll vectors per pass with all their loads issued before any store.
// Idx is the type of the flat index: 32-bit unsigned whenever the launch's
// element count fits (its divisions are a few instructions, where 64-bit ones
// by a run-time divisor are a long emulated sequence per 16-byte vector), else
// 64-bit.  Cache offsets are always 64-bit.
constexpr int kAppendUnroll = 4;

template <typename Idx>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
    // launched programmatically behind the previous kernel: wait for it to
    // complete before touching the inputs or the cache; let the next launch
    pdl_wait_prerequisites();
    pdl_launch_dependents();
    const Idx per_tok = Idx(p.num_kv_heads) * Idx(p.vec_per_row);
    const Idx total = Idx(p.num_tokens) * per_tok;
    const Idx vec = Idx(p.vec_per_row);
    const Idx stride = Idx(gridDim.x) * Idx(blockDim.x);
    for (Idx i0 = Idx(blockIdx.x) * Idx(blockDim.x) + Idx(threadIdx.x); i0 < total;
         i0 += Idx(kAppendUnroll) * stride) {
        uint4 kv[kAppendUnroll], vv[kAppendUnroll];
        int64_t slot[kAppendUnroll];
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u) {
            const Idx i = i0 + Idx(u) * stride;
            if (i < total) {
                slot[u] = __ldg(p.slots + i / per_tok);
                kv[u] = __ldg(p.k + i);
                vv[u] = __ldg(p.v + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u) {
            const Idx i = i0 + Idx(u) * stride;
            if (i >= total || slot[u] < 0) continue;      // past the end, or a padding token
            if (slot[u] >= p.num_slots) {
                flag_error(p.err, PKV_DEV_BAD_SLOT);
                continue;
            }
            const Idx t = i / per_tok;
            const Idx r = i - t * per_tok;                // (head, vector) within the token
            const int64_t blk = slot[u] / p.block_size;
            const int64_t row = slot[u] - blk * p.block_size;
            const Idx h = r / vec;
            const Idx c = r - h * vec;
            const int64_t dst =
                ((blk * p.num_kv_heads + int64_t(h)) * p.block_size + row) * p.vec_per_row + int64_t(c);
            p.k_cache[dst] = kv[u];
            p.v_cache[dst] = vv[u];
        }
    }
}

struct CopyParams {
    const int32_t* pairs;
    uint4* k_cache;
    uint4* v_cache;           // null: k_cache is one pool holding both
    int64_t vec_per_block;    // 16-byte vectors per physical block (all heads)
    int32_t num_blocks;
    int* err;
};

// blockIdx.y = pair; blockIdx.x strides over the block's vectors
__global__ void __launch_bounds__(256) copy_blocks_kernel(CopyParams p) {
    pdl_wait_prerequisites();   // as append_kernel
    pdl_launch_dependents();
    const int pair = blockIdx.y;
    const int src = __ldg(p.pairs + 2 * pair), dst = __ldg(p.pairs + 2 * pair + 1);
    if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(p.err, PKV_DEV_BAD_COPY_PAIR);
        return;
    }
    const uint4* ks = p.k_cache + int64_t(src) * p.vec_per_block;
    uint4* kd = p.k_cache + int64_t(dst) * p.vec_per_block;
    if (p.v_cache) {
        const uint4* vs = p.v_cache + int64_t(src) * p.vec_per_block;
        uint4* vd = p.v_cache + int64_t(dst) * p.vec_per_block;
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < p.vec_per_block;
             i += int64_t(gridDim.x) * blockDim.x) {
            kd[i] = ks[i];
            vd[i] = vs[i];
        }
    } else {   // one pool (the 8-bit cache: K and V tiles of a block side by side)
        for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < p.vec_per_block;
             i += int64_t(gridDim.x) * blockDim.x)
            kd[i] = ks[i];
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

// Raw bytes of one 8-element chunk of a row (16 B of bf16, 32 B of fp32).
template <typename T>
struct Chunk8 {
    uint4 w[sizeof(T) / 2];
};
template <typename T>
__device__ __forceinline__ void load_raw(const T* p, Chunk8<T>& x) {
#pragma unroll
    for (int i = 0; i < int(sizeof(T)) / 2; ++i) x.w[i] = __ldg(reinterpret_cast<const uint4*>(p) + i);
}
template <typename T>
__device__ __forceinline__ void store_raw(T* p, const Chunk8<T>& x) {
#pragma unroll
    for (int i = 0; i < int(sizeof(T)) / 2; ++i) reinterpret_cast<uint4*>(p)[i] = x.w[i];
}
__device__ __forceinline__ void widen(const Chunk8<__nv_bfloat16>& x, float (&f)[8]) {
    const uint32_t w[4] = {x.w[0].x, x.w[0].y, x.w[0].z, x.w[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void widen(const Chunk8<float>& x, float (&f)[8]) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        f[4 * i] = __uint_as_float(x.w[i].x);
        f[4 * i + 1] = __uint_as_float(x.w[i].y);
        f[4 * i + 2] = __uint_as_float(x.w[i].z);
        f[4 * i + 3] = __uint_as_float(x.w[i].w);
    }
}

// A token's rows, in order: its Hq query heads (rotated into q_out), its Hkv
// K heads (rotated into the slot) and its Hkv V heads (copied into the slot).
// One thread per (token, group of kRows rows, 8-pair chunk): it issues the
// loads of all its rows' chunks before it rotates and stores any, so each
// thread keeps kRows x 32 B (bf16) in flight, and it loads the chunk's cos
// and sin once for the group.  Eight consecutive threads cover a 256-byte
// row, so loads and stores stay coalesced.  (Idx as for append_kernel.)
template <typename T>
__host__ __device__ constexpr int rope_rows_per_thread() { return 16 / int(sizeof(T)); }

template <typename T, int D, typename Idx>
__global__ void __launch_bounds__(256, 2) append_rope_kernel(RopeParams p) {
    constexpr int kChunks = D / 16;           // 8-pair chunks per head row
    constexpr int kRows = rope_rows_per_thread<T>();
    const int hq = p.num_q_rows, hkv = p.num_kv_heads;
    const int rows = hq + 2 * hkv;
    const int groups = (rows + kRows - 1) / kRows;
    const Idx per_tok = Idx(groups) * Idx(kChunks);
    const Idx total = Idx(p.num_tokens) * per_tok;
    for (Idx i = Idx(blockIdx.x) * Idx(blockDim.x) + Idx(threadIdx.x); i < total;
         i += Idx(gridDim.x) * Idx(blockDim.x)) {
        const Idx ti = i / per_tok;
        const int r = int(i - ti * per_tok);
        const int64_t t = int64_t(ti);
        const int c = r % kChunks;
        const int row_lo = (r / kChunks) * kRows;
        const int pos = __ldg(p.positions + t);
        const bool pos_ok = pos >= 0 && pos < p.max_position;
        const int64_t slot = __ldg(p.slots + t);
        const bool slot_ok = slot >= 0 && slot < p.num_slots;
        if (row_lo == 0 && c == 0) {
            // a bad position matters to the rows that rotate: q heads, and K
            // heads whose slot is in range (a padding or out-of-range slot
            // skips K and V)
            if (!pos_ok && (hq > 0 || slot_ok)) flag_error(p.err, PKV_DEV_BAD_POSITION);
            if (slot >= p.num_slots) flag_error(p.err, PKV_DEV_BAD_SLOT);
        }
        int64_t row0 = 0;
        if (slot_ok) {
            const int64_t blk = slot / p.block_size;
            row0 = blk * hkv * p.block_size + (slot - blk * p.block_size);
        }
        // sources and destinations of the group's rows; a row that is not
        // written this step (past the token's rows, or skipped) is inactive
        Chunk8<T> x1[kRows], x2[kRows];
        const T* src[kRows];
        T* dst[kRows];
        bool act[kRows], rot[kRows];
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const int row = row_lo + j;
            if (row < hq) {
                const int64_t off = (t * hq + row) * D + 8 * c;
                src[j] = static_cast<const T*>(p.q) + off;
                dst[j] = static_cast<T*>(p.q_out) + off;
                act[j] = pos_ok;
                rot[j] = true;
            } else if (row < hq + hkv) {
                const int h = row - hq;
                src[j] = static_cast<const T*>(p.k) + (t * hkv + h) * D + 8 * c;
                dst[j] = static_cast<T*>(p.k_cache) + (row0 + int64_t(h) * p.block_size) * D + 8 * c;
                act[j] = pos_ok && slot_ok;
                rot[j] = true;
            } else {
                const int h = row - hq - hkv;
                src[j] = static_cast<const T*>(p.v) + (t * hkv + h) * D + 8 * c;
                dst[j] = static_cast<T*>(p.v_cache) + (row0 + int64_t(h) * p.block_size) * D + 8 * c;
                act[j] = slot_ok && row < rows;
                rot[j] = false;
            }
            if (act[j]) {
                load_raw<T>(src[j], x1[j]);
                load_raw<T>(src[j] + D / 2, x2[j]);
            }
        }
        float co[8], si[8];
        if (pos_ok && row_lo < hq + hkv) {
            const float* cs = p.cos_sin + int64_t(pos) * D;
            load8<float>(cs + 8 * c, co);
            load8<float>(cs + D / 2 + 8 * c, si);
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            if (!act[j]) continue;
            if (!rot[j]) {
                store_raw<T>(dst[j], x1[j]);
                store_raw<T>(dst[j] + D / 2, x2[j]);
                continue;
            }
            float a1[8], a2[8], y1[8], y2[8];
            widen(x1[j], a1);
            widen(x2[j], a2);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float a = __fmul_rn(a1[e], co[e]), b = __fmul_rn(a2[e], si[e]);
                const float s = __fmul_rn(a1[e], si[e]), f = __fmul_rn(a2[e], co[e]);
                y1[e] = __fsub_rn(a, b);
                y2[e] = __fadd_rn(s, f);
            }
            store8<T>(dst[j], y1);
            store8<T>(dst[j] + D / 2, y2);
        }
    }
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Resident 256-thread blocks per SM of a grid-stride kernel (1 if the query
// fails; its error is cleared so that it is not reported by a later launch).
template <typename K>
int resident_blocks_per_sm(K kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    return n;
}

// Grid-stride launch of the RoPE append with no more blocks than are resident
// at once (the kernel holds a group's rows in registers, so fewer than eight
// 256-thread blocks fit on an SM: two, at the bound of 128 registers).
template <typename T, int D, typename Idx>
int launch_rope(const RopeParams& p, int64_t total, void* stream) {
    static const int per_sm = resident_blocks_per_sm(append_rope_kernel<T, D, Idx>);
    const int64_t blocks =
        std::min<int64_t>((total + 255) / 256, int64_t(std::max(num_sms(), 1)) * per_sm);
    append_rope_kernel<T, D, Idx><<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cuda_status(cudaGetLastError());
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
    const int64_t sms = std::max(num_sms(), 1);
    const int64_t want = (total + 255) / 256;
    if (total < (int64_t(1) << 31)) {
        static const int per_sm = resident_blocks_per_sm(append_kernel<uint32_t>);
        const int64_t blocks = std::min<int64_t>(want, sms * per_sm);
        return cuda_status(launch_pdl(append_kernel<uint32_t>, dim3(unsigned(blocks)), dim3(256), 0,
                                      static_cast<cudaStream_t>(stream), p));
    }
    static const int per_sm = resident_blocks_per_sm(append_kernel<int64_t>);
    const int64_t blocks = std::min<int64_t>(want, sms * per_sm);
    return cuda_status(launch_pdl(append_kernel<int64_t>, dim3(unsigned(blocks)), dim3(256), 0,
                                  static_cast<cudaStream_t>(stream), p));
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
    return cuda_status(launch_pdl(copy_blocks_kernel, dim3(gx, unsigned(num_pairs)), dim3(256), 0,
                                  static_cast<cudaStream_t>(stream), p));
}

extern "C" int pkv_copy_blocks_int8(const int32_t* block_pairs, int32_t num_pairs, void* kv_pool,
                                    const pkv_cache_desc* desc, void* stream) {
    if (!desc) return PKV_ERR_INVALID;
    if (desc->dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
    pkv_cache_desc bd = *desc;
    bd.dtype = PKV_BF16;
    int st = check_desc(&bd, false);
    if (st != PKV_OK) return st;
    if (desc->block_size != 16) return PKV_ERR_UNSUPPORTED;   // the tile layout is 16 rows
    if (num_pairs < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!block_pairs || !kv_pool || !aligned16(kv_pool) ||
        (reinterpret_cast<uintptr_t>(block_pairs) & 3u))
        return PKV_ERR_INVALID;
    // whole blocks as bytes: every KV head's K and V tiles of codes and scales
    const int64_t tile_bytes = int64_t(desc->block_size) * desc->head_dim + desc->block_size * 4;
    const int64_t block_bytes = int64_t(desc->num_kv_heads) * 2 * tile_bytes;
    if (block_bytes % 16) return PKV_ERR_UNSUPPORTED;
    int* err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    CopyParams p;
    p.pairs = block_pairs;
    p.k_cache = static_cast<uint4*>(kv_pool);
    p.v_cache = nullptr;
    p.vec_per_block = block_bytes / 16;
    p.num_blocks = desc->num_blocks;
    p.err = err;
    const unsigned gx = unsigned(std::min<int64_t>((p.vec_per_block + 255) / 256, 64));
    copy_blocks_kernel<<<dim3(gx, unsigned(num_pairs)), 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cuda_status(cudaGetLastError());
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
    const bool bf = desc->dtype == PKV_BF16;
    const int rows_per_thread = bf ? rope_rows_per_thread<__nv_bfloat16>() : rope_rows_per_thread<float>();
    const int64_t groups = (p.num_q_rows + 2 * int64_t(p.num_kv_heads) + rows_per_thread - 1) /
                           rows_per_thread;
    // (token, row group, chunk) triples
    const int64_t total = int64_t(num_tokens) * groups * (desc->head_dim / 16);
    const bool narrow = total < (int64_t(1) << 31);
    if (desc->head_dim == 128) {
        if (bf) {
            if (narrow) st = launch_rope<__nv_bfloat16, 128, uint32_t>(p, total, stream);
            else st = launch_rope<__nv_bfloat16, 128, int64_t>(p, total, stream);
        } else {
            if (narrow) st = launch_rope<float, 128, uint32_t>(p, total, stream);
            else st = launch_rope<float, 128, int64_t>(p, total, stream);
        }
    } else {
        if (bf) {
            if (narrow) st = launch_rope<__nv_bfloat16, 64, uint32_t>(p, total, stream);
            else st = launch_rope<__nv_bfloat16, 64, int64_t>(p, total, stream);
        } else {
            if (narrow) st = launch_rope<float, 64, uint32_t>(p, total, stream);
            else st = launch_rope<float, 64, int64_t>(p, total, stream);
        }
    }
    return st;
}
