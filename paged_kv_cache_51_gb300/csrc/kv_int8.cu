// 8-bit KV cache: quantise on append, dequantise inside the decode gather.
//
// "大模型部署.md" §2.5 LMDeploy (2. TurboMind 推理引擎解析) keeps the KV cache in
// 8 bits, halving what decode reads from HBM.  Format (the pages give none):
// symmetric int8 with one fp32 scale per (token, KV head),
//   amax = max_d |x[d]|,  scale = amax / 127,  code = clamp(rint(x / scale), -127, 127)
// (code = 0, scale = 0 for an all-zero row), each division rounded once in
// fp32, so the stored codes are reproducible exactly.  Pools: codes
// [NB][Hkv][bs][D] int8 and scales [NB][Hkv][bs] fp32, for K and for V.
//
// Decode reads a (block, head) tile as 16·D bytes of codes plus 64 bytes of
// scales (two bulk copies each for K and V).  The score of key t is
// scale_k[t] · (q · code_k[t]), and the V scale is folded into p, so the
// dequantisation costs one multiply per key.  Everything else (work units,
// online softmax, split merge) is the bf16 decode path's.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "decode_common.cuh"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// ---------------------------------------------------------------------------
// Append: one warp per (token, KV head) row; K and V rows of a token handled
// by consecutive warps.
// ---------------------------------------------------------------------------
struct AppendI8Params {
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const int64_t* slots;
    int8_t* k_codes;
    int8_t* v_codes;
    float* k_scales;
    float* v_scales;
    int64_t num_tokens;
    int32_t num_kv_heads;
    int32_t block_size;
    int64_t num_slots;
    int* err;
};

template <int D>
__global__ void __launch_bounds__(256) append_int8_kernel(AppendI8Params p) {
    constexpr int DPL = D / 32;  // values per lane: 4 or 2
    const int lane = threadIdx.x & 31;
    const int64_t rows = p.num_tokens * p.num_kv_heads * 2;
    for (int64_t r = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5; r < rows;
         r += (int64_t(gridDim.x) * blockDim.x) >> 5) {
        const bool is_v = r & 1;
        const int64_t th = r >> 1;              // token * Hkv + head
        const int64_t t = th / p.num_kv_heads;
        const int h = int(th - t * p.num_kv_heads);
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;
        if (slot >= p.num_slots) {
            if (lane == 0) flag_error(p.err, PKV_DEV_BAD_SLOT);
            continue;
        }
        const __nv_bfloat16* src = (is_v ? p.v : p.k) + th * D + lane * DPL;
        float x[DPL];
        if constexpr (DPL == 4) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
            x[0] = __uint_as_float(u.x << 16);
            x[1] = __uint_as_float(u.x & 0xffff0000u);
            x[2] = __uint_as_float(u.y << 16);
            x[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(src));
            x[0] = __uint_as_float(u << 16);
            x[1] = __uint_as_float(u & 0xffff0000u);
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
        for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullWarp, amax, off));
        const float scale = __fdiv_rn(amax, 127.f);
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            float c = scale > 0.f ? rintf(__fdiv_rn(x[i], scale)) : 0.f;
            c = fminf(fmaxf(c, -127.f), 127.f);
            packed |= (uint32_t(int32_t(c)) & 0xffu) << (8 * i);
        }
        const int64_t blk = slot / p.block_size;
        const int64_t row = (blk * p.num_kv_heads + h) * p.block_size + (slot - blk * p.block_size);
        int8_t* dst = (is_v ? p.v_codes : p.k_codes) + row * D + lane * DPL;
        if constexpr (DPL == 4) {
            *reinterpret_cast<uint32_t*>(dst) = packed;
        } else {
            *reinterpret_cast<uint16_t*>(dst) = uint16_t(packed);
        }
        if (lane == 0) (is_v ? p.v_scales : p.k_scales)[row] = scale;
    }
}

// ---------------------------------------------------------------------------
// Decode split kernel (CUDA cores, any group size 1/2/4/8).
// ---------------------------------------------------------------------------
struct SplitI8Params {
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    const int8_t* k_codes;
    const int8_t* v_codes;
    const float* k_scales;
    const float* v_scales;
    const int32_t* block_tables;
    const int32_t* context_lens;
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
    float scale_log2;
    int* err;
};

template <int D, int G>
struct I8Cfg {
    static constexpr int kWarps = 4;
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kDPL = D / 32;
    static constexpr int kTileBytes = kBlockTokens * D;      // codes of one (block, head)
    static constexpr int kScaleBytes = kBlockTokens * 4;     // their scales
    // stage: [K codes][V codes][K scales][V scales]
    static constexpr int kStageBytes = 2 * kTileBytes + 2 * kScaleBytes;
    static constexpr int kStages = 12;
    static constexpr int kTC = G == 1 ? 16 : 32 / G;
    static constexpr int kNV = kTC * G;
    static constexpr int kNC = kBlockTokens / kTC;
    static constexpr int kPBuf = G * kBlockTokens + G;
    static constexpr int kComb = G * (D + 2);
    static constexpr int kPBufOff = kStages * kStageBytes;
    static constexpr int kCombOff = kPBufOff + kWarps * kPBuf * 4;
    static constexpr int kBarOff = (kCombOff + kWarps * kComb * 4 + 15) / 16 * 16;
    static constexpr int kQueueOff = kBarOff + 2 * kStages * 8;
    static constexpr int kSmem = kQueueOff + int(sizeof(UnitQueue));
};

template <int DPL>
__device__ __forceinline__ void load_codes(const int8_t* p, float (&out)[DPL]) {
    if constexpr (DPL == 4) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] = float(int8_t(u >> (8 * i)));
    } else {
        const uint16_t u = *reinterpret_cast<const uint16_t*>(p);
        out[0] = float(int8_t(u));
        out[1] = float(int8_t(u >> 8));
    }
}

template <int D, int G>
__global__ void __launch_bounds__(I8Cfg<D, G>::kThreads) decode_split_int8_kernel(SplitI8Params p) {
    using C = I8Cfg<D, G>;
    extern __shared__ __align__(128) unsigned char smem[];
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
    const int Hkv = p.num_kv_heads, Hq = p.num_q_heads;
    const int n_units = p.n_items[0] * Hkv;
    constexpr int kSplitBlocks = kSplitTokens / kBlockTokens;

    if (warp == C::kWarps) {
        // ---------------- producer ----------------
        uint32_t it = 0;
        bool ok = true;
        int next = uq_first_ticket(p.ticket, lane);
        for (uint32_t k = 0;; ++k) {
            const int u = uq_produce(uq, k, next, p.ticket, n_units, lane, p.err, ok);
            if (u < 0) break;
            const int2 item = p.items[u / Hkv];
            const int kvh = u % Hkv;
            const int ctx = p.context_lens[item.x];
            const int b0 = item.y * kSplitBlocks;
            const int nb = min(kSplitBlocks, (ctx + kBlockTokens - 1) / kBlockTokens - b0);
            int my_blk = 0;
            if (lane < nb) my_blk = p.block_tables[size_t(item.x) * p.table_stride + b0 + lane];
            for (int j = 0; j < nb; ++j, ++it) {
                const int blk = __shfl_sync(kFullWarp, my_blk, j);
                const int st = it % C::kStages;
                ok = __all_sync(kFullWarp, mbar_wait(&empty[st], ((it / C::kStages) & 1) ^ 1, p.err));
                if (!ok) break;
                if (lane == 0) {
                    if (blk < 0 || blk >= p.num_blocks) {
                        flag_error(p.err, PKV_DEV_BAD_BLOCK_ID);
                        mbar_arrive(&full[st]);
                    } else {
                        mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                        const size_t row = size_t(blk) * Hkv + kvh;
                        unsigned char* dst = smem + size_t(st) * C::kStageBytes;
                        bulk_g2s(dst, p.k_codes + row * C::kTileBytes, C::kTileBytes, &full[st]);
                        bulk_g2s(dst + C::kTileBytes, p.v_codes + row * C::kTileBytes,
                                 C::kTileBytes, &full[st]);
                        bulk_g2s(dst + 2 * C::kTileBytes, p.k_scales + row * kBlockTokens,
                                 C::kScaleBytes, &full[st]);
                        bulk_g2s(dst + 2 * C::kTileBytes + C::kScaleBytes,
                                 p.v_scales + row * kBlockTokens, C::kScaleBytes, &full[st]);
                    }
                }
                __syncwarp();
            }
        }
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
    const int my_head = G == 1 ? 0 : lane / TC;
    const int my_tok = G == 1 ? (lane >> 1) : lane % TC;
    float* pbuf = pbuf_all + warp * C::kPBuf;
    uint32_t it_base = 0;
    bool ok = true;
    for (uint32_t k = 0;; ++k) {
        const int u = uq_consume(uq, k, C::kWarps * 32, p.err, ok);
        if (u < 0) break;
        const int2 item = p.items[u / Hkv];
        const int seq = item.x, split = item.y;
        const int kvh = u % Hkv;
        const int ctx = p.context_lens[seq];
        const int b0 = split * kSplitBlocks;
        const int nb = min(kSplitBlocks, (ctx + kBlockTokens - 1) / kBlockTokens - b0);

        float qr[G][DPL];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float t[DPL];
            Elem<__nv_bfloat16>::template load<DPL>(p.q + (size_t(seq) * Hq + kvh * G + j) * D + lane * DPL, t);
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
            if (ok) ok = __all_sync(kFullWarp, mbar_wait(&full[st], (it / C::kStages) & 1, p.err));
            if (!ok) continue;
            const unsigned char* sb = smem + size_t(st) * C::kStageBytes;
            const int8_t* kt = reinterpret_cast<const int8_t*>(sb);
            const int8_t* vt = kt + C::kTileBytes;
            const float* ksc = reinterpret_cast<const float*>(sb + 2 * C::kTileBytes);
            const float* vsc = ksc + kBlockTokens;
            const int nvalid = min(kBlockTokens, ctx - (b0 + jb) * kBlockTokens);

            float s[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float part[NV];
#pragma unroll
                for (int tt = 0; tt < TC; ++tt) {
                    float kf[DPL];
                    load_codes<DPL>(kt + (c * TC + tt) * D + lane * DPL, kf);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        float acc = qr[j][0] * kf[0];
#pragma unroll
                        for (int d = 1; d < DPL; ++d) acc = fmaf(qr[j][d], kf[d], acc);
                        part[j * TC + tt] = acc;
                    }
                }
                const int tok = c * TC + my_tok;
                s[c] = reduce_scatter<NV>(part, lane) * ksc[tok];
                if (tok >= nvalid) s[c] = -INFINITY;
            }
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
                const int tok = c * TC + my_tok;
                pbuf[my_head * kBlockTokens + tok] = pc * vsc[tok];   // V scale folded into p
            }
            psum = group_sum<G, TC>(psum);
            l = l * alpha + psum;
            m = m_new;
            if (my_tok == 0) pbuf[G * kBlockTokens + my_head] = alpha;
            __syncwarp();
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float a = pbuf[G * kBlockTokens + j];
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[j][d] *= a;
            }
            for (int t = 0; t < nvalid; ++t) {
                float vf[DPL];
                load_codes<DPL>(vt + t * D + lane * DPL, vf);
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
        const int nsplit = (ctx + kSplitTokens - 1) / kSplitTokens;
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
                p.out[(size_t(seq) * Hq + h) * D + d] = __float2bfloat16_rn(O / L);
            } else {
                const size_t slot = (size_t(seq) * Hq + h) * p.max_splits + split;
                p.part_o[slot * D + d] = O;
                if (d == 0) p.part_ml[slot] = make_float2(M, L);
            }
        }
        consumer_sync(C::kWarps * 32);
    }
}

bool aligned(const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; }

template <int D, int G>
int launch_i8(const AttnArgs& a, const int8_t* kc, const int8_t* vc, const float* ks,
              const float* vs) {
    using C = I8Cfg<D, G>;
    auto kern = decode_split_int8_kernel<D, G>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::kThreads, C::kSmem) !=
            cudaSuccess ||
        per_sm < 1)
        return PKV_ERR_CUDA;
    const int64_t bound = int64_t(a.num_seqs) * a.ws.max_splits * a.desc->num_kv_heads;
    const int64_t grid = std::min<int64_t>(int64_t(num_sms()) * per_sm, bound);
    if (grid < 1) return PKV_OK;
    SplitI8Params p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.k_codes = kc;
    p.v_codes = vc;
    p.k_scales = ks;
    p.v_scales = vs;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
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
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    kern<<<unsigned(grid), C::kThreads, C::kSmem, a.stream>>>(p);
    return cuda_status(cudaGetLastError());
}

template <int D>
int launch_i8_d(const AttnArgs& a, int g, const int8_t* kc, const int8_t* vc, const float* ks,
                const float* vs) {
    switch (g) {
        case 1: return launch_i8<D, 1>(a, kc, vc, ks, vs);
        case 2: return launch_i8<D, 2>(a, kc, vc, ks, vs);
        case 4: return launch_i8<D, 4>(a, kc, vc, ks, vs);
        case 8: return launch_i8<D, 8>(a, kc, vc, ks, vs);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int paged_kv_append_int8(const void* k, const void* v, const int64_t* slot_mapping,
                                    int32_t num_tokens, void* k_codes, void* v_codes,
                                    float* k_scales, float* v_scales, const pkv_cache_desc* desc,
                                    void* stream) {
    if (!desc) return PKV_ERR_INVALID;
    if (desc->dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
    pkv_cache_desc bd = *desc;
    bd.dtype = PKV_BF16;
    int st = check_desc(&bd, false);
    if (st != PKV_OK) return st;
    if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_codes || !v_codes || !k_scales || !v_scales)
        return PKV_ERR_INVALID;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_codes, 16) || !aligned(v_codes, 16) ||
        !aligned(k_scales, 16) || !aligned(v_scales, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID;
    int* err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    AppendI8Params p;
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.slots = slot_mapping;
    p.k_codes = static_cast<int8_t*>(k_codes);
    p.v_codes = static_cast<int8_t*>(v_codes);
    p.k_scales = k_scales;
    p.v_scales = v_scales;
    p.num_tokens = num_tokens;
    p.num_kv_heads = desc->num_kv_heads;
    p.block_size = desc->block_size;
    p.num_slots = int64_t(desc->num_blocks) * desc->block_size;
    p.err = err;
    const int64_t warps = int64_t(num_tokens) * desc->num_kv_heads * 2;
    const int64_t blocks = std::min<int64_t>((warps * 32 + 255) / 256, int64_t(num_sms()) * 8);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (desc->head_dim == 128)
        append_int8_kernel<128><<<unsigned(blocks), 256, 0, s>>>(p);
    else
        append_int8_kernel<64><<<unsigned(blocks), 256, 0, s>>>(p);
    return cuda_status(cudaGetLastError());
}

extern "C" int paged_attention_decode_int8(void* out, const void* q, const void* k_codes,
                                           const void* v_codes, const float* k_scales,
                                           const float* v_scales, const pkv_cache_desc* desc,
                                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* context_lens, int32_t num_seqs,
                                           int32_t max_context_len, float scale, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    if (!desc) return PKV_ERR_INVALID;
    if (desc->dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
    // the attention checks on the bf16 view (q, out, group size, head_dim, block size)
    pkv_cache_desc qd = *desc;
    qd.dtype = PKV_BF16;
    int st = check_desc(&qd, true);
    if (st != PKV_OK) return st;
    if (num_seqs < 0 || max_blocks_per_seq < 1 || max_context_len < 1) return PKV_ERR_INVALID;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_codes || !v_codes || !k_scales || !v_scales || !block_tables ||
        !context_lens)
        return PKV_ERR_INVALID;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_codes, 16) || !aligned(v_codes, 16) ||
        !aligned(k_scales, 16) || !aligned(v_scales, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4))
        return PKV_ERR_INVALID;
    const size_t need = pkv_decode_workspace_bytes(&qd, num_seqs, max_context_len);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    AttnArgs a{};
    workspace_layout(&qd, num_seqs, max_context_len, 0, workspace, &a.ws);
    a.err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    a.out = out;
    a.q = q;
    a.desc = &qd;
    a.block_tables = block_tables;
    a.table_stride = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.num_seqs = num_seqs;
    a.num_query_tokens = num_seqs;
    a.max_query_len = 1;
    a.max_context_len = max_context_len;
    a.scale = scale;
    a.stream = static_cast<cudaStream_t>(stream);
    if ((st = launch_plan(a)) != PKV_OK) return st;
    const int g = qd.num_q_heads / qd.num_kv_heads;
    const auto* kc = static_cast<const int8_t*>(k_codes);
    const auto* vc = static_cast<const int8_t*>(v_codes);
    st = qd.head_dim == 128 ? launch_i8_d<128>(a, g, kc, vc, k_scales, v_scales)
                            : launch_i8_d<64>(a, g, kc, vc, k_scales, v_scales);
    if (st != PKV_OK) return st;
    return launch_decode_merge(a);
}
