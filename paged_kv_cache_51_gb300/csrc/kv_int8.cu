// 8-bit KV cache: quantise on append, dequantise inside the decode gather.
//
// "大模型部署.md" §2.5 LMDeploy (2. TurboMind 推理引擎解析) keeps the KV cache in
// 8 bits, halving what decode reads from HBM.  Format (the pages give none):
// symmetric int8 with one fp32 scale per (token, KV head),
//   amax = max_d |x[d]|,  scale = amax / 127,  code = clamp(rint(x / scale), -127, 127)
// (code = 0, scale = 0 for an all-zero row), each division rounded once in
// fp32, so the stored codes are reproducible exactly.
//
// Pool layout.  One tile holds 16 tokens of one KV head: their 16 * D codes,
// then their 16 fp32 scales (16 * D + 64 bytes).  The pool holds, per (block,
// KV head), the K tile and then the V tile, so a decode stage is one bulk copy
// of 2 * (16 * D + 64) contiguous bytes: the scales as separate 64-byte copies
// cost 13 % of the call, and K and V as two 2112-byte copies from separate
// pools 6 % more than one 4224-byte run (scattered reads of 2 KB runs keep
// the DRAM less busy than reads of 4 KB).  K codes are row-major [token][D] with
// the 16-byte chunks of row r XOR-swizzled (chunk c stored at c ^ sw(r),
// sw(r) = r & 7 for D = 128 and (r >> 1) & 3 for D = 64); V codes are
// dim-major [D][token].  Both code layouts let a warp load its tensor-core
// fragments as 32-bit words with no shared-memory bank conflicts.
//
// Decode runs both products on tensor cores (mma.sync m16n8k16, f16 in, fp32
// accumulate), which keeps the kernel on the HBM roofline for every group size:
//   * codes become f16 exactly: flipping the sign bit gives the byte c + 128, a
//     byte permute places two such bytes in the mantissas of 1024 (f16 0x64xx),
//     and one packed subtraction of 1152 leaves c;
//   * q (bf16) is exact in f16 after a power-of-two shift chosen per work unit
//     (largest |q| in [2^14, 2^15)); the shift is undone on the fp32 scores;
//   * S = K q^T (tokens x heads) is scaled per token by the K scale;
//   * the V scale is folded into P, P' = p * v_scale * 2^(127 - e_v), where e_v
//     is the running largest V-scale exponent of the unit, so P' < 2 fits f16;
//     when e_v grows the accumulator is rescaled with the softmax alpha;
//   * O^T = V^T P' (dims x heads) accumulates in the mma's fp32 registers.
// Work units, the online softmax, the warp combine and the split merge are
// the bf16 decode path's.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "decode_common.cuh"
#include "launch_cache.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// bytes of one (block, KV head) tile: codes, then scales
template <int D>
__host__ __device__ constexpr int i8_tile_bytes() {
    return kBlockTokens * D + kBlockTokens * 4;
}

// 16-byte chunk swizzle of the K tile row r
template <int D>
__host__ __device__ constexpr int k_swizzle(int r) {
    return D == 128 ? (r & 7) : ((r >> 1) & 3);
}

// ---------------------------------------------------------------------------
// Append: one warp per (token, KV head) row; K and V rows of a token handled
// by consecutive warps.
// ---------------------------------------------------------------------------
struct AppendI8Params {
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const int64_t* slots;
    unsigned char* kv_pool;
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
        int32_t code[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            float c = scale > 0.f ? rintf(__fdiv_rn(x[i], scale)) : 0.f;
            code[i] = int32_t(fminf(fmaxf(c, -127.f), 127.f));
        }
        const int64_t blk = slot / p.block_size;
        const int rr = int(slot - blk * p.block_size);           // token row within the tile
        unsigned char* tile =
            p.kv_pool + ((blk * p.num_kv_heads + h) * 2 + (is_v ? 1 : 0)) * i8_tile_bytes<D>();
        if (!is_v) {
            // row-major, 16-byte chunk (lane * DPL) / 16 swizzled by the row
            const int d0 = lane * DPL;
            unsigned char* dst = tile + rr * D + (((d0 >> 4) ^ k_swizzle<D>(rr)) << 4) + (d0 & 15);
            uint32_t packed = 0;
#pragma unroll
            for (int i = 0; i < DPL; ++i) packed |= (uint32_t(code[i]) & 0xffu) << (8 * i);
            if constexpr (DPL == 4) {
                *reinterpret_cast<uint32_t*>(dst) = packed;
            } else {
                *reinterpret_cast<uint16_t*>(dst) = uint16_t(packed);
            }
        } else {
            // dim-major: byte (d, rr) at d * 16 + rr
            unsigned char* dst = tile + rr;
#pragma unroll
            for (int i = 0; i < DPL; ++i)
                dst[(lane * DPL + i) * kBlockTokens] = static_cast<unsigned char>(code[i] & 0xff);
        }
        if (lane == 0) reinterpret_cast<float*>(tile + kBlockTokens * D)[rr] = scale;
    }
}

// ---------------------------------------------------------------------------
// Decode split kernel (tensor cores, group size 1, 2, 4 or 8).
// ---------------------------------------------------------------------------
struct SplitI8Params {
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    const unsigned char* kv_pool;
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
    static constexpr int kKB = D / 16;                       // 16-dim blocks
    static constexpr int kCodeBytes = kBlockTokens * D;      // codes of one (block, head)
    static constexpr int kTileBytes = i8_tile_bytes<D>();    // codes + their scales
    // stage: [K codes][K scales][V codes][V scales], the two tiles as stored
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = 8;
    // resident CTAs per SM the register allocation must allow (the compiler
    // otherwise takes 109 registers for D = 128, g = 1, and a fourth CTA no
    // longer fits: 0.2406 -> 0.264 ms on the Llama-2-7B batch)
    static constexpr int kMinBlocks = D == 128 ? 4 : 5;
    static constexpr int kPB = 8 * kBlockTokens * 2;         // P' per warp: f16 [8 heads][16 tokens]
    static constexpr int kComb = G * (D + 2);
    static constexpr int kQBytes = G * D * 2;                // q of one unit (bf16)
    static constexpr int kQSlots = 2;                        // units whose q is in flight
    static constexpr int kPBufOff = kStages * kStageBytes;
    static constexpr int kCombOff = kPBufOff + kWarps * kPB;
    static constexpr int kQOff = (kCombOff + kWarps * kComb * 4 + 15) / 16 * 16;
    static constexpr int kMetaOff = kQOff + kQSlots * kQBytes;
    static constexpr int kBarOff = kMetaOff + kQSlots * 16;
    // full[kStages], empty[kStages], q_full[kQSlots], q_empty[kQSlots]
    static constexpr int kQueueOff = kBarOff + (2 * kStages + 2 * kQSlots) * 8;
    static constexpr int kSmem = kQueueOff + int(sizeof(UnitQueue));
    static_assert(kStageBytes % 128 == 0 && kTileBytes % 16 == 0, "bulk copy alignment");
    // Consumer warp w takes tiles w, w + kWarps, ... of a unit and waits on a
    // stage by parity alone.  With kStages a multiple of kWarps the previous use
    // of that stage is the same warp's own (finished) tile; otherwise it can be
    // another warp's tile whose copy has not landed, the parity matches the
    // wrong phase and the wait passes early.
    static_assert(kStages % kWarps == 0, "stage ring must be a multiple of the consumer warps");
};

// four int8 codes -> two f16x2 registers, exactly (lo: bytes 0, 1; hi: bytes 2, 3)
__device__ __forceinline__ void codes_to_f16x2(uint32_t u, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = u ^ 0x80808080u;                  // byte c + 128
    const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140u);   // f16 1024 + byte (two lanes)
    const uint32_t b = __byte_perm(x, 0x64646464u, 0x4342u);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));   // - 1152
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^k for an exponent k in [-126, 127]
__device__ __forceinline__ float exp2i(int k) { return __uint_as_float(uint32_t(127 + k) << 23); }

template <int D, int G>
__global__ void __launch_bounds__(I8Cfg<D, G>::kThreads, I8Cfg<D, G>::kMinBlocks)
    decode_split_int8_kernel(SplitI8Params p) {
    using C = I8Cfg<D, G>;
    constexpr int KB = C::kKB;
    extern __shared__ __align__(128) unsigned char smem[];
    float* comb = reinterpret_cast<float*>(smem + C::kCombOff);
    unsigned char* qbuf = smem + C::kQOff;
    int4* meta = reinterpret_cast<int4*>(smem + C::kMetaOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* empty = full + C::kStages;
    uint64_t* q_full = empty + C::kStages;
    uint64_t* q_empty = q_full + C::kQSlots;
    UnitQueue* uq = reinterpret_cast<UnitQueue*>(smem + C::kQueueOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < C::kQSlots; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], C::kWarps);
        }
        uq_init(uq);
        fence_mbar_init();
    }
    __syncthreads();
    // launched right behind the planner (programmatic launch): its work list must
    // be complete before anything below reads it; the merge kernel may launch now
    pdl_wait_prerequisites();
    pdl_launch_dependents();
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
            // the unit's description and q, so the consumers start without global loads
            const int qs = k % C::kQSlots;
            ok = __all_sync(kFullWarp,
                            mbar_wait(&q_empty[qs], ((k / C::kQSlots) & 1) ^ 1, p.err));
            if (!ok) break;
            if (lane == 0) {
                meta[qs] = make_int4(item.x, item.y, ctx, kvh);
                mbar_arrive_expect_tx(&q_full[qs], C::kQBytes);
                bulk_g2s(qbuf + qs * C::kQBytes, p.q + (size_t(item.x) * Hq + kvh * G) * D,
                         C::kQBytes, &q_full[qs]);
            }
            __syncwarp();
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
                        // the (block, head) unit: K tile then V tile, one run
                        bulk_g2s(dst, p.kv_pool + row * C::kStageBytes, C::kStageBytes, &full[st]);
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
        return;   // q copies: each one completes before its unit's consumers (which wait on it) finish
    }

    // ---------------- consumer warps ----------------
    // mma fragment coordinates: lane = 4 g + t
    const int g = lane >> 2, t = lane & 3;
    uint16_t* pb = reinterpret_cast<uint16_t*>(smem + C::kPBufOff + warp * C::kPB);
    const int ksw = k_swizzle<D>(g);                  // rows g and g + 8 share it
    uint32_t it_base = 0;
    bool ok = true;
    for (uint32_t k = 0;; ++k) {
        const int u = uq_consume(uq, k, C::kWarps * 32, p.err, ok);
        if (u < 0) break;
        const int qs = k % C::kQSlots;
        if (ok) ok = __all_sync(kFullWarp, mbar_wait(&q_full[qs], (k / C::kQSlots) & 1, p.err));
        const int4 mt = meta[qs];
        const int seq = mt.x, split = mt.y, ctx = mt.z, kvh = mt.w;
        const int b0 = split * kSplitBlocks;
        const int nb = ok ? min(kSplitBlocks, (ctx + kBlockTokens - 1) / kBlockTokens - b0) : 0;

        // q as the B operand of S = K q^T: head g, dims 16 kb + 4 t .. + 3 (the
        // k index of the product is permuted the same way on the K side)
        const __nv_bfloat16* qsm = reinterpret_cast<const __nv_bfloat16*>(qbuf + qs * C::kQBytes);
        float qv[KB][4];
        float amax = 0.f;
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            uint2 w = make_uint2(0u, 0u);
            if (g < G) w = *reinterpret_cast<const uint2*>(qsm + g * D + 16 * kb + 4 * t);
            qv[kb][0] = __uint_as_float(w.x << 16);
            qv[kb][1] = __uint_as_float(w.x & 0xffff0000u);
            qv[kb][2] = __uint_as_float(w.y << 16);
            qv[kb][3] = __uint_as_float(w.y & 0xffff0000u);
#pragma unroll
            for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(qv[kb][i]));
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullWarp, amax, off));
        // shift e: amax * 2^-e in [2^14, 2^15), exact in f16
        const int e = max(int(__float_as_uint(amax) >> 23) - 141, -100);
        const float down = exp2i(-e);
        const float qf = exp2i(e) * p.scale_log2;
        uint32_t qb[KB][2];
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            qb[kb][0] = pack_f16x2(qv[kb][0] * down, qv[kb][1] * down);
            qb[kb][1] = pack_f16x2(qv[kb][2] * down, qv[kb][3] * down);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_empty[qs]);   // this warp is done with the slot

        // running state: heads 2t and 2t + 1 (m, per-lane partial l), O^T fragments
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        int ev = 0;                                   // largest V-scale exponent seen (biased)
        float o[KB][4];
#pragma unroll
        for (int mb = 0; mb < KB; ++mb)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[mb][i] = 0.f;

        for (int jb = warp; jb < nb; jb += C::kWarps) {
            const uint32_t it = it_base + jb;
            const int st = it % C::kStages;
            if (ok) ok = __all_sync(kFullWarp, mbar_wait(&full[st], (it / C::kStages) & 1, p.err));
            if (!ok) continue;
            const unsigned char* sb = smem + size_t(st) * C::kStageBytes;
            const unsigned char* kt = sb;
            const unsigned char* vt = sb + C::kTileBytes;
            const float* ksc = reinterpret_cast<const float*>(kt + C::kCodeBytes);
            const float* vsc = reinterpret_cast<const float*>(vt + C::kCodeBytes);
            const int nvalid = min(kBlockTokens, ctx - (b0 + jb) * kBlockTokens);

            // S = K q^T: rows tokens g, g + 8; columns heads 2t, 2t + 1
            float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                const int off = ((kb ^ ksw) << 4) + 4 * t;
                const uint32_t u0 = *reinterpret_cast<const uint32_t*>(kt + g * D + off);
                const uint32_t u1 = *reinterpret_cast<const uint32_t*>(kt + (g + 8) * D + off);
                uint32_t a0, a1, a2, a3;
                codes_to_f16x2(u0, a0, a2);
                codes_to_f16x2(u1, a1, a3);
                mma_f16(sacc, a0, a1, a2, a3, qb[kb][0], qb[kb][1]);
            }
            const bool val0 = g < nvalid, val1 = g + 8 < nvalid;
            const float kq0 = ksc[g] * qf, kq1 = ksc[g + 8] * qf;
            const float s0 = val0 ? sacc[0] * kq0 : -INFINITY;
            const float s1 = val0 ? sacc[1] * kq0 : -INFINITY;
            const float s2 = val1 ? sacc[2] * kq1 : -INFINITY;
            const float s3 = val1 ? sacc[3] * kq1 : -INFINITY;
            float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(kFullWarp, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(kFullWarp, mx1, off));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
            const float p2 = exp2f(s2 - mn0), p3 = exp2f(s3 - mn1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);

            // V scales of the valid tokens; the running exponent keeps P' < 2
            const float vs0 = val0 ? vsc[g] : 0.f, vs1 = val1 ? vsc[g + 8] : 0.f;
            float vm = fmaxf(vs0, vs1);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) vm = fmaxf(vm, __shfl_xor_sync(kFullWarp, vm, off));
            const int ev_new = max(ev, min(int(__float_as_uint(vm) >> 23), 253));
            const float shift = exp2i(max(ev - ev_new, -126));
            ev = ev_new;
            const float fv = exp2i(127 - ev);
            const float2 ao = make_float2(al0 * shift, al1 * shift);

            // P' (f16) through shared memory into the B-operand layout [head][token]
            pb[(2 * t) * kBlockTokens + g] = __half_as_ushort(__float2half_rn(p0 * vs0 * fv));
            pb[(2 * t + 1) * kBlockTokens + g] = __half_as_ushort(__float2half_rn(p1 * vs0 * fv));
            pb[(2 * t) * kBlockTokens + g + 8] = __half_as_ushort(__float2half_rn(p2 * vs1 * fv));
            pb[(2 * t + 1) * kBlockTokens + g + 8] = __half_as_ushort(__float2half_rn(p3 * vs1 * fv));
            __syncwarp();
            // head g, tokens 4t .. 4t + 3 (the PV product's k index, permuted as on the V side)
            const uint2 bp = *reinterpret_cast<const uint2*>(pb + g * kBlockTokens + 4 * t);

            // O^T = diag-scaled O^T + V^T P': rows dims 16 mb + g, + 8; columns heads 2t, 2t + 1.
            // The rescale is skipped when every lane's factors are exactly 1 (the
            // running max and the V-scale exponent unchanged): the same bits.
            if (__any_sync(kFullWarp, ao.x != 1.f || ao.y != 1.f)) {
#pragma unroll
                for (int mb = 0; mb < KB; ++mb) {
                    const float2 lo = __fmul2_rn(make_float2(o[mb][0], o[mb][1]), ao);
                    const float2 hi = __fmul2_rn(make_float2(o[mb][2], o[mb][3]), ao);
                    o[mb][0] = lo.x;
                    o[mb][1] = lo.y;
                    o[mb][2] = hi.x;
                    o[mb][3] = hi.y;
                }
            }
#pragma unroll
            for (int mb = 0; mb < KB; ++mb) {
                const uint32_t u0 =
                    *reinterpret_cast<const uint32_t*>(vt + (16 * mb + g) * kBlockTokens + 4 * t);
                const uint32_t u1 = *reinterpret_cast<const uint32_t*>(
                    vt + (16 * mb + g + 8) * kBlockTokens + 4 * t);
                uint32_t a0, a1, a2, a3;
                codes_to_f16x2(u0, a0, a2);
                codes_to_f16x2(u1, a1, a3);
                mma_f16(o[mb], a0, a1, a2, a3, bp.x, bp.y);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        it_base += nb;

        // ---- combine the consumer warps' states ----
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(kFullWarp, l0, off);
            l1 += __shfl_xor_sync(kFullWarp, l1, off);
        }
        const float inv_fv = ev > 0 ? __uint_as_float(uint32_t(ev) << 23) : 0.f;   // 2^(ev - 127)
        float* rec = comb + warp * C::kComb;
        const int h0 = 2 * t, h1 = 2 * t + 1;
#pragma unroll
        for (int mb = 0; mb < KB; ++mb) {
            if (h0 < G) {
                rec[h0 * D + 16 * mb + g] = o[mb][0] * inv_fv;
                rec[h0 * D + 16 * mb + g + 8] = o[mb][2] * inv_fv;
            }
            if (h1 < G) {
                rec[h1 * D + 16 * mb + g] = o[mb][1] * inv_fv;
                rec[h1 * D + 16 * mb + g + 8] = o[mb][3] * inv_fv;
            }
        }
        if (g == 0) {
            if (h0 < G) {
                rec[G * D + h0] = m0;
                rec[G * D + G + h0] = l0;
            }
            if (h1 < G) {
                rec[G * D + h1] = m1;
                rec[G * D + G + h1] = l1;
            }
        }
        consumer_sync(C::kWarps * 32);
        const int nsplit = (ctx + kSplitTokens - 1) / kSplitTokens;
        // (a failed wait leaves the unit's description unknown: write nothing)
        for (int idx = threadIdx.x; ok && idx < G * D; idx += C::kWarps * 32) {
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
                const uint64_t keep = l2_evict_last_policy();
                st_keep(p.part_o + slot * D + d, O, keep);
                if (d == 0) st_keep(p.part_ml + slot, make_float2(M, L), keep);
            }
        }
        consumer_sync(C::kWarps * 32);
    }
}

bool aligned(const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; }

template <int D, int G>
int launch_i8(const AttnArgs& a, const unsigned char* kvp) {
    using C = I8Cfg<D, G>;
    auto kern = decode_split_int8_kernel<D, G>;
    const int per_sm = kernel_occupancy<decode_split_int8_kernel<D, G>>(C::kThreads, C::kSmem);
    if (per_sm < 1) return PKV_ERR_CUDA;
    const int64_t bound = int64_t(a.num_seqs) * a.ws.max_splits * a.desc->num_kv_heads;
    const int64_t grid = std::min<int64_t>(int64_t(num_sms()) * per_sm, bound);
    if (grid < 1) return PKV_OK;
    SplitI8Params p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.kv_pool = kvp;
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

template <int D>
int launch_i8_d(const AttnArgs& a, int g, const unsigned char* kvp) {
    switch (g) {
        case 1: return launch_i8<D, 1>(a, kvp);
        case 2: return launch_i8<D, 2>(a, kvp);
        case 4: return launch_i8<D, 4>(a, kvp);
        case 8: return launch_i8<D, 8>(a, kvp);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int paged_kv_append_int8(const void* k, const void* v, const int64_t* slot_mapping,
                                    int32_t num_tokens, void* kv_pool,
                                    const pkv_cache_desc* desc, void* stream) {
    if (!desc) return PKV_ERR_INVALID;
    if (desc->dtype != PKV_INT8) return PKV_ERR_UNSUPPORTED;
    pkv_cache_desc bd = *desc;
    bd.dtype = PKV_BF16;
    int st = check_desc(&bd, false);
    if (st != PKV_OK) return st;
    if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (desc->block_size != kBlockTokens) return PKV_ERR_UNSUPPORTED;   // the tile layout is 16 rows
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !kv_pool) return PKV_ERR_INVALID;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(kv_pool, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID;
    int* err = device_error_ptr(&st);
    if (st != PKV_OK) return st;
    AppendI8Params p;
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.slots = slot_mapping;
    p.kv_pool = static_cast<unsigned char*>(kv_pool);
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

extern "C" int paged_attention_decode_int8(void* out, const void* q, const void* kv_pool,
                                           const pkv_cache_desc* desc,
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
    if (!out || !q || !kv_pool || !block_tables || !context_lens) return PKV_ERR_INVALID;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(kv_pool, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
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
    const auto* kvp = static_cast<const unsigned char*>(kv_pool);
    st = qd.head_dim == 128 ? launch_i8_d<128>(a, g, kvp) : launch_i8_d<64>(a, g, kvp);
    if (st != PKV_OK) return st;
    return launch_decode_merge(a);
}
