// Decode split kernel for grouped-query attention (group size 2, 4 or 8), bf16.
//
// Same work units, pipeline and result as decode_split_kernel in decode.cu
// (exact softmax(q K^T * scale) V over a 512-token split, online recurrence of
// "第 15 章：推理引擎与部署" §15.1 算法详解 over 16-key blocks, G query heads of
// one KV head per unit, "大模型部署.md" §4.1 4. MQA 与 GQA).  What changes is
// how a block is multiplied.  With G query heads sharing a KV head, both
// products of a block are small dense contractions:
//   S = Q K^T   (G x D) . (D x 16)      O += P V   (G x 16) . (16 x D)
// On CUDA cores the per-lane dot products need a warp-wide reduction per
// (head, key) and the kernel becomes issue-bound as G grows; here each is a
// handful of warp-level tensor-core instructions (mma.sync m16n8k16, bf16 in,
// fp32 accumulate; rows G..15 of the 16-row tile are zero padding), so the
// kernel stays bound by HBM.
//
// K and V tiles are fetched with TMA tensor copies that land 128-byte swizzled,
// so the ldmatrix reads that build the tensor-core fragments are free of bank
// conflicts.  Rows of a partial last block are zeroed in shared memory before
// the PV product (never-written cache rows may hold anything; 0 x NaN = NaN).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "launch_cache.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

struct MmaParams {
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
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

template <int D, int G>
struct MmaCfg {
    static constexpr int kWarps = 4;
    static constexpr int kThreads = (kWarps + 1) * 32;
    static constexpr int kHalves = D / 64;                 // 64-dim boxes per tile
    static constexpr int kTileBytes = kBlockTokens * D * 2;
    static constexpr int kStageBytes = 2 * kTileBytes;
    // 12 stages at 2 CTAs per SM: 192 KB of tiles in flight per SM (measured
    // 0.5 % faster than 8 stages for g = 4).  For g = 8 the consumer warps
    // combine through two records instead of four to make room.
    static constexpr int kStages = 12;
    static constexpr int kMinBlocks = G == 8 ? 2 : 1;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kComb = G * (D + 2);
    static constexpr int kCombRecords = G == 8 ? 2 : kWarps;
    static constexpr int kCombOff = kRingBytes;
    static constexpr int kQBytes = G * D * 2;               // q of one unit (bf16)
    static constexpr int kQSlots = 2;                       // units whose q is in flight
    static constexpr int kQOff = kCombOff + kCombRecords * kComb * 4;
    static constexpr int kMetaOff = kQOff + kQSlots * kQBytes;
    static constexpr int kBarOff = kMetaOff + kQSlots * 32;
    // full[kStages], empty[kStages], q_full[kQSlots], q_empty[kQSlots]
    static constexpr int kQueueOff = kBarOff + (2 * kStages + 2 * kQSlots) * 8;
    static constexpr int kSmem = kQueueOff + int(sizeof(UnitQueue)) + 1024;  // + alignment slack
    static_assert(G == 2 || G == 4 || G == 8, "group size");
    // a consumer warp waits on a stage by parity: its previous use must be the
    // same warp's own tile (tiles of a unit go to warps round-robin)
    static_assert(kStages % kWarps == 0, "stage ring must be a multiple of the consumer warps");
};

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// d += a (16x16, rows gid / gid+8) . b (16x8); rows 8..15 of a are zero here
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// shared address of 16-byte chunk `c` (0..D/8-1) of token row `t` in a swizzled tile
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int t, int c) {
    return tile + uint32_t((c >> 3) * (kBlockTokens * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Combine of a plain unit's four consumer-warp states for groups of 8 (every
// row of the tile's top half is a query head, so each lane holds the whole
// state of its row for its columns): warps 2 and 3 hand their states to warps
// 0 and 1 through two records, warp 1 hands the merged state to warp 0, and
// warp 0 writes the unit's split partials or outputs.  Two records instead of
// four leave shared memory for a deeper tile ring.
template <int D>
__device__ __forceinline__ void combine_pairwise(const MmaParams& p, float* comb,
                                                 float (&o)[D / 8][4], float& m_row,
                                                 float& l_row, bool ok, int nsplit, int seq,
                                                 int qrow, int split, int kvh) {
    using C = MmaCfg<D, 8>;
    constexpr int G = 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    auto put = [&](float* rec) {
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<float2*>(rec + gid * D + n * 8 + 2 * tig) =
                make_float2(o[n][0], o[n][1]);
        if (tig == 0) {
            rec[G * D + gid] = m_row;
            rec[G * D + G + gid] = l_row;
        }
    };
    auto merge = [&](const float* rec) {
        const float m2 = rec[G * D + gid], l2 = rec[G * D + G + gid];
        const float M = fmaxf(m_row, m2);
        const float Mx = M == -INFINITY ? 0.f : M;    // both states empty: stay empty
        const float s1 = exp2f(m_row - Mx), s2 = exp2f(m2 - Mx);
        l_row = fmaf(l2, s2, l_row * s1);
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            const float2 v = *reinterpret_cast<const float2*>(rec + gid * D + n * 8 + 2 * tig);
            o[n][0] = fmaf(v.x, s2, o[n][0] * s1);
            o[n][1] = fmaf(v.y, s2, o[n][1] * s1);
        }
        m_row = M;
    };
    if (warp >= 2) put(comb + (warp - 2) * C::kComb);
    asm volatile("bar.sync 1, %0;" ::"r"(C::kWarps * 32) : "memory");
    if (warp < 2) merge(comb + warp * C::kComb);
    asm volatile("bar.sync 1, %0;" ::"r"(C::kWarps * 32) : "memory");
    if (warp == 1) put(comb);
    asm volatile("bar.sync 1, %0;" ::"r"(C::kWarps * 32) : "memory");
    if (warp != 0) return;
    merge(comb);
    // (a failed wait leaves the unit's description unknown: write nothing)
    if (!ok) return;
    const int Hq = p.num_q_heads;
    const int h = kvh * G + gid;
    if (nsplit == 1) {
        __nv_bfloat16* dst = p.out + (size_t(qrow) * Hq + h) * D + 2 * tig;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<__nv_bfloat162*>(dst + n * 8) =
                __floats2bfloat162_rn(o[n][0] / l_row, o[n][1] / l_row);
    } else {
        const uint64_t keep = l2_evict_last_policy();
        const size_t slot = (size_t(seq) * Hq + h) * p.max_splits + split;
        float* dst = p.part_o + slot * D + 2 * tig;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            st_keep(reinterpret_cast<float2*>(dst + n * 8), make_float2(o[n][0], o[n][1]), keep);
        if (tig == 0) st_keep(p.part_ml + slot, make_float2(m_row, l_row), keep);
    }
}

// Rows gid (R = 0) or gid + 8 (R = 1) of a grouped split's accumulators: query
// head h of sequence s, as its split partial, or as its output when the split
// is the sequence's only one.
template <int D, int R>
__device__ __forceinline__ void grouped_write(const MmaParams& p, const float (&o)[D / 8][4], int s,
                                              int h, int split, float m_row, float l_row) {
    const int tig = threadIdx.x & 3;
    const int Hq = p.num_q_heads;
    const int nsplit = (p.context_lens[s] - 1) / kSplitTokens + 1;
    if (nsplit == 1) {
        __nv_bfloat16* dst = p.out + (size_t(s) * Hq + h) * D + 2 * tig;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<__nv_bfloat162*>(dst + n * 8) =
                __floats2bfloat162_rn(o[n][2 * R] / l_row, o[n][2 * R + 1] / l_row);
    } else {
        const uint64_t keep = l2_evict_last_policy();
        const size_t slot = (size_t(s) * Hq + h) * p.max_splits + split;
        float* dst = p.part_o + slot * D + 2 * tig;
#pragma unroll
        for (int n = 0; n < D / 8; ++n)
            st_keep(reinterpret_cast<float2*>(dst + n * 8),
                    make_float2(o[n][2 * R], o[n][2 * R + 1]), keep);
        if (tig == 0) st_keep(p.part_ml + slot, make_float2(m_row, l_row), keep);
    }
}

// One complete 512-token split that `count` consecutive sequences from `first`
// read block for block (groups of 8 query heads).  Every tile of the split is
// loaded once and read by all four consumer warps; warp w takes sequences
// first + 2w (tile rows 0..7, its eight query heads) and first + 2w + 1 (rows
// 8..15, the rows a single sequence leaves empty), with a running max and sum
// per row over all the split's tiles in order, and writes their split
// partials, or their outputs when the split is a sequence's only one.
template <int D>
__device__ __forceinline__ void grouped_split(const MmaParams& p, uint32_t base, uint64_t* full,
                                              uint64_t* empty, uint32_t it_base, int nb,
                                              int first, int count, int split, int kvh,
                                              bool& ok) {
    using C = MmaCfg<D, 8>;
    constexpr int G = 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int Hq = p.num_q_heads;
    const int active = (count + 1) / 2;                // warps with members
    const bool act = warp < active, has_b = 2 * warp + 1 < count;
    const int sa = first + 2 * warp, sb = has_b ? sa + 1 : sa;
    if (!act) return;   // warp 0 releases each tile for the warps without members

    // q fragments (A operand): rows gid from sequence sa, rows gid + 8 from sb
    uint32_t qa0[D / 16], qa1[D / 16], qa2[D / 16], qa3[D / 16];
    {
        const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q);
        const uint32_t* ra = q32 + (size_t(sa) * Hq + kvh * G + gid) * (D / 2);
        const uint32_t* rb = q32 + (size_t(sb) * Hq + kvh * G + gid) * (D / 2);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa0[ks] = ra[ks * 8 + tig];
            qa2[ks] = ra[ks * 8 + 4 + tig];
            qa1[ks] = has_b ? rb[ks * 8 + tig] : 0u;
            qa3[ks] = has_b ? rb[ks * 8 + 4 + tig] : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
    const uint32_t release = warp == 0 ? 1 + C::kWarps - active : 1;

    for (int jb = 0; jb < nb; ++jb) {
        const uint32_t it = it_base + jb;
        const int st = it % C::kStages;
        if (ok) ok = __all_sync(kFullMask, mbar_wait(&full[st], (it / C::kStages) & 1, p.err));
        if (!ok) continue;
        const uint32_t kt = base + st * C::kStageBytes;
        const uint32_t vt = kt + C::kTileBytes;

        // S = q K^T for both sequences' rows: two 8-key column tiles
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int mi = lane >> 3;
            const int t = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(tile_addr(kt, t, ks * 2 + (mi & 1)), r0, r1, r2, r3);
                mma16816(s0, qa0[ks], qa1[ks], qa2[ks], qa3[ks], r0, r1);
                mma16816(s1, qa0[ks], qa1[ks], qa2[ks], qa3[ks], r2, r3);
            }
        }
        // row gid (sa): keys 2tig, 2tig+1 (s0[0..1]) and 8+2tig, 9+2tig (s1[0..1]);
        // row gid + 8 (sb): the same keys in s0[2..3], s1[2..3].  Every key is valid.
        float va[4] = {s0[0], s0[1], s1[0], s1[1]};
        float vb[4] = {s0[2], s0[3], s1[2], s1[3]};
        float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            va[i] *= p.scale_log2;
            vb[i] *= p.scale_log2;
            xa = fmaxf(xa, va[i]);
            xb = fmaxf(xb, vb[i]);
        }
        xa = fmaxf(xa, __shfl_xor_sync(kFullMask, xa, 1));
        xb = fmaxf(xb, __shfl_xor_sync(kFullMask, xb, 1));
        xa = fmaxf(xa, __shfl_xor_sync(kFullMask, xa, 2));
        xb = fmaxf(xb, __shfl_xor_sync(kFullMask, xb, 2));
        const float na = fmaxf(ma, xa), nb2 = fmaxf(mb, xb);
        const float aa = exp2f(ma - na), ab = exp2f(mb - nb2);
        float pa[4], pb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            pa[i] = exp2f(va[i] - na);
            pb[i] = exp2f(vb[i] - nb2);
        }
        la = la * aa + (pa[0] + pa[1]) + (pa[2] + pa[3]);
        lb = lb * ab + (pb[0] + pb[1]) + (pb[2] + pb[3]);
        if (__any_sync(kFullMask, aa != 1.f || ab != 1.f)) {
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] *= aa;
                o[n][1] *= aa;
                o[n][2] *= ab;
                o[n][3] *= ab;
            }
        }
        ma = na;
        mb = nb2;

        // O += P V with both sequences' rows of P as the A operand
        const uint32_t p0 = pack2(pa[0], pa[1]), p1 = pack2(pb[0], pb[1]);
        const uint32_t p2 = pack2(pa[2], pa[3]), p3 = pack2(pb[2], pb[3]);
        {
            const int mi = lane >> 3;
            const int t = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
            for (int pr2 = 0; pr2 < D / 16; ++pr2) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(tile_addr(vt, t, pr2 * 2 + (mi >> 1)), r0, r1, r2, r3);
                mma16816(o[2 * pr2], p0, p1, p2, p3, r0, r1);
                mma16816(o[2 * pr2 + 1], p0, p1, p2, p3, r2, r3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cnt(&empty[st], release);
    }
    if (!ok) return;

    // per-row sums over the quad, then each sequence's partial (or output)
    la += __shfl_xor_sync(kFullMask, la, 1);
    lb += __shfl_xor_sync(kFullMask, lb, 1);
    la += __shfl_xor_sync(kFullMask, la, 2);
    lb += __shfl_xor_sync(kFullMask, lb, 2);
    grouped_write<D, 0>(p, o, sa, kvh * G + gid, split, ma, la);
    if (has_b) grouped_write<D, 1>(p, o, sb, kvh * G + gid, split, mb, lb);
}

template <int D, int G>
__global__ void __launch_bounds__(MmaCfg<D, G>::kThreads, MmaCfg<D, G>::kMinBlocks)
    decode_split_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, MmaParams p) {
    using C = MmaCfg<D, G>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* smem = smem_raw + (base - raw);
    float* comb = reinterpret_cast<float*>(smem + C::kCombOff);
    unsigned char* qbuf = smem + C::kQOff;
    int4* meta = reinterpret_cast<int4*>(smem + C::kMetaOff);   // [slot][2]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* empty = full + C::kStages;
    uint64_t* q_full = empty + C::kStages;
    uint64_t* q_empty = q_full + C::kQSlots;
    UnitQueue* uq = reinterpret_cast<UnitQueue*>(smem + C::kQueueOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            // a tile is released by its consumer warp, which arrives for all of
            // them, or (grouped units) by every consumer warp once
            mbar_init(&empty[s], C::kWarps);
        }
        for (int s = 0; s < C::kQSlots; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], C::kWarps);
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
            const int grouped = item.y >> kItemSplitBits;   // sequences reading this split
            // (a grouped split is complete for every member: the first one's table serves all)
            const SplitSpan sp = split_span(ctx, item.y & kItemSplitMask, p.window);
            const int b0 = sp.begin;
            const int nb = max(0, sp.end - b0);
            int my_blk = 0;
            if (lane < nb) my_blk = p.block_tables[size_t(item.x) * p.table_stride + b0 + lane];
            // the unit's description and q, so the consumers start without global loads
            const int qs = k % C::kQSlots;
            ok = __all_sync(kFullMask, mbar_wait(&q_empty[qs], ((k / C::kQSlots) & 1) ^ 1, p.err));
            if (!ok) break;
            if (lane == 0) {
                const int qrow = p.query_start_loc ? p.query_start_loc[item.x] : item.x;
                meta[2 * qs] = make_int4(item.x, item.y, ctx, kvh);
                meta[2 * qs + 1] = make_int4(qrow, 0, 0, 0);
                if (grouped) {
                    mbar_arrive(&q_full[qs]);   // each consumer warp loads its members' q
                } else {
                    mbar_arrive_expect_tx(&q_full[qs], C::kQBytes);
                    bulk_g2s(qbuf + qs * C::kQBytes, p.q + (size_t(qrow) * Hq + kvh * G) * D,
                             C::kQBytes, &q_full[qs]);
                }
            }
            __syncwarp();
            for (int j = 0; j < nb; ++j, ++it) {
                const int blk = __shfl_sync(kFullMask, my_blk, j);
                const int st = it % C::kStages;
                ok = __all_sync(kFullMask, mbar_wait(&empty[st], ((it / C::kStages) & 1) ^ 1, p.err));
                if (!ok) break;
                if (lane == 0) {
                    if (blk < 0 || blk >= p.num_blocks) {
                        flag_error(p.err, PKV_DEV_BAD_BLOCK_ID);
                        mbar_arrive(&full[st]);
                    } else {
                        mbar_arrive_expect_tx(&full[st], C::kStageBytes);
                        const uint32_t dst = base + st * C::kStageBytes;
                        const int row = (blk * Hkv + kvh) * kBlockTokens;
#pragma unroll
                        for (int h = 0; h < C::kHalves; ++h) {
                            tma_2d(dst + h * kBlockTokens * 128, &tmap_k, h * 64, row, &full[st]);
                            tma_2d(dst + C::kTileBytes + h * kBlockTokens * 128, &tmap_v, h * 64,
                                   row, &full[st]);
                        }
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
    const int gid = lane >> 2, tig = lane & 3;
    uint32_t it_base = 0;
    bool ok = true;
    for (uint32_t k = 0;; ++k) {
        const int u = uq_consume(uq, k, C::kWarps * 32, p.err, ok);
        if (u < 0) break;
        const int qs = k % C::kQSlots;
        if (ok) ok = __all_sync(kFullMask, mbar_wait(&q_full[qs], (k / C::kQSlots) & 1, p.err));
        const int4 mt = meta[2 * qs];
        const int seq = mt.x, split = mt.y & kItemSplitMask, ctx = mt.z, kvh = mt.w;
        const int qrow = meta[2 * qs + 1].x;
        const SplitSpan sp = split_span(ctx, split, p.window);
        const int b0 = sp.begin;
        const int nb = ok ? max(0, sp.end - b0) : 0;
        if constexpr (G == 8) {
            const int grouped = mt.y >> kItemSplitBits;
            if (grouped) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&q_empty[qs]);
                grouped_split<D>(p, base, full, empty, it_base, nb, seq, grouped, split, kvh, ok);
                it_base += nb;
                continue;
            }
        }

        // q fragments (A operand): row gid = query head gid of the group, rows >= G zero
        uint32_t qa0[D / 16], qa2[D / 16];
        {
            const uint32_t* qh = reinterpret_cast<const uint32_t*>(qbuf + qs * C::kQBytes) +
                                 (gid < G ? gid : 0) * (D / 2);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                qa0[ks] = gid < G ? qh[ks * 8 + tig] : 0u;
                qa2[ks] = gid < G ? qh[ks * 8 + 4 + tig] : 0u;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_empty[qs]);   // this warp is done with the slot
        float o[D / 8][4];
#pragma unroll
        for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m_row = -INFINITY, l_part = 0.f;

        for (int jb = warp; jb < nb; jb += C::kWarps) {
            const uint32_t it = it_base + jb;
            const int st = it % C::kStages;
            if (ok) ok = __all_sync(kFullMask, mbar_wait(&full[st], (it / C::kStages) & 1, p.err));
            if (!ok) continue;
            const uint32_t kt = base + st * C::kStageBytes;
            const uint32_t vt = kt + C::kTileBytes;
            const int nvalid = min(kBlockTokens, ctx - (b0 + jb) * kBlockTokens);
            // keys below the window's first key (its block only) are masked
            const int fvalid = b0 + jb == sp.lo / kBlockTokens ? sp.lo % kBlockTokens : 0;

            // ---- S = q K^T: two 8-key column tiles ----
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const int mi = lane >> 3;
                const int t = ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(tile_addr(kt, t, ks * 2 + (mi & 1)), r0, r1, r2, r3);
                    mma16816(s0, qa0[ks], 0u, qa2[ks], 0u, r0, r1);
                    mma16816(s1, qa0[ks], 0u, qa2[ks], 0u, r2, r3);
                }
            }
            // this thread's row gid holds keys 2tig, 2tig+1 (s0) and 8+2tig, 9+2tig (s1)
            float v[4] = {s0[0], s0[1], s1[0], s1[1]};
            const int key[4] = {2 * tig, 2 * tig + 1, 8 + 2 * tig, 9 + 2 * tig};
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[i] = key[i] < nvalid && key[i] >= fvalid ? v[i] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, v[i]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
            const float m_new = fmaxf(m_row, mx);
            const float alpha = exp2f(m_row - m_new);
            float pr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pr[i] = exp2f(v[i] - m_new);
            l_part = l_part * alpha + (pr[0] + pr[1]) + (pr[2] + pr[3]);
            if (__any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    o[n][0] *= alpha;
                    o[n][1] *= alpha;
                }
            }
            m_row = m_new;

            // zero V rows past the context (partial last block) and below the
            // window's first key before PV reads them
            if (nvalid < kBlockTokens || fvalid > 0) {
                const int nz = (kBlockTokens - nvalid + fvalid) * (D / 8);
                for (int i = lane; i < nz; i += 32) {
                    const int z = i / (D / 8), c = i % (D / 8);
                    const int t = z < fvalid ? z : nvalid + (z - fvalid);
                    const uint32_t a = tile_addr(vt, t, c);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0)
                                 : "memory");
                }
                __syncwarp();
            }

            // ---- O += P V: P is the S tile in bf16, reused as the A operand ----
            const uint32_t pa0 = pack2(pr[0], pr[1]), pa2 = pack2(pr[2], pr[3]);
            {
                const int mi = lane >> 3;
                const int t = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                for (int pr2 = 0; pr2 < D / 16; ++pr2) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(tile_addr(vt, t, pr2 * 2 + (mi >> 1)), r0, r1, r2, r3);
                    mma16816(o[2 * pr2], pa0, 0u, pa2, 0u, r0, r1);
                    mma16816(o[2 * pr2 + 1], pa0, 0u, pa2, 0u, r2, r3);
                }
            }
            if (nvalid < kBlockTokens || fvalid > 0) fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive_cnt(&empty[st], C::kWarps);
        }
        it_base += nb;

        // ---- combine the consumer warps ----
        float l_row = l_part;
        l_row += __shfl_xor_sync(kFullMask, l_row, 1);
        l_row += __shfl_xor_sync(kFullMask, l_row, 2);
        if constexpr (G == 8) {
            combine_pairwise<D>(p, comb, o, m_row, l_row, ok, sp.nsplit, seq, qrow, split, kvh);
            continue;
        }
        float* rec = comb + warp * C::kComb;
        if (gid < G) {
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                rec[gid * D + n * 8 + 2 * tig] = o[n][0];
                rec[gid * D + n * 8 + 2 * tig + 1] = o[n][1];
            }
            if (tig == 0) {
                rec[G * D + gid] = m_row;
                rec[G * D + G + gid] = l_row;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(C::kWarps * 32) : "memory");
        const int nsplit = sp.nsplit;
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
                p.out[(size_t(qrow) * Hq + h) * D + d] = __float2bfloat16_rn(O / L);
            } else {
                const size_t slot = (size_t(seq) * Hq + h) * p.max_splits + split;
                const uint64_t keep = l2_evict_last_policy();
                st_keep(p.part_o + slot * D + d, O, keep);
                if (d == 0) st_keep(p.part_ml + slot, make_float2(M, L), keep);
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(C::kWarps * 32) : "memory");
    }
    // a preceding prefill kernel overlapped this grid: finish only after it has
    if (threadIdx.x == 0) pdl_wait_prerequisites();
}

template <int D, int G>
int launch_t(const AttnArgs& a) {
    using C = MmaCfg<D, G>;
    auto kern = decode_split_mma_kernel<D, G>;
    CUtensorMap mk, mv;
    if (!make_cache_tensor_map(&mk, a.k_cache, a.desc) ||
        !make_cache_tensor_map(&mv, a.v_cache, a.desc))
        return PKV_ERR_CUDA;
    const int per_sm = kernel_occupancy<decode_split_mma_kernel<D, G>>(C::kThreads, C::kSmem);
    if (per_sm < 1) return PKV_ERR_CUDA;
    const int64_t bound = int64_t(a.num_seqs) * a.ws.max_splits * a.desc->num_kv_heads;
    const int64_t grid = std::min<int64_t>(int64_t(num_sms()) * per_sm, bound);
    if (grid < 1) return PKV_OK;
    MmaParams p;
    p.q = static_cast<const __nv_bfloat16*>(a.q);
    p.out = static_cast<__nv_bfloat16*>(a.out);
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
    return cuda_status(cudaLaunchKernelEx(&cfg, kern, mk, mv, p));
}

template <int D>
int launch_d(const AttnArgs& a, int g) {
    switch (g) {
        case 2: return launch_t<D, 2>(a);
        case 4: return launch_t<D, 4>(a);
        case 8: return launch_t<D, 8>(a);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace

bool decode_mma_eligible(const pkv_cache_desc* d) {
    const int g = d->num_q_heads / d->num_kv_heads;
    return d->dtype == PKV_BF16 && (d->head_dim == 64 || d->head_dim == 128) &&
           d->block_size == kBlockTokens && (g == 2 || g == 4 || g == 8) &&
           int64_t(d->num_blocks) * d->num_kv_heads * kBlockTokens < (int64_t(1) << 31);
}

int launch_decode_split_mma(const AttnArgs& a) {
    const int g = a.desc->num_q_heads / a.desc->num_kv_heads;
    return a.desc->head_dim == 128 ? launch_d<128>(a, g) : launch_d<64>(a, g);
}

}  // namespace pkv
