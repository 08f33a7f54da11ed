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
    // g = 8 runs 3 CTAs per SM on a 4-stage ring (measured faster on the
    // prefix-sharing batch); smaller groups run 12 stages at 2 CTAs per SM
    // (192 KB of tiles in flight per SM; measured 0.5 % faster than 8 stages)
    static constexpr int kStages = G == 8 ? 4 : 12;
    static constexpr int kMinBlocks = G == 8 ? 3 : 1;
    static constexpr int kRingBytes = kStages * kStageBytes;
    static constexpr int kComb = G * (D + 2);
    static constexpr int kCombOff = kRingBytes;
    static constexpr int kQBytes = G * D * 2;               // q of one unit (bf16)
    static constexpr int kQSlots = 2;                       // units whose q is in flight
    static constexpr int kQOff = kCombOff + kWarps * kComb * 4;
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
            const SplitSpan sp = split_span(ctx, item.y, p.window);
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
                mbar_arrive_expect_tx(&q_full[qs], C::kQBytes);
                bulk_g2s(qbuf + qs * C::kQBytes, p.q + (size_t(qrow) * Hq + kvh * G) * D, C::kQBytes,
                         &q_full[qs]);
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
        const int seq = mt.x, split = mt.y, ctx = mt.z, kvh = mt.w;
        const int qrow = meta[2 * qs + 1].x;
        const SplitSpan sp = split_span(ctx, split, p.window);
        const int b0 = sp.begin;
        const int nb = ok ? max(0, sp.end - b0) : 0;

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
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        it_base += nb;

        // ---- combine the consumer warps ----
        float l_row = l_part;
        l_row += __shfl_xor_sync(kFullMask, l_row, 1);
        l_row += __shfl_xor_sync(kFullMask, l_row, 2);
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
