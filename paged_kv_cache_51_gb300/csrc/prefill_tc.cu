// Prefill-chunk attention on the tcgen05 tensor cores (ragged mixed batches).
//
// What is computed: for a chunk of qlen new tokens of one sequence whose K/V
// are already appended after a cached prefix, query i attends causally to keys
// 0 .. ctx - qlen + i ("第 15 章：推理引擎与部署" §15.6 两阶段与 Chunked Prefill;
// "DeepSpeed-FastGen 深度解析" §3.2 动态分割融合).  Softmax is exact and is
// accumulated tile by tile with the online recurrence of §15.1 算法详解
// (running max m, running sum l, O rescaled by alpha), in base 2.
//
// With a sliding window of W keys ("大模型部署.md" §2.1 block_sliding_window;
// the reading taken: a query sees its W most recent keys), query i sees keys
// max(0, a - W + 1) .. a, a = ctx - qlen + i, over a logically ordered table:
// a unit's key tiles start at the tile holding its first token's first key,
// each row masks the keys below its own window, and V rows below the first
// token's window in that tile are zeroed before P V (they belong to other
// tokens of the ring, or were never written).
//
// Both products are dense contractions, so they run on the 5th-generation
// tensor cores:
//   S = Q K^T   M = 128 query rows, N = 128 keys, K = 128 dims
//   O += P V    M = 128 query rows, N = 128 dims, K = 128 keys
// with bf16 operands (Q, K, V in shared memory, P in TMEM) and fp32
// accumulators in TMEM.
//
// Tile shapes.  A tile's 128 rows are 128/G tokens x the G query heads of one
// KV head (GQA packing, "大模型部署.md" §4.1 4. MQA 与 GQA), so every K/V byte
// staged is used by all G heads.  A key tile is 8 paged blocks (128 keys).
// Shared-memory operands use the 128-byte-swizzled K-major layout (Q, K) and
// the 128-byte swizzled MN-major layout (V); TMA tensor copies write K and V
// blocks straight into that layout, one (block, 64-dim half) box of 16 x 128 B
// per copy.
//
// Warp roles (384 threads, one CTA per SM, persistent over work units):
//   warps 0-7  softmax: two threads per query row, one per 64-key half of each
//              key tile (warps w and w + 4 hold the same rows).  A thread reads
//              its 64 scores from TMEM, masks them, exchanges its tile maximum
//              with the other half's thread through shared memory (both then
//              hold the same running max) and with that frees the S buffer for
//              the Q K^T two tiles on; it computes P (bf16) into a P buffer of
//              its own in TMEM and keeps a partial row sum.  The P V product reads
//              P from there and accumulates both halves into one O.  S and P
//              are double-buffered, so a Q K^T waits only until the softmax has
//              loaded the scores it overwrites, not until their P V has run,
//              and the softmax of the next key tile overlaps the previous
//              products.  O is rescaled (each thread its 64 dims) only when the
//              running max grows by more than 2^8, the one case that waits for
//              the previous P V.  The epilogue adds the halves' sums; a full
//              unit's bf16 output tile is staged in the unit's Q buffer (the
//              TMA box layout) and leaves by two TMA tensor stores, so the warps
//              go on to the next unit at once (128 rows of scattered 16-byte
//              global stores kept the load/store unit busy for ~3000 cycles);
//              warp 8 issues those stores before it reuses the buffer.  A
//              partial unit writes its valid rows directly.
//   warp 8     takes work units from a ticket (the planner orders them longest
//              first) and publishes them to the other roles; TMA producer for
//              the unit's Q tile (two buffers) and for K: blocks of each key
//              tile into a 2-stage K ring; a K stage is released as soon as its
//              Q K^T product is done; sends staged output tiles out by TMA
//   warp 9     TMA producer for V: a 2-stage V ring released by the P V product
//   warp 10    TMEM owner and Q K^T issuer (one thread issues tcgen05.mma)
//   warp 11    P V issuer (one thread)
//              A thread issuing tcgen05.mma is held for the length of each
//              product, and every instruction that another warp of its SM
//              sub-partition (warp index mod 4) issues meanwhile delays the
//              next product: measured with one issuing thread and busy warps
//              beside it, a 128 x 128 x 16 product takes 64 cycles alone, 79
//              beside two warps of TMEM loads and stores, 126 beside two warps
//              of FMAs, and 64 whatever runs on the other three
//              sub-partitions.  Each sub-partition holds two softmax warps (a
//              warp reads only its own quarter of TMEM's lanes), so the two
//              products go out from two sub-partitions (2 and 3), each carrying
//              half the issue work.  Tensor-core instructions of one thread run
//              in issue order, but two threads' need not: a Q K^T into an S
//              buffer waits until the softmax has loaded the scores it
//              replaces (two tiles earlier).  The pipe works on
//              Q K^T of tile q + 1 and P V of tile q - 1 while the softmax runs
//              on tile q (across units as well).
// Every wait is bounded; on a timeout the kernel records an error, stops
// issuing work, drains its copies and MMAs and frees TMEM before it returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "launch_cache.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kRows = 128;                   // query rows per tile
constexpr int kDim = 128;                    // head dim
constexpr int kKeys = 128;                   // keys per key tile
constexpr int kBlkPerTile = kKeys / kBlockTokens;  // 8 cache blocks
// Ring depths.  A key tile's TMA copies take about a microsecond to land, about
// one tile period: K and V run 2 deep.  Q is double-buffered so the next unit's
// Q is in place before its first Q K^T; a finished unit's Q buffer then holds
// its output tile until the TMA stores have read it.
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kQBufs = 2;
static_assert(kKStages == 2 && kVStages == 2,
              "the rings are released through the two S and P buffers' barriers");
constexpr int kSub = kRows * 128;            // one 64-column half of a 128-row operand (16 KiB)
constexpr int kQBytes = 2 * kSub;            // one Q tile: 2 halves (dims 0-63, 64-127)
constexpr int kKBytes = 2 * kKeys * 128;     // one K or V tile (2 halves of 128 key rows x 128 B)
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kQBufs * kQBytes;
constexpr int kVOff = kKOff + kKStages * kKBytes;
constexpr int kStatOff = kVOff + kVStages * kKBytes;  // l per half and row, 2 sets
constexpr int kXmOff = kStatOff + 2 * 2 * kRows * 4;  // tile maxima per half and row, 2 sets
constexpr int kBarOff = kXmOff + 2 * 2 * kRows * 4;
constexpr int kSmemBytes = kBarOff + 1024 + 1024;  // barriers, unit ring + 1 KiB alignment slack
constexpr int kSoftWarps = 8;
constexpr int kKProducerWarp = 8;
constexpr int kVProducerWarp = 9;
constexpr int kMmaWarp = 10;                 // TMEM owner, Q K^T issuer
constexpr int kPvWarp = 11;                  // P V issuer
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;          // S (2 x 128) + P (2 x 64) + O (128)
constexpr uint32_t kPCol = 256;              // P buffer b at kPCol + 64 b (bf16 pairs)
constexpr uint32_t kOCol = 384;              // O: 128 columns (fp32, one per dim)
constexpr float kRescaleThreshold = 8.0f;    // log2 units: rescale O only when max grows > 2^8
constexpr int kBoxBytes = kBlockTokens * 128;  // one TMA box: 16 rows x 64 bf16

// barrier indices
enum {
    B_K_FULL = 0,
    // A K stage is free once the Q K^T that read it has completed, and a V stage
    // once its P V has: with two K stages, two V stages and two S and two P
    // buffers, stage i of each ring belongs to the tiles of buffer i, so the
    // producers wait on B_S_FULL and B_O_DONE (the next phase of either needs a
    // tile the waiting producer has not loaded yet, so a wait cannot alias).
    B_V_FULL = B_K_FULL + kKStages,
    B_S_FULL = B_V_FULL + kVStages,
    B_S_EMPTY = B_S_FULL + 2,       // [S buffer]: every softmax warp has loaded its scores
    B_P_FULL = B_S_EMPTY + 2,       // [P buffer]: every softmax warp has written its P
    B_O_DONE = B_P_FULL + 2,        // [P buffer]: that buffer's P V has completed
    B_Q_FULL = B_O_DONE + 2,        // [Q buffer]
    B_Q_EMPTY = B_Q_FULL + kQBufs,  // [Q buffer]: every softmax warp has finished its unit's
                                    // epilogue (output staged there or written directly)
    B_U_READY = B_Q_EMPTY + kQBufs, // [unit slot]
    B_U_EMPTY = B_U_READY + 4,      // [unit slot]
    B_O_EMPTY = B_U_EMPTY + 4,
    B_STAT,                         // both halves' l of the current unit are published
    B_XM,                           // [lane quarter]: both halves' tile maxima are published
    B_DRAIN = B_XM + 4,             // the Q K^T issuer's products have completed
    B_DRAIN_PV,                     // the P V issuer's products have completed
    B_COUNT
};

// instruction descriptor, kind::f16: bf16 x bf16 -> fp32, M = 128, N = 128
constexpr uint32_t idesc_bf16(bool b_mn_major) {
    return (1u << 4)                        // D format: f32
           | (1u << 7)                      // A format: bf16
           | (1u << 10)                     // B format: bf16
           | (0u << 15)                     // A K-major
           | ((b_mn_major ? 1u : 0u) << 16) // B K-major / MN-major
           | (uint32_t(kKeys >> 3) << 17)   // N / 8
           | (uint32_t(kRows >> 4) << 24);  // M / 16
}
constexpr uint32_t kIdescQK = idesc_bf16(false);
constexpr uint32_t kIdescPV = idesc_bf16(true);

// shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;  // descriptor version for tcgen05
    d |= uint64_t(2) << 61;  // SWIZZLE_128B
    return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Bursts of eight products from one asm block.  The issuing thread runs in step
// with the tensor pipe (measured: each cycle it spends between two products is a
// cycle the pipe idles), so a tile's products go out back to back with their
// descriptors computed beforehand.
//
// S = Q K^T over K = 128 dims in eight K = 16 steps; the first step overwrites D.
__device__ __forceinline__ void umma_ss8(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                         uint32_t idesc) {
    asm volatile(
        "{\n .reg .pred pz, pa;\n setp.ne.b32 pz, %17, %17;\n setp.eq.b32 pa, %17, %17;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, pz;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, pa;\n}\n" ::"r"(d),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]),
        "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
        "r"(idesc)
        : "memory");
}

// O_h += P_h V_h for both key halves h (four K = 16 steps each): D of half h at
// d + 128 h, A (P_h, bf16 pairs in TMEM) at a + 64 h + 8 kk, B descriptors
// b[4 h + kk].  The first step of each half accumulates only if `acc` is set.
__device__ __forceinline__ void umma_ts8(uint32_t d, uint32_t a, const uint64_t (&b)[8],
                                         uint32_t idesc, uint32_t acc) {
    // eight K = 16 steps over 128 keys (A from TMEM, 8 columns of bf16 pairs per
    // step) into one accumulator; the first overwrites it when acc == 0
    asm volatile(
        "{\n .reg .pred pf, pa;\n .reg .b32 a1, a2, a3, a4, a5, a6, a7;\n"
        " setp.ne.b32 pf, %10, 0;\n setp.eq.b32 pa, %10, %10;\n"
        " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n add.u32 a4, %1, 32;\n"
        " add.u32 a5, %1, 40;\n add.u32 a6, %1, 48;\n add.u32 a7, %1, 56;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %11, pf;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %3, %11, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], %4, %11, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], %5, %11, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], %6, %11, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], %7, %11, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], %8, %11, pa;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], %9, %11, pa;\n}\n" ::"r"(d),
        "r"(a), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]),
        "l"(b[7]), "r"(acc), "r"(idesc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#define PKV_R32(r)                                                                              \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),         \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),           \
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),           \
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define PKV_W32(r)                                                                          \
    "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),   \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), \
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), \
        "r"(r[29]), "r"(r[30]), "r"(r[31])

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : PKV_R32(r)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        PKV_W32(r)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // a -> low half, b -> high half
    return *reinterpret_cast<uint32_t*>(&v);
}

struct PrefillParams {
    __nv_bfloat16* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start_loc;
    const int2* items;
    const int32_t* n_items;
    const int32_t* counters;   // [2]: how many CTAs (one per SM) take prefill units
    int32_t* ticket;           // next prefill unit (reset by the planner)
    int32_t table_stride;
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t group;
    int32_t tokens_per_tile;
    int32_t window;            // sliding window in keys (0: none); tables in logical order
    float scale_log2;
    int* err;
};

// Per-unit geometry shared by all roles.  Key tiles start at table index
// kbase (0 without a window; with one, the 128-key tile holding the first key
// of the unit's first token), so tile j holds keys kbase + 128 j ..; n_keys,
// n_tiles and nblk count from kbase, and lo0 is the first token's first key
// relative to kbase.
struct Unit {
    int seq, kvh, q0, qlen, ctx, t0, nt, n_keys, n_tiles, nblk, kbase, lo0;
};

__device__ __forceinline__ Unit unit_of(const PrefillParams& p, int u) {
    Unit x;
    const int2 item = p.items[u / p.num_kv_heads];
    x.kvh = u % p.num_kv_heads;
    x.seq = item.x;
    x.q0 = p.query_start_loc[x.seq];
    x.qlen = p.query_start_loc[x.seq + 1] - x.q0;
    x.ctx = p.context_lens[x.seq];
    x.t0 = item.y * p.tokens_per_tile;
    x.nt = min(p.tokens_per_tile, x.qlen - x.t0);
    const int lo = window_first_key(x.ctx - x.qlen + x.t0, p.window);
    x.kbase = lo / kKeys * kKeys;
    x.lo0 = lo - x.kbase;
    x.n_keys = x.ctx - x.qlen + x.t0 + x.nt - x.kbase;  // up to the tile's last token's key
    x.n_tiles = (x.n_keys + kKeys - 1) / kKeys;
    x.nblk = (x.n_keys + kBlockTokens - 1) / kBlockTokens;
    return x;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// A full unit's output tile leaves shared memory by TMA tensor stores (one per
// 64-dim half), so the softmax warps do not wait for 128 rows of scattered
// global stores.  The issuing thread tracks the stores as one bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y,
                                             int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the source of every committed store has been read (the staging tile may be reused)
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed store has completed
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 2^x on the MUFU unit in one instruction (PTX ex2.approx.ftz.f32: a few ulps
// of relative error, subnormal results flushed to zero).  The softmax weights
// and rescale factors only; everything else in this file keeps IEEE fp32.
__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// max(a, b, c) in one instruction (three-input form of max.f32)
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// A wait's first attempt and another barrier's test in one go, so the two
// round trips overlap: whether the phase `wpar` of `wbar` has completed (the
// try may suspend the thread a little while it has not), and in `tested`
// whether the phase `tpar` of `tbar` has.
__device__ __forceinline__ bool mbar_try_and_test(uint64_t* wbar, uint32_t wpar, uint64_t* tbar,
                                                  uint32_t tpar, bool& tested) {
    uint32_t a, b;
    asm volatile(
        "{\n .reg .pred pa, pb;\n"
        " mbarrier.test_wait.parity.shared::cta.b64 pb, [%4], %5;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 pa, [%2], %3;\n"
        " selp.u32 %0, 1, 0, pa;\n selp.u32 %1, 1, 0, pb;\n}\n"
        : "=r"(a), "=r"(b)
        : "r"(smem_u32(wbar)), "r"(wpar), "r"(smem_u32(tbar)), "r"(tpar)
        : "memory");
    tested = b != 0;
    return a != 0;
}

// Block ids of a unit's key tiles, fetched 4 tiles (32 blocks, one per lane) at
// a time and one group ahead, so a producer never waits on the block table.
struct BlockIds {
    const int32_t* bt;
    int nblk, cur, next;
    __device__ __forceinline__ int load(int group, int lane) const {
        const int i = group * 32 + lane;
        return i < nblk ? bt[i] : -1;
    }
    __device__ __forceinline__ void start(const int32_t* table, int n, int lane) {
        bt = table;
        nblk = n;
        cur = load(0, lane);
        next = load(1, lane);
    }
    // block id of block i (0..7) of key tile j for lanes i < 8; call for j = 0, 1, 2, ...
    __device__ __forceinline__ int tile(int j, int lane) {
        if (j > 0 && (j & 3) == 0) {
            cur = next;
            next = load((j >> 2) + 1, lane);
        }
        return __shfl_sync(0xffffffffu, cur, ((j & 3) << 3) + (lane & 7));
    }
};

// Unit ring: the K producer takes units from the ticket (the planner ordered
// the items longest first) and publishes them; the V producer, the two MMA
// issuers and the 8 softmax warps read each one and release its slot.
constexpr int kUnitSlots = 4;
constexpr int kUnitReaders = 1 + 2 + kSoftWarps;

// A published unit: its id (-1: no more work) and geometry, computed once by
// the K producer so the other roles start a unit without global loads.
struct UnitSlot {
    int u;
    Unit x;
};
// barriers, TMEM address, abort flag and unit ring share the 1 KiB after kBarOff
static_assert(B_COUNT * 8 + 16 + kUnitSlots * sizeof(UnitSlot) <= 1024, "barrier area");

__device__ __forceinline__ int unit_read(uint64_t* bars, const UnitSlot* ring, uint32_t k,
                                         int* err, bool& ok, Unit& x) {
    const int slot = k % kUnitSlots;
    int u = -1;
    if (ok && mbar_wait(&bars[B_U_READY + slot], (k / kUnitSlots) & 1, err)) {
        u = ring[slot].u;
        x = ring[slot].x;
    } else {
        ok = false;
    }
    return u;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_o, PrefillParams p) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;           // 1 KiB aligned for the swizzle
    unsigned char* smem = smem_raw + (base - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + B_COUNT * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + B_COUNT * 8 + 4);
    UnitSlot* unit_ring = reinterpret_cast<UnitSlot*>(smem + kBarOff + B_COUNT * 8 + 16);
    float* stat = reinterpret_cast<float*>(smem + kStatOff);  // [set][half][row]
    float* xm = reinterpret_cast<float*>(smem + kXmOff);      // [tile parity][half][row]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Shared-memory set-up needs nothing from the plan, so it runs while the
    // planner still works.  Zero the operand area once so no stale bit pattern
    // can be NaN.
    for (int i = threadIdx.x; i < kStatOff / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars[B_K_FULL + s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&bars[B_V_FULL + s], 1);
        }
        for (int s = 0; s < kQBufs; ++s) {
            mbar_init(&bars[B_Q_FULL + s], 1);
            mbar_init(&bars[B_Q_EMPTY + s], kSoftWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_S_FULL + s], 1);
            mbar_init(&bars[B_S_EMPTY + s], kSoftWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_P_FULL + s], kSoftWarps);
            mbar_init(&bars[B_O_DONE + s], 1);
        }
        for (int s = 0; s < kUnitSlots; ++s) {
            mbar_init(&bars[B_U_READY + s], 1);
            mbar_init(&bars[B_U_EMPTY + s], kUnitReaders);
        }
        mbar_init(&bars[B_O_EMPTY], kSoftWarps);
        mbar_init(&bars[B_STAT], kSoftWarps);
        for (int s = 0; s < 4; ++s) mbar_init(&bars[B_XM + s], 2);
        mbar_init(&bars[B_DRAIN], 1);
        mbar_init(&bars[B_DRAIN_PV], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }

    // Launched right behind the planner (programmatic launch): wait for the plan.
    // The planner gives the prefill chunks only as many SMs as their share of
    // the batch's work; the other CTAs leave at once, and the decode kernel that
    // follows in the stream may start right away on the SMs they free (it reads
    // the plan without waiting, so the trigger comes after this grid's wait).
    pdl_wait_prerequisites();
    pdl_launch_dependents();
    const int active = min(p.counters[2], int(gridDim.x));
    if (int(blockIdx.x) >= active) return;
    const int n_units = p.n_items[0] * p.num_kv_heads;

    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kKProducerWarp) {
        // ------- unit tickets, Q tiles, output stores and the K ring (one warp) -------
        // Q buffer b holds unit k's Q and then, once its epilogue has staged it,
        // unit k's output tile.  Before loading unit k + 2's Q there, this warp
        // sends the staged tile out by TMA and waits until it has been read; the
        // last two units' tiles go out after the loop.
        uint32_t kt = 0;
        bool ok = true;
        bool out_staged[kQBufs] = {false, false};   // per Q buffer: its last unit was staged
        int out_y[kQBufs] = {0, 0}, out_z[kQBufs] = {0, 0};
        uint32_t k = 0;
        auto send_output = [&](int qb) {
            if (lane == 0 && out_staged[qb]) {
                const uint32_t src = base + kQOff + qb * kQBytes;
                tma_store_3d(&tmap_o, src, 0, out_y[qb], out_z[qb]);
                tma_store_3d(&tmap_o, src + kSub, 64, out_y[qb], out_z[qb]);
                bulk_commit();
                bulk_wait_read();   // the buffer may take the next Q after this
            }
            out_staged[qb] = false;
        };
        // A CTA's first unit is its own index (units come longest first, one for
        // each active CTA, with no atomic before the first copies); later units
        // come from the ticket, after them.  The next unit's ticket is taken when
        // this unit's last K tile is issued, not when the unit starts: a CTA that
        // reserved its next unit at the start of a long one would take a long or
        // medium unit that a CTA finishing sooner should get (measured on the
        // SplitFuse chunks: CTAs ending at 33 and at 44 us).  The atomic's latency
        // still hides behind the unit's last products and epilogue.
        int next = int(blockIdx.x);
        for (;; ++k) {
            const int slot = k % kUnitSlots;
            ok = ok && __all_sync(0xffffffffu, mbar_wait(&bars[B_U_EMPTY + slot],
                                                         ((k / kUnitSlots) & 1) ^ 1, p.err));
            int u = -1;
            if (lane == 0 && ok && !*abort_flag && next < n_units) u = next;
            u = __shfl_sync(0xffffffffu, u, 0);
            Unit x = {};
            if (u >= 0) x = unit_of(p, u);
            if (lane == 0) {
                unit_ring[slot].u = u;
                unit_ring[slot].x = x;
                mbar_arrive(&bars[B_U_READY + slot]);
            }
            if (u < 0) break;
            // Q tile of the unit (two 64-dim halves); the buffer's previous unit
            // has staged its output (or written it directly) by now
            const int qb = k % kQBufs;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars[B_Q_EMPTY + qb], ((k / kQBufs) & 1) ^ 1, p.err));
            if (!ok) break;
            send_output(qb);
            out_staged[qb] = x.nt == p.tokens_per_tile;
            out_y[qb] = x.kvh * p.group;
            out_z[qb] = x.q0 + x.t0;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[B_Q_FULL + qb], 2 * kSub);
                const uint32_t qd = base + kQOff + qb * kQBytes;
                tma_load_3d(qd, &tmap_q, 0, x.kvh * p.group, x.q0 + x.t0, &bars[B_Q_FULL + qb]);
                tma_load_3d(qd + kSub, &tmap_q, 64, x.kvh * p.group, x.q0 + x.t0,
                            &bars[B_Q_FULL + qb]);
            }
            __syncwarp();
            BlockIds ids;
            ids.start(p.block_tables + size_t(x.seq) * p.table_stride + x.kbase / kBlockTokens,
                      x.nblk, lane);
            for (int j = 0; j < x.n_tiles && ok; ++j, ++kt) {
                const int st = kt % kKStages;
                const int nb = min(kBlkPerTile, x.nblk - j * kBlkPerTile);
                const int blk = ids.tile(j, lane);
                if (j == x.n_tiles - 1 && lane == 0) next = active + atomicAdd(p.ticket, 1);
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bars[B_S_FULL + st], ((kt / kKStages) & 1) ^ 1, p.err));
                if (!ok || *abort_flag) {
                    ok = false;
                    break;
                }
                const bool good = lane < nb && blk >= 0 && blk < p.num_blocks;
                if (lane < nb && !good) flag_error(p.err, PKV_DEV_BAD_BLOCK_ID);
                const unsigned mask = __ballot_sync(0xffffffffu, good);
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars[B_K_FULL + st], uint32_t(__popc(mask)) * 2u * kBoxBytes);
                __syncwarp();
                if (good) {
                    const uint32_t dst = base + kKOff + st * kKBytes + uint32_t(lane) * kBoxBytes;
                    const int row = (blk * p.num_kv_heads + x.kvh) * kBlockTokens;
                    tma_load_2d(dst, &tmap_k, 0, row, &bars[B_K_FULL + st]);
                    tma_load_2d(dst + kKeys * 128, &tmap_k, 64, row, &bars[B_K_FULL + st]);
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        // the last units' output tiles (k units were loaded)
        for (uint32_t kk = k >= kQBufs ? k - kQBufs : 0; ok && kk < k; ++kk) {
            const int qb = kk % kQBufs;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars[B_Q_EMPTY + qb], (kk / kQBufs) & 1, p.err));
            if (ok) send_output(qb);
        }
        if (!ok) *abort_flag = 1;
        // never leave with copies in flight: wait for the last fill of each stage,
        // and for the output stores to complete
        if (lane == 0) {
            for (int k = 0; k < kKStages && uint32_t(k) < kt; ++k) {
                const uint32_t last = kt - 1 - k;
                mbar_wait(&bars[B_K_FULL + last % kKStages], (last / kKStages) & 1, p.err);
            }
            bulk_wait_all();
        }
    } else if (warp == kVProducerWarp) {
        // ------------------------------ V ring ------------------------------
        uint32_t kt = 0;
        bool ok = true;
        for (uint32_t k = 0;; ++k) {
            Unit x;
            const int u = unit_read(bars, unit_ring, k, p.err, ok, x);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_U_EMPTY + k % kUnitSlots]);
            if (u < 0 || !ok) break;
            BlockIds ids;
            ids.start(p.block_tables + size_t(x.seq) * p.table_stride + x.kbase / kBlockTokens,
                      x.nblk, lane);
            for (int j = 0; j < x.n_tiles && ok; ++j, ++kt) {
                const int st = kt % kVStages;
                const int nb = min(kBlkPerTile, x.nblk - j * kBlkPerTile);
                const int blk = ids.tile(j, lane);
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bars[B_O_DONE + st], ((kt / kVStages) & 1) ^ 1, p.err));
                if (!ok || *abort_flag) {
                    ok = false;
                    break;
                }
                const bool good = lane < nb && blk >= 0 && blk < p.num_blocks;
                const unsigned mask = __ballot_sync(0xffffffffu, good);
                if (lane == 0)
                    mbar_arrive_expect_tx(&bars[B_V_FULL + st], uint32_t(__popc(mask)) * 2u * kBoxBytes);
                __syncwarp();
                if (good) {
                    const uint32_t dst = base + kVOff + st * kKBytes + uint32_t(lane) * kBoxBytes;
                    const int row = (blk * p.num_kv_heads + x.kvh) * kBlockTokens;
                    tma_load_2d(dst, &tmap_v, 0, row, &bars[B_V_FULL + st]);
                    tma_load_2d(dst + kKeys * 128, &tmap_v, 64, row, &bars[B_V_FULL + st]);
                }
                __syncwarp();
            }
        }
        if (!ok) *abort_flag = 1;
        if (lane == 0) {
            for (int k = 0; k < kVStages && uint32_t(k) < kt; ++k) {
                const uint32_t last = kt - 1 - k;
                mbar_wait(&bars[B_V_FULL + last % kVStages], (last / kVStages) & 1, p.err);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------- Q K^T issuer ----------------------------
        // Key tiles are numbered over the CTA's whole sequence of units.  Q K^T
        // of tile q writes S buffer q & 1, which held S(q - 2): it waits until
        // every softmax warp has loaded those scores, then for its K stage and
        // (first tile of a unit) its Q buffer.  The pipe
        // idles for every instruction this thread runs between two products,
        // so the waits come first, then one fence and the eight products in one
        // burst; descriptors come from per-CTA bases plus constant offsets
        // (shared-memory addresses stay below 256 KiB: adding to the 14-bit
        // start field never carries).  The abort flag is read once per unit; a
        // wait that can no longer be satisfied ends on its time limit.
        if (lane == 0) {
            bool ok = true;
            uint64_t qd[8];  // Q buffer 0: K-major, 128-byte swizzle
            {
                const uint64_t q0 = sdesc(base + kQOff, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    qd[kk] = q0 + uint64_t(((kk >> 2) * kSub + (kk & 3) * 32) >> 4);
            }
            const uint64_t kd_base = sdesc(base + kKOff, 16, 1024);
            uint32_t q = 0;                      // Q K^T tiles issued
            for (uint32_t k = 0;; ++k) {
                Unit x;
                const int u = unit_read(bars, unit_ring, k, p.err, ok, x);
                mbar_arrive(&bars[B_U_EMPTY + k % kUnitSlots]);
                if (u < 0 || !ok || *abort_flag) break;
                const uint32_t qb = k & 1;
                const uint64_t qoff = uint64_t(qb) * (kQBytes >> 4);
                for (int j = 0; j < x.n_tiles; ++j, ++q) {
                    uint64_t qa[8], kd[8];
                    const uint64_t k0 = kd_base + uint64_t((q % kKStages) * (kKBytes >> 4));
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        qa[i] = qd[i] + qoff;
                        kd[i] = k0 + uint64_t(((i >> 2) * (kKeys * 128) + (i & 3) * 32) >> 4);
                    }
                    ok = (q < 2 || mbar_wait(&bars[B_S_EMPTY + (q & 1)], ((q - 2) >> 1) & 1, p.err)) &&
                         (j != 0 || mbar_wait(&bars[B_Q_FULL + qb], (k >> 1) & 1, p.err)) &&
                         mbar_wait(&bars[B_K_FULL + q % kKStages], (q / kKStages) & 1, p.err);
                    if (!ok) break;
                    tc_after();
                    umma_ss8(tmem + (q & 1) * kKeys, qa, kd, kIdescQK);
                    umma_commit(&bars[B_S_FULL + (q & 1)]);
                }
                if (!ok) break;
            }
            if (!ok) *abort_flag = 1;
            // wait until every MMA issued here has completed before TMEM is freed
            umma_commit(&bars[B_DRAIN]);
            mbar_wait(&bars[B_DRAIN], 0, p.err);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ----------------------------- P V issuer -----------------------------
        // P V of tile t (both 64-key halves into the one O accumulator) once the
        // softmax warps have published P(t), the tile's V has landed and, for a
        // unit's first tile, the previous unit's epilogue has read O (its first
        // products overwrite O).  Products of this thread run in order, so a
        // completed O_DONE of tile t also covers every earlier P V.
        if (lane == 0) {
            bool ok = true;
            const uint64_t vd_base = sdesc(base + kVOff, kKeys * 128, 1024);
            uint32_t t = 0;                      // P V tiles issued
            for (uint32_t k = 0;; ++k) {
                Unit x;
                const int u = unit_read(bars, unit_ring, k, p.err, ok, x);
                mbar_arrive(&bars[B_U_EMPTY + k % kUnitSlots]);
                if (u < 0 || !ok || *abort_flag) break;
                for (int j = 0; j < x.n_tiles; ++j, ++t) {
                    uint64_t vd[8];
                    const uint64_t v0 = vd_base + uint64_t((t % kVStages) * (kKBytes >> 4));
#pragma unroll
                    for (int i = 0; i < 8; ++i) vd[i] = v0 + uint64_t((i * 16 * 128) >> 4);
                    ok = mbar_wait(&bars[B_P_FULL + (t & 1)], (t >> 1) & 1, p.err) &&
                         mbar_wait(&bars[B_V_FULL + t % kVStages], (t / kVStages) & 1, p.err) &&
                         (j != 0 || mbar_wait(&bars[B_O_EMPTY], (k & 1) ^ 1u, p.err));
                    if (!ok) break;
                    tc_after();
                    umma_ts8(tmem + kOCol, tmem + kPCol + (t & 1) * 64, vd, kIdescPV, j == 0 ? 0u : 1u);
                    umma_commit(&bars[B_O_DONE + (t & 1)]);
                }
                if (!ok) break;
            }
            if (!ok) *abort_flag = 1;
            umma_commit(&bars[B_DRAIN_PV]);
            mbar_wait(&bars[B_DRAIN_PV], 0, p.err);
        }
        __syncwarp();
    } else {
        // -------------- softmax: thread = (query row r, key half h) --------------
        const int r = (warp & 3) * 32 + lane;            // query row = TMEM lane
        const int h = warp >> 2;                          // key half of each 128-key tile
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        const int G = p.group;
        uint32_t kt = 0;
        bool ok = true;
        for (uint32_t k = 0;; ++k) {
            Unit x;
            const int u = unit_read(bars, unit_ring, k, p.err, ok, x);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_U_EMPTY + k % kUnitSlots]);
            if (u < 0 || !ok || *abort_flag) break;
            const int tok = r / G, g_head = r % G;
            const bool row_valid = tok < x.nt;
            const int t = x.t0 + tok;
            // this row's visible keys, as indices from the unit's first key tile:
            // lower .. limit (the window's first key .. the row's own position)
            const int last = row_valid ? x.ctx - x.qlen + t : x.ctx - 1;
            const int limit = last - x.kbase;
            const int lower = row_valid ? window_first_key(last, p.window) - x.kbase : x.lo0;

            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < x.n_tiles; ++j) {
                const uint32_t g = kt + j;
                // S(g), and whether the P V of tile g - 2 (the last reader of P
                // buffer g & 1) has completed, tested without waiting (it nearly
                // always has; the bounded wait runs before P is stored only if it
                // has not)
                bool p_done;
                bool s_full = mbar_try_and_test(&bars[B_S_FULL + (g & 1)], (g >> 1) & 1,
                                                &bars[B_O_DONE + (g & 1)], ((g - 2) >> 1) & 1, p_done);
                if (!s_full) s_full = mbar_wait(&bars[B_S_FULL + (g & 1)], (g >> 1) & 1, p.err);
                ok = __all_sync(0xffffffffu, s_full);
                if (!ok) break;
                tc_after();
                float s[64];
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem + lane_base + (g & 1) * kKeys + h * 64, v0);
                    tmem_ld32(tmem + lane_base + (g & 1) * kKeys + h * 64 + 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        s[i] = __uint_as_float(v0[i]);
                        s[32 + i] = __uint_as_float(v1[i]);
                    }
                }
                const bool p_free = g < 2 || p_done;

                // mask keys beyond this row's causal limit and below its window;
                // max on the raw scores
                const int key0 = j * kKeys + h * 64;
                if (key0 + 63 > limit || key0 < lower) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        s[c] = (key0 + c <= limit && key0 + c >= lower) ? s[c] : -INFINITY;
                }
                // eight independent partial maxima instead of one 64-long chain
                // (three-input maxima: half the instructions of a two-input tree)
                float mx8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = max3f(s[i], s[i + 8], s[i + 16]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = max3f(mx8[i], s[i + 24], s[i + 32]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = max3f(mx8[i], s[i + 40], s[i + 48]);
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[i + 56]);
                const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                                       fmaxf(mx8[6], mx8[7])) * p.scale_log2;
                // the row's two halves share one O, so they share the running max:
                // exchange this tile's maxima with the other half's thread (warp
                // warp ^ 4, same TMEM lanes) through shared memory, a slot per tile
                // parity; both then take identical decisions from identical values
                float* xslot = xm + (g & 1) * 2 * kRows;
                xslot[h * kRows + r] = mx;
                // the scores are in registers: Q K^T of tile g + 2 may overwrite them
                tc_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars[B_XM + (warp & 3)]);
                    mbar_arrive(&bars[B_S_EMPTY + (g & 1)]);
                }
                ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_XM + (warp & 3)], g & 1, p.err));
                if (!ok) break;
                const float m_new = fmaxf(m, fmaxf(mx, xslot[(h ^ 1) * kRows + r]));
                const bool need = m_new > m + kRescaleThreshold;  // first visible keys included
                float alpha = 1.f;
                if (need) {
                    alpha = ex2_approx(m - m_new);
                    m = m_new;
                    l *= alpha;
                }
                // P = 2^(s * scale - m) in bf16; the exponent arguments and the row
                // sum use packed fp32x2 arithmetic (two lanes per instruction)
                const float neg_m = m == -INFINITY ? 0.f : -m;
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                const float2 nm2 = make_float2(neg_m, neg_m);
                uint32_t w[32];
                float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                  make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float2 e = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), sc2, nm2);
                    const float p0 = ex2_approx(e.x), p1 = ex2_approx(e.y);
                    sum4[c & 3] = __fadd2_rn(sum4[c & 3], make_float2(p0, p1));
                    w[c] = pack_bf16(p0, p1);
                }
                l += ((sum4[0].x + sum4[0].y) + (sum4[1].x + sum4[1].y)) +
                     ((sum4[2].x + sum4[2].y) + (sum4[3].x + sum4[3].y));
                const bool warp_need = __any_sync(0xffffffffu, need);
                if (j > 0 && warp_need) {
                    // rescale O_h: wait for the previous P V (buffer (g - 1) & 1;
                    // the P V products run in issue order on one thread, so every
                    // older one has completed too)
                    const uint32_t gp = g - 1;
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + (gp & 1)],
                                                           (gp >> 1) & 1, p.err));
                    if (!ok) break;
                    tc_after();
                    // this thread's 64 dims of the row's O (the other half's thread
                    // takes the other 64, with the same alpha)
#pragma unroll 1
                    for (int c2 = 0; c2 < 2; ++c2) {
                        uint32_t v[32];
                        const uint32_t ta = tmem + lane_base + kOCol + h * 64 + c2 * 32;
                        tmem_ld32(ta, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        tmem_st32(ta, v);
                    }
                }
                // P (bf16 pairs) into P buffer g & 1, columns 32 h .. 32 h + 31, once
                // the P V of tile g - 2 (the buffer's last reader) has completed
                if (!__all_sync(0xffffffffu, p_free)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_O_DONE + (g & 1)],
                                                           ((g - 2) >> 1) & 1, p.err));
                    if (!ok) break;
                }
                tc_after();
                tmem_st32(tmem + lane_base + kPCol + (g & 1) * 64 + h * 32, w);
                // rows of the last staged block that lie beyond the context were
                // never written: zero their V so 0 * (anything) cannot become NaN.
                // The half whose keys hold that block does it before its P V.
                const int rows_last = x.ctx - x.kbase - (x.nblk - 1) * kBlockTokens;  // 1..16+
                const int slot = (x.nblk - 1) - j * kBlkPerTile;
                const bool zero_v = j == x.n_tiles - 1 && rows_last < kBlockTokens && (slot >> 2) == h;
                // in the unit's first tile, the rows below its first token's window
                // hold other tokens of the ring (or were never written): zero their V
                // too; this half's keys h * 64 .. h * 64 + z_lo - 1
                const int z_lo = j == 0 ? max(0, min(x.lo0, h * 64 + 64) - h * 64) : 0;
                if (zero_v || z_lo > 0) {
                    // the V tile must have landed before its rows are overwritten (its
                    // stage cannot be refilled before this tile's P V has been issued)
                    ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_V_FULL + g % kVStages],
                                                           (g / kVStages) & 1, p.err));
                    if (!ok) break;
                    unsigned char* vs = smem + kVOff + (g % kVStages) * kKBytes;
                    const int nz = zero_v ? (kBlockTokens - rows_last) * 2 * 8 : 0;  // rows x halves x chunks
                    for (int i = r; i < nz; i += kRows) {
                        const int row = rows_last + i / 16, half = (i / 8) & 1, c = i & 7;
                        *reinterpret_cast<uint4*>(vs + half * (kKeys * 128) +
                                                  (slot * kBlockTokens + row) * 128 + c * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    for (int i = r; i < z_lo * 16; i += kRows) {
                        const int key = h * 64 + i / 16, half = (i / 8) & 1, c = i & 7;
                        *reinterpret_cast<uint4*>(vs + half * (kKeys * 128) + key * 128 + c * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_async_smem();   // the zeroed V rows, before the P V reads them
                }
                tmem_wait_st();
                tc_before();
                __syncwarp();
                if (!ok) break;
                if (lane == 0) mbar_arrive(&bars[B_P_FULL + (g & 1)]);
            }
            if (!ok) break;
            // ---- epilogue: O / l -> out (this thread: dims 64h..64h+63; l is the sum
            // of both halves' partial sums, taken against the shared running max) ----
            const uint32_t glast = kt + x.n_tiles - 1;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars[B_O_DONE + (glast & 1)], (glast >> 1) & 1, p.err));
            if (!ok) break;
            tc_after();
            // A full unit (every row a query) leaves through its own Q buffer, which
            // its last Q K^T has finished with (these warps read that product's
            // scores), and TMA stores; a partial one writes its valid rows
            // directly.  Either way the buffer is handed back to the Q producer at
            // the end.
            const bool staged = x.nt == p.tokens_per_tile;
            const uint32_t qbuf = k % kQBufs;
            float* st_set = stat + (k & 1) * 2 * kRows;
            st_set[h * kRows + r] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_STAT]);
            ok = __all_sync(0xffffffffu, mbar_wait(&bars[B_STAT], k & 1, p.err));
            if (!ok) break;
            const float inv = 1.f / (st_set[r] + st_set[kRows + r]);
            // this thread's 64 output dims (bf16 pairs): chunk c = dims 8c .. 8c + 7
            uint32_t packed[32];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kOCol + h * 64 + c2 * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    packed[c2 * 16 + i] = pack_bf16(__uint_as_float(v[2 * i]) * inv,
                                                    __uint_as_float(v[2 * i + 1]) * inv);
            }
            // O has been read: the next unit's first P V may overwrite it
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_O_EMPTY]);
            if (staged) {
                // row r of half h, 128-byte swizzled like the TMA box of the output map
                unsigned char* row = smem + kQOff + qbuf * kQBytes + h * kSub + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) * 16)) =
                        make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                   packed[4 * c + 3]);
                fence_async_smem();   // generic-proxy writes, before the TMA reads them
            } else if (row_valid) {
                uint4* dst = reinterpret_cast<uint4*>(
                    p.out + (size_t(x.q0 + t) * p.num_q_heads + x.kvh * G + g_head) * kDim + h * 64);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2],
                                        packed[4 * c + 3]);
            }
            // the unit is done with its Q buffer; a staged tile in it goes out with
            // the producer's next use of the buffer
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_Q_EMPTY + qbuf]);
            kt += x.n_tiles;
        }
        if (!ok) *abort_flag = 1;
    }

    tc_before();
    __syncthreads();
    tc_after();
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---- host side -------------------------------------------------------------

}  // namespace

int prefill_supported(const pkv_cache_desc* d) {
    const int g = d->num_q_heads / d->num_kv_heads;
    return d->dtype == PKV_BF16 && d->head_dim == kDim && d->block_size == kBlockTokens &&
           (g == 1 || g == 2 || g == 4 || g == 8) &&
           int64_t(d->num_blocks) * d->num_kv_heads * kBlockTokens < (int64_t(1) << 31);
}

int prefill_item_bound(int32_t num_seqs, int32_t num_query_tokens, int32_t group) {
    const int32_t tokens_per_tile = kPrefillRows / group;
    return ceil_div(num_query_tokens, tokens_per_tile) + num_seqs;
}

int launch_prefill(const AttnArgs& a) {
    const pkv_cache_desc* d = a.desc;
    if (!prefill_supported(d)) return PKV_ERR_UNSUPPORTED;
    const int group = d->num_q_heads / d->num_kv_heads;
    CUtensorMap mk, mv, mq, mo;
    // the output has the query's shape: the same box serves the output tile's stores
    if (!make_cache_tensor_map(&mk, a.k_cache, d) || !make_cache_tensor_map(&mv, a.v_cache, d) ||
        !make_query_tensor_map(&mq, a.q, a.num_query_tokens, d->num_q_heads, group) ||
        !make_query_tensor_map(&mo, a.out, a.num_query_tokens, d->num_q_heads, group))
        return PKV_ERR_CUDA;
    PrefillParams p;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.query_start_loc = a.query_start_loc;
    p.items = a.ws.prefill_items;
    p.n_items = a.ws.counters + 1;
    p.counters = a.ws.counters;
    p.ticket = a.ws.counters + 4;
    p.table_stride = a.table_stride;
    p.num_blocks = d->num_blocks;
    p.num_kv_heads = d->num_kv_heads;
    p.num_q_heads = d->num_q_heads;
    p.group = group;
    p.tokens_per_tile = kPrefillRows / p.group;
    p.window = a.window;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.err = a.err;
    if (kernel_occupancy<prefill_kernel>(kThreads, kSmemBytes) < 1) return PKV_ERR_CUDA;
    const int64_t bound = int64_t(a.ws.max_prefill_items) * d->num_kv_heads;
    const int64_t grid = std::min<int64_t>(num_sms(), bound);
    if (grid < 1) return PKV_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cuda_status(cudaLaunchKernelEx(&cfg, prefill_kernel, mk, mv, mq, mo, p));
}

}  // namespace pkv
