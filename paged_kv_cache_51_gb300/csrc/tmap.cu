// Host helper: TMA tensor maps over a paged cache pool.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.h"

namespace pkv {

namespace {
// Encoded maps depend only on the address and the shape, so the last few are
// kept: a serving loop calls with the same pools (and often the same q) every step.
struct MapKey {
    int kind;
    const void* ptr;
    int64_t a, b, c, d;
    bool operator==(const MapKey& o) const {
        return kind == o.kind && ptr == o.ptr && a == o.a && b == o.b && c == o.c && d == o.d;
    }
};
constexpr int kMapCache = 16;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
CUtensorMap g_map_val[kMapCache];
bool g_map_used[kMapCache];
int g_map_next = 0;

bool map_lookup(const MapKey& k, CUtensorMap* m) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCache; ++i)
        if (g_map_used[i] && g_map_key[i] == k) {
            *m = g_map_val[i];
            return true;
        }
    return false;
}
void map_store(const MapKey& k, const CUtensorMap& m) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    const int i = g_map_next;
    g_map_next = (g_map_next + 1) % kMapCache;
    g_map_key[i] = k;
    g_map_val[i] = m;
    g_map_used[i] = true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}
}  // namespace

// The pool [num_blocks][Hkv][bs][D] (bf16) as a 2-D tensor of rows of D
// elements; a box is the bs rows of one (block, head) tile by 64 columns, so a
// 128-dim tile is two boxes.  Copies land 128-byte swizzled (16-byte chunk c of
// row r at chunk position c ^ (r % 8)), the layout the tensor-core operand
// descriptors and conflict-free ldmatrix reads expect.
bool make_cache_tensor_map(CUtensorMap* m, const void* cache, const pkv_cache_desc* d) {
    const MapKey key{0, cache, d->num_blocks, d->num_kv_heads, d->block_size, d->head_dim};
    if (d->dtype == PKV_BF16 && map_lookup(key, m)) return true;
    auto fn = encode_fn();
    if (!fn || d->dtype != PKV_BF16 || (d->head_dim != 64 && d->head_dim != 128)) return false;
    const cuuint64_t rows = cuuint64_t(d->num_blocks) * d->num_kv_heads * d->block_size;
    if (rows >= (cuuint64_t(1) << 31)) return false;
    const cuuint64_t gdim[2] = {cuuint64_t(d->head_dim), rows};
    const cuuint64_t gstride[1] = {cuuint64_t(d->head_dim) * 2};
    const cuuint32_t box[2] = {64, cuuint32_t(d->block_size)};
    const cuuint32_t estride[2] = {1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), gdim, gstride, box,
           estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, *m);
    return true;
}

// Queries [num_tokens][num_q_heads][128] (bf16) as a 3-D tensor (dims, heads,
// tokens).  A box is 64 dims x G heads x 128 / G tokens: the 128 rows
// (token, head of the group) of one 64-dim half of a prefill Q tile, 128 B
// each, landing 128-byte swizzled like the cache tiles.  Tokens past the end
// read as zero.
bool make_query_tensor_map(CUtensorMap* m, const void* q, int32_t num_tokens, int32_t num_q_heads,
                           int32_t group) {
    const MapKey key{1, q, num_tokens, num_q_heads, group, 0};
    if (map_lookup(key, m)) return true;
    auto fn = encode_fn();
    if (!fn || num_tokens < 1 || group < 1 || kPrefillRows % group) return false;
    const cuuint64_t gdim[3] = {128, cuuint64_t(num_q_heads), cuuint64_t(num_tokens)};
    const cuuint64_t gstride[2] = {128 * 2, cuuint64_t(num_q_heads) * 128 * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(kPrefillRows / group)};
    const cuuint32_t estride[3] = {1, 1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), gdim, gstride, box,
           estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    map_store(key, *m);
    return true;
}

}  // namespace pkv
