// Decode attention without a caller-provided workspace.
//
// paged_attention_decode keeps its split-K partial results in a workspace the
// caller allocates.  Some callers cannot allocate device memory when they
// call: a plugin or custom op living inside a host engine that owns all device
// memory through its own arena and hands plugins no scratch allocator; a
// serving process that gave the whole remaining HBM to its KV-cache pool at
// start-up, so any later cudaMalloc fails; or a step loop that must not call
// cudaMalloc/cudaFree at all because those calls can synchronize the device.
// For them this file keeps a fixed scratch area in the library's own device
// memory (a file-scope array, PKV_NOALLOC_SCRATCH_BYTES per device that loads
// the library, held until the process exits) and runs the same decode path
// on it.  Nothing here allocates.
#include <cuda_runtime.h>
#include <mutex>

#include "pkv_internal.h"

// The scratch area: the work list, the split partials and their (max, sum).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch, looked up once per device with that
// device current.  In host code the array's name is only a host-side stand-in,
// never a device address, so it is never passed to a kernel directly.  The
// address stays valid while the device's primary context lives; a
// cudaDeviceReset would unload the module, and the header rules out calls on
// that device afterwards.
int scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[128] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const pkv_cache_desc* desc,
                                              const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, int32_t num_seqs,
                                              int32_t max_context_len, float scale,
                                              void* stream) {
    if (pkv::check_desc(desc, true) != PKV_OK) return pkv::check_desc(desc, true);
    if (num_seqs < 0 || max_context_len < 1) return PKV_ERR_INVALID;
    // Reject batches whose partials do not fit before touching the device.
    const size_t need = pkv_decode_workspace_bytes(desc, num_seqs, max_context_len);
    if (need == 0 || need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    if (num_seqs == 0) return PKV_OK;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
    // Nothing in the scratch has to start at zero: the planner rewrites the
    // work-list counters on every call and every partial is written before it
    // is read, so the previous call's contents are never used.
    return paged_attention_decode(out, q, k_cache, v_cache, desc, block_tables,
                                  max_blocks_per_seq, context_lens, num_seqs, max_context_len,
                                  scale, scratch, PKV_NOALLOC_SCRATCH_BYTES, stream);
}
