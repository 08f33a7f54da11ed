// Prefill-chunk attention for ragged mixed batches (placeholder until the
// tensor-core kernel lands): reports the shape as unsupported.
#include "pkv_internal.h"

namespace pkv {

int prefill_supported(const pkv_cache_desc*) { return 0; }

int prefill_item_bound(int32_t num_seqs, int32_t num_query_tokens, int32_t group) {
    const int32_t tokens_per_tile = kPrefillRows / group;
    return ceil_div(num_query_tokens, tokens_per_tile) + num_seqs;
}

int launch_prefill(const AttnArgs&) { return PKV_ERR_UNSUPPORTED; }

}  // namespace pkv
