// Token-budget composition of one forward pass (Dynamic SplitFuse).
//
// "DeepSpeed-FastGen 深度解析" §3.2 动态分割融合: long prompts are split into
// chunks over several forward passes and short prompts are fused, so every
// pass carries the same token budget.  "第 15 章：推理引擎与部署" §15.6 两阶段与
// Chunked Prefill: sum(prefill chunk tokens) + decode sequences <= budget,
// decode tokens served first.  Prompts are served in arrival order with
// chunk = min(remaining, budget left), so only the last prompt served in a
// pass is split.
#include "pagedkv.h"

extern "C" int pkv_splitfuse_compose(int32_t token_budget, int32_t num_decode,
                                     int32_t num_prompts, const int32_t* prompt_remaining,
                                     int32_t* chunk_out, int32_t* decode_admitted,
                                     int32_t* tokens_used) {
    if (token_budget < 0 || num_decode < 0 || num_prompts < 0 || !decode_admitted ||
        (num_prompts > 0 && (!prompt_remaining || !chunk_out)))
        return PKV_ERR_INVALID;
    for (int32_t i = 0; i < num_prompts; ++i)
        if (prompt_remaining[i] < 0) return PKV_ERR_INVALID;
    int64_t left = token_budget;
    const int64_t dec = num_decode < left ? num_decode : left;
    left -= dec;
    for (int32_t i = 0; i < num_prompts; ++i) {
        const int64_t c = prompt_remaining[i] < left ? prompt_remaining[i] : left;
        chunk_out[i] = int32_t(c);
        left -= c;
    }
    *decode_admitted = int32_t(dec);
    if (tokens_used) *tokens_used = int32_t(token_budget - left);
    return PKV_OK;
}
