"""Token-budget composition of one forward pass (oracle; test infrastructure only).

[FastGen §3.2 动态分割融合]: long prompts are split into chunks spread over
several forward passes, short prompts are fused so that each pass carries a
fixed token budget.  [Ch15 §15.6 两阶段与 Chunked Prefill]: the budget is
shared as sum(prefill chunk tokens) + number of decode sequences <= budget,
decode tokens first (scenario B: 8192 - 256 decode tokens = 7936 left for the
prompt chunk), and a long prompt continues in the next pass (scenario A:
10000 -> 8192, then 1808).

Reading where the pages are silent: decodes are admitted in the given order
while the budget lasts; prompts are served in arrival order, each chunk being
min(remaining tokens, budget left), so only the last prompt served in a pass
can be split.
"""


def compose(token_budget, num_decode, prompt_remaining):
    """Return (decode_admitted, chunks, tokens_used)."""
    if token_budget < 0 or num_decode < 0 or any(r < 0 for r in prompt_remaining):
        raise ValueError("negative input")
    left = token_budget
    decode_admitted = min(num_decode, left)
    left -= decode_admitted
    chunks = []
    for r in prompt_remaining:
        c = min(r, left)
        chunks.append(c)
        left -= c
    return decode_admitted, chunks, token_budget - left
