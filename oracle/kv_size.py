"""Closed-form KV-cache size (oracle; test infrastructure only).

bytes = 2 (K and V) x layers x batch x seq x kv_heads x head_dim x dtype_bytes
[Infra 一、2 (cache显存 = 2*层数*批大小*序列长*隐藏层维度*精度字节); Ch15 §15.6
"KV Cache 大小计算" (per token, with N_kv KV heads); Ch7 §2.1 (per layer)].
With kv_heads x head_dim equal to the hidden size this is the MHA form.
"""


def kv_cache_bytes(layers, batch, seq, kv_heads, head_dim, dtype_bytes):
    for x in (layers, batch, seq, kv_heads, head_dim, dtype_bytes):
        if int(x) != x or x < 0:
            raise ValueError("sizes must be non-negative integers")
    return 2 * layers * batch * seq * kv_heads * head_dim * dtype_bytes


def pool_bytes(num_blocks, kv_heads, block_size, head_dim, dtype_bytes):
    """Bytes of one layer's K and V block pools of ``num_blocks`` blocks."""
    return kv_cache_bytes(1, num_blocks, block_size, kv_heads, head_dim, dtype_bytes)


def tokens_that_fit(cache_bytes, layers, kv_heads, head_dim, dtype_bytes):
    return cache_bytes // kv_cache_bytes(layers, 1, 1, kv_heads, head_dim, dtype_bytes)
