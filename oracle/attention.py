"""Exact attention over a paged KV cache, in float64 (oracle; test infrastructure only).

Definition followed: O = softmax(Q K^T / sqrt(d)) V, with the row maximum
subtracted before exponentiation (which leaves softmax unchanged)
[Ch15 §15.1 "标准 Attention 的瓶颈" and "Flash Attention 的两大创新";
Ch7 §2.2.2 传统注意力计算; Deploy §4.1].

The keys and values of a sequence are not contiguous: logical token ``p`` lives
in physical block ``block_table[p // block_size]`` at row ``p % block_size``
[Ch15 §15.6 "PagedAttention：分页 KV Cache" (Block Table / 页表 and the
block_size=4 example); Deploy §2.1 "4. PageAttention 内存管理技术详解" (逻辑块通过 block table
映射到非连续物理块)].  The oracle first walks the block table into a dense
token-major array and only then applies the plain definition; it never uses
the online recurrence.

Readings of points the pages leave open:
  * Cache layout is ``[num_blocks, num_kv_heads, block_size, head_dim]`` (one
    contiguous tile per (block, kv head)); K and V are separate pools.
  * GQA: query head ``h`` reads KV head ``h // (Hq // Hkv)`` (contiguous groups)
    [Deploy §4.1 "4. MQA 与 GQA": a group of Q heads shares one KV head].
  * ``context_lens[s]`` already counts this step's tokens: the new token's K/V
    are written to the cache before attention [Infra 一、推理两阶段 2、解码: 将
    KtVt 更新到 kv cache 中, then attend].  A decode query therefore attends to
    keys 0 .. ctx-1, itself included.
  * A span of ``qlen`` queries of one sequence (a prefill chunk over a cached
    prefix) holds absolute positions ctx-qlen .. ctx-1; query i attends keys
    0 .. ctx-qlen+i (causal) [Ch15 §15.6 两阶段与 Chunked Prefill;
    FastGen §3.2 动态分割融合].
  * scale defaults to 1/sqrt(head_dim).
  * Sliding window ``window`` = W > 0 [Deploy §2.1 block_sliding_window: the
    pages keep only a window of blocks per sequence and say nothing about the
    mask]: a query attends the W most recent keys up to and including its own
    position, i.e. table indices max(0, a - W + 1) .. a for a query at table
    index a.  The table must list the sequence's blocks in logical order (it
    may start past logical block 0, so table index = position - first
    position of the table); W = 0 means no window.
"""

import math

import numpy as np

from .numerics import widen


def gather_sequence(cache, table_row, ctx, block_size):
    """Walk one block table: return the sequence's first ``ctx`` tokens as [ctx, Hkv, D].

    ``cache`` is [num_blocks, Hkv, block_size, D] in the cache's storage dtype.
    """
    if ctx < 0:
        raise ValueError("negative context length")
    nblk = -(-ctx // block_size)
    rows = []
    for j in range(nblk):
        b = int(table_row[j])
        if not 0 <= b < cache.shape[0]:
            raise IndexError(f"block id {b} outside the pool")
        # [Hkv, bs, D] -> [bs, Hkv, D]: tokens of this block in logical order
        rows.append(np.swapaxes(cache[b], 0, 1))
    if not rows:
        return cache[:0, :, :0, :].reshape(0, cache.shape[1], cache.shape[3])
    dense = np.concatenate(rows, axis=0)
    return dense[:ctx]


def softmax_attention(q, k, v, scale, n_visible=None, first_visible=None):
    """Exact attention for a set of query rows against one key/value sequence.

    q: [nq, D] float64; k, v: [n, D] float64.  ``n_visible[i]`` (optional) is
    how many leading keys query row i may see (causal masking); all keys if
    None.  ``first_visible[i]`` (optional) is the first key row i may see (a
    sliding window); key 0 if None.  Returns [nq, D] float64.
    """
    s = (q @ k.T) * scale
    if n_visible is not None:
        n_visible = np.asarray(n_visible)
        if np.any(n_visible < 1) or np.any(n_visible > k.shape[0]):
            raise ValueError("every query must see between 1 and n keys")
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols < n_visible[:, None], s, -np.inf)
    if first_visible is not None:
        first_visible = np.asarray(first_visible)
        last = (np.asarray(n_visible) if n_visible is not None
                else np.full(q.shape[0], k.shape[0]))
        if np.any(first_visible < 0) or np.any(first_visible >= last):
            raise ValueError("every query must see at least one key")
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols >= first_visible[:, None], s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return (p @ v) / p.sum(axis=1, keepdims=True)


def _check_heads(num_q_heads, num_kv_heads):
    if num_kv_heads < 1 or num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    return num_q_heads // num_kv_heads


def _first_visible(last, window):
    """First key a query whose last visible key is ``last`` attends (table indices)."""
    return np.maximum(0, np.asarray(last) - window + 1) if window else None


def decode(q, k_cache, v_cache, block_tables, context_lens, block_size, dtype, scale=None,
           window=0):
    """One query token per sequence.

    q: [S, Hq, D] (cache dtype storage); caches [NB, Hkv, bs, D];
    block_tables [S, W] int; context_lens [S] (>= 1, includes the query's own
    token); ``window`` > 0: a sliding window of that many keys.  Returns
    float64 [S, Hq, D].
    """
    S, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = _check_heads(Hq, Hkv)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qf = widen(q, dtype)
    out = np.empty((S, Hq, D), dtype=np.float64)
    for s in range(S):
        ctx = int(context_lens[s])
        if ctx < 1:
            raise ValueError("context length must be >= 1")
        kd = widen(gather_sequence(k_cache, block_tables[s], ctx, block_size), dtype)
        vd = widen(gather_sequence(v_cache, block_tables[s], ctx, block_size), dtype)
        first = _first_visible([ctx - 1], window)
        for h in range(Hq):
            kvh = h // g
            out[s, h] = softmax_attention(qf[s, h][None, :], kd[:, kvh], vd[:, kvh], scale,
                                          first_visible=first)[0]
    return out


def varlen(q, k_cache, v_cache, block_tables, query_start_loc, context_lens, block_size,
           dtype, scale=None, window=0):
    """Ragged batch: sequence s owns query rows query_start_loc[s] .. query_start_loc[s+1]-1.

    Rows of a sequence are its last ``qlen`` positions; row i sees keys
    0 .. ctx-qlen+i (with a sliding window W > 0: from max(0, ctx-qlen+i-W+1)).
    A sequence with qlen == 1 is a decode row.  Returns float64 [Tq, Hq, D].
    """
    Tq, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    g = _check_heads(Hq, Hkv)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qf = widen(q, dtype)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    S = len(context_lens)
    if qsl.shape != (S + 1,) or qsl[0] != 0 or qsl[-1] != Tq or np.any(np.diff(qsl) < 0):
        raise ValueError("query_start_loc must be a non-decreasing prefix sum from 0 to Tq")
    out = np.full((Tq, Hq, D), np.nan, dtype=np.float64)
    for s in range(S):
        r0, r1 = int(qsl[s]), int(qsl[s + 1])
        qlen = r1 - r0
        if qlen == 0:
            continue
        ctx = int(context_lens[s])
        if qlen > ctx:
            raise ValueError("a sequence cannot have more queries than context tokens")
        kd = widen(gather_sequence(k_cache, block_tables[s], ctx, block_size), dtype)
        vd = widen(gather_sequence(v_cache, block_tables[s], ctx, block_size), dtype)
        n_visible = ctx - qlen + 1 + np.arange(qlen)
        first = _first_visible(n_visible - 1, window)
        for h in range(Hq):
            kvh = h // g
            out[r0:r1, h] = softmax_attention(qf[r0:r1, h], kd[:, kvh], vd[:, kvh], scale,
                                              n_visible, first)
    return out
