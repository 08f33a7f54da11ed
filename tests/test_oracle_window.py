"""Pins for the oracle's sliding-window attention and its chunk-capable ring
(CPU only).

The pages keep a sliding window of blocks per sequence ("大模型部署.md" §2.1
block_sliding_window: logical block j >= W_b reuses table entry j mod W_b) and
leave the attention mask open; the reading taken is that a query at position p
sees keys max(0, p - W + 1) .. p.  A chunk of C queries then needs C + W - 1
keys at once, so a pool serving chunks keeps W_b + ceil((C - 1) / bs) ring
blocks and exports logically ordered tables.  These tests pin that chain to
brute force on the unpaged rows: a plausible mistake in the ring size, the
export's first block, the context it reports or the window mask fails one.
"""

import numpy as np
import pytest

import workloads
from oracle import attention
from oracle.block_pool import OK, PoolError
from oracle.prefix_cache import SlidingWindowPool
from oracle.run import execute, execute_window_trace
from tests import bruteforce


def _lens_after(tr):
    lens, out = {}, []
    for step in tr.steps:
        for seq, qlen in step:
            lens[seq] = lens.get(seq, 0) + qlen
        out.append(dict(lens))
    return out


@pytest.mark.parametrize("dtype,bs,window,chunk", [("f32", 4, 8, 6), ("bf16", 4, 12, 1),
                                                   ("bf16", 8, 16, 9), ("f32", 4, 8, 13)])
def test_chunked_windowed_trace_matches_brute_force(dtype, bs, window, chunk):
    tr = workloads.window_trace(3, dtype, 4, 2, 8, bs, window, chunk, prompts=(23, 5, 40),
                                gens=(4, 9, 2), scale=1.0)
    outs, _, _ = execute_window_trace(tr)
    lens = _lens_after(tr)
    assert len(tr.steps) > 3
    for i, out in enumerate(outs):
        ref = np.array(bruteforce.window_trace_step(tr, i, lens[i]))
        assert np.abs(out - ref).max() <= 1e-12, i


def test_window_off_by_one_is_detected():
    tr = workloads.window_trace(4, "f32", 4, 2, 8, 4, 8, 6, prompts=(30,), gens=(3,), scale=1.0)
    lens = _lens_after(tr)
    for wrong in (tr.window - 1, tr.window + 1):
        tr2 = workloads.window_trace(4, "f32", 4, 2, 8, 4, 8, 6, prompts=(30,), gens=(3,),
                                     scale=1.0)
        tr2.window = wrong
        try:
            outs, _, _ = execute_window_trace(tr2)
        except PoolError:
            continue                       # a narrower ring refuses the chunk outright
        worst = max(np.abs(out - np.array(bruteforce.window_trace_step(tr, i, lens[i]))).max()
                    for i, out in enumerate(outs))
        assert worst > 1e-3


def test_window_covering_the_context_changes_nothing():
    w = workloads.random_varlen(5, "f32", 8, 4, 16, 4, [(0, 9), (13, 6), (30, 1)])
    ost, ref = execute(w)
    bt, ctx, qsl = ost.batch_metadata()
    got = attention.varlen(w.q, ost.k_cache, ost.v_cache, bt, qsl, ctx, w.block_size, w.dtype,
                           window=int(ctx.max()))
    assert np.array_equal(got, ref)
    dec = workloads.random_decode(6, "f32", 8, 4, 16, 4, [5, 17])
    ost, ref = execute(dec)
    bt, ctx, _ = ost.batch_metadata()
    got = attention.decode(dec.q, ost.k_cache, ost.v_cache, bt, ctx, 4, "f32", window=17)
    assert np.array_equal(got, ref)


def test_window_of_one_returns_the_query_own_value():
    w = workloads.random_varlen(7, "f32", 4, 2, 8, 4, [(6, 5), (0, 3)])
    ost, _ = execute(w)
    bt, ctx, qsl = ost.batch_metadata()
    got = attention.varlen(w.q, ost.k_cache, ost.v_cache, bt, qsl, ctx, w.block_size, w.dtype,
                           window=1)
    rows = bruteforce.dense_sequences(w)
    r = 0
    for seq, qlen in w.batch:
        toks = rows[seq]
        for i in range(qlen):
            own = toks[len(toks) - qlen + i]
            for h in range(4):
                assert np.array_equal(got[r, h], w.v_rows[own, h // 2].astype(np.float64))
            r += 1


def test_ring_size_and_logical_export():
    # bs 4, window 8 (W_b = 2), chunks of up to 6: ring = 2 + ceil(5 / 4) = 4 blocks
    p = SlidingWindowPool(32, 4, 8, max_chunk=6)
    assert p.ring == 4 and p.capacity == 16
    st, slots = p.add_sequence("s", 6)
    assert st == OK and -1 not in slots
    for _ in range(6):
        p.append_slot("s")
    # 12 tokens, next step's queries are its last 6: keys from position 12 - 6 - 8 + 1 = -1 -> 0
    t, c = p.logical_table("s", 6)
    assert c == 12 and len(t) == 3
    for _ in range(9):
        p.append_slot("s")
    # 21 tokens; last 6 queries attend from 21 - 6 - 8 + 1 = 8 -> block 2; context 21 - 8 = 13
    t, c = p.logical_table("s", 6)
    assert c == 13 and t == [p.tables["s"][j % 4] for j in (2, 3, 4, 5)]
    # one decode query: from position 13 -> block 3 (rows 1.. of it), context 21 - 12 = 9
    t, c = p.logical_table("s", 1)
    assert c == 9 and t == [p.tables["s"][j % 4] for j in (3, 4, 5)]
    # a span the ring cannot hold is refused; so is the rotated export on this ring
    with pytest.raises(PoolError):
        p.logical_table("s", 10)
    with pytest.raises(PoolError):
        p.window_table("s")
    # the pages' ring (max_chunk 1) is unchanged
    q = SlidingWindowPool(32, 4, 8)
    assert q.ring == 2 and q.capacity == 8


def test_prompt_longer_than_the_ring_skips_only_overwritten_tokens():
    p = SlidingWindowPool(32, 4, 8, max_chunk=5)         # ring 2 + 1 = 3 blocks, 12 tokens
    st, slots = p.add_sequence("a", 20)
    assert st == OK and slots[:8] == [-1] * 8 and -1 not in slots[8:]
    assert len(set(slots[8:])) == 12
