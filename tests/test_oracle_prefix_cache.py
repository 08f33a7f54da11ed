"""Pins for the prefix-caching and sliding-window pool models (CPU only)."""

import random

import pytest

from oracle.block_pool import LATER, NEVER, OK
from oracle.prefix_cache import PrefixCachingPool, SlidingWindowPool, block_hash, fnv1a64


def test_fnv1a64_published_vectors():
    # test vectors published with the FNV-1a definition (offset basis, "a", "foobar")
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_is_chained_over_the_whole_prefix():
    a = block_hash(0, [1, 2, 3, 4])
    b = block_hash(a, [5, 6, 7, 8])
    # same block content after a different first block: different hash
    assert block_hash(block_hash(0, [9, 2, 3, 4]), [5, 6, 7, 8]) != b
    # the bytes hashed are prev (8 bytes LE) + tokens (4 bytes LE each)
    raw = (0).to_bytes(8, "little") + b"".join(t.to_bytes(4, "little") for t in (1, 2, 3, 4))
    assert a == fnv1a64(raw)


def _toks(*blocks, tail=()):
    out = []
    for b in blocks:
        out += [b * 100 + i for i in range(4)]
    return out + list(tail)


def test_shared_prefix_blocks_are_reused_and_the_tail_is_private():
    p = PrefixCachingPool(32, 4)
    st, slots_a, cached_a = p.add_sequence("a", _toks(1, 2, 3, tail=(7, 7)))
    assert st == OK and cached_a == 0
    st, slots_b, cached_b = p.add_sequence("b", _toks(1, 2, 9, tail=(7, 7)))
    ta, tb = p.block_table("a"), p.block_table("b")
    assert ta[:2] == tb[:2] and ta[2] != tb[2] and ta[3] != tb[3]     # partial tail never shared
    assert cached_b == 8 and slots_b[:8] == slots_a[:8]
    assert [p.ref[x] for x in ta] == [2, 2, 1, 1]
    # a different first block shares nothing, even when later blocks match
    st, _, cached_c = p.add_sequence("c", _toks(5, 2, 3))
    assert cached_c == 0 and not set(p.block_table("c")) & set(ta)
    # conservation: every block is free, parked or referenced
    used = {x for t in p.tables.values() for x in t}
    assert len(used) + p.num_free() == 32
    assert sum(p.ref) == sum(len(t) for t in p.tables.values())


def test_freed_prefix_is_parked_and_taken_back():
    p = PrefixCachingPool(8, 4)
    p.add_sequence("a", _toks(1, 2, tail=(5,)))
    ta = p.block_table("a")
    p.set_clock(3)
    p.free_sequence("a")
    # the two hashed blocks are parked, the partial one is free again
    assert p.num_evictable() == 2 and p.num_free() == 8
    assert p.free[-1] == ta[2]
    st, slots, cached = p.add_sequence("b", _toks(1, 2, tail=(6,)))
    assert cached == 8 and p.block_table("b")[:2] == ta[:2] and p.num_evictable() == 0


def test_evictor_order_oldest_then_most_tokens_then_first_parked():
    p = PrefixCachingPool(4, 2)
    p.add_sequence("x", [1, 1, 2, 2, 3, 3])         # 3 hashed blocks, 2/4/6 tokens
    p.add_sequence("y", [9, 9])                     # 1 hashed block
    tx, ty = p.block_table("x"), p.block_table("y")
    p.set_clock(10)
    p.free_sequence("y")                            # parked at 10
    p.set_clock(5)
    p.free_sequence("x")                            # parked at 5 (older), in table order
    assert p.num_evictable() == 4 and not p.free
    # new content: evicts clock-5 blocks first, the one covering 6 tokens first
    p.set_clock(20)
    p.add_sequence("z", [7, 7])
    assert p.block_table("z") == [tx[2]]
    p.add_sequence("w", [8, 8, 8, 8])
    assert p.block_table("w") == [tx[1], tx[0]]
    # the clock-10 block is the last one left, and its prefix still hits
    st, _, cached = p.add_sequence("v", [9, 9])
    assert p.block_table("v")[0] == ty[0] and cached == 2
    # nothing left: admission says LATER, and NEVER for more than the pool
    assert p.can_allocate(2) == LATER and p.can_allocate(9) == NEVER


def test_filled_block_is_promoted_to_an_existing_copy():
    p = PrefixCachingPool(16, 4)
    p.add_sequence("a", _toks(1, 2))                # two hashed blocks
    p.add_sequence("b", _toks(1, tail=(200, 201, 202)))
    tb = p.block_table("b")
    assert p.block_table("a")[0] == tb[0]
    private = tb[1]
    slot, cow = p.append_token("b", 203)            # fills block 1 with a's tokens
    assert cow is None and p.block_table("b")[1] == p.block_table("a")[1]
    assert slot == p.block_table("a")[1] * 4 + 3 and p.free[-1] == private
    # no match: the filled block is registered and shared with the next prompt
    p.add_sequence("c", _toks(1, tail=(200, 201)))
    p.append_token("c", 777)
    p.append_token("c", 778)
    h = block_hash(block_hash(0, _toks(1)), [200, 201, 777, 778])
    assert p.cached[h] == p.block_table("c")[1]
    st, _, cached = p.add_sequence("d", _toks(1) + [200, 201, 777, 778, 5])
    assert cached == 8 and p.block_table("d")[1] == p.block_table("c")[1]


def test_copy_on_write_in_a_shared_partial_block_then_promotion_cancels_it():
    p = PrefixCachingPool(16, 4)
    p.add_sequence("a", [1, 2, 3, 4, 5, 6, 7, 8])
    p.add_sequence("b", [1, 2, 3, 4, 5, 6, 9])
    p.fork("b", "b2")
    shared = p.block_table("b")[1]
    slot, cow = p.append_token("b", 10)             # shared partial block: copy
    assert cow == (shared, p.block_table("b")[1]) and p.ref[shared] == 1
    # b's copy, now full, was registered under the hash of 1..6, 9, 10; b2 (sole
    # owner of the old block) fills it with the same tokens and switches to b's copy
    slot, cow = p.append_token("b2", 10)
    assert cow is None and p.block_table("b2")[1] == p.block_table("b")[1]
    assert p.ref[shared] == 0 and p.free[-1] == shared
    # a fork whose shared tail is filled to a known block: copy cancelled
    p.add_sequence("e", [1, 2, 3, 4, 5, 6, 7])
    p.fork("e", "e2")
    slot, cow = p.append_token("e2", 8)
    assert cow is None and p.block_table("e2")[1] == p.block_table("a")[1]


def test_prefix_pool_random_traces_keep_invariants():
    rng = random.Random(0)
    for trial in range(30):
        bs = rng.choice([1, 2, 4])
        p = PrefixCachingPool(40, bs, rng.choice([0, 2]), rng.sample(range(40), 40))
        live, nxt = [], 0
        for step in range(120):
            p.set_clock(step // 3)
            op = rng.random()
            if op < 0.3 or not live:
                toks = [rng.choice([1, 2, 3]) for _ in range(rng.randint(1, 12))]
                st, slots, cached = p.add_sequence(nxt, toks)
                if st == OK:
                    assert cached % bs == 0 and cached <= len(toks)
                    assert len(set(slots)) == len(slots)
                    live.append(nxt)
                nxt += 1
            elif op < 0.75:
                s = rng.choice(live)
                p.append_token(s, rng.choice([1, 2, 3]))
            elif op < 0.85:
                p.fork(rng.choice(live), nxt)
                live.append(nxt)
                nxt += 1
            else:
                s = live.pop(rng.randrange(len(live)))
                p.free_sequence(s)
            used = {x for t in p.tables.values() for x in t}
            assert len(used) + len(p.free) + len(p.evictor) == 40
            assert not used & set(p.free) and not used & set(p.evictor)
            for b in range(40):
                assert p.ref[b] == sum(t.count(b) for t in p.tables.values())
            # every full block of every sequence holds the hash of its prefix
            for s, t in p.tables.items():
                toks, prev = p.tokens[s], 0
                for j in range(len(toks) // bs):
                    prev = block_hash(prev, toks[j * bs:(j + 1) * bs])
                    assert p.hash_of[t[j]] in (prev, None)


def test_sliding_window_worked_example():
    # bs 4, window 8 (2 ring blocks), prompt of 10 tokens
    p = SlidingWindowPool(16, 4, 8, free_order=[5, 6] + [b for b in range(16) if b not in (5, 6)])
    st, slots = p.add_sequence("s", 10)
    assert st == OK and p.tables["s"] == [5, 6]
    assert slots == [-1, -1, 22, 23, 24, 25, 26, 27, 20, 21]
    assert p.window_table("s") == ([6, 5], 8)
    slot, cow = p.append_slot("s")                  # position 10 -> block 5 row 2
    assert slot == 22 and cow is None
    assert p.can_allocate(100) == OK and p.blocks_needed(100) == 2


def test_sliding_window_holds_exactly_the_last_window_tokens():
    rng = random.Random(1)
    for trial in range(40):
        bs = rng.choice([1, 2, 4, 16])
        window = bs * rng.randint(1, 6)
        p = SlidingWindowPool(64, bs, window)
        n0 = rng.randint(1, 3 * window)
        st, slots = p.add_sequence(0, n0)
        holder = {}
        for pos, s in enumerate(slots):
            if s >= 0:
                assert s not in holder
                holder[s] = pos
        for _ in range(rng.randint(0, 3 * window)):
            pos = p.context_len(0)
            s, cow = p.append_slot(0)
            holder[s] = pos
        n = p.context_len(0)
        table, ctx = p.window_table(0)
        held = sorted(holder[table[i // bs] * bs + i % bs] for i in range(ctx))
        assert held == list(range(n - ctx, n)) and ctx == min(n, window)


def test_sliding_window_fork_copies_a_shared_ring_block():
    p = SlidingWindowPool(16, 2, 4)
    p.add_sequence("a", 6)                          # ring full: [b0, b1], next write into b0
    p.fork("a", "b")
    ring = list(p.tables["b"])
    slot, cow = p.append_slot("a")                  # position 6: logical block 3 -> ring entry 1
    assert cow == (ring[1], p.tables["a"][1]) and p.tables["b"] == ring
    assert slot == p.tables["a"][1] * 2 and p.ref[ring[1]] == 1
    with pytest.raises(Exception):
        SlidingWindowPool(16, 4, 6)                 # window not a multiple of block_size
