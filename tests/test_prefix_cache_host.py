"""The C++ pool's prefix-caching and sliding-window variants against the oracle
models, operation by operation on random traces (host only, no GPU)."""

import random

import pytest

from oracle.block_pool import LATER, NEVER, OK
from oracle.prefix_cache import PrefixCachingPool, SlidingWindowPool

_ST = {0: OK, -2: LATER, -3: NEVER}


def _compare_state(lib, cpp, ora, live, n_blocks, window=False):
    assert cpp.num_free() == ora.num_free()
    for b in range(n_blocks):
        assert cpp.ref_count(b) == ora.ref[b]
    if live:
        width = max(len(ora.tables[s]) for s in live) + 1
        tables, ctx = cpp.block_tables(live, width)
        for i, s in enumerate(live):
            if window:
                want, wctx = ora.window_table(s)
            else:
                want, wctx = ora.tables[s], ora.context_len(s)
            assert tables[i, :len(want)].tolist() == want
            assert int(ctx[i]) == wctx


@pytest.mark.parametrize("seed", range(12))
def test_prefix_caching_pool_matches_oracle(lib, seed):
    rng = random.Random(seed)
    nb = rng.choice([12, 24, 40])
    bs = rng.choice([1, 2, 4, 16])
    wm = rng.choice([0, 0, 2])
    order = rng.sample(range(nb), nb)
    cpp = lib.BlockPool(nb, bs, wm, order, prefix_caching=True)
    ora = PrefixCachingPool(nb, bs, wm, order)
    vocab = [rng.randint(-3, 3) for _ in range(3)]
    live, nxt = [], 0
    for step in range(150):
        now = step // 4
        cpp.set_clock(now)
        ora.set_clock(now)
        op = rng.random()
        if op < 0.3 or not live:
            toks = [rng.choice(vocab) for _ in range(rng.randint(1, 3 * bs + 2))]
            st, slots, cached = cpp.add_tokens(nxt, toks)
            ost, oslots, ocached = ora.add_sequence(nxt, toks)
            assert _ST[st] == ost
            if ost == OK:
                assert slots == oslots and cached == ocached
                live.append(nxt)
            nxt += 1
        elif op < 0.75:
            s = rng.choice(live)
            t = rng.choice(vocab)
            st, slot, cow = cpp.append_token(s, t)
            oslot, ocow = ora.append_token(s, t)
            if oslot is None:
                assert st == -2
            else:
                assert st == 0 and slot == oslot and cow == ocow
        elif op < 0.85:
            p = rng.choice(live)
            cpp.fork(p, nxt)
            ora.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        else:
            s = live.pop(rng.randrange(len(live)))
            cpp.free(s)
            ora.free_sequence(s)
        assert cpp.num_evictable() == ora.num_evictable()
        for b in range(nb):
            assert cpp.block_hash(b) == ora.hash_of[b]
        _compare_state(lib, cpp, ora, live, nb)


@pytest.mark.parametrize("seed", range(12))
def test_sliding_window_pool_matches_oracle(lib, seed):
    rng = random.Random(100 + seed)
    nb = rng.choice([8, 16, 40])
    bs = rng.choice([1, 2, 4, 16])
    window = bs * rng.randint(1, 4)
    order = rng.sample(range(nb), nb)
    cpp = lib.BlockPool(nb, bs, 0, order, sliding_window=window)
    ora = SlidingWindowPool(nb, bs, window, 0, order)
    live, nxt = [], 0
    for step in range(150):
        op = rng.random()
        if op < 0.25 or not live:
            n = rng.randint(1, 3 * window)
            st, slots = cpp.add_status(nxt, n)
            ost, oslots = ora.add_sequence(nxt, n)
            assert _ST[st] == ost
            if ost == OK:
                assert slots == oslots
                live.append(nxt)
            nxt += 1
        elif op < 0.8:
            s = rng.choice(live)
            st, slot, cow = cpp.append_slot_status(s)
            oslot, ocow = ora.append_slot(s)
            if oslot is None:
                assert st == -2
            else:
                assert st == 0 and slot == oslot and cow == ocow
        elif op < 0.88:
            p = rng.choice(live)
            cpp.fork(p, nxt)
            ora.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        else:
            s = live.pop(rng.randrange(len(live)))
            cpp.free(s)
            ora.free_sequence(s)
        _compare_state(lib, cpp, ora, live, nb, window=True)


def test_variant_rules_at_the_boundary(lib):
    L = lib.lib()
    import ctypes

    h = ctypes.c_void_p()
    # the pages refuse prefix caching with a sliding window
    assert L.pkv_pool_create_ex(16, 4, 0, None, 1, 8, ctypes.byref(h)) == lib.PKV_ERR_UNSUPPORTED
    assert L.pkv_pool_create_ex(16, 4, 0, None, 0, 6, ctypes.byref(h)) == lib.PKV_ERR_INVALID
    assert L.pkv_pool_create_ex(16, 4, 0, None, 4, 0, ctypes.byref(h)) == lib.PKV_ERR_INVALID
    pool = lib.BlockPool(16, 4, prefix_caching=True)
    # count-only calls need token ids on a prefix-caching pool
    assert lib.lib().pkv_seq_add(pool._h, 1, 5, None) == lib.PKV_ERR_UNSUPPORTED
    st, slots, cached = pool.add_tokens(1, [1, 2, 3, 4, 5])
    assert st == 0 and cached == 0
    slot = ctypes.c_int64()
    assert L.pkv_seq_append_slot(pool._h, 1, ctypes.byref(slot), None, None) == \
        lib.PKV_ERR_UNSUPPORTED
    # a plain pool takes token ids too, and reports nothing cached
    plain = lib.BlockPool(16, 4)
    st, slots, cached = plain.add_tokens(7, [1, 2, 3, 4, 5])
    tables, ctx = plain.block_tables([7], 2)
    t = tables[0].tolist()
    assert st == 0 and cached == 0 and int(ctx[0]) == 5
    assert slots == [t[p // 4] * 4 + p % 4 for p in range(5)]


def _compare_window_tables(lib, cpp, ora, live):
    """pkv_window_tables against the oracle's logical export, for random query spans."""
    rng = random.Random(len(live) * 7 + 1)
    ids, qlens, want = [], [], []
    for s in live:
        n = ora.context_len(s)
        top = min(n, ora.capacity - ora.window + 1)
        q = rng.randint(1, top)
        ids.append(s)
        qlens.append(q)
        want.append(ora.logical_table(s, q))
    width = max(len(t) for t, _ in want) + 1
    tables, ctx = cpp.window_tables(ids, qlens, width)
    for i, (t, c) in enumerate(want):
        assert tables[i, :len(t)].tolist() == t and int(ctx[i]) == c
        assert (tables[i, len(t):] == -1).all()


@pytest.mark.parametrize("seed", range(12))
def test_chunked_window_pool_matches_oracle(lib, seed):
    """Rings with room for prefill chunks: sequences added with a chunk and grown by
    chunks or single tokens, forked and freed, in the C++ pool and the oracle."""
    rng = random.Random(300 + seed)
    bs = rng.choice([1, 2, 4, 16])
    window = bs * rng.randint(1, 4)
    chunk = rng.randint(2, 3 * window)
    ring = window // bs + -(-(chunk - 1) // bs)
    nb = ring * rng.randint(2, 6)
    order = rng.sample(range(nb), nb)
    cpp = lib.BlockPool(nb, bs, 0, order, sliding_window=window, max_chunk=chunk)
    ora = SlidingWindowPool(nb, bs, window, 0, order, max_chunk=chunk)
    live, nxt = [], 0
    for step in range(150):
        op = rng.random()
        if op < 0.2 or not live:
            n = rng.randint(1, chunk)
            st, slots = cpp.add_status(nxt, n)
            ost, oslots = ora.add_sequence(nxt, n)
            assert _ST[st] == ost
            if ost == OK:
                assert slots == oslots and -1 not in slots
                live.append(nxt)
            nxt += 1
        elif op < 0.8:
            s = rng.choice(live)
            for _ in range(rng.choice([1, 1, rng.randint(1, chunk)])):
                st, slot, cow = cpp.append_slot_status(s)
                oslot, ocow = ora.append_slot(s)
                if oslot is None:
                    assert st == -2
                    break
                assert st == 0 and slot == oslot and cow == ocow
        elif op < 0.88:
            p = rng.choice(live)
            cpp.fork(p, nxt)
            ora.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        else:
            s = live.pop(rng.randrange(len(live)))
            cpp.free(s)
            ora.free_sequence(s)
        assert cpp.num_free() == ora.num_free()
        for b in range(nb):
            assert cpp.ref_count(b) == ora.ref[b]
        if live:
            _compare_window_tables(lib, cpp, ora, live)


def test_window_table_rules_at_the_boundary(lib):
    import ctypes

    L = lib.lib()
    h = ctypes.c_void_p()
    assert L.pkv_pool_create_window(16, 4, 0, None, 0, 4, ctypes.byref(h)) == lib.PKV_ERR_INVALID
    assert L.pkv_pool_create_window(16, 4, 0, None, 6, 4, ctypes.byref(h)) == lib.PKV_ERR_INVALID
    assert L.pkv_pool_create_window(16, 4, 0, None, 8, 0, ctypes.byref(h)) == lib.PKV_ERR_INVALID
    pool = lib.BlockPool(32, 4, 0, sliding_window=8, max_chunk=6)   # ring 2 + 2 blocks
    assert pool.add_status(1, 6)[0] == 0
    # the exact-window export does not exist on a ring with chunk room
    with pytest.raises(lib.PagedKVError) as e:
        pool.block_tables([1], 4)
    assert e.value.status == lib.PKV_ERR_UNSUPPORTED
    # a span the ring cannot hold (6 + 8 - 1 <= 16 is the most), a span above the length
    tables, ctx = pool.window_tables([1], [6], 4)
    assert int(ctx[0]) == 6
    for q in (7, 0):
        with pytest.raises(lib.PagedKVError) as e:
            pool.window_tables([1], [q], 4)
        assert e.value.status == lib.PKV_ERR_INVALID
    for _ in range(20):
        pool.append_slot(1)
    with pytest.raises(lib.PagedKVError):
        pool.window_tables([1], [10], 8)
    # a pool without a window has no window export
    plain = lib.BlockPool(8, 4)
    plain.add(1, 3)
    with pytest.raises(lib.PagedKVError) as e:
        plain.window_tables([1], [1], 2)
    assert e.value.status == lib.PKV_ERR_UNSUPPORTED
