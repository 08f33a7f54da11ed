"""Pins for the block-pool model and the cache mirror (CPU only)."""

import numpy as np
import pytest

from oracle import cache
from oracle.block_pool import LATER, NEVER, OK, BlockPoolModel
from tests.conftest import read_kv, read_rows


def test_paging_example_block_size_4():
    g = read_kv("paging_example_bs4.txt")
    bs = int(g["block_size"])
    head = [int(x) for x in g["free_order_head"].split()]
    order = head + [b for b in range(16) if b not in head]
    pool = BlockPoolModel(16, bs, 0, order)
    st, slots = pool.add_sequence(0, int(g["prompt_tokens"]))
    assert st == OK
    assert pool.block_table(0) == [int(x) for x in g["prompt_table"].split()]
    assert slots == [int(x) for x in g["prompt_slots"].split()]
    slot, cow = pool.append_slot(0)
    assert cow is None
    assert slot == int(g["next_token_slot"])
    assert slot // bs == int(g["next_token_block"]) and slot % bs == 0
    assert pool.block_table(0) == [int(x) for x in g["table_after"].split()]


def test_internal_fragmentation_example():
    g = read_kv("fragmentation_example.txt")
    bs, n = int(g["block_size"]), int(g["tokens"])
    pool = BlockPoolModel(4, bs)
    assert pool.blocks_needed(n) == int(g["blocks"])
    assert pool.blocks_needed(n) * bs == int(g["capacity"])
    assert pool.blocks_needed(n) * bs - n == int(g["wasted"])


@pytest.mark.parametrize("row", read_rows("admission_cases.txt"))
def test_admission_cases(row):
    total, wm, used, bs, tokens = (int(x) for x in row[:5])
    want = row[5]
    pool = BlockPoolModel(total, bs, wm)
    if used:
        assert pool.add_sequence(99, used * bs)[0] == OK
    assert pool.num_free() == total - used
    assert pool.can_allocate(tokens) == want
    st, slots = pool.add_sequence(1, tokens)
    assert st == want
    assert (slots is not None) == (want == OK)


def test_fork_and_copy_on_write_of_shared_tail():
    bs = 16
    pool = BlockPoolModel(300, bs)
    pool.add_sequence(0, 3000)              # 187 full blocks + 8 tokens in block 188
    tail = pool.block_table(0)[-1]
    for c in range(1, 9):
        pool.fork(0, c)
    pool.free_sequence(0)
    assert pool.ref[tail] == 8
    pairs = []
    for c in range(1, 9):
        slot, cow = pool.append_slot(c)
        pairs.append(cow)
        assert slot // bs == pool.block_table(c)[-1] and slot % bs == 3000 % bs
    # the first seven appenders copy the shared tail; the last holder writes in place
    assert all(p is not None and p[0] == tail for p in pairs[:7])
    assert pairs[7] is None and pool.block_table(8)[-1] == tail
    assert len({p[1] for p in pairs[:7]}) == 7
    # every full prompt block is still shared by all eight branches
    for b in pool.block_table(1)[:-1]:
        assert pool.ref[b] == 8
    _check_invariants(pool)


def test_exhaustion_changes_nothing():
    pool = BlockPoolModel(2, 4)
    pool.add_sequence(0, 8)
    before = (pool.block_table(0), pool.context_len(0), pool.num_free())
    assert pool.append_slot(0) == (None, None)
    assert (pool.block_table(0), pool.context_len(0), pool.num_free()) == before
    assert pool.can_allocate(1) == LATER
    assert pool.can_allocate(9) == NEVER


def _check_invariants(pool):
    refs = [0] * pool.num_blocks
    for t in pool.tables.values():
        for b in t:
            refs[b] += 1
    assert refs == pool.ref
    live = sum(1 for r in pool.ref if r > 0)
    assert live + pool.num_free() == pool.num_blocks
    for s, t in pool.tables.items():
        assert len(t) == pool.blocks_needed(pool.context_len(s))


def test_random_operation_invariants():
    rng = np.random.default_rng(7)
    pool = BlockPoolModel(200, 8, 0, rng.permutation(200))
    next_id = 0
    for _ in range(3000):
        op = rng.integers(0, 4)
        seqs = list(pool.tables)
        if op == 0 or not seqs:
            if pool.add_sequence(next_id, int(rng.integers(1, 40)))[0] == OK:
                next_id += 1
        elif op == 1:
            pool.append_slot(seqs[rng.integers(len(seqs))])
        elif op == 2 and len(seqs) < 40:
            pool.fork(seqs[rng.integers(len(seqs))], next_id)
            next_id += 1
        elif op == 3:
            pool.free_sequence(seqs[rng.integers(len(seqs))])
        _check_invariants(pool)


def test_cache_append_places_tokens_and_skips_padding():
    bs, nb, hkv, d = 4, 5, 2, 3
    kc = np.zeros((nb, hkv, bs, d), dtype=np.float32)
    vc = np.zeros_like(kc)
    k = np.arange(3 * hkv * d, dtype=np.float32).reshape(3, hkv, d) + 1
    v = -k
    cache.append(kc, vc, k, v, [13, -1, 2], bs)
    assert np.array_equal(kc[3, :, 1, :], k[0]) and np.array_equal(vc[3, :, 1, :], v[0])
    assert np.array_equal(kc[0, :, 2, :], k[2])
    assert np.count_nonzero(kc) == 2 * hkv * d
    with pytest.raises(ValueError):
        cache.append(kc, vc, k[:2], v[:2], [7, 7], bs)
    with pytest.raises(IndexError):
        cache.append(kc, vc, k[:1], v[:1], [nb * bs], bs)
    with pytest.raises(TypeError):
        cache.append(kc, vc, k.astype(np.float64), v, [1, 2, 3], bs)


def test_copy_blocks_copies_whole_block():
    kc = np.random.default_rng(0).standard_normal((4, 2, 4, 3)).astype(np.float32)
    vc = kc + 1
    k0, v0 = kc.copy(), vc.copy()
    cache.copy_blocks(kc, vc, [(1, 3), (0, 2)])
    assert np.array_equal(kc[3], k0[1]) and np.array_equal(vc[2], v0[0])
    assert np.array_equal(kc[:2], k0[:2])
