"""Pins for the attention oracle (CPU only).

Each check compares the oracle with something other than itself: brute force
on unpaged data, exact special cases, the pages' own fp32 check, invariants of
the block table, and a negative control.
"""

import math

import numpy as np
import pytest

import workloads
from oracle import attention, numerics, online, sketch
from oracle.run import OracleState, execute
from tests import bruteforce
from tests.conftest import read_kv


def _max_err(out, ref):
    err = 0.0
    for r, heads in enumerate(ref):
        for h, vec in enumerate(heads):
            err = max(err, float(np.max(np.abs(out[r, h] - np.array(vec)))))
    return err


def test_config1_decode_matches_bruteforce_on_unpaged_data():
    w = workloads.config1()
    _, out = execute(w)
    ref = bruteforce.run(w)
    assert _max_err(out, ref) <= 1e-13


@pytest.mark.parametrize("ctx", [[1, 16, 17, 33], [5, 48, 2, 31]])
def test_bf16_gqa_decode_matches_bruteforce(ctx):
    w = workloads.random_decode(3, "bf16", 8, 2, 32, 16, ctx, scale=0.5)
    _, out = execute(w)
    assert _max_err(out, bruteforce.run(w)) <= 1e-13


def test_varlen_causal_matches_bruteforce():
    # (cached prefix, new query tokens): chunk over prefix, chunk from empty,
    # decode row, chunk that ends exactly on a block boundary
    spans = [(7, 3), (0, 5), (20, 1), (3, 13), (16, 16)]
    w = workloads.random_varlen(5, "bf16", 4, 2, 16, 4, spans, scale=0.7)
    _, out = execute(w)
    assert _max_err(out, bruteforce.run(w)) <= 1e-13


def test_varlen_row_equals_decode_at_that_position():
    spans = [(9, 6)]
    w = workloads.random_varlen(8, "f32", 4, 4, 8, 4, spans)
    st, out = execute(w)
    bt, ctx, _ = st.batch_metadata()
    for i in range(6):
        single = attention.decode(w.q[i:i + 1], st.k_cache, st.v_cache, bt, [9 + i + 1], 4, "f32")
        assert np.max(np.abs(single[0] - out[i])) <= 1e-14


def test_block_permutation_invariance_is_bitwise():
    w = workloads.random_decode(11, "bf16", 4, 4, 16, 4, [3, 9, 27, 40], scale=1.0)
    st, out = execute(w)
    bt, ctx, _ = st.batch_metadata()
    rng = np.random.default_rng(0)
    perm = rng.permutation(w.num_blocks)          # new id of old block b is perm[b]
    k2 = np.empty_like(st.k_cache)
    v2 = np.empty_like(st.v_cache)
    k2[perm] = st.k_cache
    v2[perm] = st.v_cache
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    out2 = attention.decode(w.q, k2, v2, bt2, ctx, 4, "bf16")
    assert np.array_equal(out, out2)


def test_shared_prefix_branches():
    """Two branches forked from one prompt share its blocks; identical private tokens
    give identical outputs, and each output equals dense attention over prompt + private."""
    bs = 4
    rng = np.random.default_rng(2)
    prompt, priv = 10, 3
    hq = hkv = 2
    d = 8
    k_rows = rng.standard_normal((prompt + priv, hkv, d), dtype=np.float32)
    v_rows = rng.standard_normal((prompt + priv, hkv, d), dtype=np.float32)
    q = np.repeat(rng.standard_normal((1, hq, d), dtype=np.float32), 2, axis=0)
    setup = [("add", 0, prompt, 0), ("fork", 0, 1), ("fork", 0, 2), ("free", 0),
             ("grow", 1, priv, prompt), ("grow", 2, priv, prompt)]
    w = workloads.Workload("branches", "f32", hq, hkv, d, bs, 16, np.arange(16, dtype=np.int32),
                           setup, [], [(1, 1), (2, 1)], q, k_rows, v_rows)
    st, out = execute(w)
    assert np.array_equal(out[0], out[1])
    bt, _, _ = st.batch_metadata()
    assert bt[0][0] == bt[1][0] and bt[0][1] == bt[1][1]      # full prompt blocks shared
    assert bt[0][2] != bt[1][2]                                # partial tail was copied
    rows = {1: list(range(prompt + priv)), 2: list(range(prompt + priv))}
    assert _max_err(out, bruteforce.run(w, rows)) <= 1e-13


def test_special_cases():
    d = 16
    rng = np.random.default_rng(1)
    k = rng.standard_normal((9, d))
    v = rng.standard_normal((9, d))
    q = rng.standard_normal((1, d))
    # one key: output is that value row, exactly
    assert np.array_equal(attention.softmax_attention(q, k[:1], v[:1], 0.25)[0], v[0])
    # zero query: uniform weights, output is the mean of V
    o = attention.softmax_attention(np.zeros((1, d)), k, v, 0.25)[0]
    assert np.max(np.abs(o - v.mean(axis=0))) <= 1e-15
    # constant V rows: output is that row
    vc = np.tile(v[3], (9, 1))
    assert np.max(np.abs(attention.softmax_attention(q, k, vc, 0.25)[0] - v[3])) <= 1e-15
    # one key scoring 60 above all others dominates to within e^-60
    kk = np.zeros((9, d))
    qq = np.zeros((1, d))
    qq[0, 0] = 1.0
    kk[5, 0] = 60.0
    o = attention.softmax_attention(qq, kk, v, 1.0)[0]
    assert np.max(np.abs(o - v[5])) <= 8 * math.exp(-60) * np.max(np.abs(v)) * 2


def test_widen_bf16_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [1.0, -1.0, 0.0, 3.140625, 3.3895313892515355e38, 9.183549615799121e-41]
    assert numerics.widen(bits, "bf16").tolist() == want
    assert numerics.bf16_bits_from_f64_exact([1.0, -2.5]).tolist() == [0x3F80, 0xC020]
    with pytest.raises(ValueError):
        numerics.bf16_bits_from_f64_exact([1.0 + 2 ** -10])


def test_negative_control_per_block_sketch_is_not_attention():
    rng = np.random.default_rng(4)
    d, bs = 16, 4
    k = rng.standard_normal((13, d))
    v = rng.standard_normal((13, d))
    q = rng.standard_normal(d)
    exact = attention.softmax_attention(q[None], k, v, 0.25)[0]
    bad = sketch.per_block_softmax(q, k, v, 0.25, bs)
    assert np.max(np.abs(exact - bad)) > 0.1
    # with a single block the sketch coincides with attention
    one = sketch.per_block_softmax(q, k[:bs], v[:bs], 0.25, bs)
    assert np.max(np.abs(one - attention.softmax_attention(q[None], k[:bs], v[:bs], 0.25)[0])) < 1e-14


@pytest.mark.parametrize("tile", [1, 3, 16, 64, 1000])
def test_online_recurrence_equals_exact(tile):
    rng = np.random.default_rng(tile)
    q = rng.standard_normal((5, 32))
    k = rng.standard_normal((203, 32)) * 2
    v = rng.standard_normal((203, 32))
    ref = attention.softmax_attention(q, k, v, 0.3)
    assert np.max(np.abs(online.attention_online(q, k, v, 0.3, tile) - ref)) <= 1e-12


@pytest.mark.parametrize("split", [1, 16, 50, 512])
def test_split_merge_equals_exact(split):
    rng = np.random.default_rng(split)
    q = rng.standard_normal((4, 16))
    k = rng.standard_normal((300, 16)) * 3
    v = rng.standard_normal((300, 16))
    ref = attention.softmax_attention(q, k, v, 0.25)
    assert np.max(np.abs(online.attention_split(q, k, v, 0.25, 16, split) - ref)) <= 1e-12


def test_pages_fp32_tiled_check():
    """Rerun the page's experiment: tiled online softmax vs standard attention, fp32,
    N=128, d=64, tiles of 32, seed 42; the page prints a max difference of 2.98e-07
    and asserts atol 1e-5."""
    torch = pytest.importorskip("torch")
    g = read_kv("online_softmax_check.txt")
    n, d, tile = int(g["N"]), int(g["d"]), int(g["tile_cols"])
    torch.manual_seed(int(g["seed"]))
    Q, K, V = (torch.randn(n, d).numpy() for _ in range(3))
    scale = 1.0 / math.sqrt(d)
    s = (Q @ K.T) * np.float32(scale)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    std = (p / p.sum(axis=1, keepdims=True)) @ V
    tiled = np.concatenate([online.attention_online(Q[i:i + tile], K, V, scale, tile)
                            for i in range(0, n, tile)])
    assert tiled.dtype == np.float32
    diff = float(np.max(np.abs(std - tiled)))
    assert diff <= float(g["asserted_atol"])
    # same order of magnitude as the printed value (fp32 rounding only)
    assert float(g["printed_max_difference"]) / 20 <= diff <= float(g["printed_max_difference"]) * 20
    # and in float64 the two agree to rounding
    Q64, K64, V64 = (x.astype(np.float64) for x in (Q, K, V))
    assert np.max(np.abs(online.attention_online(Q64, K64, V64, scale, tile)
                         - attention.softmax_attention(Q64, K64, V64, scale))) < 1e-13


def test_gather_walks_block_table_in_logical_order():
    bs, hkv, d = 4, 2, 3
    cache = np.arange(6 * hkv * bs * d, dtype=np.float32).reshape(6, hkv, bs, d)
    table = [5, 0, 3]
    dense = attention.gather_sequence(cache, table, 10, bs)
    assert dense.shape == (10, hkv, d)
    for p in range(10):
        assert np.array_equal(dense[p], cache[table[p // bs], :, p % bs, :])


def test_oracle_state_step_records_slots_and_cow():
    w = workloads.config5(groups=1, branches=3, prompt=20, max_private=3, n_long=1,
                          long_ctx=40)
    st = OracleState(w)
    st.run_setup()
    st.run_step()
    assert len(st.step_slots) == len(w.batch)
    assert len(set(st.step_slots)) == len(st.step_slots)
