"""Pins for the closed-form KV-cache size (values the pages print)."""

import pytest

import workloads
from oracle import kv_size
from tests.conftest import read_kv, read_rows


@pytest.mark.parametrize("row", read_rows("kv_size_examples.txt"))
def test_printed_examples(row):
    layers, batch, seq, kvh, d, nbytes, want = (int(x) for x in row[1:8])
    assert kv_size.kv_cache_bytes(layers, batch, seq, kvh, d, nbytes) == want


def test_capacity_example():
    g = read_kv("kv_pool_capacity.txt")
    per_tok = kv_size.kv_cache_bytes(28, 1, 1, 4, 128, 2)
    assert per_tok == int(g["bytes_per_token"])
    fit = int(float(g["pool_gib"]) * 2 ** 30) // per_tok
    assert fit == int(g["tokens_fit"])
    blocks_tokens = int(g["num_gpu_blocks"]) * int(g["block_size"])
    assert blocks_tokens == int(g["block_tokens"]) and blocks_tokens <= fit


def test_pool_bytes_matches_allocation_for_configs():
    # one layer's two pools [NB, Hkv, bs, D] in the cache dtype
    w = workloads.config1()
    want = 2 * w.num_blocks * w.num_kv_heads * w.block_size * w.head_dim * 4
    assert kv_size.pool_bytes(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, 4) == want
