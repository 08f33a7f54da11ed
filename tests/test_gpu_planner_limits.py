"""GPU parity at the planner's size limits.

The planner scans the batch in passes of 1024 sequences (one thread each,
carrying the work-list offsets across passes), and orders prefill items
longest first only up to 2048 items (longer lists keep their order).  These
cases cross both limits and are checked against the float64 oracle.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from tests.gpu_parity import TOL, cache_bytes_equal, errors, run_both  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rt(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import runner

    lib.device_error(clear=True)
    return runner


def _check(w, rt, lib):
    ost, oout, dc, step, out = run_both(w, rt)
    assert lib.device_error() == 0
    assert cache_bytes_equal(dc.k_cache, ost.k_cache), "K cache bytes differ"
    assert cache_bytes_equal(dc.v_cache, ost.v_cache), "V cache bytes differ"
    mx, mean = errors(out, oout)
    tmax, tmean = TOL[w.dtype]
    assert mx <= tmax and mean <= tmean, (mx, mean)


def test_decode_more_sequences_than_a_planner_pass_gqa(rt, lib):
    # 1100 decode rows (two planner passes), one to three splits each, g = 4
    rng = np.random.default_rng(31)
    ctx = rng.integers(1, 1100, size=1100)
    _check(workloads.random_decode(31, "bf16", 8, 2, 128, 16, ctx, scale=0.5), rt, lib)


def test_decode_more_sequences_than_a_planner_pass_g1_d64(rt, lib):
    # 1100 decode rows, g = 1, head_dim 64 (the CUDA-core split kernel)
    rng = np.random.default_rng(32)
    ctx = rng.integers(1, 1600, size=1100)
    _check(workloads.random_decode(32, "bf16", 4, 4, 64, 16, ctx, scale=0.5), rt, lib)


def test_prefill_items_beyond_the_sort_capacity(rt, lib):
    # 140 chunks of 256 tokens at g = 8 (16 tokens per row tile): 2240 prefill
    # items, more than the planner reorders, plus decode rows in between
    rng = np.random.default_rng(33)
    spans = []
    for i in range(140):
        spans.append((int(rng.integers(0, 300)), 256))
        if i % 10 == 0:
            spans.append((int(rng.integers(1, 900)), 1))
    _check(workloads.random_varlen(33, "bf16", 8, 1, 128, 16, spans, scale=0.5), rt, lib)
