"""GPU parity for sliding-window attention over prompt chunks and decode rows.

A windowed run adds each prompt chunk by chunk to a window pool whose ring has
room for the chunk ("大模型部署.md" §2.1 block_sliding_window, with the reading
that a query sees its window of most recent keys), appends every step's K/V,
and attends with one windowed varlen call over logically ordered tables.  Each
step's output is compared with the oracle's windowed run of the same trace
(float64, its own pool, cache mirror and masks), and the final caches byte for
byte.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle.run import execute, execute_window_trace  # noqa: E402
from tests.gpu_parity import TOL, cache_bytes_equal, out_f64  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rt(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import runner

    lib.device_error(clear=True)
    return runner


def _check_trace(tr, rt, lib):
    outs, kc, vc = rt.run_window_trace(tr)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    ref, okc, ovc = execute_window_trace(tr)
    tmax, tmean = TOL[tr.dtype]
    for i, (o, r) in enumerate(zip(outs, ref)):
        d = np.abs(out_f64(o) - r)
        assert float(d.max()) <= tmax and float(d.mean()) <= tmean, (i, float(d.max()))
    assert cache_bytes_equal(kc, okc) and cache_bytes_equal(vc, ovc)
    return len(tr.steps)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 8), (64, 8)])
def test_chunked_prompts_longer_than_the_window(rt, lib, hq, hkv):
    # window 256 < prompts 700 and 1000; chunks of up to 200 tokens; the 130-token
    # prompt stays inside its window; decode steps follow each prompt
    tr = workloads.window_trace(21, "bf16", hq, hkv, 128, 16, 256, 200,
                                prompts=(700, 130, 1000), gens=(3, 40, 2))
    assert _check_trace(tr, rt, lib) > 5


@pytest.mark.parametrize("window,chunk", [(48, 300), (128, 129), (16, 64), (512, 512)])
def test_windows_against_tile_edges(rt, lib, window, chunk):
    # windows below, at and above a 128-key tile; chunks larger than the window,
    # so rows of one prefill tile start their windows in different key tiles
    tr = workloads.window_trace(22 + window, "bf16", 32, 8, 128, 16, window, chunk,
                                prompts=(900, 333), gens=(5, 3))
    _check_trace(tr, rt, lib)


def test_head_dim_64_and_decode_only_steps(rt, lib):
    tr = workloads.window_trace(23, "bf16", 16, 4, 64, 16, 64, 1, prompts=(1, 1, 1),
                                gens=(600, 90, 1200))
    _check_trace(tr, rt, lib)


def test_fp32_decode_rows_under_a_window(rt, lib):
    # fp32 caches have no prefill path: one-token chunks, decode rows only
    tr = workloads.window_trace(24, "f32", 8, 2, 128, 16, 80, 1, prompts=(1, 1),
                                gens=(700, 300), scale=1.0)
    _check_trace(tr, rt, lib)


def test_keys_below_every_window_never_reach_the_output(rt, lib):
    """Rows below each query's window may hold anything (here NaN): the same
    outputs as with the real values there, for prefill chunks and decode rows."""
    from paged_kv_cache_51_gb300 import paged_attention_varlen

    W = 100
    spans = [(400, 150), (700, 1), (90, 40), (1500, 1)]
    w = workloads.random_varlen(25, "bf16", 32, 8, 128, 16, spans, scale=0.5)
    dc, step = rt.prepare(w)
    step.write_kv()
    # a window leaves out the first (ctx - qlen - W + 1) keys of each sequence:
    # poison them in both pools (plain tables are in logical order already)
    ctx = step.ctx.cpu().tolist()
    tables = step.tables.cpu().numpy()
    for s, (c, (_, qlen)) in enumerate(zip(ctx, w.batch)):
        first = max(0, c - qlen - W + 1)
        for pos in range(first):
            b = tables[s, pos // 16]
            dc.k_cache[b, :, pos % 16] = float("nan")
            dc.v_cache[b, :, pos % 16] = float("nan")
    out = torch.empty_like(step.q)
    paged_attention_varlen(out, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables, step.qsl,
                           step.ctx, step.max_qlen, step.max_ctx, window=W)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    from oracle import attention

    ost, _ = execute(w)
    bt, octx, qsl = ost.batch_metadata()
    ref = attention.varlen(w.q, ost.k_cache, ost.v_cache, bt, qsl, octx, 16, "bf16", window=W)
    got = out_f64(out)
    assert np.isfinite(got).all()
    d = np.abs(got - ref)
    assert float(d.max()) <= TOL["bf16"][0] and float(d.mean()) <= TOL["bf16"][1]


def test_window_zero_and_negative(rt, lib):
    from paged_kv_cache_51_gb300 import PagedKVError, paged_attention_varlen

    w = workloads.random_varlen(26, "bf16", 16, 8, 128, 16, [(40, 20), (9, 1)], scale=0.5)
    dc, step = rt.prepare(w)
    step.write_kv()
    a = torch.empty_like(step.q)
    b = torch.empty_like(step.q)
    step.attend()
    paged_attention_varlen(a, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables, step.qsl,
                           step.ctx, step.max_qlen, step.max_ctx, window=0)
    # a window wider than every context is the unwindowed result, bit for bit
    paged_attention_varlen(b, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables, step.qsl,
                           step.ctx, step.max_qlen, step.max_ctx, window=10 ** 6)
    torch.cuda.synchronize()
    assert torch.equal(a, step.out) and torch.equal(b, step.out)
    with pytest.raises(PagedKVError) as e:
        paged_attention_varlen(a, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables,
                               step.qsl, step.ctx, step.max_qlen, step.max_ctx, window=-1)
    assert e.value.status == lib.PKV_ERR_INVALID
