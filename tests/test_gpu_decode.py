"""GPU parity: append, copy-on-write and decode attention through the C ABI vs the oracle.

Cache writes are compared byte for byte over the whole pool; attention within
the tolerances in tests/gpu_parity.py.  Every call's device error word must
stay clear unless a test plants a bad input on purpose (which the kernels'
own bounds checks turn into an error code; nothing out of bounds is touched).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from tests.gpu_parity import (TOL, assert_within_derived_bound, cache_bytes_equal,  # noqa: E402
                              errors, out_f64, run_both)

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
    return ost, oout, dc, step, out


def test_config1_tiny_f32(rt, lib):
    _check(workloads.config1(), rt, lib)


def test_config2_llama2_7b_decode_full(rt, lib):
    _check(workloads.config2(), rt, lib)


def test_config3_llama3_8b_gqa_decode_full(rt, lib):
    _check(workloads.config3(), rt, lib)


def test_config5_prefix_sharing_and_long_context_full(rt, lib):
    ost, oout, dc, step, out = _check(workloads.config5(), rt, lib)
    # copy-on-write happened in setup or in the step, and the step copied what the oracle copied
    assert step.pairs.shape[0] == len(ost.step_cow)
    # branches of one group share their prompt blocks
    tables = step.tables.cpu().numpy()
    assert np.array_equal(tables[0, :187], tables[1, :187])


@pytest.mark.parametrize("ctx", [
    [1], [16], [17], [2, 511, 512, 513], [1024, 1025, 33, 5000], [40000],
])
def test_split_boundaries_bf16(rt, lib, ctx):
    _check(workloads.random_decode(1, "bf16", 8, 8, 128, 16, ctx, scale=0.5), rt, lib)


@pytest.mark.parametrize("dtype,hq,hkv,d", [
    ("bf16", 16, 8, 128), ("bf16", 32, 8, 128), ("bf16", 64, 8, 128),
    ("bf16", 8, 8, 64), ("bf16", 32, 4, 64), ("f32", 16, 2, 128), ("f32", 8, 1, 64),
    ("f32", 16, 16, 128),
])
def test_head_shapes(rt, lib, dtype, hq, hkv, d):
    ctx = [3, 100, 700, 1600]
    _check(workloads.random_decode(2, dtype, hq, hkv, d, 16, ctx, scale=0.5), rt, lib)


def test_large_scores_stay_finite(rt, lib):
    # queries of scale 64 over N(0,1) keys give scores of standard deviation 64,
    # a few hundred at the maximum: exp without the max subtraction would
    # overflow fp32.  Keys and values keep config 1's magnitudes, so only the
    # score-rounding term of the derived bound grows.
    w = workloads.random_decode(4, "f32", 8, 8, 64, 16, [300, 1200], scale=1.0, q_scale=64.0)
    ost, oout, dc, step, out = run_both(w, rt)
    assert lib.device_error() == 0
    got = out_f64(out)
    assert np.isfinite(got).all()
    assert_within_derived_bound(w, ost, oout, got)


def test_batch_invariance_bitwise(rt, lib):
    """The same sequence decoded in two different batches gives identical bits."""
    from paged_kv_cache_51_gb300 import runner

    a = workloads.random_decode(7, "bf16", 32, 8, 128, 16, [1500], scale=0.5)
    _, step_a = runner.prepare(a)
    out_a = step_a.run().clone()
    # a bigger batch whose first sequence has the same values
    b = workloads.random_decode(7, "bf16", 32, 8, 128, 16, [1500], scale=0.5)
    b2 = workloads.random_decode(9, "bf16", 32, 8, 128, 16, [900, 4000, 17], scale=0.5)
    # append b2's sequences after b's one
    nrow = b.k_rows.shape[0]
    b.k_rows = np.concatenate([b.k_rows, b2.k_rows])
    b.v_rows = np.concatenate([b.v_rows, b2.v_rows])
    b.q = np.concatenate([b.q, b2.q])
    shift = lambda ops, ds: [(op[0], op[1] + ds, op[2], op[3] + nrow) for op in ops]  # noqa
    b.setup = b.setup + shift(b2.setup, 1)
    b.step = b.step + shift(b2.step, 1)
    b.batch = b.batch + [(s + 1, q) for s, q in b2.batch]
    b.num_blocks = b.num_blocks + b2.num_blocks
    b.free_order = np.concatenate([b.free_order, b2.free_order + a.num_blocks]).astype(np.int32)
    _, step_b = runner.prepare(b)
    out_b = step_b.run()
    torch.cuda.synchronize()
    assert torch.equal(out_a[0], out_b[0])
    assert lib.device_error() == 0


def test_block_permutation_gives_identical_bits(rt, lib):
    from paged_kv_cache_51_gb300 import paged_attention_decode

    w = workloads.random_decode(5, "bf16", 16, 4, 128, 16, [700, 1300, 90], scale=0.5)
    dc, step = rt.prepare(w)
    out1 = step.run().clone()
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(0))
    permd = perm.to(dc.k_cache.device)
    k2 = torch.empty_like(dc.k_cache)
    v2 = torch.empty_like(dc.v_cache)
    k2[permd] = dc.k_cache
    v2[permd] = dc.v_cache
    t = step.tables.long()
    t2 = torch.where(t >= 0, permd[t.clamp(min=0)], t).int().contiguous()
    out2 = torch.empty_like(out1)
    paged_attention_decode(out2, step.q, k2, v2, dc.desc, t2, step.ctx, step.max_ctx)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_bad_block_id_is_flagged_not_faulted(rt, lib):
    from paged_kv_cache_51_gb300 import paged_attention_decode

    w = workloads.random_decode(6, "bf16", 8, 8, 128, 16, [40, 40], scale=0.5)
    dc, step = rt.prepare(w)
    step.run()
    assert lib.device_error() == 0
    bad = step.tables.clone()
    bad[1, 0] = w.num_blocks + 5          # outside the pool: must be skipped, not read
    paged_attention_decode(step.out, step.q, dc.k_cache, dc.v_cache, dc.desc, bad, step.ctx,
                           step.max_ctx)
    assert lib.device_error() == 1        # PKV_DEV_BAD_BLOCK_ID
    assert lib.device_error() == 0        # cleared


def test_bad_slot_and_context_are_flagged(rt, lib):
    from paged_kv_cache_51_gb300 import paged_attention_decode, paged_kv_append

    w = workloads.random_decode(6, "bf16", 8, 8, 128, 16, [40], scale=0.5)
    dc, step = rt.prepare(w)
    before = dc.k_cache.clone()
    slots = torch.tensor([w.num_blocks * 16 + 3], dtype=torch.int64, device="cuda")
    paged_kv_append(step.k_new, step.v_new, slots, dc.k_cache, dc.v_cache, dc.desc)
    assert lib.device_error() == 3        # PKV_DEV_BAD_SLOT
    assert torch.equal(before, dc.k_cache)
    # negative slot = padding: nothing written, no error
    paged_kv_append(step.k_new, step.v_new, -slots, dc.k_cache, dc.v_cache, dc.desc)
    assert lib.device_error() == 0 and torch.equal(before, dc.k_cache)
    # context longer than the promised maximum is rejected by the planner
    ctx = step.ctx.clone()
    ctx[0] = step.max_ctx + 1
    paged_attention_decode(step.out, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables, ctx,
                           step.max_ctx)
    assert lib.device_error() == 2        # PKV_DEV_BAD_CONTEXT_LEN


def test_copy_blocks_bit_exact(rt, lib):
    from paged_kv_cache_51_gb300 import pkv_copy_blocks

    w = workloads.random_decode(8, "bf16", 8, 8, 128, 16, [200], scale=0.5)
    dc, step = rt.prepare(w)
    step.run()
    pairs = torch.tensor([[step.tables[0, 0].item(), w.num_blocks - 1],
                          [step.tables[0, 3].item(), w.num_blocks - 2]], dtype=torch.int32,
                         device="cuda")
    pkv_copy_blocks(pairs, dc.k_cache, dc.v_cache, dc.desc)
    torch.cuda.synchronize()
    for s, d in pairs.tolist():
        assert torch.equal(dc.k_cache[s], dc.k_cache[d]) and torch.equal(dc.v_cache[s], dc.v_cache[d])
    assert lib.device_error() == 0


def test_varlen_with_only_decode_rows_matches_decode(rt, lib):
    from paged_kv_cache_51_gb300 import paged_attention_varlen

    w = workloads.random_decode(3, "bf16", 32, 8, 128, 16, [5, 600, 2100], scale=0.5)
    dc, step = rt.prepare(w)
    out_dec = step.run().clone()
    out_var = torch.empty_like(out_dec)
    paged_attention_varlen(out_var, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables,
                           step.qsl, step.ctx, 1, step.max_ctx)
    torch.cuda.synchronize()
    assert torch.equal(out_dec, out_var)
    assert lib.device_error() == 0


@pytest.mark.parametrize("hq,hkv,dtype", [(8, 8, "bf16"), (32, 8, "bf16"), (64, 8, "bf16"),
                                          (16, 8, "bf16"), (8, 8, "f32")])
def test_never_written_rows_may_hold_nan_decode(rt, lib, hq, hkv, dtype):
    """Rows of a partial last block past the context were never written; whatever they
    hold (NaN here) must not reach the output of any decode path."""
    from oracle.run import execute

    w = workloads.random_decode(21, dtype, hq, hkv, 128, 16, [3, 17, 530, 1000], scale=0.5)
    _, ref = execute(w)
    dc = rt.DeviceCache(w)
    dc.k_cache.fill_(float("nan"))
    dc.v_cache.fill_(float("nan"))
    dc.run_setup()
    step = rt.Step(dc, dc.plan_step())
    out = step.run()
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert np.isfinite(out_f64(out)).all()
    mx, mean = errors(out, ref)
    assert mx <= TOL[dtype][0] and mean <= TOL[dtype][1]


def test_bad_query_layout_is_flagged_and_nothing_runs(rt, lib):
    """query_start_loc must run from 0 to num_query_tokens: otherwise the planner
    flags PKV_DEV_BAD_QUERY_LAYOUT and plans no work (the output is not written)."""
    from paged_kv_cache_51_gb300 import paged_attention_varlen

    w = workloads.random_varlen(61, "bf16", 16, 8, 128, 16, [(30, 2), (9, 1)], scale=0.5)
    dc, step = rt.prepare(w)
    step.write_kv()
    lib.device_error(clear=True)
    bad_qsl = torch.tensor([0, 2, 2], dtype=torch.int32, device="cuda")   # ends at 2, not 3
    out = torch.full_like(step.q, 7.0)
    paged_attention_varlen(out, step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables, bad_qsl,
                           step.ctx, step.max_qlen, step.max_ctx)
    assert lib.device_error() == 5                                   # PKV_DEV_BAD_QUERY_LAYOUT
    assert bool((out == 7.0).all())
    # the same call with the right layout is unaffected
    step.attend()
    torch.cuda.synchronize()
    assert lib.device_error() == 0


def test_empty_inputs_are_no_ops(rt, lib):
    """No sequences, no query tokens, no new tokens, no copy pairs: each call
    returns at once, touches no output and records no device error."""
    from paged_kv_cache_51_gb300 import (paged_attention_decode, paged_attention_varlen,
                                         paged_kv_append, pkv_copy_blocks)

    w = workloads.random_decode(71, "bf16", 16, 8, 128, 16, [40, 7], scale=0.5)
    dc, step = rt.prepare(w)
    step.write_kv()
    lib.device_error(clear=True)
    k_before, v_before = dc.k_cache.clone(), dc.v_cache.clone()
    q0 = step.q[:0]
    out0 = torch.empty_like(q0)
    paged_attention_decode(out0, q0, dc.k_cache, dc.v_cache, dc.desc, step.tables[:0],
                           step.ctx[:0], step.max_ctx)
    # varlen with sequences that have no query rows: nothing is written
    sentinel = torch.full_like(step.q, 3.0)
    qsl_empty = torch.zeros(len(w.batch) + 1, dtype=torch.int32, device="cuda")
    paged_attention_varlen(sentinel[:0], q0, dc.k_cache, dc.v_cache, dc.desc, step.tables,
                           qsl_empty, step.ctx, 0, step.max_ctx)
    rows = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    paged_kv_append(rows, rows, torch.empty(0, dtype=torch.int64, device="cuda"), dc.k_cache,
                    dc.v_cache, dc.desc)
    pkv_copy_blocks(torch.empty((0, 2), dtype=torch.int32, device="cuda"), dc.k_cache,
                    dc.v_cache, dc.desc)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert torch.equal(dc.k_cache, k_before) and torch.equal(dc.v_cache, v_before)
    assert bool((sentinel == 3.0).all())


@pytest.mark.parametrize("hq,hkv", [(8, 8), (64, 8)])
def test_longest_context_many_split_passes(rt, lib, hq, hkv):
    """131072 keys: 256 splits, so the merge folds eight passes of 32 splits."""
    w = workloads.random_decode(72, "bf16", hq, hkv, 128, 16, [131072, 1000], scale=0.5)
    _check(w, rt, lib)
