"""GPU: every attention call sees the device work queued before it on its stream.

The library's kernels are chained with programmatic dependent launch: the
planner, the append and the block copies start while the kernel before them on
the stream finishes, and the kernels behind the planner (prefill, decode split,
merge, 8-bit split) start early too; each waits for its predecessor before it
reads or writes anything.  Here q is rewritten on the device (an exact sign
flip) right before each of several calls, with no host synchronisation in
between, and every call's result is checked against the float64 oracle for the
q it must have read; and the step's new K/V rows are rewritten by the
library's own append between calls, so nothing but its kernels separates one
call from the next.  A kernel that read q, the cache or the plan before the
writes ahead of it had finished would fail this.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import attention as oatt  # noqa: E402
from oracle import quant  # noqa: E402
from tests.gpu_parity import TOL, errors, run_both  # noqa: E402

pytestmark = pytest.mark.gpu

CALLS = 5


@pytest.fixture(scope="module")
def rt(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import runner

    lib.device_error(clear=True)
    return runner


def _neg_bits(q, dtype):
    """The oracle's copy of -q (bf16 is stored as uint16 bit patterns)."""
    return q ^ np.uint16(0x8000) if dtype == "bf16" else -q


def _oracle(ost, q):
    w = ost.w
    bt, ctx, qsl = ost.batch_metadata()
    if all(n == 1 for _, n in w.batch):
        return oatt.decode(q, ost.k_cache, ost.v_cache, bt, ctx, w.block_size, w.dtype)
    return oatt.varlen(q, ost.k_cache, ost.v_cache, bt, qsl, ctx, w.block_size, w.dtype)


def _alternating_calls(w, rt, lib):
    ost, oout, dc, step, out = run_both(w, rt)
    ref = {+1: oout, -1: _oracle(ost, _neg_bits(w.q, w.dtype))}
    outs = []
    for _ in range(CALLS):
        step.q.neg_()            # queued on the stream, no host synchronisation
        step.attend()
        outs.append(step.out.clone())
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    tmax, tmean = TOL[w.dtype]
    for i, o in enumerate(outs):
        sign = -1 if i % 2 == 0 else +1
        mx, mean = errors(o, ref[sign])
        assert mx <= tmax and mean <= tmean, (i, sign, mx, mean)


def test_decode_g1_sees_each_new_q(rt, lib):
    _alternating_calls(workloads.config2(batch=8), rt, lib)


def test_decode_gqa_sees_each_new_q(rt, lib):
    _alternating_calls(workloads.config3(batch=8), rt, lib)


def test_mixed_batch_sees_each_new_q(rt, lib):
    spans = [(0, 130), (700, 64), (300, 1), (1500, 1), (2500, 1), (90, 33)]
    _alternating_calls(workloads.random_varlen(21, "bf16", 32, 8, 128, 16, spans, scale=0.5),
                       rt, lib)


def test_int8_decode_sees_each_new_q(rt, lib):
    import paged_kv_cache_51_gb300 as pkv

    w = workloads.config2(batch=8)
    ost, _, dc, step, _ = run_both(w, rt)
    nb, hkv, bs, d = dc.k_cache.shape
    ic = pkv.Int8Cache(nb, hkv, bs, d, w.num_q_heads)

    def rows(c):
        return c.transpose(1, 2).reshape(nb * bs, hkv, d).contiguous()

    pkv.paged_kv_append_int8(rows(dc.k_cache), rows(dc.v_cache),
                             torch.arange(nb * bs, dtype=torch.int64, device="cuda"), ic)
    kq, ks = quant.quantize_rows(ost.k_cache, "bf16")
    vq, vs = quant.quantize_rows(ost.v_cache, "bf16")
    bt, ctx, _ = ost.batch_metadata()
    ref = {+1: quant.decode_int8(w.q, kq, ks, vq, vs, bt, ctx, bs, "bf16"),
           -1: quant.decode_int8(_neg_bits(w.q, "bf16"), kq, ks, vq, vs, bt, ctx, bs, "bf16")}
    q = step.q.clone()
    out = torch.empty_like(q)
    outs = []
    for _ in range(CALLS):
        q.neg_()
        pkv.paged_attention_decode_int8(out, q, ic, step.tables, step.ctx, step.max_ctx)
        outs.append(out.clone())
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    tmax, tmean = TOL["bf16"]
    for i, o in enumerate(outs):
        sign = -1 if i % 2 == 0 else +1
        mx, mean = errors(o, ref[sign])
        assert mx <= tmax and mean <= tmean, (i, sign, mx, mean)


def test_attention_sees_each_append_before_it(rt, lib):
    """append (variant i) -> attention -> append (variant i + 1) -> ..., queued
    back to back: each call must see its own append's rows."""
    from oracle import cache as ocache
    from paged_kv_cache_51_gb300 import paged_attention_decode, paged_kv_append

    w = workloads.config3(batch=8)
    ost, _, dc, step, _ = run_both(w, rt)
    rng = np.random.default_rng(71)
    variants = [workloads._values(rng, tuple(step.k_new.shape), "bf16", 0.5) for _ in range(4)]
    dev = [torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).cuda()
           for v in variants]
    slots = step.slot_mapping.cpu().numpy()
    outs = [torch.empty_like(step.q) for _ in variants]
    torch.cuda.synchronize()
    for i in range(len(variants)):
        # K takes variant i, V variant i + 1 (mod n): a stale row of either shows
        paged_kv_append(dev[i], dev[(i + 1) % len(dev)], step.slot_mapping, dc.k_cache,
                        dc.v_cache, dc.desc)
        paged_attention_decode(outs[i], step.q, dc.k_cache, dc.v_cache, dc.desc, step.tables,
                               step.ctx, step.max_ctx, ws=step.ws)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    tmax, tmean = TOL["bf16"]
    bt, ctx, _ = ost.batch_metadata()
    for i in range(len(variants)):
        kc, vc = ost.k_cache.copy(), ost.v_cache.copy()
        ocache.append(kc, vc, variants[i], variants[(i + 1) % len(variants)], slots,
                      w.block_size)
        ref = oatt.decode(w.q, kc, vc, bt, ctx, w.block_size, "bf16")
        mx, mean = errors(outs[i], ref)
        assert mx <= tmax and mean <= tmean, (i, mx, mean)
