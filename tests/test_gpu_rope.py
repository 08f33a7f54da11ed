"""GPU parity for the rotary-embedding append: rotated q and cache bytes exact, then
decode over the rotated values within tolerance."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import attention, cache, rope  # noqa: E402
from oracle.run import OracleState  # noqa: E402
from tests.gpu_parity import (TOL, assert_within_derived_bound, cache_bytes_equal,  # noqa: E402
                              out_f64)

pytestmark = pytest.mark.gpu


def _torch_rows(rows, dtype):
    from paged_kv_cache_51_gb300.runner import _torch_rows as f

    return f(rows, dtype)


@pytest.mark.parametrize("dtype,hq,hkv,d", [("bf16", 32, 8, 128), ("bf16", 16, 16, 64),
                                            ("f32", 8, 2, 128), ("f32", 8, 8, 64)])
def test_append_rope_bit_exact_then_decode(lib, dtype, hq, hkv, d):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import paged_attention_decode, paged_kv_append_rope, runner

    lib.device_error(clear=True)
    w = workloads.random_decode(31, dtype, hq, hkv, d, 16, [5, 200, 1031, 2999], scale=1.0)
    max_pos = 4096
    tab = rope.rope_table(max_pos, d)
    # history on both sides (plain appends), then the step's tokens through the rotary append
    dc = runner.DeviceCache(w)
    dc.run_setup()
    planned = dc.plan_step()
    ost = OracleState(w)
    ost.run_setup()
    # oracle: its own pool gives the step's slots and positions
    o_slots = []
    for kind, seq, n, row in w.step:
        if kind == "add":
            o_slots += ost.pool.add_sequence(seq, n)[1]
        else:
            for _ in range(n):
                o_slots.append(ost.pool.append_slot(seq)[0])
    slots = np.array(o_slots, dtype=np.int64)
    assert np.array_equal(slots, planned["slot_mapping"].numpy())
    rows = np.concatenate([np.arange(row, row + n) for _, _, n, row in w.step])
    positions = np.array([ost.pool.context_len(s) - 1 for s, _ in w.batch], dtype=np.int32)
    q_ref = rope.append_rope(ost.k_cache, ost.v_cache, w.q, w.k_rows[rows], w.v_rows[rows],
                             slots, positions, tab, w.block_size, w.dtype, cache.append)
    # device
    dev = "cuda"
    q = _torch_rows(w.q, dtype).to(dev)
    k_new = planned["k"].to(dev)
    v_new = planned["v"].to(dev)
    pos_d = torch.tensor([dc.pool.seq_len(s) - 1 for s, _ in w.batch], dtype=torch.int32,
                         device=dev)
    tab_d = torch.from_numpy(tab).to(dev)
    q_out = torch.empty_like(q)
    paged_kv_append_rope(k_new, v_new, planned["slot_mapping"].to(dev), pos_d, tab_d, dc.k_cache,
                         dc.v_cache, dc.desc, q=q, q_out=q_out)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    got_q = q_out.cpu()
    got_q = got_q.numpy() if dtype == "f32" else got_q.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_q.view(np.uint8), np.ascontiguousarray(q_ref).view(np.uint8))
    assert cache_bytes_equal(dc.k_cache, ost.k_cache)
    assert cache_bytes_equal(dc.v_cache, ost.v_cache)
    # in place rotation gives the same bytes
    q2 = q.clone()
    paged_kv_append_rope(k_new, v_new, planned["slot_mapping"].to(dev), pos_d, tab_d, dc.k_cache,
                         dc.v_cache, dc.desc, q=q2)
    torch.cuda.synchronize()
    assert torch.equal(q2, q_out)
    # decode over the rotated cache and query
    tables, ctx, _ = dc.batch_metadata()
    out = torch.empty_like(q)
    paged_attention_decode(out, q_out, dc.k_cache, dc.v_cache, dc.desc, tables.to(dev),
                           ctx.to(dev), int(ctx.max()))
    torch.cuda.synchronize()
    bt, octx, _ = ost.batch_metadata()
    ref = attention.decode(q_ref, ost.k_cache, ost.v_cache, bt, octx, w.block_size, w.dtype)
    if dtype == "f32":
        # values N(0,1) as config 1, but 128 dimensions and up to 3000 keys:
        # the derived bound (stated tolerance + first-order score rounding)
        assert_within_derived_bound(w, ost, ref, out_f64(out), q=q_ref)
    else:
        d_ = np.abs(out_f64(out) - ref)
        tmax, tmean = TOL[dtype]
        assert float(d_.max()) <= tmax and float(d_.mean()) <= tmean


def test_bad_rotary_position_is_flagged(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import cache_desc, paged_kv_append_rope

    kc = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    desc = cache_desc(kc, 2)
    k = torch.ones((1, 2, 64), dtype=torch.bfloat16, device="cuda")
    tab = torch.from_numpy(rope.rope_table(8, 64)).cuda()
    pos = torch.tensor([8], dtype=torch.int32, device="cuda")       # table has 0..7
    slots = torch.tensor([3], dtype=torch.int64, device="cuda")
    lib.device_error(clear=True)
    paged_kv_append_rope(k, k, slots, pos, tab, kc, vc, desc)
    assert lib.device_error() == 8                                  # PKV_DEV_BAD_POSITION
    assert torch.count_nonzero(kc) == 0                             # K row skipped


def _dev(x, dtype):
    return _torch_rows(x, dtype).to("cuda")


def _host_bits(t, dtype):
    t = t.cpu()
    return t.numpy() if dtype == "f32" else t.view(torch.int16).numpy().view(np.uint16)


# Head counts whose rows (q heads + 2 x KV heads) leave the kernel's last row
# group part-filled (8 rows a thread for bf16, 4 for f32), with padding tokens,
# and the form without q.
@pytest.mark.parametrize("dtype,hq,hkv,d,with_q", [("bf16", 6, 3, 128, True),
                                                  ("bf16", 10, 5, 64, False),
                                                  ("f32", 3, 1, 64, True),
                                                  ("bf16", 32, 8, 128, True)])
def test_append_rope_ragged_row_groups_and_padding(lib, dtype, hq, hkv, d, with_q):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import cache_desc, paged_kv_append_rope

    nb, bs, max_pos, T = 400, 16, 2048, 3000
    q, k, v, slots, pos = workloads.append_inputs(41 + hq, dtype, T, hq if with_q else 0, hkv, d,
                                                  nb * bs, max_pos, pad_every=7)
    tab = rope.rope_table(max_pos, d)
    sdt = np.float32 if dtype == "f32" else np.uint16
    ok = np.zeros((nb, hkv, bs, d), dtype=sdt)
    ov = np.zeros_like(ok)
    q_ref = rope.append_rope(ok, ov, q, k, v, slots, pos, tab, bs, dtype, cache.append)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    kc = torch.zeros((nb, hkv, bs, d), dtype=tdt, device="cuda")
    vc = torch.zeros_like(kc)
    desc = cache_desc(kc, hq)
    q_d = _dev(q, dtype) if with_q else None
    q_out = torch.empty_like(q_d) if with_q else None
    lib.device_error(clear=True)
    paged_kv_append_rope(_dev(k, dtype), _dev(v, dtype), torch.from_numpy(slots).cuda(),
                         torch.from_numpy(pos).cuda(), torch.from_numpy(tab).cuda(), kc, vc, desc,
                         q=q_d, q_out=q_out)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert cache_bytes_equal(kc, ok)
    assert cache_bytes_equal(vc, ov)
    if with_q:
        assert np.array_equal(_host_bits(q_out, dtype).view(np.uint8),
                              np.ascontiguousarray(q_ref).view(np.uint8))


def test_plain_append_several_grid_passes(lib):
    # 6000 tokens x 8 KV heads x 16 vectors: more 16-byte vectors than one
    # unrolled pass of the resident grid covers, with padding tokens
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import cache_desc, paged_kv_append

    nb, bs, hkv, d, T = 600, 16, 8, 128, 6000
    _, k, v, slots, _ = workloads.append_inputs(43, "bf16", T, 0, hkv, d, nb * bs, 1, pad_every=5)
    ok = np.zeros((nb, hkv, bs, d), dtype=np.uint16)
    ov = np.zeros_like(ok)
    cache.append(ok, ov, k, v, slots, bs)
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    lib.device_error(clear=True)
    paged_kv_append(_dev(k, "bf16"), _dev(v, "bf16"), torch.from_numpy(slots).cuda(), kc, vc,
                    cache_desc(kc, hkv))
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    assert cache_bytes_equal(kc, ok)
    assert cache_bytes_equal(vc, ov)
