"""GPU parity for the 8-bit KV cache: codes and scales bit-exact against the
oracle's quantiser, decode within the bf16 tolerance of exact attention over
the dequantised cache."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import quant  # noqa: E402
from oracle.run import execute  # noqa: E402
from tests.gpu_parity import TOL, out_f64  # noqa: E402

pytestmark = pytest.mark.gpu


def _bf16_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _logical_codes(k_phys, v_phys):
    """Device tile layout -> logical [NB, Hkv, 16, D] (the layout the header
    defines: K rows with 16-byte chunks XOR-swizzled by the row, V dim-major)."""
    k = k_phys.cpu().numpy()
    v = v_phys.cpu().numpy()
    nb, hkv, bs, d = k.shape
    r = np.arange(bs)
    sw = (r & 7) if d == 128 else ((r >> 1) & 3)
    chunks = k.reshape(nb, hkv, bs, d // 16, 16)
    kl = np.empty_like(chunks)
    for row in range(bs):
        for c in range(d // 16):
            kl[:, :, row, c] = chunks[:, :, row, c ^ sw[row]]
    vl = np.ascontiguousarray(np.swapaxes(v.reshape(nb, hkv, d, bs), 2, 3))
    return kl.reshape(nb, hkv, bs, d), vl


def _pool_rows(c):
    """[NB, Hkv, bs, D] -> rows [NB * bs, Hkv, D] (row index = slot)."""
    nb, hkv, bs, d = c.shape
    return np.ascontiguousarray(np.swapaxes(c, 1, 2).reshape(nb * bs, hkv, d))


def _fill(lib, w, ost, slot_perm_seed):
    """Quantise the oracle's final bf16 cache (every slot, in shuffled order) into a
    device 8-bit cache; returns it with the oracle's codes and scales."""
    ic = lib.Int8Cache(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim, w.num_q_heads)
    k_rows = _pool_rows(ost.k_cache)
    v_rows = _pool_rows(ost.v_cache)
    n = k_rows.shape[0]
    order = np.random.default_rng(slot_perm_seed).permutation(n)
    slots = order.astype(np.int64)
    slots[::7] = -1                                             # padding rows are skipped
    keep = slots >= 0
    lib.paged_kv_append_int8(_bf16_tensor(k_rows[order]).cuda(), _bf16_tensor(v_rows[order]).cuda(),
                             torch.from_numpy(slots).cuda(), ic)
    # the skipped slots take a second pass, in their own order
    rest = order[~keep]
    lib.paged_kv_append_int8(_bf16_tensor(k_rows[rest]).cuda(), _bf16_tensor(v_rows[rest]).cuda(),
                             torch.from_numpy(rest.astype(np.int64)).cuda(), ic)
    shape = ost.k_cache.shape
    kq = np.zeros(shape, np.int8)
    vq = np.zeros(shape, np.int8)
    ks = np.zeros(shape[:3], np.float32)
    vs = np.zeros(shape[:3], np.float32)
    quant.append_int8(kq, ks, vq, vs, k_rows, v_rows, np.arange(n), w.block_size, "bf16")
    return ic, (kq, ks, vq, vs)


@pytest.mark.parametrize("hq,hkv,d", [(32, 32, 128), (32, 8, 128), (16, 8, 64), (64, 8, 128),
                                      (8, 8, 64)])
def test_int8_append_bit_exact_and_decode(lib, hq, hkv, d):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib.device_error(clear=True)
    w = workloads.random_decode(41 + hq + d, "bf16", hq, hkv, d, 16, [1, 5, 16, 17, 200, 513,
                                                                     1031, 2999], scale=2.0)
    ost, _ = execute(w, with_attention=False)
    ic, (kq, ks, vq, vs) = _fill(lib, w, ost, hq * 7 + d)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    kl, vl = _logical_codes(ic.k_codes, ic.v_codes)
    assert np.array_equal(kl, kq)
    assert np.array_equal(vl, vq)
    assert np.array_equal(ic.k_scales.cpu().numpy().view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(ic.v_scales.cpu().numpy().view(np.uint32), vs.view(np.uint32))
    bt, ctx, _ = ost.batch_metadata()
    q = _bf16_tensor(w.q).cuda()
    out = torch.empty_like(q)
    lib.paged_attention_decode_int8(out, q, ic, torch.from_numpy(bt).cuda(),
                                    torch.from_numpy(ctx).cuda(), int(ctx.max()))
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    ref = quant.decode_int8(w.q, kq, ks, vq, vs, bt, ctx, w.block_size, "bf16")
    diff = np.abs(out_f64(out) - ref)
    tmax, tmean = TOL["bf16"]
    assert float(diff.max()) <= tmax and float(diff.mean()) <= tmean


def test_int8_extremes_and_zero_rows(lib):
    """All-zero rows (scale 0), a row of one spike, bf16 subnormals and the
    largest bf16 values quantise exactly as the oracle does."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hkv, d = 2, 128
    rng = np.random.default_rng(3)
    x = rng.standard_normal((12, hkv, d)).astype(np.float32)
    x[0] = 0.0
    x[1] = 0.0
    x[1, :, 5] = -3.0
    x[2] *= 1e-39                                               # subnormal range
    x[3] *= 1e37                                                # near the top of the range
    x[4, 0, :] = 1.0                                            # constant row
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ic = lib.Int8Cache(2, hkv, 16, d, hkv)
    slots = np.arange(12, dtype=np.int64) + 3
    lib.device_error(clear=True)
    lib.paged_kv_append_int8(_bf16_tensor(bits).cuda(), _bf16_tensor(bits[::-1]).cuda(),
                             torch.from_numpy(slots).cuda(), ic)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    kq = np.zeros((2, hkv, 16, d), np.int8)
    vq = np.zeros_like(kq)
    ks = np.zeros((2, hkv, 16), np.float32)
    vs = np.zeros_like(ks)
    quant.append_int8(kq, ks, vq, vs, bits, np.ascontiguousarray(bits[::-1]), slots, 16, "bf16")
    kl, vl = _logical_codes(ic.k_codes, ic.v_codes)
    assert np.array_equal(kl, kq)
    assert np.array_equal(vl, vq)
    assert np.array_equal(ic.k_scales.cpu().numpy().view(np.uint32), ks.view(np.uint32))
    assert np.array_equal(ic.v_scales.cpu().numpy().view(np.uint32), vs.view(np.uint32))
    assert ks[0, 0, 3] == 0 and np.all(kq[0, :, 3] == 0)


def test_int8_bad_slot_is_flagged(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ic = lib.Int8Cache(2, 2, 16, 64, 2)
    k = torch.ones((2, 2, 64), dtype=torch.bfloat16, device="cuda")
    lib.device_error(clear=True)
    lib.paged_kv_append_int8(k, k, torch.tensor([1, 32], dtype=torch.int64, device="cuda"), ic)
    assert lib.device_error() == 3                                  # PKV_DEV_BAD_SLOT
    assert int(torch.count_nonzero(ic.k_codes)) == 2 * 64           # slot 1 written, 32 skipped


@pytest.mark.parametrize("d", [128, 64])
def test_int8_copy_on_write_moves_codes_and_scales(lib, d):
    """Block copies through pkv_copy_blocks_int8 equal the oracle's whole-block copy
    (tiles of 2112 and 1088 bytes: codes, then scales)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from oracle import cache as ocache

    hkv, nb = 4, 12
    rng = np.random.default_rng(9)
    x = rng.standard_normal((nb * 16, hkv, d)).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ic = lib.Int8Cache(nb, hkv, 16, d, hkv * 2)
    slots = np.arange(nb * 16, dtype=np.int64)
    lib.paged_kv_append_int8(_bf16_tensor(bits).cuda(), _bf16_tensor(bits[::-1].copy()).cuda(),
                             torch.from_numpy(slots).cuda(), ic)
    kq = np.zeros((nb, hkv, 16, d), np.int8)
    vq = np.zeros_like(kq)
    ks = np.zeros((nb, hkv, 16), np.float32)
    vs = np.zeros_like(ks)
    quant.append_int8(kq, ks, vq, vs, bits, bits[::-1].copy(), slots, 16, "bf16")
    pairs = [(3, 7), (0, 11), (5, 2)]
    ocache.copy_blocks(kq, vq, pairs)
    ocache.copy_blocks(ks[..., None], vs[..., None], pairs)
    lib.device_error(clear=True)
    lib.pkv_copy_blocks_int8(torch.tensor(pairs, dtype=torch.int32, device="cuda"), ic)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    kl, vl = _logical_codes(ic.k_codes, ic.v_codes)
    assert np.array_equal(kl, kq) and np.array_equal(vl, vq)
    assert np.array_equal(ic.k_scales.cpu().numpy(), ks)
    assert np.array_equal(ic.v_scales.cpu().numpy(), vs)


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_int8_full_size_sampled(lib, cfg):
    """The benchmark's full batches (Llama-2-7B decode, Llama-3-8B GQA decode,
    g = 8 prefix sharing with 32k-token rows): every slot of the step's bf16
    pools quantised on the device, then the int8 decode call as timed; six
    sequences and the longest one checked against the oracle, which quantises
    those sequences' blocks itself (codes and scales bit-exact, attention within
    the bf16 tolerance)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_51_gb300 import runner

    w = workloads.make(cfg)
    dc, step = runner.prepare(w)
    step.run()
    torch.cuda.synchronize()
    nb, hkv, bs, d = dc.k_cache.shape
    ic = lib.Int8Cache(nb, hkv, bs, d, w.num_q_heads)

    def rows(c):
        return c.transpose(1, 2).reshape(nb * bs, hkv, d).contiguous()

    lib.device_error(clear=True)
    lib.paged_kv_append_int8(rows(dc.k_cache), rows(dc.v_cache),
                             torch.arange(nb * bs, dtype=torch.int64, device="cuda"), ic)
    out = torch.empty_like(step.q)
    lib.paged_attention_decode_int8(out, step.q, ic, step.tables, step.ctx, step.max_ctx)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    ost, _ = execute(w, with_attention=False)
    bt, ctx, _ = ost.batch_metadata()
    assert np.array_equal(bt[:, :step.tables.shape[1]], step.tables.cpu().numpy())
    q_bits = step.q.cpu().view(torch.int16).numpy().view(np.uint16)
    got = out_f64(out)
    rng = np.random.default_rng(cfg)
    picks = set(int(i) for i in rng.choice(len(ctx), size=6, replace=False))
    picks.add(int(np.argmax(ctx)))
    for s in sorted(picks):
        n = -(-int(ctx[s]) // bs)
        blocks = bt[s, :n]
        kq, ks = quant.quantize_rows(ost.k_cache[blocks], "bf16")
        vq, vs = quant.quantize_rows(ost.v_cache[blocks], "bf16")
        idx = torch.from_numpy(blocks.astype(np.int64)).cuda()
        kl, vl = _logical_codes(ic.k_codes[idx], ic.v_codes[idx])
        assert np.array_equal(kl, kq) and np.array_equal(vl, vq)
        assert np.array_equal(ic.k_scales[idx].cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(ic.v_scales[idx].cpu().numpy().view(np.uint32), vs.view(np.uint32))
        ref = quant.decode_int8(q_bits[s:s + 1], kq, ks, vq, vs, np.arange(n)[None], [int(ctx[s])],
                                bs, "bf16")
        diff = np.abs(got[s:s + 1] - ref)
        tmax, tmean = TOL["bf16"]
        assert float(diff.max()) <= tmax and float(diff.mean()) <= tmean
