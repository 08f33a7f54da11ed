"""GPU parity for the block-table variants: prefix-cached blocks shared between
sequences, and sliding-window rings, feeding the unchanged attention kernels.
Expected values are float64 dense attention over each sequence's unpaged rows."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads  # noqa: E402
from oracle import attention, numerics  # noqa: E402
from tests.gpu_parity import TOL, out_f64  # noqa: E402

pytestmark = pytest.mark.gpu


def _t(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _dense(q_bits, k_bits, v_bits, g):
    """Exact attention of q [hq, d] over k, v [n, hkv, d] (bf16 bits)."""
    q = numerics.widen(q_bits, "bf16")
    k = numerics.widen(k_bits, "bf16")
    v = numerics.widen(v_bits, "bf16")
    d = q.shape[-1]
    return np.stack([attention.softmax_attention(q[h][None], k[:, h // g], v[:, h // g],
                                                 1 / np.sqrt(d))[0] for h in range(q.shape[0])])


def _check(out, ref):
    diff = np.abs(out_f64(out) - ref)
    tmax, tmean = TOL["bf16"]
    assert float(diff.max()) <= tmax and float(diff.mean()) <= tmean


def test_prefix_cached_blocks_feed_decode_and_prefill(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hq, hkv, d, bs, nb = 32, 8, 128, 16, 64
    g = hq // hkv
    tv = workloads.TokenValues(5, 50, 1024, hkv, d)
    rng = np.random.default_rng(6)
    pool = lib.BlockPool(nb, bs, 0, rng.permutation(nb), prefix_caching=True)
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    desc = lib.cache_desc(kc, hq)
    toks = {}

    def add(sid, t):
        st, slots, cached = pool.add_tokens(sid, t)
        assert st == 0
        k, v = tv.rows(t[cached:], range(cached, len(t)))
        lib.paged_kv_append(_t(k), _t(v), torch.tensor(slots[cached:], device="cuda"), kc, vc,
                            desc)
        toks[sid] = t
        return cached

    a = rng.integers(0, 50, 200).tolist()
    b = a[:160] + rng.integers(0, 50, 50).tolist()
    c = a[:100] + rng.integers(0, 50, 30).tolist()
    lib.device_error(clear=True)
    assert add(0, a) == 0
    assert add(1, b) == 160
    assert add(2, c) == 96
    tables, ctx = pool.block_tables([0, 1, 2], 16)
    assert tables[0, :10].tolist() == tables[1, :10].tolist()
    assert tables[0, :6].tolist() == tables[2, :6].tolist() and tables[0, 6] != tables[2, 6]
    # one call: decode rows for a and c, a 50-token prefill chunk of b over its cached 160
    qa = workloads._values(rng, (1, hq, d), "bf16", 0.5)
    qb = workloads._values(rng, (50, hq, d), "bf16", 0.5)
    qc = workloads._values(rng, (1, hq, d), "bf16", 0.5)
    q = _t(np.concatenate([qa, qb, qc]))
    out = torch.empty_like(q)
    qsl = torch.tensor([0, 1, 51, 52], dtype=torch.int32, device="cuda")
    lib.paged_attention_varlen(out, q, kc, vc, desc, tables.cuda(), qsl, ctx.cuda(), 50,
                               int(ctx.max()))
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    rows = {s: tv.rows(t, range(len(t))) for s, t in toks.items()}
    _check(out[0:1], _dense(qa[0], *rows[0], g)[None])
    _check(out[51:52], _dense(qc[0], *rows[2], g)[None])
    ref_b = np.stack([_dense(qb[i], rows[1][0][:161 + i], rows[1][1][:161 + i], g)
                      for i in range(50)])
    _check(out[1:51], ref_b)
    # a's full blocks are parked when it finishes, and a new copy of its prompt takes them back
    pool.set_clock(7)
    pool.free(0)
    assert pool.num_evictable() == 2            # blocks 10, 11 of a (0..9 still used by b)
    assert add(3, a) == 192
    tables, ctx = pool.block_tables([3], 16)
    qd = workloads._values(rng, (1, hq, d), "bf16", 0.5)
    out = torch.empty((1, hq, d), dtype=torch.bfloat16, device="cuda")
    lib.paged_attention_decode(out, _t(qd), kc, vc, desc, tables.cuda(), ctx.cuda(), 200)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    _check(out, _dense(qd[0], *tv.rows(a, range(200)), g)[None])


def test_sliding_window_rings_feed_decode(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hq, hkv, d, bs, window, nb = 16, 4, 128, 16, 256, 96
    g = hq // hkv
    tv = workloads.TokenValues(8, 64, 2048, hkv, d)
    rng = np.random.default_rng(9)
    pool = lib.BlockPool(nb, bs, 0, rng.permutation(nb), sliding_window=window)
    kc = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    desc = lib.cache_desc(kc, hq)
    toks = {}
    lib.device_error(clear=True)

    def write(tok, pos, slots):
        k, v = tv.rows(tok, pos)
        lib.paged_kv_append(_t(k), _t(v), torch.tensor(slots, device="cuda"), kc, vc, desc)

    # a prompt longer than the window: its first tokens are skipped (slot -1)
    for sid, n in ((0, 100), (2, 700)):
        st, slots = pool.add_status(sid, n)
        assert st == 0 and (slots.count(-1) == max(0, n - window))
        toks[sid] = rng.integers(0, 64, n).tolist()
        write(toks[sid], range(n), slots)
    # grow token by token; fork 0 at length 600 and grow both (ring blocks copied on write)
    for step in range(900):
        if step == 500:
            pool.fork(0, 1)
            toks[1] = list(toks[0])
        live = [s for s in (0, 1, 2) if s in toks and len(toks[s]) < {0: 1000, 1: 800, 2: 900}[s]]
        slots, pairs, tk, ps = [], [], [], []
        for s in live:
            slot, cow = pool.append_slot(s)
            if cow:
                pairs.append(cow)
            t = int(rng.integers(0, 64))
            tk.append(t)
            ps.append(len(toks[s]))
            toks[s].append(t)
            slots.append(slot)
        if not live:
            break
        if pairs:
            lib.pkv_copy_blocks(torch.tensor(pairs, dtype=torch.int32, device="cuda"), kc, vc,
                                desc)
        write(tk, ps, slots)
    ids = [0, 1, 2]
    tables, ctx = pool.block_tables(ids, window // bs)
    assert ctx.tolist() == [window] * 3
    q = workloads._values(rng, (3, hq, d), "bf16", 0.5)
    out = torch.empty((3, hq, d), dtype=torch.bfloat16, device="cuda")
    lib.paged_attention_decode(out, _t(q), kc, vc, desc, tables.cuda(), ctx.cuda(), window)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    for i, s in enumerate(ids):
        n = len(toks[s])
        k, v = tv.rows(toks[s][n - window:], range(n - window, n))
        _check(out[i:i + 1], _dense(q[i], k, v, g)[None])
