"""C-ABI library on the host (no GPU needed): exports and the C++ block pool.

The C++ pool is checked operation by operation against the oracle's pool model
(a separate implementation): slots, copy-on-write pairs, block tables,
reference counts and admission statuses must match exactly.
"""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

from oracle.block_pool import LATER, NEVER, OK, BlockPoolModel
from tests.conftest import ROOT, read_kv, read_rows


def _declared_functions():
    with open(os.path.join(ROOT, "include", "pagedkv.h"), encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^PKV_API\s+(?:const\s+)?\w+\*?\s+\**(\w+)\s*\(", text,
                                 flags=re.M)))


def test_library_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert len(declared) >= 19
    L = ctypes.CDLL(lib.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), f"{name} declared in pagedkv.h but not exported"
    assert sorted(lib.EXPORTS) == declared


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.status_string(st) not in ("", "unknown status")
    assert lib.status_string(-99) == "unknown status"


_STATUS = {0: OK, -2: LATER, -3: NEVER}


def test_paging_example_through_abi(lib):
    g = read_kv("paging_example_bs4.txt")
    head = [int(x) for x in g["free_order_head"].split()]
    order = head + [b for b in range(16) if b not in head]
    pool = lib.BlockPool(16, int(g["block_size"]), 0, order)
    assert pool.add(0, int(g["prompt_tokens"])) == [int(x) for x in g["prompt_slots"].split()]
    slot, cow = pool.append_slot(0)
    assert cow is None and slot == int(g["next_token_slot"])
    tables, ctx = pool.block_tables([0], 4)
    assert tables[0, :2].tolist() == [int(x) for x in g["table_after"].split()]
    assert tables[0, 2:].tolist() == [-1, -1] and ctx.tolist() == [5]


@pytest.mark.parametrize("row", read_rows("admission_cases.txt"))
def test_admission_cases_through_abi(lib, row):
    total, wm, used, bs, tokens = (int(x) for x in row[:5])
    pool = lib.BlockPool(total, bs, wm)
    if used:
        pool.add(99, used * bs)
    assert _STATUS[pool.can_allocate(tokens)] == row[5]
    st, _ = pool.add_status(1, tokens)
    assert _STATUS[st] == row[5]


def test_cpp_pool_matches_oracle_model_on_random_traces(lib):
    rng = np.random.default_rng(11)
    for trial in range(6):
        nb, bs = int(rng.integers(20, 120)), int(rng.choice([1, 4, 16]))
        order = rng.permutation(nb)
        wm = int(rng.integers(0, 3))
        ref = BlockPoolModel(nb, bs, wm, order)
        cpp = lib.BlockPool(nb, bs, wm, order)
        next_id = 0
        for _ in range(1500):
            op = int(rng.integers(0, 4))
            seqs = sorted(ref.tables)
            if op == 0 or not seqs:
                n = int(rng.integers(1, 5 * bs + 2))
                st_ref, slots_ref = ref.add_sequence(next_id, n)
                st_cpp, slots_cpp = cpp.add_status(next_id, n)
                assert _STATUS[st_cpp] == st_ref
                assert slots_cpp == slots_ref
                if st_ref == OK:
                    next_id += 1
            elif op == 1:
                s = seqs[int(rng.integers(len(seqs)))]
                slot_ref, cow_ref = ref.append_slot(s)
                st, slot, cow = cpp.append_slot_status(s)
                if slot_ref is None:
                    assert st == lib.PKV_ERR_NO_BLOCKS
                else:
                    assert st == 0 and slot == slot_ref and cow == cow_ref
            elif op == 2 and len(seqs) < 30:
                p = seqs[int(rng.integers(len(seqs)))]
                ref.fork(p, next_id)
                cpp.fork(p, next_id)
                next_id += 1
            elif op == 3:
                s = seqs[int(rng.integers(len(seqs)))]
                ref.free_sequence(s)
                cpp.free(s)
            assert cpp.num_free() == ref.num_free()
        live = sorted(ref.tables)
        if live:
            width = max(len(t) for t in ref.tables.values())
            tables, ctx = cpp.block_tables(live, width)
            for i, s in enumerate(live):
                t = ref.block_table(s)
                assert tables[i, :len(t)].tolist() == t
                assert ctx[i] == ref.context_len(s)
        for b in range(nb):
            assert cpp.ref_count(b) == ref.ref[b]


def test_pool_errors_leave_state_unchanged(lib):
    pool = lib.BlockPool(2, 4)
    pool.add(0, 8)
    st, slot, cow = pool.append_slot_status(0)
    assert st == lib.PKV_ERR_NO_BLOCKS
    assert pool.seq_len(0) == 8 and pool.num_free() == 0
    with pytest.raises(lib.PagedKVError):
        pool.fork(5, 6)             # unknown parent
    with pytest.raises(lib.PagedKVError):
        pool.add(0, 1)              # existing id
    with pytest.raises(lib.PagedKVError):
        pool.block_tables([0], 1)   # table wider than max_blocks
    with pytest.raises(lib.PagedKVError):
        lib.BlockPool(4, 4, 0, [0, 1, 1, 2])  # not a permutation


def test_workspace_sizes_are_host_computable(lib):
    import torch

    desc = lib.CacheDesc(lib.PKV_BF16, 100, 16, 8, 32, 128)
    a = lib.decode_workspace_bytes(desc, 64, 4096)
    b = lib.decode_workspace_bytes(desc, 64, 512)
    assert a > b > 0 and a % 256 == 0
    # 64 seqs x 32 heads x 8 splits x (128 floats + (m, l))
    assert a >= 64 * 32 * 8 * (128 * 4 + 8)
    assert lib.varlen_workspace_bytes(desc, 515, 2048, 512, 3584) > 0
    bad = lib.CacheDesc(7, 100, 16, 8, 32, 128)
    assert lib.decode_workspace_bytes(bad, 1, 1) == 0
    del torch


def test_device_calls_reject_bad_arguments_before_launch(lib):
    """Host-side validation returns an error without touching a GPU."""
    L = lib.lib()
    desc = lib.CacheDesc(lib.PKV_BF16, 100, 16, 8, 32, 128)
    ref = ctypes.byref
    # null pointers
    assert L.paged_kv_append(None, None, None, 4, None, None, ref(desc), None) == lib.PKV_ERR_INVALID
    assert L.paged_attention_decode(None, None, None, None, ref(desc), None, 4, None, 1, 16,
                                    0.1, None, 0, None) == lib.PKV_ERR_INVALID
    # unsupported shapes for attention
    odd = lib.CacheDesc(lib.PKV_BF16, 100, 32, 8, 32, 128)   # block_size 32
    fake = ctypes.c_void_p(1 << 20)
    assert L.paged_attention_decode(fake, fake, fake, fake, ref(odd), fake, 4, fake, 1, 16, 0.1,
                                    fake, 1 << 20, None) == lib.PKV_ERR_UNSUPPORTED
    g3 = lib.CacheDesc(lib.PKV_BF16, 100, 16, 8, 24, 128)    # group of 3
    assert L.paged_attention_decode(fake, fake, fake, fake, ref(g3), fake, 4, fake, 1, 16, 0.1,
                                    fake, 1 << 20, None) == lib.PKV_ERR_UNSUPPORTED
    # workspace too small
    assert L.paged_attention_decode(fake, fake, fake, fake, ref(desc), fake, 4, fake, 64, 4096,
                                    0.1, fake, 256, None) == lib.PKV_ERR_WORKSPACE
    # zero-sized work is a no-op
    assert L.paged_kv_append(None, None, None, 0, None, None, ref(desc), None) == 0
    assert L.pkv_copy_blocks(None, 0, None, None, ref(desc), None) == 0
    # an empty attention batch is a no-op whatever its pointers hold (zero-sized
    # tensors often have a null data pointer); its descriptor is still checked
    assert L.paged_attention_decode(None, None, None, None, ref(desc), None, 4, None, 0, 16,
                                    0.1, None, 0, None) == 0
    assert L.paged_attention_decode(None, None, None, None, ref(odd), None, 4, None, 0, 16,
                                    0.1, None, 0, None) == lib.PKV_ERR_UNSUPPORTED
    assert L.paged_attention_varlen(None, None, None, None, ref(desc), None, 4, None, None, 2, 0,
                                    0, 16, 0.1, None, 0, None) == 0
    assert L.paged_attention_varlen(None, None, None, None, ref(desc), None, 4, None, None, 0, 0,
                                    0, 16, 0.1, None, 0, None) == 0


def test_int8_entry_points_validate_on_the_host(lib):
    L = lib.lib()
    ref = ctypes.byref
    i8 = lib.CacheDesc(lib.PKV_INT8, 100, 16, 8, 32, 128)
    bf = lib.CacheDesc(lib.PKV_BF16, 100, 16, 8, 32, 128)
    fake = ctypes.c_void_p(1 << 20)
    # the split partials do not depend on the cache type
    assert lib.decode_workspace_bytes(i8, 64, 4096) == lib.decode_workspace_bytes(bf, 64, 4096)
    # a tile is the 16 rows' codes and then their fp32 scales
    assert lib.int8_tile_bytes(128) == 16 * 128 + 64 and lib.int8_tile_bytes(64) == 1088
    # the 8-bit calls take only PKV_INT8, the others never take it
    assert L.paged_kv_append_int8(fake, fake, fake, 4, fake, ref(bf),
                                  None) == lib.PKV_ERR_UNSUPPORTED
    assert L.paged_attention_decode_int8(fake, fake, fake, ref(bf), fake, 4,
                                         fake, 1, 16, 0.1, fake, 1 << 20,
                                         None) == lib.PKV_ERR_UNSUPPORTED
    assert L.paged_kv_append(fake, fake, fake, 4, fake, fake, ref(i8), None) == \
        lib.PKV_ERR_UNSUPPORTED
    assert L.paged_attention_decode(fake, fake, fake, fake, ref(i8), fake, 4, fake, 1, 16, 0.1,
                                    fake, 1 << 20, None) == lib.PKV_ERR_UNSUPPORTED
    # null pointers, a misaligned pool, head_dim, workspace, empty work
    assert L.paged_kv_append_int8(None, fake, fake, 4, fake, ref(i8),
                                  None) == lib.PKV_ERR_INVALID
    assert L.paged_kv_append_int8(fake, fake, fake, 4, None, ref(i8),
                                  None) == lib.PKV_ERR_INVALID
    assert L.paged_kv_append_int8(fake, fake, fake, 4, ctypes.c_void_p((1 << 20) + 4),
                                  ref(i8), None) == lib.PKV_ERR_INVALID
    assert L.paged_attention_decode_int8(fake, fake, ctypes.c_void_p((1 << 20) + 8),
                                         ref(i8), fake, 4, fake, 1, 16, 0.1, fake, 1 << 20,
                                         None) == lib.PKV_ERR_INVALID
    assert L.paged_attention_decode_int8(fake, fake, None, ref(i8), fake, 4, fake, 1, 16, 0.1,
                                         fake, 1 << 20, None) == lib.PKV_ERR_INVALID
    d96 = lib.CacheDesc(lib.PKV_INT8, 100, 16, 8, 32, 96)
    assert L.paged_kv_append_int8(fake, fake, fake, 4, fake, ref(d96),
                                  None) == lib.PKV_ERR_UNSUPPORTED
    assert L.paged_attention_decode_int8(fake, fake, fake, ref(i8), fake, 4,
                                         fake, 64, 4096, 0.1, fake, 256,
                                         None) == lib.PKV_ERR_WORKSPACE
    assert L.paged_attention_decode_int8(fake, fake, fake, ref(i8), fake, 4,
                                         fake, 1, 16, float("nan"), fake, 1 << 20,
                                         None) == lib.PKV_ERR_INVALID
    assert L.paged_kv_append_int8(None, None, None, 0, None, ref(i8), None) == 0
    # copy-on-write for the 8-bit cache takes only PKV_INT8, with 16-row tiles
    assert L.pkv_copy_blocks_int8(fake, 2, fake, ref(bf), None) == \
        lib.PKV_ERR_UNSUPPORTED
    b8 = lib.CacheDesc(lib.PKV_INT8, 100, 8, 8, 32, 128)
    assert L.pkv_copy_blocks_int8(fake, 2, fake, ref(b8), None) == \
        lib.PKV_ERR_UNSUPPORTED
    assert L.pkv_copy_blocks_int8(None, 2, fake, ref(i8), None) == \
        lib.PKV_ERR_INVALID
    assert L.pkv_copy_blocks_int8(fake, 2, ctypes.c_void_p((1 << 20) + 4), ref(i8), None) == \
        lib.PKV_ERR_INVALID
    assert L.pkv_copy_blocks_int8(None, 0, None, ref(i8), None) == 0


def test_int8_cache_views_follow_the_tile_layout(lib):
    """The binding's code and scale views alias the one pool as the header lays
    it out: per (block, KV head) the K tile and then the V tile, each 16 rows of
    codes and then the 16 rows' fp32 scales."""
    import numpy as np
    import torch

    for d in (128, 64):
        c = lib.Int8Cache(3, 2, 16, d, 4, device="cpu")
        tile = lib.int8_tile_bytes(d)
        assert tuple(c.kv_pool.shape) == (3, 2, 2, tile) and c.kv_pool.dtype == torch.uint8
        assert c.kv_pool.is_contiguous()
        assert tuple(c.k_pool.shape) == (3, 2, tile) and c.k_pool.dtype == torch.uint8
        assert tuple(c.k_codes.shape) == (3, 2, 16, d) and c.k_codes.dtype == torch.int8
        assert tuple(c.v_scales.shape) == (3, 2, 16) and c.v_scales.dtype == torch.float32
        c.k_codes[2, 1, 5, 7] = -3
        c.v_scales[1, 0, 9] = 0.25
        flat = c.kv_pool.numpy().reshape(-1)
        unit = 2 * tile                                   # one (block, head): K then V
        assert flat[(2 * 2 + 1) * unit + 5 * d + 7].view(np.int8) == -3
        at = (1 * 2 + 0) * unit + tile + 16 * d + 4 * 9
        assert flat[at:at + 4].view(np.float32)[0] == 0.25
        assert np.count_nonzero(flat) == 3                # -3, and 0.25 = 0x3e800000
        (kv,) = c.tensors()
        assert kv is c.kv_pool


def test_binding_refuses_values_outside_int32(lib):
    """Token ids, prompt lengths and the free order cross the ABI as int32; the
    binding raises on a value outside int32 instead of letting it wrap, and on a
    free order of the wrong length instead of letting the pool read past it."""
    pool = lib.BlockPool(64, 16, 0, prefix_caching=True)
    with pytest.raises(ValueError):
        pool.add_tokens(1, [5, 1 << 31])
    with pytest.raises(ValueError):
        pool.add_tokens(1, [-(1 << 31) - 1])
    st, slots, cached = pool.add_tokens(1, [5, (1 << 31) - 1, -(1 << 31)])
    assert st == lib.PKV_OK and len(slots) == 3 and cached == 0
    with pytest.raises(ValueError):
        lib.pkv_splitfuse_compose(16, 0, [3, 1 << 32])
    with pytest.raises(ValueError):
        lib.BlockPool(4, 16, 0, [0, 1, 2])
    with pytest.raises(TypeError):
        lib.pkv_splitfuse_compose(16, 0, np.array([1.5, 2.0]))
    # integers beyond int64 and inputs without len() (generators) are handled too
    with pytest.raises(ValueError):
        pool.add_tokens(1, [7, 1 << 63])
    with pytest.raises(ValueError):
        lib.pkv_splitfuse_compose(16, 0, (x for x in [3, 1 << 40]))
    st, slots, cached = pool.add_tokens(2, (t for t in [9, 8, 7]))
    assert st == lib.PKV_OK and len(slots) == 3
    assert lib.pkv_splitfuse_compose(16, 0, (x for x in [3, 4]))[1] == [3, 4]


class _FakeStream:
    def __init__(self, index):
        self.device = torch.device("cuda", index)
        self.cuda_stream = 0


class _FakeTensor:
    """Stands in for a CUDA tensor on device `index` (no memory, no kernel)."""

    def __init__(self, index, dtype, shape):
        self.device = torch.device("cuda", index)
        self.dtype = dtype
        self.shape = shape
        self.is_cuda = True

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return 0

    def numel(self):
        return 1 << 20


def test_binding_refuses_tensors_off_the_current_device(lib, monkeypatch):
    """The kernels run on the current device (its stream, its error word, its
    scratch array), so a tensor or stream of another GPU is refused on the host
    before the C call, and nothing is launched."""
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: _FakeStream(0))
    called = []
    monkeypatch.setattr(lib, "lib", lambda: called.append(1) or (_ for _ in ()).throw(
        AssertionError("the C library was called")))
    bf = torch.bfloat16
    desc = lib.CacheDesc(lib.PKV_BF16, 64, 16, 8, 32, 128)

    def args(dev_of_q, dev_of_tables=0):
        return dict(out=_FakeTensor(0, bf, (4, 32, 128)), q=_FakeTensor(dev_of_q, bf, (4, 32, 128)),
                    k_cache=_FakeTensor(0, bf, (64, 8, 16, 128)),
                    v_cache=_FakeTensor(0, bf, (64, 8, 16, 128)), desc=desc,
                    block_tables=_FakeTensor(dev_of_tables, torch.int32, (4, 8)),
                    context_lens=_FakeTensor(0, torch.int32, (4,)), max_context_len=100,
                    ws=_FakeTensor(0, torch.uint8, (1 << 20,)))

    with pytest.raises(ValueError, match="q is on cuda:1"):
        lib.paged_attention_decode(**args(1))
    with pytest.raises(ValueError, match="block_tables is on cuda:3"):
        lib.paged_attention_decode(**args(0, 3))
    a = args(0)
    a.pop("ws")
    a["q"] = _FakeTensor(2, bf, (4, 32, 128))
    with pytest.raises(ValueError, match="q is on cuda:2"):
        lib.paged_attention_decode_noalloc(**a)
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        lib.paged_attention_decode(**args(0), stream=_FakeStream(1))
    k = _FakeTensor(0, bf, (4, 8, 128))
    with pytest.raises(ValueError, match="slot_mapping is on cuda:1"):
        lib.paged_kv_append(k, k, _FakeTensor(1, torch.int64, (4,)),
                            _FakeTensor(0, bf, (64, 8, 16, 128)),
                            _FakeTensor(0, bf, (64, 8, 16, 128)), desc)
    assert not called
    # the pure check itself
    lib._devices_agree([("a", torch.device("cuda", 0))], 0, torch.device("cuda", 0))
    with pytest.raises(ValueError):
        lib._devices_agree([("a", torch.device("cpu"))], 0, torch.device("cuda", 0))
