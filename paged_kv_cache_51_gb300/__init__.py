"""Paged KV-cache attention for GB300 (sm_103a): thin Python binding of libpagedkv.so.

Every function here only marshals arguments (tensor data pointers, sizes and
the current CUDA stream) into the C ABI declared in include/pagedkv.h; all work
runs in the library's CUDA kernels or its C++ block pool.  There is no fallback:
if the library is missing or was built for another machine, calls raise.

PyTorch supplies device memory and streams only.
"""

import ctypes
import math
import os

import numpy as np

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PKV_OK = 0
PKV_ERR_INVALID = -1
PKV_ERR_NO_BLOCKS = -2
PKV_ERR_NEVER = -3
PKV_ERR_UNSUPPORTED = -4
PKV_ERR_CUDA = -5
PKV_ERR_WORKSPACE = -6
PKV_ERR_HOST = -7

PKV_F32 = 0
PKV_BF16 = 1
PKV_INT8 = 2

DEVICE_ERRORS = {
    0: "ok", 1: "bad block id", 2: "bad context length", 3: "bad slot", 4: "bad copy pair",
    5: "bad query layout", 6: "pipeline wait timeout", 7: "block table too narrow",
    8: "bad rotary position",
}

# every symbol the header declares (checked by the tests)
EXPORTS = (
    "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_num_free", "pkv_pool_can_allocate",
    "pkv_seq_add", "pkv_seq_fork", "pkv_seq_append_slot", "pkv_seq_free", "pkv_seq_len",
    "pkv_block_ref_count", "pkv_block_tables", "pkv_copy_blocks", "paged_kv_append",
    "paged_kv_append_rope",
    "pkv_decode_workspace_bytes", "paged_attention_decode", "paged_attention_decode_noalloc",
    "pkv_varlen_workspace_bytes",
    "paged_attention_varlen", "pkv_device_error", "pkv_status_string", "pkv_splitfuse_compose",
    "paged_kv_append_int8", "paged_attention_decode_int8", "pkv_copy_blocks_int8",
    "pkv_pool_create_ex", "pkv_pool_num_evictable", "pkv_pool_set_clock", "pkv_seq_add_tokens",
    "pkv_seq_append_token", "pkv_block_hash", "pkv_pool_create_window", "pkv_window_tables",
    "paged_attention_varlen_window",
)

PKV_POOL_PREFIX_CACHING = 1


class PagedKVError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class CacheDesc(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


_lib = None


def lib():
    """Load libpagedkv.so (built by paged_kv_cache_51_gb300._build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run paged_kv_cache_51_gb300._build.build()")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, p, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "pkv_pool_create": (ctypes.c_int, [i32, i32, i32, p, P(p)]),
        "pkv_pool_create_ex": (ctypes.c_int, [i32, i32, i32, p, i32, i32, P(p)]),
        "pkv_pool_create_window": (ctypes.c_int, [i32, i32, i32, p, i32, i32, P(p)]),
        "pkv_window_tables": (ctypes.c_int, [p, p, p, i32, i32, p, p]),
        "paged_attention_varlen_window": (ctypes.c_int, [p, p, p, p, P(CacheDesc), p, i32, p, p,
                                                         i32, i32, i32, i32, i32, ctypes.c_float,
                                                         p, sz, p]),
        "pkv_pool_num_evictable": (ctypes.c_int, [p, P(i32)]),
        "pkv_pool_set_clock": (ctypes.c_int, [p, i64]),
        "pkv_seq_add_tokens": (ctypes.c_int, [p, i64, p, i32, p, P(i32)]),
        "pkv_seq_append_token": (ctypes.c_int, [p, i64, i32, P(i64), P(i32), P(i32)]),
        "pkv_block_hash": (ctypes.c_int, [p, i32, P(ctypes.c_uint64), P(i32)]),
        "pkv_pool_destroy": (ctypes.c_int, [p]),
        "pkv_pool_num_free": (ctypes.c_int, [p, P(i32)]),
        "pkv_pool_can_allocate": (ctypes.c_int, [p, i32]),
        "pkv_seq_add": (ctypes.c_int, [p, i64, i32, p]),
        "pkv_seq_fork": (ctypes.c_int, [p, i64, i64]),
        "pkv_seq_append_slot": (ctypes.c_int, [p, i64, P(i64), P(i32), P(i32)]),
        "pkv_seq_free": (ctypes.c_int, [p, i64]),
        "pkv_seq_len": (ctypes.c_int, [p, i64, P(i32)]),
        "pkv_block_ref_count": (ctypes.c_int, [p, i32, P(i32)]),
        "pkv_block_tables": (ctypes.c_int, [p, p, i32, i32, p, p]),
        "pkv_copy_blocks": (ctypes.c_int, [p, i32, p, p, P(CacheDesc), p]),
        "paged_kv_append": (ctypes.c_int, [p, p, p, i32, p, p, P(CacheDesc), p]),
        "paged_kv_append_rope": (ctypes.c_int, [p, p, p, p, p, p, p, i32, i32, p, p,
                                                P(CacheDesc), p]),
        "pkv_decode_workspace_bytes": (sz, [P(CacheDesc), i32, i32]),
        "paged_attention_decode": (ctypes.c_int, [p, p, p, p, P(CacheDesc), p, i32, p, i32, i32,
                                                  ctypes.c_float, p, sz, p]),
        "paged_attention_decode_noalloc": (ctypes.c_int, [p, p, p, p, P(CacheDesc), p, i32, p,
                                                          i32, i32, ctypes.c_float, p]),
        "pkv_varlen_workspace_bytes": (sz, [P(CacheDesc), i32, i32, i32, i32]),
        "paged_attention_varlen": (ctypes.c_int, [p, p, p, p, P(CacheDesc), p, i32, p, p, i32,
                                                  i32, i32, i32, ctypes.c_float, p, sz, p]),
        "pkv_device_error": (ctypes.c_int, [P(i32), i32]),
        "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "pkv_splitfuse_compose": (ctypes.c_int, [i32, i32, i32, p, p, P(i32), P(i32)]),
        "paged_kv_append_int8": (ctypes.c_int, [p, p, p, i32, p, P(CacheDesc), p]),
        "pkv_copy_blocks_int8": (ctypes.c_int, [p, i32, p, P(CacheDesc), p]),
        "paged_attention_decode_int8": (ctypes.c_int, [p, p, p, P(CacheDesc), p, i32, p, i32,
                                                       i32, ctypes.c_float, p, sz, p]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def status_string(status):
    try:
        return lib().pkv_status_string(status).decode()
    except Exception:
        return "status"


_I32_MIN, _I32_MAX = -(1 << 31), (1 << 31) - 1


def _host_int32(values, name):
    """A contiguous host int32 copy of `values` (a sequence of ints or an integer
    array); a value outside int32 raises ValueError instead of wrapping."""
    if isinstance(values, np.ndarray):
        a = values
    else:
        vals = values if isinstance(values, (list, tuple)) else list(values)
        if len(vals) == 0:
            return np.zeros(0, dtype=np.int32)
        try:
            a = np.asarray(vals)
        except OverflowError as e:
            raise ValueError(f"{name}: a value is outside int32") from e
        if a.dtype.kind in "fO":
            # numpy widens ints beyond int64 (or int64 mixed with uint64) to
            # object or float: out of range if every element is an int
            if all(isinstance(x, (int, np.integer)) and not isinstance(x, bool) for x in vals):
                raise ValueError(f"{name}: a value is outside int32")
            raise TypeError(f"{name}: integers expected")
    if a.dtype.kind not in "iu":
        raise TypeError(f"{name}: integers expected, got {a.dtype}")
    if a.size and (int(a.min()) < _I32_MIN or int(a.max()) > _I32_MAX):
        raise ValueError(f"{name}: a value is outside int32")
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(status, what):
    if status != PKV_OK:
        raise PagedKVError(status, what)


# ----------------------------------------------------------------------------
# host block pool
# ----------------------------------------------------------------------------
class BlockPool:
    """Host block pool (C++): ref-counted blocks, block tables, copy-on-write."""

    def __init__(self, num_blocks, block_size, watermark_blocks=0, free_order=None,
                 prefix_caching=False, sliding_window=0, max_chunk=1):
        """``sliding_window`` > 0 with ``max_chunk`` > 1: a window pool whose ring
        also holds the keys of prefill chunks of up to max_chunk tokens
        (pkv_pool_create_window)."""
        self._h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            order = _host_int32(free_order, "free_order")
            if order.shape != (num_blocks,):
                raise ValueError(f"free_order: {order.shape[0]} entries, expected {num_blocks}")
        optr = None if order is None else order.ctypes.data
        if max_chunk != 1:
            if prefix_caching or sliding_window < 1:
                raise ValueError("max_chunk applies to sliding-window pools only")
            _check(lib().pkv_pool_create_window(num_blocks, block_size, watermark_blocks, optr,
                                                sliding_window, max_chunk, ctypes.byref(self._h)),
                   "pkv_pool_create_window")
        else:
            flags = PKV_POOL_PREFIX_CACHING if prefix_caching else 0
            _check(lib().pkv_pool_create_ex(num_blocks, block_size, watermark_blocks, optr, flags,
                                            sliding_window, ctypes.byref(self._h)),
                   "pkv_pool_create_ex")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.prefix_caching = prefix_caching
        self.sliding_window = sliding_window
        self.max_chunk = max_chunk

    def close(self):
        if self._h:
            lib().pkv_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self):
        out = ctypes.c_int32()
        _check(lib().pkv_pool_num_free(self._h, ctypes.byref(out)), "pkv_pool_num_free")
        return out.value

    def can_allocate(self, num_tokens):
        """PKV_OK, PKV_ERR_NO_BLOCKS (LATER) or PKV_ERR_NEVER."""
        return lib().pkv_pool_can_allocate(self._h, num_tokens)

    def add(self, seq_id, num_tokens):
        """Returns the slots of the prompt's tokens (list of int)."""
        slots = np.empty(max(num_tokens, 1), dtype=np.int64)
        _check(lib().pkv_seq_add(self._h, seq_id, num_tokens, slots.ctypes.data), "pkv_seq_add")
        return slots[:num_tokens].tolist()

    def add_status(self, seq_id, num_tokens):
        slots = (ctypes.c_int64 * max(num_tokens, 1))()
        st = lib().pkv_seq_add(self._h, seq_id, num_tokens, slots)
        return st, (list(slots)[:num_tokens] if st == PKV_OK else None)

    def add_tokens(self, seq_id, token_ids):
        """Returns (status, slots or None, num_cached_tokens)."""
        toks = _host_int32(token_ids, "token_ids")
        n = int(toks.shape[0])
        if n == 0:
            toks = np.zeros(1, dtype=np.int32)
        slots = np.empty(max(n, 1), dtype=np.int64)
        cached = ctypes.c_int32()
        st = lib().pkv_seq_add_tokens(self._h, seq_id, toks.ctypes.data, n, slots.ctypes.data,
                                      ctypes.byref(cached))
        return st, (slots[:n].tolist() if st == PKV_OK else None), cached.value

    def append_token(self, seq_id, token_id):
        """Returns (status, slot, cow) with cow = (src, dst) or None."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        st = lib().pkv_seq_append_token(self._h, seq_id, int(token_id), ctypes.byref(slot),
                                        ctypes.byref(src), ctypes.byref(dst))
        return st, slot.value, ((src.value, dst.value) if st == PKV_OK and src.value >= 0 else None)

    def set_clock(self, now):
        _check(lib().pkv_pool_set_clock(self._h, int(now)), "pkv_pool_set_clock")

    def num_evictable(self):
        out = ctypes.c_int32()
        _check(lib().pkv_pool_num_evictable(self._h, ctypes.byref(out)), "pkv_pool_num_evictable")
        return out.value

    def block_hash(self, block):
        """The registered hash of a block, or None."""
        h, reg = ctypes.c_uint64(), ctypes.c_int32()
        _check(lib().pkv_block_hash(self._h, block, ctypes.byref(h), ctypes.byref(reg)),
               "pkv_block_hash")
        return h.value if reg.value else None

    def fork(self, parent, child):
        _check(lib().pkv_seq_fork(self._h, parent, child), "pkv_seq_fork")

    def append_slot(self, seq_id):
        """Returns (slot, cow) with cow = (src, dst) or None."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().pkv_seq_append_slot(self._h, seq_id, ctypes.byref(slot), ctypes.byref(src),
                                         ctypes.byref(dst)), "pkv_seq_append_slot")
        return slot.value, ((src.value, dst.value) if src.value >= 0 else None)

    def append_slot_status(self, seq_id):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        st = lib().pkv_seq_append_slot(self._h, seq_id, ctypes.byref(slot), ctypes.byref(src),
                                       ctypes.byref(dst))
        return st, slot.value, ((src.value, dst.value) if st == PKV_OK and src.value >= 0 else None)

    def free(self, seq_id):
        _check(lib().pkv_seq_free(self._h, seq_id), "pkv_seq_free")

    def seq_len(self, seq_id):
        out = ctypes.c_int32()
        _check(lib().pkv_seq_len(self._h, seq_id, ctypes.byref(out)), "pkv_seq_len")
        return out.value

    def ref_count(self, block):
        out = ctypes.c_int32()
        _check(lib().pkv_block_ref_count(self._h, block, ctypes.byref(out)), "pkv_block_ref_count")
        return out.value

    def block_tables(self, seq_ids, max_blocks):
        """Returns (tables int32 tensor [n, max_blocks] padded with -1, ctx int32 tensor [n])."""
        n = len(seq_ids)
        ids = torch.tensor(list(seq_ids), dtype=torch.int64)
        tables = torch.empty((n, max_blocks), dtype=torch.int32)
        ctx = torch.empty(n, dtype=torch.int32)
        _check(lib().pkv_block_tables(self._h, ids.data_ptr(), n, max_blocks, tables.data_ptr(),
                                      ctx.data_ptr()), "pkv_block_tables")
        return tables, ctx


    def window_tables(self, seq_ids, query_lens, max_blocks):
        """Logically ordered tables of a sliding-window pool for a step whose last
        query_lens[i] tokens of sequence seq_ids[i] are queries (pkv_window_tables).
        Returns (tables int32 tensor [n, max_blocks] padded with -1, ctx int32 [n])."""
        n = len(seq_ids)
        ids = torch.tensor(list(seq_ids), dtype=torch.int64)
        ql = _host_int32(query_lens, "query_lens")
        if ql.shape != (n,):
            raise ValueError("query_lens: one entry per sequence")
        tables = torch.empty((n, max_blocks), dtype=torch.int32)
        ctx = torch.empty(n, dtype=torch.int32)
        _check(lib().pkv_window_tables(self._h, ids.data_ptr(), ql.ctypes.data if n else None, n,
                                       max_blocks, tables.data_ptr(), ctx.data_ptr()),
               "pkv_window_tables")
        return tables, ctx


def pkv_splitfuse_compose(token_budget, num_decode, prompt_remaining):
    """Token-budget composition of one forward pass (C++).

    Returns (decode_admitted, chunks, tokens_used): the first decode_admitted
    decode sequences take one token each, prompt i takes chunks[i] tokens."""
    rem = _host_int32(prompt_remaining, "prompt_remaining")
    n = int(rem.shape[0])
    if n == 0:
        rem = np.zeros(1, dtype=np.int32)
    out = np.zeros(max(n, 1), dtype=np.int32)
    dec, used = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().pkv_splitfuse_compose(token_budget, num_decode, n, rem.ctypes.data,
                                       out.ctypes.data, ctypes.byref(dec), ctypes.byref(used)),
           "pkv_splitfuse_compose")
    return dec.value, out[:n].tolist(), used.value


# ----------------------------------------------------------------------------
# device entry points
# ----------------------------------------------------------------------------
_TORCH_DTYPE = {PKV_F32: torch.float32, PKV_BF16: torch.bfloat16}


def cache_desc(k_cache, num_q_heads):
    """Descriptor of a cache tensor [num_blocks, num_kv_heads, block_size, head_dim]."""
    nb, hkv, bs, d = k_cache.shape
    dt = {torch.float32: PKV_F32, torch.bfloat16: PKV_BF16}.get(k_cache.dtype)
    if dt is None:
        raise TypeError("cache dtype must be float32 or bfloat16")
    return CacheDesc(dt, nb, bs, hkv, num_q_heads, d)


def _devices_agree(named_devices, current, stream_device):
    """Raise ValueError unless every (name, torch.device) pair and the stream's
    device are the current CUDA device: the library's kernels run on the
    current device and its device-side state (error word, scratch array) is
    looked up there, so a pointer into another GPU's memory would fault or be
    read over the peer link."""
    if stream_device.type != "cuda" or stream_device.index != current:
        raise ValueError(f"stream is on {stream_device}, but the current device is cuda:{current}")
    for name, dev in named_devices:
        if dev.type != "cuda" or dev.index != current:
            raise ValueError(f"{name} is on {dev}, but the current device is cuda:{current}; "
                             f"call under torch.cuda.device({dev})")


def _stream_on_device(stream, *named):
    """The stream handle for a launch, after checking that the stream and every
    named tensor (name, tensor or None) are on the current CUDA device."""
    if stream is None:
        stream = torch.cuda.current_stream()
    _devices_agree([(n, t.device) for n, t in named if t is not None],
                   torch.cuda.current_device(), stream.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, dtype, name):
    if not t.is_cuda or not t.is_contiguous() or t.dtype != dtype:
        raise TypeError(f"{name} must be a contiguous CUDA {dtype} tensor")


def pkv_copy_blocks(block_pairs, k_cache, v_cache, desc, stream=None):
    """block_pairs: CUDA int32 [n, 2] (src, dst)."""
    n = block_pairs.shape[0] if block_pairs is not None else 0
    if n == 0:
        return
    _need(block_pairs, torch.int32, "block_pairs")
    st = _stream_on_device(stream, ("block_pairs", block_pairs), ("k_cache", k_cache),
                           ("v_cache", v_cache))
    _check(lib().pkv_copy_blocks(_ptr(block_pairs), n, _ptr(k_cache), _ptr(v_cache),
                                 ctypes.byref(desc), st), "pkv_copy_blocks")


def paged_kv_append(k, v, slot_mapping, k_cache, v_cache, desc, stream=None):
    """k, v: CUDA [T, Hkv, D] in the cache dtype; slot_mapping: CUDA int64 [T]."""
    T = k.shape[0]
    dt = _TORCH_DTYPE[desc.dtype]
    for t, nm in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, dt, nm)
    _need(slot_mapping, torch.int64, "slot_mapping")
    st = _stream_on_device(stream, ("k", k), ("v", v), ("slot_mapping", slot_mapping),
                           ("k_cache", k_cache), ("v_cache", v_cache))
    _check(lib().paged_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache),
                                 _ptr(v_cache), ctypes.byref(desc), st),
           "paged_kv_append")


def paged_kv_append_rope(k, v, slot_mapping, positions, cos_sin, k_cache, v_cache, desc,
                         q=None, q_out=None, stream=None):
    """Append with rotary embedding fused in: k rotated at `positions` (CUDA int32
    [T]) using `cos_sin` (CUDA fp32 [max_position, D]); v copied; q (optional,
    [T, Hq, D]) rotated into q_out (defaults to q, in place)."""
    T = k.shape[0]
    dt = _TORCH_DTYPE[desc.dtype]
    for t, nm in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, dt, nm)
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(positions, torch.int32, "positions")
    _need(cos_sin, torch.float32, "cos_sin")
    if q is not None:
        _need(q, dt, "q")
        q_out = q if q_out is None else q_out
        _need(q_out, dt, "q_out")
    st = _stream_on_device(stream, ("q", q), ("q_out", q_out), ("k", k), ("v", v),
                           ("slot_mapping", slot_mapping), ("positions", positions),
                           ("cos_sin", cos_sin), ("k_cache", k_cache), ("v_cache", v_cache))
    _check(lib().paged_kv_append_rope(_ptr(q), _ptr(q_out), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                      _ptr(positions), _ptr(cos_sin), cos_sin.shape[0], T,
                                      _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
                                      st), "paged_kv_append_rope")
    return q_out


def decode_workspace_bytes(desc, num_seqs, max_context_len):
    return int(lib().pkv_decode_workspace_bytes(ctypes.byref(desc), num_seqs, max_context_len))


def varlen_workspace_bytes(desc, num_seqs, num_query_tokens, max_query_len, max_context_len):
    return int(lib().pkv_varlen_workspace_bytes(ctypes.byref(desc), num_seqs, num_query_tokens,
                                                max_query_len, max_context_len))


def workspace(nbytes, device=None):
    """A workspace buffer (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def paged_attention_decode(out, q, k_cache, v_cache, desc, block_tables, context_lens,
                           max_context_len, scale=None, ws=None, stream=None):
    """out, q: CUDA [S, Hq, D]; block_tables int32 [S, W]; context_lens int32 [S]."""
    S = q.shape[0]
    dt = _TORCH_DTYPE[desc.dtype]
    for t, nm in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, dt, nm)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    if scale is None:
        scale = 1.0 / math.sqrt(desc.head_dim)
    st = _stream_on_device(stream, ("out", out), ("q", q), ("k_cache", k_cache),
                           ("v_cache", v_cache), ("block_tables", block_tables),
                           ("context_lens", context_lens), ("ws", ws))
    if ws is None:
        ws = workspace(decode_workspace_bytes(desc, S, max_context_len), q.device)
    _check(lib().paged_attention_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        ctypes.byref(desc), _ptr(block_tables),
                                        block_tables.shape[1], _ptr(context_lens), S,
                                        max_context_len, scale, _ptr(ws), ws.numel(),
                                        st), "paged_attention_decode")
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, desc, block_tables, context_lens,
                                   max_context_len, scale=None, stream=None):
    """paged_attention_decode without a workspace argument, for callers that cannot
    allocate device memory when they call (see include/pagedkv.h).  The library
    keeps a fixed NOALLOC_SCRATCH_BYTES scratch area per device instead; batches
    whose split partials need more raise PagedKVError(PKV_ERR_WORKSPACE).  Calls
    share that area, so calls that overlap on the GPU race: serialize them."""
    S = q.shape[0]
    dt = _TORCH_DTYPE[desc.dtype]
    for t, nm in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, dt, nm)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    if scale is None:
        scale = 1.0 / math.sqrt(desc.head_dim)
    st = _stream_on_device(stream, ("out", out), ("q", q), ("k_cache", k_cache),
                           ("v_cache", v_cache), ("block_tables", block_tables),
                           ("context_lens", context_lens))
    _check(lib().paged_attention_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                ctypes.byref(desc), _ptr(block_tables),
                                                block_tables.shape[1], _ptr(context_lens), S,
                                                max_context_len, scale, st),
           "paged_attention_decode_noalloc")
    return out


def paged_attention_varlen(out, q, k_cache, v_cache, desc, block_tables, query_start_loc,
                           context_lens, max_query_len, max_context_len, scale=None, ws=None,
                           stream=None, window=0):
    """out, q: CUDA [Tq, Hq, D]; query_start_loc int32 [S+1]; context_lens int32 [S].
    ``window`` > 0: sliding-window attention (paged_attention_varlen_window) over
    logically ordered tables (BlockPool.window_tables)."""
    Tq = q.shape[0]
    S = context_lens.shape[0]
    dt = _TORCH_DTYPE[desc.dtype]
    for t, nm in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, dt, nm)
    for t, nm in ((block_tables, "block_tables"), (query_start_loc, "query_start_loc"),
                  (context_lens, "context_lens")):
        _need(t, torch.int32, nm)
    if scale is None:
        scale = 1.0 / math.sqrt(desc.head_dim)
    st = _stream_on_device(stream, ("out", out), ("q", q), ("k_cache", k_cache),
                           ("v_cache", v_cache), ("block_tables", block_tables),
                           ("query_start_loc", query_start_loc), ("context_lens", context_lens),
                           ("ws", ws))
    if ws is None:
        ws = workspace(varlen_workspace_bytes(desc, S, Tq, max_query_len, max_context_len),
                       q.device)
    if window:
        _check(lib().paged_attention_varlen_window(
            _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
            _ptr(block_tables), block_tables.shape[1], _ptr(query_start_loc), _ptr(context_lens),
            S, Tq, max_query_len, max_context_len, int(window), scale, _ptr(ws), ws.numel(), st),
            "paged_attention_varlen_window")
        return out
    _check(lib().paged_attention_varlen(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        ctypes.byref(desc), _ptr(block_tables),
                                        block_tables.shape[1], _ptr(query_start_loc),
                                        _ptr(context_lens), S, Tq, max_query_len, max_context_len,
                                        scale, _ptr(ws), ws.numel(), st),
           "paged_attention_varlen")
    return out


def int8_tile_bytes(head_dim, block_size=16):
    """Bytes of one (block, KV head) tile of the 8-bit cache: codes, then scales."""
    return block_size * head_dim + block_size * 4


class Int8Cache:
    """The pool of an 8-bit KV cache: uint8 [NB, Hkv, 2, tile], per (block, KV
    head) a K tile and then a V tile, each holding its bs x D codes and then
    their bs fp32 scales (see paged_kv_append_int8 in include/pagedkv.h for the
    format).  k_pool / v_pool (uint8 [NB, Hkv, tile]), k_codes / v_codes (int8
    [NB, Hkv, bs, D]) and k_scales / v_scales (fp32 [NB, Hkv, bs]) are views
    into it."""

    def __init__(self, num_blocks, num_kv_heads, block_size, head_dim, num_q_heads,
                 device="cuda"):
        tile = int8_tile_bytes(head_dim, block_size)
        ncode = block_size * head_dim
        self.kv_pool = torch.zeros((num_blocks, num_kv_heads, 2, tile), dtype=torch.uint8,
                                   device=device)
        self.k_pool = self.kv_pool[:, :, 0]
        self.v_pool = self.kv_pool[:, :, 1]
        self.k_codes, self.k_scales = self._views(self.k_pool, ncode, block_size, head_dim)
        self.v_codes, self.v_scales = self._views(self.v_pool, ncode, block_size, head_dim)
        self.desc = CacheDesc(PKV_INT8, num_blocks, block_size, num_kv_heads, num_q_heads,
                              head_dim)

    @staticmethod
    def _views(pool, ncode, block_size, head_dim):
        codes = pool[:, :, :ncode].view(torch.int8).unflatten(-1, (block_size, head_dim))
        scales = pool[:, :, ncode:].view(torch.float32)
        return codes, scales

    def tensors(self):
        return (self.kv_pool,)


def _need_int8_cache(c):
    d = c.desc
    shape = (d.num_blocks, d.num_kv_heads, 2, int8_tile_bytes(d.head_dim, d.block_size))
    _need(c.kv_pool, torch.uint8, "kv_pool")
    if tuple(c.kv_pool.shape) != shape:
        raise ValueError(f"kv_pool: shape {tuple(c.kv_pool.shape)}, expected {shape}")


def paged_kv_append_int8(k, v, slot_mapping, cache, stream=None):
    """Quantise k, v (CUDA bf16 [T, Hkv, D]) into the 8-bit cache through
    slot_mapping (CUDA int64 [T])."""
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need_int8_cache(cache)
    st = _stream_on_device(stream, ("k", k), ("v", v), ("slot_mapping", slot_mapping),
                           ("kv_pool", cache.kv_pool))
    _check(lib().paged_kv_append_int8(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0],
                                      _ptr(cache.kv_pool), ctypes.byref(cache.desc), st),
           "paged_kv_append_int8")


def pkv_copy_blocks_int8(block_pairs, cache, stream=None):
    """Copy-on-write for the 8-bit cache; block_pairs: CUDA int32 [n, 2] (src, dst)."""
    n = block_pairs.shape[0] if block_pairs is not None else 0
    if n == 0:
        return
    _need(block_pairs, torch.int32, "block_pairs")
    _need_int8_cache(cache)
    st = _stream_on_device(stream, ("block_pairs", block_pairs), ("kv_pool", cache.kv_pool))
    _check(lib().pkv_copy_blocks_int8(_ptr(block_pairs), n, _ptr(cache.kv_pool),
                                      ctypes.byref(cache.desc), st), "pkv_copy_blocks_int8")


def paged_attention_decode_int8(out, q, cache, block_tables, context_lens, max_context_len,
                                scale=None, ws=None, stream=None):
    """Decode attention over the 8-bit cache; out, q: CUDA bf16 [S, Hq, D]."""
    S = q.shape[0]
    _need(out, torch.bfloat16, "out")
    _need(q, torch.bfloat16, "q")
    _need_int8_cache(cache)
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    desc = cache.desc
    if scale is None:
        scale = 1.0 / math.sqrt(desc.head_dim)
    st = _stream_on_device(stream, ("out", out), ("q", q), ("kv_pool", cache.kv_pool),
                           ("block_tables", block_tables), ("context_lens", context_lens),
                           ("ws", ws))
    if ws is None:
        ws = workspace(decode_workspace_bytes(desc, S, max_context_len), q.device)
    _check(lib().paged_attention_decode_int8(_ptr(out), _ptr(q), _ptr(cache.kv_pool),
                                             ctypes.byref(desc),
                                             _ptr(block_tables), block_tables.shape[1],
                                             _ptr(context_lens), S, max_context_len, scale,
                                             _ptr(ws), ws.numel(), st),
           "paged_attention_decode_int8")
    return out


def device_error(clear=True):
    """The device error word (0 = none); synchronizes the device."""
    code = ctypes.c_int32()
    _check(lib().pkv_device_error(ctypes.byref(code), 1 if clear else 0), "pkv_device_error")
    return code.value
