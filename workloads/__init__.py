"""Seeded synthetic inputs for paged-KV attention (shared by the oracle side and the CUDA side).

This module only draws random numbers and lays out a script of block-pool
operations; it holds none of the method's arithmetic (no slot computation, no
attention, no copy-on-write logic).  Each side executes the script with its
own pool and cache code.

A workload is:
  * shapes: dtype ('f32' or 'bf16'), Hq, Hkv, head_dim D, block_size
  * a pool: ``num_blocks`` and ``free_order`` (a seeded permutation; the first
    entry is handed out first)
  * ``setup``: operations run before the measured step
        ("add",  seq, n, row)   new sequence whose n tokens take K/V rows row..row+n-1
        ("grow", seq, n, row)   append n tokens one at a time (rows row..row+n-1)
        ("fork", parent, child) share all of parent's blocks
        ("free", seq)
  * ``step``: the same kinds of operation for this step's new tokens (their K/V
    are appended before attention)
  * ``batch``: [(seq, qlen)] in query-row order; qlen = 1 is a decode row, a
    larger qlen is a prefill chunk (the sequence's last qlen tokens)
  * ``q`` [Tq, Hq, D] and the token value rows ``k_rows``/``v_rows`` [N, Hkv, D]
    in the storage dtype (float32, or bf16 bit patterns as uint16).

Context lengths quoted for a configuration are the attended lengths: they count
the step's own token(s), which are appended first.
"""

from dataclasses import dataclass, field

import numpy as np

CONFIG_NAMES = {
    1: "tiny-decode-f32",
    2: "llama2-7b-decode",
    3: "llama3-8b-gqa-decode",
    4: "splitfuse-2048",
    5: "prefix-sharing-longctx",
}


@dataclass
class Workload:
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    free_order: np.ndarray
    setup: list
    step: list
    batch: list
    q: np.ndarray
    k_rows: np.ndarray
    v_rows: np.ndarray
    notes: dict = field(default_factory=dict)

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2

    @property
    def num_tokens_q(self):
        return sum(q for _, q in self.batch)


def _bf16_bits(x32):
    """Round float32 to bf16 (round-to-nearest-even) with torch; return uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _values(rng, shape, dtype, scale):
    """Normal(0, 1) * scale in the storage dtype, drawn in bounded chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32 if dtype == "f32" else np.uint16)
    chunk = 1 << 24
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        x = rng.standard_normal(b - a, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[a:b] = x if dtype == "f32" else _bf16_bits(x)
    return out.reshape(shape)


def _blocks(n, bs):
    return -(-n // bs)


def _decode_workload(name, rng, dtype, hq, hkv, d, bs, ctx, scale, pool=None, slack=0.1,
                     q_scale=None, values=True):
    """One query token per sequence; sequence s holds ctx[s]-1 cached tokens before the step.
    Queries are drawn at ``q_scale`` (default: ``scale``).  ``values=False``
    leaves the value rows to the caller (see ``_no_values``)."""
    ctx = [int(c) for c in ctx]
    need = sum(_blocks(c, bs) for c in ctx)
    nb = pool if pool is not None else int(np.ceil(need * (1.0 + slack)))
    free_order = rng.permutation(nb).astype(np.int32)
    setup, step, row = [], [], 0
    for s, c in enumerate(ctx):
        if c - 1 > 0:
            setup.append(("add", s, c - 1, row))
            row += c - 1
    for s, c in enumerate(ctx):
        if c - 1 > 0:
            step.append(("grow", s, 1, row))
        else:
            step.append(("add", s, 1, row))
        row += 1
    batch = [(s, 1) for s in range(len(ctx))]
    notes = {"context_lens": ctx}
    if not values:
        return _no_values(Workload(name, dtype, hq, hkv, d, bs, nb, free_order, setup, step,
                                   batch, None, None, None, notes=notes), row, scale)
    k_rows = _values(rng, (row, hkv, d), dtype, scale)
    v_rows = _values(rng, (row, hkv, d), dtype, scale)
    q = _values(rng, (len(ctx), hq, d), dtype, scale if q_scale is None else q_scale)
    return Workload(name, dtype, hq, hkv, d, bs, nb, free_order, setup, step, batch, q,
                    k_rows, v_rows, notes=notes)


def _no_values(w, n_rows, scale):
    """A workload whose structure (lengths, pool, operations, batch) is drawn but
    whose value rows are not: ``k_rows``, ``v_rows`` and ``q`` are None and the
    notes give the row count and the value scale, for a consumer that draws
    values of the same distribution itself (timing runs, whose speed does not
    depend on the values)."""
    w.notes["value_rows"] = int(n_rows)
    w.notes["value_scale"] = float(scale)
    return w


def config1(seed=0):
    """Tiny decode: fp32, 4 seqs, 8/8 heads, D=64, bs=16, ctx {17,64,131,200}, pool of 64."""
    rng = np.random.default_rng(seed)
    return _decode_workload(CONFIG_NAMES[1], rng, "f32", 8, 8, 64, 16, [17, 64, 131, 200],
                            1.0, pool=64)


def config2(seed=0, batch=64):
    """Llama-2-7B-shaped decode: bf16, 32/32 heads, D=128, bs=16, ctx ~ U[512, 4096]."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(512, 4096, size=batch, endpoint=True)
    return _decode_workload(CONFIG_NAMES[2], rng, "bf16", 32, 32, 128, 16, ctx, 0.5)


def config3(seed=0, batch=256, values=True):
    """Llama-3-8B-shaped GQA decode: bf16, 32/8 heads, ctx log-uniform in [1024, 8192]."""
    rng = np.random.default_rng(seed)
    ctx = np.rint(np.exp(rng.uniform(np.log(1024), np.log(8192), size=batch))).astype(int)
    return _decode_workload(CONFIG_NAMES[3], rng, "bf16", 32, 8, 128, 16, ctx, 0.5,
                            values=values)


def config4(seed=0, n_decode=512, chunk=512, prefixes=(0, 1024, 3072)):
    """SplitFuse mixed batch: 3 prefill chunks of 512 over cached prefixes 0/1024/3072
    plus 512 decode sequences with ctx ~ U[256, 4096]; 2048 query tokens in all."""
    rng = np.random.default_rng(seed)
    hq, hkv, d, bs = 32, 8, 128, 16
    dec_ctx = [int(c) for c in rng.integers(256, 4096, size=n_decode, endpoint=True)]
    chunk_ctx = [p + chunk for p in prefixes]
    need = sum(_blocks(c, bs) for c in chunk_ctx + dec_ctx)
    nb = int(np.ceil(need * 1.1))
    free_order = rng.permutation(nb).astype(np.int32)
    setup, step, row = [], [], 0
    n_chunk = len(prefixes)
    for s, p in enumerate(prefixes):
        if p > 0:
            setup.append(("add", s, p, row))
            row += p
    for i, c in enumerate(dec_ctx):
        setup.append(("add", n_chunk + i, c - 1, row))
        row += c - 1
    for s, p in enumerate(prefixes):
        step.append(("grow", s, chunk, row) if p > 0 else ("add", s, chunk, row))
        row += chunk
    for i in range(n_decode):
        step.append(("grow", n_chunk + i, 1, row))
        row += 1
    k_rows = _values(rng, (row, hkv, d), "bf16", 0.5)
    v_rows = _values(rng, (row, hkv, d), "bf16", 0.5)
    batch = [(s, chunk) for s in range(n_chunk)] + [(n_chunk + i, 1) for i in range(n_decode)]
    q = _values(rng, (sum(x for _, x in batch), hq, d), "bf16", 0.5)
    return Workload(CONFIG_NAMES[4], "bf16", hq, hkv, d, bs, nb, free_order, setup, step, batch,
                    q, k_rows, v_rows,
                    notes={"context_lens": chunk_ctx + dec_ctx, "prefixes": list(prefixes)})


def config5(seed=0, groups=8, branches=8, prompt=3000, max_private=200, n_long=4,
            long_ctx=32768, values=True):
    """Parallel sampling + long context: bf16, 64/8 heads.  Each group's prompt is
    forked into ``branches`` branches that share its blocks; the prompt sequence is
    then freed; each branch generates U{1..max_private} private tokens, the last of
    which is this step's token.  Plus ``n_long`` sequences at ``long_ctx``."""
    rng = np.random.default_rng(seed)
    hq, hkv, d, bs = 64, 8, 128, 16
    priv = rng.integers(1, max_private, size=(groups, branches), endpoint=True)
    # pool: prompts + every branch's private blocks + one copy per branch + long seqs
    need = groups * _blocks(prompt, bs)
    need += sum(_blocks(int(p) + bs, bs) + 1 for p in priv.ravel())
    need += n_long * _blocks(long_ctx, bs)
    nb = int(np.ceil(need * 1.1))
    free_order = rng.permutation(nb).astype(np.int32)
    setup, step, batch, row = [], [], [], 0
    ctx = []
    sid = 0
    branch_ids = []
    for gi in range(groups):
        parent = sid
        sid += 1
        setup.append(("add", parent, prompt, row))
        row += prompt
        kids = []
        for _ in range(branches):
            setup.append(("fork", parent, sid))
            kids.append(sid)
            sid += 1
        setup.append(("free", parent))
        for bi, kid in enumerate(kids):
            n = int(priv[gi, bi])
            if n > 1:
                setup.append(("grow", kid, n - 1, row))
                row += n - 1
            branch_ids.append((kid, n))
    for kid, n in branch_ids:
        step.append(("grow", kid, 1, row))
        row += 1
        batch.append((kid, 1))
        ctx.append(prompt + n)
    for _ in range(n_long):
        setup.append(("add", sid, long_ctx - 1, row))
        row += long_ctx - 1
        step.append(("grow", sid, 1, row))
        row += 1
        batch.append((sid, 1))
        ctx.append(long_ctx)
        sid += 1
    if not values:
        return _no_values(Workload(CONFIG_NAMES[5], "bf16", hq, hkv, d, bs, nb, free_order,
                                   setup, step, batch, None, None, None,
                                   notes={"context_lens": ctx}), row, 0.5)
    k_rows = _values(rng, (row, hkv, d), "bf16", 0.5)
    v_rows = _values(rng, (row, hkv, d), "bf16", 0.5)
    q = _values(rng, (len(batch), hq, d), "bf16", 0.5)
    return Workload(CONFIG_NAMES[5], "bf16", hq, hkv, d, bs, nb, free_order, setup, step, batch,
                    q, k_rows, v_rows, notes={"context_lens": ctx})


def make(config, seed=0, **kw):
    return {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}[config](seed=seed, **kw)


def random_decode(seed, dtype, hq, hkv, d, bs, ctx, scale=1.0, pool=None, slack=0.1,
                  q_scale=None):
    """A decode workload with explicit context lengths (for edge-case tests);
    ``q_scale`` draws the queries at another scale than the keys and values."""
    rng = np.random.default_rng(seed)
    return _decode_workload(f"decode-{dtype}-{hq}x{hkv}x{d}", rng, dtype, hq, hkv, d, bs, ctx,
                            scale, pool=pool, slack=slack, q_scale=q_scale)


def random_varlen(seed, dtype, hq, hkv, d, bs, spans, scale=1.0, slack=0.1, q_scale=None):
    """A mixed batch from explicit (cached_prefix, qlen) spans (for edge-case tests);
    ``q_scale`` draws the queries at another scale than the keys and values."""
    rng = np.random.default_rng(seed)
    need = sum(_blocks(p + q, bs) for p, q in spans)
    nb = int(np.ceil(need * (1.0 + slack))) + 1
    free_order = rng.permutation(nb).astype(np.int32)
    setup, step, row = [], [], 0
    for s, (p, _) in enumerate(spans):
        if p > 0:
            setup.append(("add", s, p, row))
            row += p
    for s, (p, qn) in enumerate(spans):
        step.append(("grow", s, qn, row) if p > 0 else ("add", s, qn, row))
        row += qn
    k_rows = _values(rng, (row, hkv, d), dtype, scale)
    v_rows = _values(rng, (row, hkv, d), dtype, scale)
    batch = [(s, qn) for s, (_, qn) in enumerate(spans)]
    q = _values(rng, (sum(qn for _, qn in spans), hq, d), dtype,
                scale if q_scale is None else q_scale)
    return Workload(f"varlen-{dtype}", dtype, hq, hkv, d, bs, nb, free_order, setup, step, batch,
                    q, k_rows, v_rows,
                    notes={"context_lens": [p + qn for p, qn in spans]})


def append_inputs(seed, dtype, num_tokens, hq, hkv, d, num_slots, max_pos, pad_every=0,
                  scale=1.0):
    """Inputs of one (rotary) append, for edge-case tests of the append kernels.

    q [T, hq, d] (None when hq is 0), k, v [T, hkv, d] in the storage dtype;
    slots: T distinct slots drawn from [0, num_slots), every pad_every-th token
    padding (-1) when pad_every > 0; positions drawn from [0, max_pos)."""
    rng = np.random.default_rng(seed)
    q = _values(rng, (num_tokens, hq, d), dtype, scale) if hq > 0 else None
    k = _values(rng, (num_tokens, hkv, d), dtype, scale)
    v = _values(rng, (num_tokens, hkv, d), dtype, scale)
    slots = rng.permutation(num_slots)[:num_tokens].astype(np.int64)
    if pad_every > 0:
        slots[::pad_every] = -1
    positions = rng.integers(0, max_pos, size=num_tokens).astype(np.int32)
    return q, k, v, slots, positions


@dataclass
class ServingTrace:
    """Requests for a multi-step run: prompt length, tokens to generate, the step at
    which each arrives, and value rows indexed by (request, position)."""
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    free_order: np.ndarray
    prompt_len: list
    gen_len: list
    arrival: list
    row_offset: list
    k_rows: np.ndarray
    v_rows: np.ndarray
    q_rows: np.ndarray


def serving_trace(seed=0, n_requests=6, prompt_range=(20, 700), gen_range=(1, 6), arrive_every=1,
                  hq=32, hkv=8, d=128, bs=16, scale=0.5):
    """A seeded stream of requests (values N(0,1) * scale, bf16)."""
    rng = np.random.default_rng(seed)
    prompt = [int(x) for x in rng.integers(prompt_range[0], prompt_range[1], size=n_requests,
                                           endpoint=True)]
    gen = [int(x) for x in rng.integers(gen_range[0], gen_range[1], size=n_requests,
                                        endpoint=True)]
    arrival = [i * arrive_every for i in range(n_requests)]
    offs, row = [], 0
    for p, g in zip(prompt, gen):
        offs.append(row)
        row += p + g
    need = sum(_blocks(p + g, bs) for p, g in zip(prompt, gen))
    nb = int(np.ceil(need * 1.1)) + 2
    free_order = rng.permutation(nb).astype(np.int32)
    k_rows = _values(rng, (row, hkv, d), "bf16", scale)
    v_rows = _values(rng, (row, hkv, d), "bf16", scale)
    q_rows = _values(rng, (row, hq, d), "bf16", scale)
    return ServingTrace("bf16", hq, hkv, d, bs, nb, free_order, prompt, gen, arrival, offs,
                        k_rows, v_rows, q_rows)


@dataclass
class WindowTrace:
    """A multi-step run of sequences under a sliding window.

    ``steps[i]`` lists (seq, qlen) in query-row order: a sequence's first
    entry adds its first prompt chunk, later entries append qlen tokens (the
    rest of the prompt in chunks of at most ``max_chunk``, then one token per
    decode step), and every entry's qlen new tokens are that step's queries.
    Token p of sequence s has K/V rows ``row_offset[s] + p``; step i's query
    rows are ``q_rows[q_offset[i]:q_offset[i + 1]]``."""
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    window: int
    max_chunk: int
    num_blocks: int
    free_order: np.ndarray
    steps: list
    row_offset: list
    q_offset: list
    k_rows: np.ndarray
    v_rows: np.ndarray
    q_rows: np.ndarray


def window_trace(seed=0, dtype="bf16", hq=32, hkv=8, d=128, bs=16, window=256, max_chunk=200,
                 prompts=(700, 130, 1000), gens=(3, 40, 2), scale=0.5):
    """A seeded windowed run: every step, each unfinished prompt takes a chunk of
    U{1..max_chunk} tokens (at most what is left) and each finished one decodes
    one token, until every sequence has its prompt and generated tokens."""
    rng = np.random.default_rng(seed)
    lengths = [p + g for p, g in zip(prompts, gens)]
    done = [0] * len(prompts)
    steps = []
    while any(n < L for n, L in zip(done, lengths)):
        step = []
        for s, (p, L) in enumerate(zip(prompts, lengths)):
            if done[s] >= L:
                continue
            if done[s] < p:
                c = min(int(rng.integers(1, max_chunk, endpoint=True)), p - done[s])
            else:
                c = 1
            step.append((s, c))
            done[s] += c
        steps.append(step)
    ring = window // bs + _blocks(max_chunk - 1, bs)
    nb = len(prompts) * ring + 4
    free_order = rng.permutation(nb).astype(np.int32)
    offs = [int(x) for x in np.concatenate([[0], np.cumsum(lengths)[:-1]])]
    q_off = [int(x) for x in np.concatenate([[0], np.cumsum([sum(q for _, q in st)
                                                              for st in steps])])]
    k_rows = _values(rng, (sum(lengths), hkv, d), dtype, scale)
    v_rows = _values(rng, (sum(lengths), hkv, d), dtype, scale)
    q_rows = _values(rng, (q_off[-1], hq, d), dtype, scale)
    return WindowTrace(dtype, hq, hkv, d, bs, window, max_chunk, nb, free_order, steps, offs,
                       q_off, k_rows, v_rows, q_rows)


class TokenValues:
    """K/V rows that depend only on (token id, position), as a model's K/V depend
    on the token prefix: row(t, p) = bf16(E[t] + P[p]) with E, P seeded normal
    tables.  Sequences that share a token prefix get bit-identical rows there,
    which is what lets cached blocks be shared."""

    def __init__(self, seed, vocab, max_pos, hkv, d, scale=0.5):
        rng = np.random.default_rng(seed)
        self.ek = rng.standard_normal((vocab, hkv, d), dtype=np.float32) * np.float32(scale)
        self.ev = rng.standard_normal((vocab, hkv, d), dtype=np.float32) * np.float32(scale)
        self.pk = rng.standard_normal((max_pos, hkv, d), dtype=np.float32) * np.float32(scale)
        self.pv = rng.standard_normal((max_pos, hkv, d), dtype=np.float32) * np.float32(scale)

    def rows(self, token_ids, positions):
        """(k, v) bf16 bit patterns [len, hkv, d] for the given tokens at the given positions."""
        t = np.asarray(token_ids, dtype=np.int64)
        p = np.asarray(positions, dtype=np.int64)
        return _bf16_bits(self.ek[t] + self.pk[p]), _bf16_bits(self.ev[t] + self.pv[p])
