"""Execute a workload script with the oracle's own pool, cache mirror and attention.

Test infrastructure only.  A workload (see the ``workloads`` package, which
this module does not import) supplies shapes, a pool, ``setup``/``step``
operation lists, the query batch and the token value rows.  Each operation is
applied in order, one token at a time, exactly as the pages describe the block
manager and cache engine; copy-on-write copies happen before the token that
needed them is written.
"""

import numpy as np

from . import attention, cache
from .block_pool import OK, BlockPoolModel


class OracleState:
    def __init__(self, w):
        self.w = w
        self.pool = BlockPoolModel(w.num_blocks, w.block_size, 0, w.free_order)
        dt = np.float32 if w.dtype == "f32" else np.uint16
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        self.k_cache = np.zeros(shape, dtype=dt)
        self.v_cache = np.zeros(shape, dtype=dt)
        self.step_slots = []
        self.step_cow = []
        self.step_rows = []

    def _apply(self, op, record):
        w, pool = self.w, self.pool
        kind = op[0]
        if kind == "add":
            _, seq, n, row = op
            st, slots = pool.add_sequence(seq, n)
            if st != OK:
                raise RuntimeError(f"pool refused a sequence of {n} tokens: {st}")
            cache.append(self.k_cache, self.v_cache, w.k_rows[row:row + n], w.v_rows[row:row + n],
                         slots, w.block_size)
            if record:
                self.step_slots += slots
                self.step_rows += list(range(row, row + n))
        elif kind == "grow":
            _, seq, n, row = op
            for i in range(n):
                slot, cow = pool.append_slot(seq)
                if slot is None:
                    raise RuntimeError("pool exhausted")
                if cow is not None:
                    cache.copy_blocks(self.k_cache, self.v_cache, [cow])
                    if record:
                        self.step_cow.append(cow)
                cache.append(self.k_cache, self.v_cache, w.k_rows[row + i:row + i + 1],
                             w.v_rows[row + i:row + i + 1], [slot], w.block_size)
                if record:
                    self.step_slots.append(slot)
                    self.step_rows.append(row + i)
        elif kind == "fork":
            pool.fork(op[1], op[2])
        elif kind == "free":
            pool.free_sequence(op[1])
        else:
            raise ValueError(f"unknown operation {kind!r}")

    def run_setup(self):
        for op in self.w.setup:
            self._apply(op, record=False)

    def run_step(self):
        for op in self.w.step:
            self._apply(op, record=True)

    def batch_metadata(self, width=None):
        """Block tables [S, W] (padded with -1), context lengths [S], query_start_loc [S+1]."""
        seqs = [s for s, _ in self.w.batch]
        tables = [self.pool.block_table(s) for s in seqs]
        W = width if width is not None else max(len(t) for t in tables)
        bt = np.full((len(seqs), W), -1, dtype=np.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = t
        ctx = np.array([self.pool.context_len(s) for s in seqs], dtype=np.int32)
        qsl = np.zeros(len(seqs) + 1, dtype=np.int32)
        qsl[1:] = np.cumsum([q for _, q in self.w.batch])
        return bt, ctx, qsl

    def attention(self, scale=None):
        bt, ctx, qsl = self.batch_metadata()
        w = self.w
        if all(q == 1 for _, q in w.batch):
            return attention.decode(w.q, self.k_cache, self.v_cache, bt, ctx, w.block_size,
                                    w.dtype, scale)
        return attention.varlen(w.q, self.k_cache, self.v_cache, bt, qsl, ctx, w.block_size,
                                w.dtype, scale)


def execute(w, with_attention=True, scale=None):
    st = OracleState(w)
    st.run_setup()
    st.run_step()
    out = st.attention(scale) if with_attention else None
    return st, out


def execute_window_trace(tr):
    """Run a sliding-window trace (``workloads.WindowTrace``) with the oracle's
    window pool (ring with room for ``max_chunk`` queries), cache mirror and
    windowed attention.  Returns (per-step float64 outputs [Tq, Hq, D], final
    K cache, final V cache)."""
    from .prefix_cache import SlidingWindowPool

    pool = SlidingWindowPool(tr.num_blocks, tr.block_size, tr.window, 0, tr.free_order,
                             tr.max_chunk)
    dt = np.float32 if tr.dtype == "f32" else np.uint16
    shape = (tr.num_blocks, tr.num_kv_heads, tr.block_size, tr.head_dim)
    kc, vc = np.zeros(shape, dtype=dt), np.zeros(shape, dtype=dt)
    lens, outs = {}, []
    for i, step in enumerate(tr.steps):
        for seq, qlen in step:
            n = lens.get(seq, 0)
            rows = tr.row_offset[seq] + np.arange(n, n + qlen)
            if n == 0:
                st, slots = pool.add_sequence(seq, qlen)
                if st != OK:
                    raise RuntimeError(f"window pool refused a chunk: {st}")
            else:
                slots = []
                for _ in range(qlen):
                    slot, cow = pool.append_slot(seq)
                    if slot is None:
                        raise RuntimeError("window pool exhausted")
                    if cow is not None:
                        cache.copy_blocks(kc, vc, [cow])
                    slots.append(slot)
            cache.append(kc, vc, tr.k_rows[rows], tr.v_rows[rows], slots, tr.block_size)
            lens[seq] = n + qlen
        tabs = [pool.logical_table(seq, qlen) for seq, qlen in step]
        width = max(len(t) for t, _ in tabs)
        bt = np.full((len(step), width), -1, dtype=np.int32)
        for j, (t, _) in enumerate(tabs):
            bt[j, :len(t)] = t
        ctx = np.array([c for _, c in tabs], dtype=np.int32)
        qsl = np.zeros(len(step) + 1, dtype=np.int32)
        qsl[1:] = np.cumsum([q for _, q in step])
        q = tr.q_rows[tr.q_offset[i]:tr.q_offset[i + 1]]
        outs.append(attention.varlen(q, kc, vc, bt, qsl, ctx, tr.block_size, tr.dtype,
                                     window=tr.window))
    return outs, kc, vc
