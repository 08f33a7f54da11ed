"""Drive a batch through the library: host block pool -> copy-on-write -> append -> attention.

``DeviceCache`` owns one layer's K and V pools on the GPU and a host
``BlockPool``.  Pool operations are planned on the host; the device work they
imply (copy-on-write block copies, then K/V appends) is queued and issued in
batches: all copies of a batch before all of its appends.  That order equals
applying the operations one token at a time because, between two flushes, a
block that is copied from is shared and therefore not written in place, and a
copy destination is fresh.  A fork or a free makes blocks shared or reusable,
so pending work is flushed before either.

Operations use the tuple format of the ``workloads`` package:
("add", seq, n, row), ("grow", seq, n, row), ("fork", parent, child), ("free", seq).
"""

import math

import numpy as np
import torch

from . import (BlockPool, cache_desc, paged_attention_decode, paged_attention_varlen,
               paged_kv_append, pkv_copy_blocks, varlen_workspace_bytes, decode_workspace_bytes,
               workspace)


def _torch_rows(rows, dtype):
    """Host value rows (float32, or uint16 bf16 bits) -> torch tensor of the cache dtype."""
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(rows))
    return torch.from_numpy(np.ascontiguousarray(rows).view(np.int16)).view(torch.bfloat16)


class DeviceCache:
    def __init__(self, w, device="cuda", value_seed=0):
        """A workload without value rows (``k_rows`` None) gets its K/V rows and
        queries drawn on the device: N(0,1) times the workload's value scale,
        rounded to the cache dtype, from a torch generator seeded with
        ``value_seed``.  Timing runs use this; parity runs use the host rows."""
        self.w = w
        self.device = torch.device(device)
        tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        self.k_cache = torch.zeros(shape, dtype=tdt, device=self.device)
        self.v_cache = torch.zeros(shape, dtype=tdt, device=self.device)
        self.desc = cache_desc(self.k_cache, w.num_q_heads)
        self.pool = BlockPool(w.num_blocks, w.block_size, 0, w.free_order)
        self._slots, self._rows, self._pairs = [], [], []
        self.step_slots, self.step_rows, self.step_pairs = [], [], []
        self._dev_rows = None
        if w.k_rows is None:
            g = torch.Generator(device=self.device)
            g.manual_seed(value_seed)
            sc = w.notes["value_scale"]
            n = w.notes["value_rows"]

            def draw(shape_):
                x = torch.randn(shape_, generator=g, device=self.device, dtype=torch.float32)
                return (x * sc).to(tdt)

            self._dev_rows = (draw((n, w.num_kv_heads, w.head_dim)),
                              draw((n, w.num_kv_heads, w.head_dim)),
                              draw((sum(q for _, q in w.batch), w.num_q_heads, w.head_dim)))

    def _value_rows(self, rows):
        """K and V rows (indices into the workload's value rows) in the cache dtype."""
        w = self.w
        if self._dev_rows is not None:
            idx = torch.as_tensor(np.asarray(rows, dtype=np.int64)).to(self.device)
            return self._dev_rows[0][idx], self._dev_rows[1][idx]
        r = np.asarray(rows)
        return _torch_rows(w.k_rows[r], w.dtype), _torch_rows(w.v_rows[r], w.dtype)

    # ---- planning -------------------------------------------------------
    def _apply(self, op, record):
        kind = op[0]
        if kind == "add":
            _, seq, n, row = op
            slots = self.pool.add(seq, n)
            self._slots += slots
            self._rows += range(row, row + n)
            if record:
                self.step_slots += slots
                self.step_rows += range(row, row + n)
        elif kind == "grow":
            _, seq, n, row = op
            for i in range(n):
                slot, cow = self.pool.append_slot(seq)
                if cow is not None:
                    self._pairs.append(cow)
                    if record:
                        self.step_pairs.append(cow)
                self._slots.append(slot)
                self._rows.append(row + i)
                if record:
                    self.step_slots.append(slot)
                    self.step_rows.append(row + i)
        elif kind == "fork":
            self.flush()
            self.pool.fork(op[1], op[2])
        elif kind == "free":
            self.flush()
            self.pool.free(op[1])
        else:
            raise ValueError(f"unknown operation {kind!r}")

    # ---- device work ----------------------------------------------------
    def flush(self, chunk_tokens=1 << 16):
        if self._pairs:
            pairs = torch.tensor(self._pairs, dtype=torch.int32).to(self.device)
            pkv_copy_blocks(pairs, self.k_cache, self.v_cache, self.desc)
        self._pairs = []
        slots, rows = self._slots, self._rows
        for a in range(0, len(slots), chunk_tokens):
            s = torch.tensor(slots[a:a + chunk_tokens], dtype=torch.int64).to(self.device)
            k, v = self._value_rows(rows[a:a + chunk_tokens])
            paged_kv_append(k.to(self.device), v.to(self.device), s, self.k_cache, self.v_cache,
                            self.desc)
        self._slots, self._rows = [], []

    def run_setup(self):
        for op in self.w.setup:
            self._apply(op, record=False)
        self.flush()

    def plan_step(self, ops=None):
        """Plan the step's pool operations (the workload's own step, or `ops`); returns
        the step's device inputs (not yet applied to the cache)."""
        self.step_slots, self.step_rows, self.step_pairs = [], [], []
        for op in (self.w.step if ops is None else ops):
            self._apply(op, record=True)
        # the step's copies and appends stay queued: hand them to the caller
        self._slots, self._rows, self._pairs = [], [], []
        k, v = self._value_rows(self.step_rows)
        return {
            "slot_mapping": torch.tensor(self.step_slots, dtype=torch.int64),
            "k": k,
            "v": v,
            "pairs": torch.tensor(self.step_pairs, dtype=torch.int32).reshape(-1, 2),
        }

    def batch_metadata(self, batch=None):
        """Block tables [S, W] (padded -1), context lengths [S], query_start_loc [S+1] (host)."""
        w = self.w
        batch = w.batch if batch is None else batch
        seqs = [s for s, _ in batch]
        width = max(math.ceil(self.pool.seq_len(s) / w.block_size) for s in seqs)
        tables, ctx = self.pool.block_tables(seqs, width)
        qsl = torch.zeros(len(seqs) + 1, dtype=torch.int32)
        qsl[1:] = torch.cumsum(torch.tensor([q for _, q in batch], dtype=torch.int32), 0)
        return tables, ctx, qsl

    def q_tensor(self):
        if self._dev_rows is not None:
            return self._dev_rows[2]
        return _torch_rows(self.w.q, self.w.dtype)


class Step:
    """Device-resident inputs of one step and the calls that run it."""

    def __init__(self, dc, planned, batch=None, q=None):
        """`batch` ([(seq, qlen)]) and `q` (host rows [Tq, Hq, D]) default to the workload's."""
        w = dc.w
        batch = w.batch if batch is None else batch
        dev = dc.device
        self.dc = dc
        self.slot_mapping = planned["slot_mapping"].to(dev)
        self.k_new = planned["k"].to(dev)
        self.v_new = planned["v"].to(dev)
        self.pairs = planned["pairs"].to(dev)
        tables, ctx, qsl = dc.batch_metadata(batch)
        self.tables = tables.to(dev)
        self.ctx = ctx.to(dev)
        self.qsl = qsl.to(dev)
        self.max_ctx = int(ctx.max())
        self.max_qlen = max(q for _, q in batch)
        self.decode_only = self.max_qlen == 1
        self.q = (dc.q_tensor() if q is None else _torch_rows(q, w.dtype)).to(dev)
        self.out = torch.empty_like(self.q)
        S = len(batch)
        if self.decode_only:
            nbytes = decode_workspace_bytes(dc.desc, S, self.max_ctx)
        else:
            nbytes = varlen_workspace_bytes(dc.desc, S, self.q.shape[0], self.max_qlen,
                                            self.max_ctx)
        self.ws = workspace(nbytes, dev)

    def write_kv(self, stream=None):
        dc = self.dc
        pkv_copy_blocks(self.pairs, dc.k_cache, dc.v_cache, dc.desc, stream)
        paged_kv_append(self.k_new, self.v_new, self.slot_mapping, dc.k_cache, dc.v_cache, dc.desc,
                        stream)

    def attend(self, stream=None):
        dc = self.dc
        if self.decode_only:
            return paged_attention_decode(self.out, self.q, dc.k_cache, dc.v_cache, dc.desc,
                                          self.tables, self.ctx, self.max_ctx, ws=self.ws,
                                          stream=stream)
        return paged_attention_varlen(self.out, self.q, dc.k_cache, dc.v_cache, dc.desc,
                                      self.tables, self.qsl, self.ctx, self.max_qlen, self.max_ctx,
                                      ws=self.ws, stream=stream)

    def run(self, stream=None):
        self.write_kv(stream)
        return self.attend(stream)


def prepare(w, device="cuda"):
    """Set up a workload on the device; returns (DeviceCache, Step) ready to run."""
    dc = DeviceCache(w, device)
    dc.run_setup()
    step = Step(dc, dc.plan_step())
    return dc, step


def run_window_trace(tr, device="cuda"):
    """Run a sliding-window trace (``workloads.WindowTrace``) through the library:
    the C++ window pool with room for ``max_chunk`` queries, copy-on-write and
    append of each step's tokens, then one windowed varlen call over the step's
    prompt chunks and decode rows with the pool's logically ordered tables.
    Returns (list of per-step outputs on the device, K cache, V cache)."""
    dev = torch.device(device)
    tdt = torch.float32 if tr.dtype == "f32" else torch.bfloat16
    shape = (tr.num_blocks, tr.num_kv_heads, tr.block_size, tr.head_dim)
    kc = torch.zeros(shape, dtype=tdt, device=dev)
    vc = torch.zeros_like(kc)
    desc = cache_desc(kc, tr.num_q_heads)
    pool = BlockPool(tr.num_blocks, tr.block_size, 0, tr.free_order,
                     sliding_window=tr.window, max_chunk=tr.max_chunk)
    lens, outs = {}, []
    for i, step in enumerate(tr.steps):
        slots, rows, pairs = [], [], []
        for seq, qlen in step:
            n = lens.get(seq, 0)
            if n == 0:
                slots += pool.add(seq, qlen)
            else:
                for _ in range(qlen):
                    slot, cow = pool.append_slot(seq)
                    if cow is not None:
                        pairs.append(cow)
                    slots.append(slot)
            rows += range(tr.row_offset[seq] + n, tr.row_offset[seq] + n + qlen)
            lens[seq] = n + qlen
        if pairs:
            pkv_copy_blocks(torch.tensor(pairs, dtype=torch.int32).to(dev), kc, vc, desc)
        r = np.asarray(rows)
        paged_kv_append(_torch_rows(tr.k_rows[r], tr.dtype).to(dev),
                        _torch_rows(tr.v_rows[r], tr.dtype).to(dev),
                        torch.tensor(slots, dtype=torch.int64).to(dev), kc, vc, desc)
        seqs = [seq for seq, _ in step]
        qlens = [q for _, q in step]
        width = max(math.ceil(lens[s] / tr.block_size) for s in seqs) + 1
        tables, ctx = pool.window_tables(seqs, qlens, width)
        qsl = torch.zeros(len(step) + 1, dtype=torch.int32)
        qsl[1:] = torch.cumsum(torch.tensor(qlens, dtype=torch.int32), 0)
        q = _torch_rows(tr.q_rows[tr.q_offset[i]:tr.q_offset[i + 1]], tr.dtype).to(dev)
        out = torch.empty_like(q)
        paged_attention_varlen(out, q, kc, vc, desc, tables.to(dev), qsl.to(dev), ctx.to(dev),
                               max(qlens), int(ctx.max()), window=tr.window)
        outs.append(out)
    return outs, kc, vc
