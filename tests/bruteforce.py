"""Brute-force attention on UNPAGED data, in pure Python (tests only).

Independent of ``oracle``: it never sees a block table or a cache; it works on
the dense token sequences rebuilt straight from a workload script (the values
as they were drawn, before anything was scattered into a pool), widens bf16 by
its own route (struct), and sums with math.fsum.
"""

import math
import struct


def widen_scalar(x, dtype):
    if dtype == "f32":
        return float(x)
    return struct.unpack("<f", struct.pack("<I", int(x) << 16))[0]


def dense_sequences(w):
    """seq id -> list of K/V row indices in token order, for scripts without forks."""
    rows = {}
    for op in list(w.setup) + list(w.step):
        if op[0] in ("add", "grow"):
            _, seq, n, row = op
            rows.setdefault(seq, []).extend(range(row, row + n))
        else:
            raise ValueError("brute force handles scripts without fork/free only")
    return rows


def attend(qvec, keys, vals, scale):
    scores = [scale * math.fsum(a * b for a, b in zip(qvec, k)) for k in keys]
    mx = max(scores)
    wts = [math.exp(s - mx) for s in scores]
    tot = math.fsum(wts)
    d = len(vals[0])
    return [math.fsum(wts[j] * vals[j][i] for j in range(len(keys))) / tot for i in range(d)]


def run(w, rows_by_seq=None, scale=None, window=0):
    """Return out[qrow][head] = list of D floats for every query row of the batch
    (``window`` > 0: each query sees only its ``window`` most recent tokens)."""
    rows_by_seq = rows_by_seq or dense_sequences(w)
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    g = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = []
    r = 0
    for seq, qlen in w.batch:
        toks = rows_by_seq[seq]
        ctx = len(toks)
        for i in range(qlen):
            last = ctx - qlen + i
            visible = toks[max(0, last - window + 1) if window else 0:last + 1]
            heads = []
            for h in range(hq):
                kv = h // g
                qv = [widen_scalar(x, w.dtype) for x in w.q[r, h]]
                ks = [[widen_scalar(x, w.dtype) for x in w.k_rows[t, kv]] for t in visible]
                vs = [[widen_scalar(x, w.dtype) for x in w.v_rows[t, kv]] for t in visible]
                heads.append(attend(qv, ks, vs, scale))
            out.append(heads)
            r += 1
    return out


def window_trace_step(tr, step_index, lens_after):
    """Dense windowed attention of one step of a sliding-window trace, straight
    from the trace's unpaged rows: query i of (seq, qlen) sits at position
    lens_after[seq] - qlen + i and sees positions max(0, pos - window + 1) .. pos."""
    hq, hkv, d = tr.num_q_heads, tr.num_kv_heads, tr.head_dim
    g = hq // hkv
    scale = 1.0 / math.sqrt(d)
    out = []
    r = tr.q_offset[step_index]
    for seq, qlen in tr.steps[step_index]:
        n = lens_after[seq]
        for i in range(qlen):
            pos = n - qlen + i
            first = max(0, pos - tr.window + 1)
            rows = [tr.row_offset[seq] + t for t in range(first, pos + 1)]
            heads = []
            for h in range(hq):
                kv = h // g
                qv = [widen_scalar(x, tr.dtype) for x in tr.q_rows[r, h]]
                ks = [[widen_scalar(x, tr.dtype) for x in tr.k_rows[t, kv]] for t in rows]
                vs = [[widen_scalar(x, tr.dtype) for x in tr.v_rows[t, kv]] for t in rows]
                heads.append(attend(qv, ks, vs, scale))
            out.append(heads)
            r += 1
    return out
