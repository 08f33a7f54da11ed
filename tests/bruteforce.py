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


def run(w, rows_by_seq=None, scale=None):
    """Return out[qrow][head] = list of D floats for every query row of the batch."""
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
            visible = toks[:ctx - qlen + i + 1]
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
