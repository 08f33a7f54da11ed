"""8-bit KV cache: quantise on append, dequantise in the gather (oracle; test infrastructure only).

[Deploy §2.5 LMDeploy, "2. TurboMind 推理引擎解析"]: TurboMind keeps the KV
cache in 8 bits, which halves the bytes decode reads.  The pages give no
format; the reading taken here is symmetric int8 with one float32 scale per
(token, KV head):

    amax  = max_d |x[d]|                 (exact)
    scale = amax / 127                   (float32 division, rounded once)
    code  = clamp(rint(x[d] / scale), -127, 127)   (float32 division, ties to even)
    code  = 0 and scale = 0 when amax = 0

and a stored row reads back as code * scale.  The codes are a decision of the
float32 arithmetic, so this module computes them exactly as the kernel does
(numpy float32 is IEEE with one rounding per operation).

Cache layout: codes [num_blocks, Hkv, block_size, D] int8 and scales
[num_blocks, Hkv, block_size] float32, separately for K and V.
"""

import numpy as np

from .numerics import widen


def quantize_rows(x, dtype):
    """x [..., D] in the storage dtype (float32, or bf16 bits) -> (codes int8, scales float32)."""
    f = widen(x, dtype).astype(np.float32)  # exact: bf16 and float32 values are float32
    amax = np.max(np.abs(f), axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = np.rint(f / safe[..., None])
    q = np.where(scale[..., None] > 0, q, 0.0)
    codes = np.clip(q, -127, 127).astype(np.int8)
    return codes, scale


def dequantize(codes, scales):
    """float64 values code * scale (exact)."""
    return codes.astype(np.float64) * scales.astype(np.float64)[..., None]


def append_int8(kq, ks, vq, vs, k, v, slot_mapping, block_size, dtype):
    """Quantise k, v ([T, Hkv, D], storage dtype) and write codes and scales to their slots."""
    slots = np.asarray(slot_mapping, dtype=np.int64)
    kc, kscale = quantize_rows(k, dtype)
    vc, vscale = quantize_rows(v, dtype)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        b, r = divmod(int(slot), block_size)
        kq[b, :, r, :] = kc[t]
        vq[b, :, r, :] = vc[t]
        ks[b, :, r] = kscale[t]
        vs[b, :, r] = vscale[t]


def decode_int8(q, kq, ks, vq, vs, block_tables, context_lens, block_size, q_dtype, scale=None):
    """Exact attention (float64) over the dequantised cache; one query per sequence."""
    import math

    S, Hq, D = q.shape
    Hkv = kq.shape[1]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qf = widen(q, q_dtype)
    out = np.empty((S, Hq, D))
    for s in range(S):
        ctx = int(context_lens[s])
        nblk = -(-ctx // block_size)
        blocks = [int(b) for b in block_tables[s][:nblk]]
        kd = np.concatenate([np.swapaxes(dequantize(kq[b], ks[b]), 0, 1) for b in blocks])[:ctx]
        vd = np.concatenate([np.swapaxes(dequantize(vq[b], vs[b]), 0, 1) for b in blocks])[:ctx]
        for h in range(Hq):
            sc = (kd[:, h // g] @ qf[s, h]) * scale
            p = np.exp(sc - sc.max())
            out[s, h] = (p @ vd[:, h // g]) / p.sum()
    return out
