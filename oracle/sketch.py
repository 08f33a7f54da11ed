"""The per-block-normalised sketch from [Ch7 §2.2.2 注意力计算的重构] (negative control).

The sketch normalises each block's scores on their own and adds up the blocks'
outputs: sum_b softmax(q K_b^T * scale) V_b.  With more than one block this is
not attention (the weights sum to the number of blocks, and blocks are not
weighted against each other).  The tests use it only to show that the exact
oracle differs from it; nothing in the product computes it.
"""

import numpy as np


def per_block_softmax(q, k, v, scale, block_size):
    """q [D]; k, v [n, D] float64 -> [D]."""
    out = np.zeros(q.shape[0])
    for b0 in range(0, k.shape[0], block_size):
        s = (k[b0:b0 + block_size] @ q) * scale
        p = np.exp(s - s.max())
        out += (p / p.sum()) @ v[b0:b0 + block_size]
    return out
