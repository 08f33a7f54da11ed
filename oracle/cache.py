"""Cache mirror operations (oracle; test infrastructure only).

* ``append``: each new token's K/V goes to the physical slot the host planned
  for it: block ``slot // block_size``, row ``slot % block_size``
  [Infra 一、2、解码 (KtVt 更新到 kv cache); Deploy §2.1 ("真正的分配物理块号":
  the block manager only plans, the cache engine writes)].  A negative slot
  means "no write" (padding), a reading the pages leave open.
* ``copy_blocks``: copy-on-write copies a whole physical block (every row, K
  and V, all KV heads) from ``src`` to ``dst``: a shared last block gets a
  private copy before the write [Deploy §2.1 append_slots; Infra 二、2
  copy-on-write].

The cache dtype is the input dtype (float32 or bf16 bit patterns); an append is
a bit copy, so the mirror is exact byte for byte.
"""

import numpy as np


def append(k_cache, v_cache, k, v, slot_mapping, block_size):
    """Write k[t], v[t] ([T, Hkv, D]) to slot_mapping[t] in place."""
    slots = np.asarray(slot_mapping, dtype=np.int64)
    if k.dtype != k_cache.dtype or v.dtype != v_cache.dtype:
        raise TypeError("append is a bit copy: input dtype must equal cache dtype")
    live = slots >= 0
    s = slots[live]
    if len(np.unique(s)) != len(s):
        raise ValueError("two tokens map to the same slot")
    nb = k_cache.shape[0]
    if np.any(s >= nb * block_size):
        raise IndexError("slot outside the pool")
    blk = s // block_size
    row = s % block_size
    # one token at a time, in order; each write is [Hkv, D]
    for i, t in enumerate(np.nonzero(live)[0]):
        k_cache[blk[i], :, row[i], :] = k[t]
        v_cache[blk[i], :, row[i], :] = v[t]


def copy_blocks(k_cache, v_cache, pairs):
    """For each (src, dst): cache[dst] = cache[src], whole block, K and V."""
    for src, dst in pairs:
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
