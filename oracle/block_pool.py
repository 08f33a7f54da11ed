"""Reference model of the ref-counted physical block pool (oracle; test infrastructure only).

Semantics, in the pages' order:

* A sequence of L tokens needs ceil(L / block_size) blocks [Ch7 §2.2.1 块分配机制;
  Deploy §2.1 _allocate_sequence: one physical block per logical block, logical
  index from 0].
* Admission with a watermark [Deploy §2.1 "3. vLLM 调度策略与显存块管理", can_allocate]: NEVER when the pool
  could not hold the request even empty (total - need < watermark); OK when the
  free blocks cover it with the watermark left over (free - need >= watermark);
  LATER otherwise.
* Growing a sequence by one token [Deploy §2.1 append_slots; Infra 二、2 (每个
  逻辑块仅在前一个块被填满后才会分配新的物理块)]: a new block is taken only when
  the last block is full; otherwise the token goes into the last block, and if
  that block is shared (ref count > 1) it is first copied to a fresh block
  (copy-on-write): the sequence's table points at the copy, the old block loses
  one reference, and the (old, new) pair is returned so the device can copy.
* Forking a sequence (parallel sampling) shares every block: ref count + 1
  [Deploy §2.1 "4. PageAttention 内存管理技术详解" (引用计数 / 写时复制); Infra 二、2].
* Freeing drops one reference per block; a block with no references returns to
  the free list [Infra 二 (全局空闲物理块列表)].

Readings where the pages are silent (also used by the C++ pool, which is a
separate implementation):
  * The free list is a stack.  ``free_order`` lists the initial stack from the
    top: its first entry is handed out first.  A freed block goes on top
    (LIFO, as the Ch7 §2.3 sketch's ``free_blocks.pop()``).
  * A sequence's blocks are released in table order.
  * Adding a sequence applies the admission rule (NEVER / LATER / OK); growing
    one needs only a free block.
"""

OK, LATER, NEVER = "OK", "LATER", "NEVER"


class PoolError(Exception):
    pass


class BlockPoolModel:
    def __init__(self, num_blocks, block_size, watermark_blocks=0, free_order=None):
        if num_blocks < 1 or block_size < 1 or watermark_blocks < 0:
            raise PoolError("bad pool parameters")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.watermark_blocks = watermark_blocks
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise PoolError("free_order must be a permutation of the block ids")
        self._stack = list(reversed(order))  # top of stack = end of list
        self.ref = [0] * num_blocks
        self.tables = {}
        self.lens = {}

    # -- queries -----------------------------------------------------------
    def num_free(self):
        return len(self._stack)

    def blocks_needed(self, n_tokens):
        return -(-n_tokens // self.block_size)

    def can_allocate(self, n_tokens):
        need = self.blocks_needed(n_tokens)
        if self.num_blocks - need < self.watermark_blocks:
            return NEVER
        if self.num_free() - need >= self.watermark_blocks:
            return OK
        return LATER

    def block_table(self, seq_id):
        return list(self.tables[seq_id])

    def context_len(self, seq_id):
        return self.lens[seq_id]

    def slot_of(self, seq_id, pos):
        """Physical slot of logical token ``pos``: table[pos // bs] * bs + pos % bs."""
        t = self.tables[seq_id]
        return t[pos // self.block_size] * self.block_size + pos % self.block_size

    # -- mutations ---------------------------------------------------------
    def _take(self):
        b = self._stack.pop()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _drop(self, b):
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            self._stack.append(b)

    def add_sequence(self, seq_id, n_tokens):
        """Allocate a prompt of ``n_tokens`` tokens; return its slots in order."""
        if seq_id in self.tables:
            raise PoolError("sequence exists")
        if n_tokens < 1:
            raise PoolError("empty prompt")
        st = self.can_allocate(n_tokens)
        if st != OK:
            return st, None
        table = [self._take() for _ in range(self.blocks_needed(n_tokens))]
        self.tables[seq_id] = table
        self.lens[seq_id] = n_tokens
        return OK, [self.slot_of(seq_id, p) for p in range(n_tokens)]

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            raise PoolError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def append_slot(self, seq_id):
        """Grow a sequence by one token.

        Returns (slot, cow) where cow is None or the (src, dst) block pair the
        device must copy before writing the token.  Returns (None, None) and
        changes nothing when a block is needed but none is free.
        """
        table = self.tables[seq_id]
        pos = self.lens[seq_id]
        if pos % self.block_size == 0:  # last block full (or none yet): new block
            if not self._stack:
                return None, None
            table.append(self._take())
            self.lens[seq_id] = pos + 1
            return self.slot_of(seq_id, pos), None
        last = table[-1]
        if self.ref[last] == 1:
            self.lens[seq_id] = pos + 1
            return self.slot_of(seq_id, pos), None
        if not self._stack:
            return None, None
        new = self._take()
        table[-1] = new
        self._drop(last)
        self.lens[seq_id] = pos + 1
        return self.slot_of(seq_id, pos), (last, new)

    def free_sequence(self, seq_id):
        for b in self.tables.pop(seq_id):
            self._drop(b)
        del self.lens[seq_id]
