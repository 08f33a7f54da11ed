"""Prefix caching and sliding-window block tables (oracle; test infrastructure only).

Two host-side variants of the block table from "大模型部署.md" §2.1 (3. vLLM 调度策略
与显存块管理: BlockSpaceManager with ``enable_caching`` or ``sliding_window``;
CachedBlockAllocator and its LRU evictor).  The pages allow one or the other,
never both.

Prefix caching, as the pages describe it:
  * a full logical block is identified by a hash of every token of the sequence
    up to the end of that block; a block with that hash that is in use is
    shared (reference count + 1), one parked in the evictor is taken back;
  * a block whose last reference goes away keeps its hash and moves to the
    evictor instead of the free list, so a later prompt with the same prefix
    can reuse it;
  * a new block comes from the free list, else the evictor gives one up:
    least recently accessed first; among equals, the one whose hash covers the
    most tokens; among those, any (here: the one parked first);
  * when decoding fills a block, its hash is computed; if a block with that
    hash already exists the sequence switches to it and the filled copy is
    released, otherwise the block is registered under the hash.

Sliding window, as the pages describe it: with W_b = ceil(window / block_size),
logical block j >= W_b reuses table[j % W_b], so a table is a ring of W_b
physical blocks; admission counts min(blocks, W_b); a shared ring block is
copied before it is written (copy-on-write).

Readings where the pages are silent:
  * The hash of logical block j is FNV-1a (64 bit, its published offset basis
    and prime) over the 8 little-endian bytes of the previous block's hash
    (0 for block 0) followed by the block's token ids as 4-byte little-endian
    integers.  Only full blocks have a hash.
  * ``num_cached_tokens`` of a new prompt is block_size times the number of
    leading logical blocks that were found (in use or in the evictor).
  * The access clock is the caller's (``set_clock``); a block is stamped when
    it is handed to a sequence and when it is parked in the evictor.
  * The free count used for admission is free list + evictor.
  * If a decode step both copies a shared block and then finds the filled
    block's hash, the copy is cancelled: the sequence switches to the found
    block, which already holds the tokens.
  * Sliding window: the window is a multiple of block_size, so the last
    ``window`` tokens fill the W_b ring blocks exactly; prompt tokens whose slot
    a later token of the same prompt takes get slot -1 (skip); the exported
    table lists the physical blocks of the last W_b logical blocks in logical
    order, with context min(len, window).
  * Sliding window with prefill chunks: a chunk of C queries needs the C + W - 1
    most recent keys at once, more than a ring of exactly W tokens holds, so a
    pool that serves chunks of up to ``max_chunk`` tokens keeps
    R_b = W_b + ceil((max_chunk - 1) / block_size) ring blocks (max_chunk = 1:
    the pages' ring).  The ring then holds the last R_b * block_size tokens.
    For a step whose last ``qlen`` tokens are queries, ``logical_table`` lists
    the ring entries of logical blocks first .. last in logical order, where
    ``first`` holds the first key any of those queries attends, with context
    = len - first * block_size; attention then applies the window as a mask
    (the rows below the window in the first entry may hold newer tokens).
"""

import math

from .block_pool import LATER, NEVER, OK, PoolError

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data):
    """FNV-1a, 64 bit, over a bytes object."""
    h = FNV_OFFSET
    for b in data:
        h ^= b
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(prev_hash, tokens):
    """Chained hash of one full block: FNV-1a over prev_hash (8 bytes LE) + tokens (int32 LE)."""
    data = int(prev_hash).to_bytes(8, "little")
    for t in tokens:
        data += int(t).to_bytes(4, "little", signed=True)
    return fnv1a64(data)


class PrefixCachingPool:
    """Block pool with prefix caching (hash-shared full blocks + LRU evictor)."""

    def __init__(self, num_blocks, block_size, watermark_blocks=0, free_order=None):
        if num_blocks < 1 or block_size < 1 or watermark_blocks < 0:
            raise PoolError("bad pool parameters")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.watermark_blocks = watermark_blocks
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise PoolError("free_order must be a permutation of the block ids")
        self.free = list(reversed(order))      # stack: end of list is handed out next
        self.ref = [0] * num_blocks
        self.hash_of = [None] * num_blocks     # hash of a registered block
        self.hashed_tokens = [0] * num_blocks
        self.last_accessed = [0] * num_blocks
        self.cached = {}                       # hash -> block (in use or in the evictor)
        self.evictor = []                      # parked blocks, in the order they were parked
        self.clock = 0
        self.tables = {}
        self.tokens = {}
        self.hashes = {}                       # seq -> hashes of its full blocks

    # -- queries -----------------------------------------------------------
    def num_free(self):
        return len(self.free) + len(self.evictor)

    def num_evictable(self):
        return len(self.evictor)

    def blocks_needed(self, n):
        return -(-n // self.block_size)

    def can_allocate(self, n):
        need = self.blocks_needed(n)
        if self.num_blocks - need < self.watermark_blocks:
            return NEVER
        if self.num_free() - need >= self.watermark_blocks:
            return OK
        return LATER

    def block_table(self, seq):
        return list(self.tables[seq])

    def context_len(self, seq):
        return len(self.tokens[seq])

    def slot_of(self, seq, pos):
        return self.tables[seq][pos // self.block_size] * self.block_size + pos % self.block_size

    # -- block sources -----------------------------------------------------
    def set_clock(self, now):
        self.clock = int(now)

    def _evict(self):
        """Take a block out of the evictor: oldest access, then most hashed tokens, then first parked."""
        best = None
        for b in self.evictor:
            if best is None or self.last_accessed[b] < self.last_accessed[best] or (
                    self.last_accessed[b] == self.last_accessed[best]
                    and self.hashed_tokens[b] > self.hashed_tokens[best]):
                best = b
        self.evictor.remove(best)
        del self.cached[self.hash_of[best]]
        self.hash_of[best] = None
        self.hashed_tokens[best] = 0
        return best

    def _fresh(self):
        """An unhashed block with one reference: free list first, else evicted."""
        b = self.free.pop() if self.free else self._evict()
        self.ref[b] = 1
        self.last_accessed[b] = self.clock
        return b

    def _lookup(self, h):
        """The block registered under h with one more reference, or None."""
        b = self.cached.get(h)
        if b is None:
            return None
        if self.ref[b] == 0:
            self.evictor.remove(b)
        self.ref[b] += 1
        self.last_accessed[b] = self.clock
        return b

    def _register(self, b, h, n_tokens):
        self.hash_of[b] = h
        self.hashed_tokens[b] = n_tokens
        self.cached[h] = b

    def _release(self, b):
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            if self.hash_of[b] is not None:
                self.last_accessed[b] = self.clock
                self.evictor.append(b)
            else:
                self.free.append(b)

    # -- sequence operations -----------------------------------------------
    def add_sequence(self, seq, token_ids):
        """Returns (status, slots, num_cached_tokens)."""
        token_ids = [int(t) for t in token_ids]
        n = len(token_ids)
        if seq in self.tables or n < 1:
            raise PoolError("bad sequence")
        st = self.can_allocate(n)
        if st != OK:
            return st, None, None
        bs = self.block_size
        table, hashes, prev, leading, run = [], [], 0, 0, True
        for j in range(self.blocks_needed(n)):
            if (j + 1) * bs <= n:
                h = block_hash(prev, token_ids[j * bs:(j + 1) * bs])
                hashes.append(h)
                prev = h
                b = self._lookup(h)
                if b is None:
                    run = False
                    b = self._fresh()
                    self._register(b, h, (j + 1) * bs)
                elif run:
                    leading += 1
            else:
                run = False
                b = self._fresh()
            table.append(b)
        self.tables[seq] = table
        self.tokens[seq] = token_ids
        self.hashes[seq] = hashes
        return OK, [self.slot_of(seq, p) for p in range(n)], leading * bs

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            raise PoolError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.tokens[child] = list(self.tokens[parent])
        self.hashes[child] = list(self.hashes[parent])
        for b in self.tables[child]:
            self.ref[b] += 1

    def append_token(self, seq, token_id):
        """Grow by one token.  Returns (slot, cow) or (None, None) when no block is free."""
        table, toks = self.tables[seq], self.tokens[seq]
        bs, pos = self.block_size, len(toks)
        j = pos // bs
        cow = None
        if pos % bs == 0:
            if self.num_free() == 0:
                return None, None
            table.append(self._fresh())
        elif self.ref[table[j]] > 1:
            if self.num_free() == 0:
                return None, None
            old = table[j]
            table[j] = self._fresh()
            self._release(old)
            cow = (old, table[j])
        toks.append(int(token_id))
        if (pos + 1) % bs == 0:
            prev = self.hashes[seq][j - 1] if j > 0 else 0
            h = block_hash(prev, toks[j * bs:(j + 1) * bs])
            self.hashes[seq].append(h)
            found = self._lookup(h)
            if found is not None:
                self._release(table[j])
                table[j] = found
                cow = None
            else:
                self._register(table[j], h, (j + 1) * bs)
        return self.slot_of(seq, pos), cow

    def free_sequence(self, seq):
        for b in self.tables.pop(seq):
            self._release(b)
        del self.tokens[seq]
        del self.hashes[seq]


class SlidingWindowPool:
    """Block pool whose tables are rings of window / block_size blocks, plus
    ceil((max_chunk - 1) / block_size) for pools that serve prefill chunks."""

    def __init__(self, num_blocks, block_size, window, watermark_blocks=0, free_order=None,
                 max_chunk=1):
        if num_blocks < 1 or block_size < 1 or watermark_blocks < 0 or max_chunk < 1:
            raise PoolError("bad pool parameters")
        if window < block_size or window % block_size:
            raise PoolError("window must be a positive multiple of block_size")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.window = window
        self.max_chunk = max_chunk
        self.ring = window // block_size + math.ceil((max_chunk - 1) / block_size)
        self.capacity = self.ring * block_size    # tokens the ring holds
        self.watermark_blocks = watermark_blocks
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise PoolError("free_order must be a permutation of the block ids")
        self.free = list(reversed(order))
        self.ref = [0] * num_blocks
        self.tables = {}                       # physical ring, at most W_b entries
        self.lens = {}

    def num_free(self):
        return len(self.free)

    def blocks_needed(self, n):
        return min(-(-n // self.block_size), self.ring)

    def can_allocate(self, n):
        need = self.blocks_needed(n)
        if self.num_blocks - need < self.watermark_blocks:
            return NEVER
        if self.num_free() - need >= self.watermark_blocks:
            return OK
        return LATER

    def context_len(self, seq):
        return self.lens[seq]

    def slot_of(self, seq, pos):
        bs = self.block_size
        return self.tables[seq][(pos // bs) % self.ring] * bs + pos % bs

    def _take(self):
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def _release(self, b):
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            self.free.append(b)

    def add_sequence(self, seq, n):
        """Returns (status, slots); a token whose slot a later prompt token takes gets -1."""
        if seq in self.tables or n < 1:
            raise PoolError("bad sequence")
        st = self.can_allocate(n)
        if st != OK:
            return st, None
        self.tables[seq] = [self._take() for _ in range(self.blocks_needed(n))]
        self.lens[seq] = n
        return OK, [self.slot_of(seq, p) if p + self.capacity >= n else -1 for p in range(n)]

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            raise PoolError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def append_slot(self, seq):
        table, pos, bs = self.tables[seq], self.lens[seq], self.block_size
        j = pos // bs
        cow = None
        if pos % bs == 0 and j < self.ring:
            if not self.free:
                return None, None
            table.append(self._take())
        else:
            r = j % self.ring
            if self.ref[table[r]] > 1:
                if not self.free:
                    return None, None
                old = table[r]
                table[r] = self._take()
                self._release(old)
                cow = (old, table[r])
        self.lens[seq] = pos + 1
        return self.slot_of(seq, pos), cow

    def free_sequence(self, seq):
        for b in self.tables.pop(seq):
            self._release(b)
        del self.lens[seq]

    def window_table(self, seq):
        """(physical blocks of the last W_b logical blocks in logical order, context length):
        exactly the last ``window`` tokens, for decode without a mask; only a ring of
        exactly W_b blocks (max_chunk = 1) has that property."""
        if self.ring != self.window // self.block_size:
            raise PoolError("a ring with chunk room needs logical_table and a window mask")
        n, bs = self.lens[seq], self.block_size
        nb = -(-n // bs)
        first = max(0, nb - self.ring)
        return [self.tables[seq][j % self.ring] for j in range(first, nb)], min(n, self.window)

    def logical_table(self, seq, qlen=1):
        """(ring entries of logical blocks first .. last in logical order, context) for a
        step whose last ``qlen`` tokens are queries under the window: ``first`` is the
        block of the first key the first query attends, context = len - first * bs."""
        n, bs = self.lens[seq], self.block_size
        if not 1 <= qlen <= n:
            raise PoolError("query span must be 1 .. sequence length")
        if qlen + self.window - 1 > self.capacity:
            raise PoolError("the ring cannot hold the keys of that many queries")
        first = max(0, n - qlen - self.window + 1) // bs
        nb = -(-n // bs)
        return [self.tables[seq][j % self.ring] for j in range(first, nb)], n - first * bs
