"""Host block manager with prefix sharing, clone-N and copy-on-write (test oracle).

What the pages give, and the readings taken where they stop:

* nano-vllm "Model Runner" notes, section "prepare Prefill": the block manager
  is CPU-side bookkeeping run at schedule time, before the model.
  ``can_allocate`` consults the prefix cache to know how many blocks a
  sequence needs, ``allocate`` writes physical block ids into the sequence's
  block table, and ``num_cached_tokens`` counts the prompt tokens whose K/V
  are already in the cache (``cu_seqlens_k = scheduled + cached``, section
  "prefix cache").
* nanochat "04 · Engine 推理与工具调用", sections 2-3: one prefill, then the
  cache is cloned for N samples.  Here a clone shares the blocks (reference
  counts) instead of copying them.

Readings (the pages are silent on the internals):

* Free blocks form a FIFO, initially 0, 1, ..., num_blocks - 1; allocation
  takes the front, a block whose count drops to 0 goes to the back.
* A full block is identified by (the physical block before it in the table,
  or -1, and its block_size token ids): an exact key, no hash collisions.
  A freed block keeps its key until it is handed out again, so a later
  prompt with the same prefix can reclaim it from the free list.
* A prompt looks up its full blocks in order and stops at the first miss;
  a block is looked up only if at least one prompt token lies after it (the
  last token is always computed).  ``cached_tokens`` = block_size x hits.
* Appending a token (decode) that starts a new block takes a fresh block.
  A token that lands in a shared last block (count > 1, e.g. after a fork)
  first copies that block: a fresh block receives its existing rows
  (copy-on-write), the shared block loses one reference.  A block that
  becomes full registers its key.
* Allocation that needs more free blocks than there are changes nothing and
  reports "no space".
"""
from __future__ import annotations


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        self.nb, self.bs = int(num_blocks), int(block_size)
        self.free = list(range(self.nb))        # FIFO: front = index 0
        self.ref = [0] * self.nb
        self.key_of = [None] * self.nb          # key a block is registered under
        self.cache = {}                         # key -> block

    def _key(self, parent: int, tokens) -> tuple:
        return (int(parent),) + tuple(int(t) for t in tokens)

    def _take(self) -> int:
        b = self.free.pop(0)
        if self.key_of[b] is not None:          # stale content: forget it
            del self.cache[self.key_of[b]]
            self.key_of[b] = None
        self.ref[b] = 1
        return b

    def _register(self, b: int, parent: int, tokens) -> None:
        k = self._key(parent, tokens)
        if k in self.cache:                     # an equal block exists: keep the first
            return
        self.cache[k] = b
        self.key_of[b] = k

    def num_free(self) -> int:
        return len(self.free)

    def allocate(self, tokens):
        """Block table and cached token count for a new prompt, or None (no space)."""
        n, bs = len(tokens), self.bs
        nblk = -(-n // bs)
        hits, parent = [], -1
        for i in range(nblk):
            if (i + 1) * bs > n - 1:            # keep at least the last token to compute
                break
            b = self.cache.get(self._key(parent, tokens[i * bs:(i + 1) * bs]))
            if b is None:
                break
            hits.append(b)
            parent = b
        need = (nblk - len(hits)) + sum(1 for b in hits if self.ref[b] == 0)
        if need > len(self.free):
            return None
        table = []
        for b in hits:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
            table.append(b)
        parent = table[-1] if table else -1
        for i in range(len(hits), nblk):
            b = self._take()
            if (i + 1) * bs <= n:               # full block: register its content
                self._register(b, parent, tokens[i * bs:(i + 1) * bs])
            table.append(b)
            parent = b
        return table, bs * len(hits)

    def append(self, tokens, table):
        """The sequence now holds ``tokens`` (one more than before).  Returns
        (table, copy) with copy = (src, dst, rows) for copy-on-write or None;
        None for the table when no block is free."""
        n, bs = len(tokens), self.bs
        p = n - 1                               # position of the new token
        table = list(table)
        copy = None
        if p % bs == 0:                         # a new block
            if not self.free:
                return None, None
            table.append(self._take())
        else:
            last = table[-1]
            if self.ref[last] > 1:              # shared: copy before writing
                if not self.free:
                    return None, None
                b = self._take()
                self.ref[last] -= 1
                copy = (last, b, p % bs)
                table[-1] = b
        if p % bs == bs - 1:                    # the last block is now full
            i = p // bs
            parent = table[i - 1] if i > 0 else -1
            self._register(table[i], parent, tokens[i * bs:(i + 1) * bs])
        return table, copy

    def fork(self, table) -> list:
        """A clone of the sequence: every block gains a reference."""
        for b in table:
            self.ref[b] += 1
        return list(table)

    def release(self, table) -> None:
        """The sequence ends: its blocks lose a reference (last block first)."""
        for b in reversed(table):
            self.ref[b] -= 1
            assert self.ref[b] >= 0
            if self.ref[b] == 0:
                self.free.append(b)
