"""Host semantics of the KV block allocator, written as a plain Python model.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The C++ allocator in
the library is checked against this model operation by operation, bit-exact.

What the pages fix ("PagedAttention (vLLM) -- Virtual memory cho AI"):
* section "Co che Block Table": the cache is cut into fixed blocks (typically
  16 tokens); each sequence has a table from logical block i (tokens
  16i..16i+15) to a physical block anywhere in memory; a block is handed out
  only when a token actually needs it (100 tokens -> 7 blocks = 112 slots
  instead of 256 blocks for a 4096-token reservation); freed blocks, even small
  ones released mid-run, are reused at once with no defragmentation.
* section "Copy-on-Write cho Beam Search": branches of beam search / parallel
  sampling share the physical blocks of their common prefix and split a block
  only when their tokens start to differ.

Readings where the pages are silent (each listed in the design notes):
* free list: a LIFO stack that hands out block 0 first, then 1, 2, ...; a
  freed sequence pushes its blocks in table order (so its last block is the
  next one handed out);
* copy-on-write happens on ``append_slot`` into a partially filled last block
  whose reference count is above one: a fresh block is taken, the pair
  (src, dst) is reported for the device copy and src loses one reference; the
  last remaining holder writes in place; a shared *full* block is never copied;
* running out of blocks returns ERR_OOM and changes nothing;
* waste = 1 - occupied slots / allocated slots, every physical block counted
  once however many sequences share it.

Prefix caching ("vLLM PagedAttention: Buoc dot pha ve thong luong suy luan
LLM", list of advanced features: the KV cache of a prompt prefix shared by
several requests is reused instead of recomputed).  The pages give no
mechanism; the reading modelled here (and listed in the design notes):
* only full blocks of prompts added with ``add_seq_cached`` are registered,
  each under its whole token prefix (here the prefix itself is the key; the
  library uses a hash of it plus an exact comparison of the block's tokens);
* a prompt shares its leading full blocks whose prefixes are registered
  (reference count + 1) and allocates the rest; ``cached_tokens`` = shared
  blocks x block_size;
* a registered block left without holders stays registered in an evictable
  queue; a freed prompt's blocks join it last block first; blocks are taken
  from the free stack first, then from the front of the queue (unregistering
  them); ``num_free`` counts both;
* ``cache_clear`` moves the evictable blocks (front first) to the free stack
  and forgets every registration.

Truncation (rolling back drafted tokens that verification rejected -- same
page, speculative decoding): ``truncate(seq, n)`` keeps the first n tokens;
the reading modelled here is in its docstring.
"""
from __future__ import annotations

OK = 0
ERR_INVALID = 1
ERR_OOM = 2


class BlockAllocatorModel:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        # top of the stack is the list's end: block 0 is handed out first
        self._free = list(range(self.num_blocks - 1, -1, -1))
        self._ref = [0] * self.num_blocks
        self._seqs = {}  # seq id -> [table (list of block ids), num_tokens]
        self._cache = {}      # token prefix (tuple) -> block
        self._key = {}        # registered block -> its token prefix
        self._evictable = []  # registered blocks without holders, front = released longest ago
        self.hits = 0
        self.misses = 0

    # -- internal -----------------------------------------------------------
    def _available(self) -> int:
        return len(self._free) + len(self._evictable)

    def _take(self) -> int:
        if self._free:
            b = self._free.pop()
        else:
            b = self._evictable.pop(0)
            del self._cache[self._key.pop(b)]
        self._ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self._ref[b] -= 1
        if self._ref[b] == 0 and b not in self._key:
            self._free.append(b)

    # -- operations (return a status, plus results) --------------------------
    def add_seq(self, seq: int, num_tokens: int) -> int:
        """A new sequence holding ``num_tokens`` tokens (a prompt)."""
        if seq in self._seqs or num_tokens < 0:
            return ERR_INVALID
        need = -(-num_tokens // self.block_size)
        if need > self._available():
            return ERR_OOM
        table = [self._take() for _ in range(need)]
        self._seqs[seq] = [table, num_tokens]
        return OK

    def add_seq_cached(self, seq: int, tokens):
        """A prompt with known token ids.  Returns (status, cached_tokens)."""
        tokens = [int(t) for t in tokens]
        if seq in self._seqs:
            return ERR_INVALID, 0
        B = self.block_size
        n = len(tokens)
        nfull, need = n // B, -(-n // B)
        hit = []
        for i in range(nfull):
            b = self._cache.get(tuple(tokens[:(i + 1) * B]))
            if b is None:
                break
            hit.append(b)
        revived = sum(1 for b in hit if self._ref[b] == 0)
        if need - len(hit) > self._available() - revived:
            return ERR_OOM, 0
        table = []
        for b in hit:
            if self._ref[b] == 0:
                self._evictable.remove(b)
            self._ref[b] += 1
            table.append(b)
        for i in range(len(hit), need):
            b = self._take()
            table.append(b)
            key = tuple(tokens[:(i + 1) * B])
            if i < nfull and key not in self._cache:
                self._cache[key] = b
                self._key[b] = key
        self._seqs[seq] = [table, n]
        self.hits += len(hit)
        self.misses += nfull - len(hit)
        return OK, len(hit) * B

    def cache_stats(self):
        return {"hits": self.hits, "misses": self.misses, "cached_blocks": len(self._cache),
                "evictable_blocks": len(self._evictable)}

    def cache_clear(self) -> int:
        for b in self._evictable:
            self._free.append(b)
        self._evictable = []
        self._cache = {}
        self._key = {}
        return OK

    def append_slot(self, seq: int):
        """Room for one more token of ``seq``.  Returns (status, slot, cow_src,
        cow_dst); cow_src/cow_dst are -1 when no copy is needed."""
        if seq not in self._seqs:
            return ERR_INVALID, -1, -1, -1
        table, n = self._seqs[seq]
        offset = n % self.block_size
        src = dst = -1
        if offset == 0:
            # last block full (or no block yet): a fresh block for this token
            if not self._available():
                return ERR_OOM, -1, -1, -1
            table.append(self._take())
        elif self._ref[table[-1]] > 1:
            # the partially filled last block is shared: copy before writing
            if not self._available():
                return ERR_OOM, -1, -1, -1
            src = table[-1]
            dst = self._take()
            self._ref[src] -= 1
            table[-1] = dst
        slot = table[-1] * self.block_size + offset
        self._seqs[seq][1] = n + 1
        return OK, slot, src, dst

    def fork(self, parent: int, child: int) -> int:
        """``child`` starts as ``parent``, sharing every block by reference."""
        if parent not in self._seqs or child in self._seqs or parent == child:
            return ERR_INVALID
        table, n = self._seqs[parent]
        for b in table:
            self._ref[b] += 1
        self._seqs[child] = [list(table), n]
        return OK

    def free_seq(self, seq: int) -> int:
        if seq not in self._seqs:
            return ERR_INVALID
        table, _ = self._seqs.pop(seq)
        for b in table:
            self._release(b)
        # registered blocks left without holders: evictable, last block first
        for b in reversed(table):
            if self._ref[b] == 0 and b in self._key:
                self._evictable.append(b)
        return OK

    def extend(self, seq: int, count: int):
        """Room for ``count`` more tokens of ``seq`` at once (a prefill chunk):
        the same slots and copy pair as ``count`` calls of append_slot, but all
        or nothing.  Returns (status, slots, cow_src, cow_dst)."""
        if seq not in self._seqs or count < 0:
            return ERR_INVALID, [], -1, -1
        table, n = self._seqs[seq]
        B = self.block_size
        shared_partial = n % B != 0 and self._ref[table[-1]] > 1
        need = -(-(n + count) // B) - -(-n // B) + (1 if shared_partial and count > 0 else 0)
        if need > self._available():
            return ERR_OOM, [], -1, -1
        slots, src, dst = [], -1, -1
        for _ in range(count):
            st, slot, s_, d_ = self.append_slot(seq)
            assert st == OK
            slots.append(slot)
            if s_ >= 0:
                src, dst = s_, d_
        return OK, slots, src, dst

    def truncate(self, seq: int, num_tokens: int) -> int:
        """Keep the first ``num_tokens`` tokens of ``seq`` (drafted tokens that
        verification rejected, for instance).  Blocks wholly past the new end
        are released in table order; registered ones left without holders join
        the evictable queue, the later block first.  A registered block that
        becomes the partially filled last block of its only holder loses its
        registration: the next append writes into it."""
        if seq not in self._seqs:
            return ERR_INVALID
        table, n = self._seqs[seq]
        if num_tokens < 0 or num_tokens > n:
            return ERR_INVALID
        keep = -(-num_tokens // self.block_size)
        dropped = table[keep:]
        del table[keep:]
        for b in dropped:
            self._release(b)
        for b in reversed(dropped):
            if self._ref[b] == 0 and b in self._key:
                self._evictable.append(b)
        self._seqs[seq][1] = num_tokens
        if keep and num_tokens % self.block_size and table[-1] in self._key and self._ref[table[-1]] == 1:
            del self._cache[self._key.pop(table[-1])]
        return OK

    # -- queries --------------------------------------------------------------
    def block_table(self, seq: int):
        return list(self._seqs[seq][0])

    def num_tokens(self, seq: int) -> int:
        return self._seqs[seq][1]

    def num_free(self) -> int:
        return self._available()

    def refcount(self, block: int) -> int:
        return self._ref[block]

    def sequences(self):
        return sorted(self._seqs)

    def waste(self):
        """(occupied slots, allocated slots) with each live block counted once."""
        fill = {}
        for table, n in self._seqs.values():
            for i, b in enumerate(table):
                used = min(self.block_size, max(0, n - i * self.block_size))
                fill[b] = max(fill.get(b, 0), used)
        return sum(fill.values()), len(fill) * self.block_size
