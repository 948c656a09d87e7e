"""TEST INFRASTRUCTURE ONLY: the BlockManager of "P06 BlockManager", in plain Python.

Followed step by step from that page ("three operations, one ledger, invariants"
table and the L2 hints), with fork + copy-on-write added from "ans20xx day 31"
(`fork_sequence`, `ensure_private_last_block`, `append_with_cow`).

Ledger (the page's L2 table):
  free_blocks    deque of unhashed free blocks, popleft to take, append to return
  ref            reference count per physical block
  block_hash     hash registered for each block (None = not in the cache)
  hash_to_block  hash -> block, for hits
  evictable      OrderedDict of ref==0 blocks that still carry a hash; insertion
                 order is LRU order (oldest first)
  tables/tokens/hashes/cached   per-sequence records

Readings where the pages are silent or ambiguous:
  * The chained hash is Python's hash of (parent, tuple(block tokens)) with
    parent None for the first block (the page's own suggestion).  Its values are
    never observable; only equal/unequal matters.
  * Registering a hash that already maps to another block sets
    block_hash[b] = h but keeps the old map entry ("keep the old one").
  * fork(parent, child) copies the parent's table, tokens, hash chain and cached
    count and adds one reference to every block (day-31 `fork_sequence`).
  * append_slot into a partial last block whose ref > 1 is a copy-on-write: take
    a new block (the only step that can fail, so it comes first), drop one
    reference from the old block, put the new block in the table and queue the
    (old, new) pair for copy_blocks (day-31 `ensure_private_last_block`).
"""
from collections import OrderedDict, deque


class OutOfBlocks(Exception):
    """Not enough free + evictable blocks; the manager's state is unchanged."""


class BlockManager:
    def __init__(self, num_blocks, block_size, enable_prefix_cache=True,
                 initial_free_order=None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.enable_prefix_cache = bool(enable_prefix_cache)
        order = list(range(self.num_blocks)) if initial_free_order is None \
            else [int(b) for b in initial_free_order]
        if sorted(order) != list(range(self.num_blocks)):
            raise ValueError("initial_free_order must be a permutation of the pool")
        self.free_blocks = deque(order)
        self.ref = [0] * self.num_blocks
        self.block_hash = [None] * self.num_blocks
        self.hash_to_block = {}
        self.evictable = OrderedDict()
        self.tables, self.tokens, self.hashes, self.cached = {}, {}, {}, {}
        self.cow_pairs = []

    # -- queries -------------------------------------------------------------
    @property
    def num_free_blocks(self):
        return len(self.free_blocks) + len(self.evictable)

    def can_allocate(self, num_tokens):
        """The coarse check: ceil(n / bs) <= num_free_blocks (ignores hits)."""
        return -(-int(num_tokens) // self.block_size) <= self.num_free_blocks

    def slot(self, seq, pos):
        table = self.tables[seq]
        return table[pos // self.block_size] * self.block_size + pos % self.block_size

    def block_table(self, seq):
        return list(self.tables[seq])

    def num_cached_tokens(self, seq):
        return self.cached[seq]

    def take_cow_pairs(self):
        pairs, self.cow_pairs = self.cow_pairs, []
        return pairs

    # -- helpers -------------------------------------------------------------
    def _chain(self, tokens):
        """Chained hashes of the len // bs full blocks of ``tokens``."""
        bs = self.block_size
        out, parent = [], None
        for i in range(len(tokens) // bs):
            parent = hash((parent, tuple(tokens[i * bs:(i + 1) * bs])))
            out.append(parent)
        return out

    def _take_block(self):
        if self.free_blocks:
            b = self.free_blocks.popleft()
        elif self.evictable:
            b, _ = self.evictable.popitem(last=False)   # oldest end
            h = self.block_hash[b]
            if self.hash_to_block.get(h) == b:
                del self.hash_to_block[h]
            self.block_hash[b] = None
        else:
            raise OutOfBlocks("no free or evictable block")
        self.ref[b] = 1
        return b

    def _register(self, b, h):
        self.block_hash[b] = h
        self.hash_to_block.setdefault(h, b)

    # -- operations ----------------------------------------------------------
    def allocate(self, seq, tokens):
        if seq in self.tables:
            raise ValueError("sequence %r already allocated" % (seq,))
        tokens = [int(t) for t in tokens]
        bs = self.block_size
        n_blocks = -(-len(tokens) // bs)
        # (1) chained hashes of the full blocks only
        chain = self._chain(tokens) if self.enable_prefix_cache else []
        # (2) consecutive hits within the first (len - 1) // bs blocks
        hits = []
        if self.enable_prefix_cache and tokens:
            for h in chain[:(len(tokens) - 1) // bs]:
                b = self.hash_to_block.get(h)
                if b is None:
                    break
                hits.append(b)
        # (3) exact capacity check, before any write
        new_needed = n_blocks - len(hits)
        revived = sum(1 for b in hits if self.ref[b] == 0)
        if new_needed > self.num_free_blocks - revived:
            raise OutOfBlocks("need %d new blocks, %d usable"
                              % (new_needed, self.num_free_blocks - revived))
        # (4) hits leave the evictable pool and gain a reference
        for b in hits:
            if self.ref[b] == 0:
                del self.evictable[b]
            self.ref[b] += 1
        # (5) the rest are taken fresh
        table = hits + [self._take_block() for _ in range(new_needed)]
        # (6) register the full blocks that were not hits
        for i in range(len(hits), len(chain)):
            self._register(table[i], chain[i])
        # (7) per-sequence records
        self.tables[seq] = table
        self.tokens[seq] = tokens
        self.hashes[seq] = chain
        self.cached[seq] = len(hits) * bs
        return list(table)

    def append_slot(self, seq, token):
        bs = self.block_size
        table, toks = self.tables[seq], self.tokens[seq]
        pos = len(toks)
        # (1) take a block first -- the only step that can raise
        if pos // bs == len(table):
            table.append(self._take_block())
        elif self.ref[table[-1]] > 1:
            new = self._take_block()
            old = table[-1]
            self.ref[old] -= 1
            table[-1] = new
            self.cow_pairs.append((old, new))
        # (2) then the token
        toks.append(int(token))
        # (3) a block that just became full is hashed onto the chain and registered
        if self.enable_prefix_cache and (pos + 1) % bs == 0:
            chain = self.hashes[seq]
            h = hash((chain[-1] if chain else None, tuple(toks[pos + 1 - bs:pos + 1])))
            chain.append(h)
            self._register(table[pos // bs], h)
        return self.slot(seq, pos)

    def fork(self, parent, child):
        if child in self.tables:
            raise ValueError("sequence %r already allocated" % (child,))
        self.tables[child] = list(self.tables[parent])
        for b in self.tables[child]:
            self.ref[b] += 1
        self.tokens[child] = list(self.tokens[parent])
        self.hashes[child] = list(self.hashes[parent])
        self.cached[child] = self.cached[parent]

    def free(self, seq):
        table = self.tables.get(seq)
        if table is None:
            return
        for b in reversed(table):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if self.block_hash[b] is not None:
                    self.evictable[b] = None      # newest end
                else:
                    self.free_blocks.append(b)
        for rec in (self.tables, self.tokens, self.hashes, self.cached):
            del rec[seq]

    # -- invariants I1-I5 of the page ----------------------------------------
    def check_invariants(self):
        free_set, ev_set = set(self.free_blocks), set(self.evictable)
        assert len(free_set) == len(self.free_blocks), "duplicate in free list"
        assert not (free_set & ev_set), "I1: free and evictable overlap"
        assert self.num_free_blocks == len(self.free_blocks) + len(self.evictable)
        for b in free_set | ev_set:
            assert self.ref[b] == 0, "I1: block %d free with ref %d" % (b, self.ref[b])
        for b in range(self.num_blocks):
            in_ev = b in ev_set
            assert in_ev == (self.ref[b] == 0 and self.block_hash[b] is not None), \
                "I2 fails for block %d" % b
        for h, b in self.hash_to_block.items():
            assert self.block_hash[b] == h, "I3 fails for hash -> block %d" % b
        counts = [0] * self.num_blocks
        for table in self.tables.values():
            for b in table:
                counts[b] += 1
        assert counts == self.ref, "I4: ref != number of tables holding the block"
        if not self.tables:
            assert self.num_free_blocks == self.num_blocks, "I4: blocks leaked"
        for seq, c in self.cached.items():
            assert c % self.block_size == 0 and (c < len(self.tokens[seq]) or c == 0), \
                "I5 fails for %r" % (seq,)
        # every block is in exactly one place: in use, free or evictable
        in_use = {b for t in self.tables.values() for b in t}
        assert len(in_use | free_set | ev_set) == self.num_blocks
