"""Python face of the native BlockManager (pkv_bm_* in libpagedkv.so)."""
import ctypes

import numpy as np

from ._lib import PKV_ERR_OUT_OF_BLOCKS, PKV_OK, PagedKVError, check, lib


class OutOfBlocks(PagedKVError):
    """Not enough free + evictable blocks; the manager's state is unchanged."""


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class BlockManager:
    """Free list (FIFO), ref counts, chained-hash prefix cache, LRU evictable pool,
    atomic allocate/append, fork + copy-on-write.  Host-only, single-threaded."""

    def __init__(self, num_blocks, block_size=16, enable_prefix_cache=True,
                 initial_free_order=None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = None if initial_free_order is None else _i32(initial_free_order)
        self._h = lib().pkv_bm_create(self.num_blocks, self.block_size,
                                      1 if enable_prefix_cache else 0,
                                      _p(order) if order is not None else None)
        if not self._h:
            raise ValueError("pkv_bm_create rejected its arguments")
        self._keep = order

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().pkv_bm_destroy(h)
            self._h = None

    def _check(self, rc, what):
        if rc == PKV_ERR_OUT_OF_BLOCKS:
            raise OutOfBlocks(rc, what)
        return check(rc, what)

    def allocate(self, seq, tokens):
        """Blocks for a new sequence's prompt: the physical block table (list of
        ints).  Leading full blocks found in the prefix cache (at most
        (len - 1) // block_size of them) are reused; raises OutOfBlocks with
        the state unchanged when the pool cannot hold the rest."""
        toks = _i32(tokens)
        cap = -(-len(toks) // self.block_size)
        table = np.empty(max(cap, 1), dtype=np.int32)
        nt, nc = ctypes.c_int64(), ctypes.c_int64()
        rc = lib().pkv_bm_allocate(self._h, int(seq), _p(toks), len(toks), _p(table), cap,
                                   ctypes.byref(nt), ctypes.byref(nc))
        self._check(rc, "allocate")
        return table[:nt.value].tolist()

    def append_slot(self, seq, token):
        """Append one token: the slot (block * block_size + offset) it goes to.
        Takes a new block when the last is full, or a private copy of a shared
        last block (copy-on-write, pair queued for take_cow_pairs); raises
        OutOfBlocks with the state unchanged."""
        slot = ctypes.c_int64()
        self._check(lib().pkv_bm_append_slot(self._h, int(seq), int(token), ctypes.byref(slot)),
                    "append_slot")
        return slot.value

    def append_slots(self, seqs, tokens):
        """One append per listed sequence, in order; returns int64 slots."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        toks = _i32(tokens)
        slots = np.empty(len(seqs), dtype=np.int64)
        done = ctypes.c_int64()
        rc = lib().pkv_bm_append_slots(self._h, _p(seqs), _p(toks), len(seqs), _p(slots),
                                       ctypes.byref(done))
        self._check(rc, "append_slots (%d done)" % done.value)
        return slots

    def append_slots_partial(self, seqs, tokens):
        """Like append_slots, but stops at the first failure instead of raising:
        returns (slots int64 [n], number appended, status of the failing append
        or PKV_OK)."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        toks = _i32(tokens)
        slots = np.empty(len(seqs), dtype=np.int64)
        done = ctypes.c_int64()
        rc = lib().pkv_bm_append_slots(self._h, _p(seqs), _p(toks), len(seqs), _p(slots),
                                       ctypes.byref(done))
        return slots, int(done.value), int(rc)

    def fork(self, parent, child):
        """child shares every block of parent (reference counts + 1)."""
        self._check(lib().pkv_bm_fork(self._h, int(parent), int(child)), "fork")

    def free(self, seq):
        """Release a sequence's blocks, last first: hashed blocks whose count
        drops to 0 join the evictable pool, the others the free list."""
        self._check(lib().pkv_bm_free(self._h, int(seq)), "free")

    def slot(self, seq, pos):
        """table[pos // block_size] * block_size + pos % block_size."""
        out = ctypes.c_int64()
        self._check(lib().pkv_bm_slot(self._h, int(seq), int(pos), ctypes.byref(out)), "slot")
        return out.value

    @property
    def num_free_blocks(self):
        """Blocks an allocation may take: the free list plus the evictable pool."""
        return int(lib().pkv_bm_num_free_blocks(self._h))

    @property
    def utilization(self):
        """Share of the pool in use: 1 - free / num_blocks ("qaqbuyan: vLLM
        PagedAttention", the block allocator's utilisation), free counting
        the evictable cached blocks an allocation may reclaim; 0 for an empty
        pool."""
        if self.num_blocks == 0:
            return 0.0
        return 1.0 - self.num_free_blocks / self.num_blocks

    def can_allocate(self, num_tokens):
        """The coarse check ceil(num_tokens / block_size) <= num_free_blocks
        (prefix-cache hits not counted)."""
        return bool(lib().pkv_bm_can_allocate(self._h, int(num_tokens)))

    def block_table(self, seq):
        """The sequence's physical block ids, logical order."""
        n = lib().pkv_bm_block_table(self._h, int(seq), None, 0)
        if n < 0:
            raise PagedKVError(int(n), "block_table")
        out = np.empty(max(n, 1), dtype=np.int32)
        lib().pkv_bm_block_table(self._h, int(seq), _p(out), n)
        return out[:n].tolist()

    def num_tokens(self, seq):
        """Tokens the sequence holds (prompt + appended)."""
        n = lib().pkv_bm_num_tokens(self._h, int(seq))
        if n < 0:
            raise PagedKVError(int(n), "num_tokens")
        return int(n)

    def num_cached_tokens(self, seq):
        """Prompt tokens its allocate found in the prefix cache (a multiple of
        block_size)."""
        n = lib().pkv_bm_num_cached_tokens(self._h, int(seq))
        if n < 0:
            raise PagedKVError(int(n), "num_cached_tokens")
        return int(n)

    def block_tables(self, seqs, max_blocks=None, pad=-1):
        """int32 [n, max_blocks] tables and int32 [n] token counts of ``seqs``."""
        seqs = np.ascontiguousarray(seqs, dtype=np.int64)
        if max_blocks is None:
            max_blocks = max([lib().pkv_bm_block_table(self._h, int(s), None, 0) for s in seqs]
                             + [1])
        tables = np.empty((len(seqs), max_blocks), dtype=np.int32)
        lens = np.empty(len(seqs), dtype=np.int32)
        rc = lib().pkv_bm_fill_block_tables(self._h, _p(seqs), len(seqs), _p(tables), max_blocks,
                                            int(pad), _p(lens))
        self._check(rc, "block_tables")
        return tables, lens

    def take_cow_pairs(self):
        """The (src, dst) block pairs queued by copy-on-write appends since the
        last call, for copy_blocks; the queue is emptied."""
        n = lib().pkv_bm_take_cow_pairs(self._h, None, 0)
        out = np.empty((max(n, 1), 2), dtype=np.int64)
        lib().pkv_bm_take_cow_pairs(self._h, _p(out), n)
        return [tuple(r) for r in out[:n].tolist()]

    def _list(self, fn):
        n = fn(self._h, None, 0)
        out = np.empty(max(n, 1), dtype=np.int32)
        fn(self._h, _p(out), n)
        return out[:n].tolist()

    def free_list(self):
        return self._list(lib().pkv_bm_free_list)

    def evictable_list(self):
        return self._list(lib().pkv_bm_evictable_list)

    def ref_counts(self):
        return self._list(lib().pkv_bm_ref_counts)

    def check_invariants(self):
        rc = lib().pkv_bm_check_invariants(self._h)
        if rc != PKV_OK:
            raise AssertionError("BlockManager invariant I%d violated" % rc)
