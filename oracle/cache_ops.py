"""TEST INFRASTRUCTURE ONLY: the cache-consistency operations, by definition.

slot          "P06 BlockManager", problem summary: the K/V of token ``pos`` of a
              sequence lives at slot = table[pos // bs] * bs + pos % bs.
reshape_and_cache
              "ans20xx day 31", block-table paragraph: a decoded token is written
              into the last, not-yet-full block of its sequence; with the cache
              laid out [num_blocks, bs, Hkv, D] ("qaqbuyan", `paged_attention`
              docstring) that is row slot % bs of block slot // bs.  Reading where
              the pages are silent: a negative slot means "no write".
copy_blocks   "ans20xx day 31", toy COW append: when a shared block is made
              private the old block's KV bytes are copied into the new one.
              Reading: the whole block is copied, for K and V of every layer,
              pairs applied in order.

All of these move fp16 values as raw 16-bit patterns, so results are compared
bit for bit.
"""
import numpy as np


def slot(table, pos: int, block_size: int) -> int:
    """Physical slot of logical position ``pos`` through ``table``."""
    return int(table[pos // block_size]) * block_size + pos % block_size


def _bits(a):
    a = np.asarray(a)
    return a.view(np.uint16) if a.dtype == np.float16 else a


def reshape_and_cache(k, v, slot_mapping, k_cache, v_cache):
    """Write k[i], v[i] ([T, Hkv, D]) at slot_mapping[i] of the caches, in place.

    k_cache/v_cache: [num_blocks, bs, Hkv, D].  Raises IndexError on a slot past
    the pool, like the kernel's error status.
    """
    kb, vb = _bits(k), _bits(v)
    kcb, vcb = _bits(k_cache), _bits(v_cache)
    num_blocks, bs = kcb.shape[0], kcb.shape[1]
    for i, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        if s >= num_blocks * bs:
            raise IndexError("slot %d outside a pool of %d slots" % (s, num_blocks * bs))
        block, offset = divmod(s, bs)
        kcb[block, offset] = kb[i]
        vcb[block, offset] = vb[i]


def copy_blocks(k_caches, v_caches, pairs):
    """For every (src, dst) in order and every layer: cache[dst] = cache[src]."""
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2).tolist():
        for kc, vc in zip(k_caches, v_caches):
            kcb, vcb = _bits(kc), _bits(vc)
            n = kcb.shape[0]
            if not (0 <= src < n and 0 <= dst < n):
                raise IndexError("block pair (%d, %d) outside a pool of %d" % (src, dst, n))
            kcb[dst] = kcb[src]
            vcb[dst] = vcb[src]
