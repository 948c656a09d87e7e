"""TEST INFRASTRUCTURE ONLY: the oracle's own decode-batch metadata.

Plays a workload's op script (from the shared seeded generator) on the oracle
BlockManager and returns block tables, context lengths, the slot of every new
token (by the page's slot formula) and the copy-on-write pairs.
"""
import numpy as np

from paged_kv_cache_138_gb300 import workloads as wl

from . import cache_ops
from .block_manager import BlockManager


def _play(bm, ops):
    slots = []
    for op in ops:
        if op[0] == "allocate":
            bm.allocate(op[1], op[2])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        else:
            slots.append(bm.append_slot(op[1], op[2]))
    return slots


def oracle_batch(w):
    """(tables [S, max_blocks] padded with -1, context lens, new-token slots,
    cow pairs [P, 2], pool size)."""
    if w.name == "prefix-sharing":
        nb = wl.pool_blocks(w)
        bm = BlockManager(nb, w.block_size, True, wl.free_order(w, nb))
        sc = wl.prefix_sharing_script(w)
        _play(bm, sc.setup)
        _play(bm, sc.cow_step)
        cow = bm.take_cow_pairs()
        _play(bm, sc.fill)
        slots = _play(bm, sc.step)
    else:
        lens = wl.context_lengths(w)
        nb = wl.pool_blocks(w, lens)
        bm = BlockManager(nb, w.block_size, False, wl.free_order(w, nb))
        sc = wl.decode_script(w, lens)
        _play(bm, sc.setup)
        slots = _play(bm, sc.step)
        cow = []
    tabs = [bm.block_table(s) for s in sc.batch]
    mb = max(len(t) for t in tabs)
    tables = np.full((len(tabs), mb), -1, dtype=np.int32)
    for i, t in enumerate(tabs):
        tables[i, :len(t)] = t
    lens = np.array([len(bm.tokens[s]) for s in sc.batch], dtype=np.int32)
    for i in range(len(sc.batch)):
        if slots[i] != cache_ops.slot(tabs[i], int(lens[i]) - 1, w.block_size):
            raise AssertionError("append_slot disagrees with the slot formula")
    return (tables, lens, np.array(slots, dtype=np.int64),
            np.array(cow, dtype=np.int64).reshape(-1, 2), nb)
