"""Builds the metadata of one decode batch with the native BlockManager.

For each workload the op script of ``workloads`` is played on a
``block_manager.BlockManager`` whose free list starts in the workload's shuffled
order, so physical placement is random and FIFO-allocated.  The result is what
the kernels consume: block tables, context lengths, the slot of every new
token and, for the prefix-sharing workload, the copy-on-write pairs.
"""
from dataclasses import dataclass

import numpy as np

from . import workloads as wl
from .block_manager import BlockManager


@dataclass
class DecodeBatch:
    workload: wl.Workload
    num_blocks: int
    block_tables: np.ndarray   # int32 [S, max_blocks], -1 past each table
    context_lens: np.ndarray   # int32 [S], the new token included
    slot_mapping: np.ndarray   # int64 [S], slot of each new token
    cow_pairs: np.ndarray      # int64 [P, 2] (src, dst) for copy_blocks
    manager: BlockManager

    @property
    def num_seqs(self):
        return len(self.context_lens)

    @property
    def max_blocks(self):
        return self.block_tables.shape[1]


def _play(bm, ops):
    for op in ops:
        if op[0] == "allocate":
            bm.allocate(op[1], op[2])
        elif op[0] == "fork":
            bm.fork(op[1], op[2])
        elif op[0] == "append":
            bm.append_slot(op[1], op[2])
        else:
            raise ValueError(op[0])


def _append_batch(bm, ops):
    seqs = np.array([op[1] for op in ops], dtype=np.int64)
    toks = np.array([op[2] for op in ops], dtype=np.int32)
    return bm.append_slots(seqs, toks)


def prepare_batch(w: wl.Workload, max_blocks=None) -> DecodeBatch:
    if w.name == "prefix-sharing":
        nb = wl.pool_blocks(w)
        bm = BlockManager(nb, w.block_size, True, wl.free_order(w, nb))
        sc = wl.prefix_sharing_script(w)
        _play(bm, sc.setup)
        _append_batch(bm, sc.cow_step)
        cow = bm.take_cow_pairs()
        if sc.fill:
            _append_batch(bm, sc.fill)
        if bm.take_cow_pairs():
            raise RuntimeError("unexpected copy-on-write after the first private token")
        slots = _append_batch(bm, sc.step)
    else:
        lens = wl.context_lengths(w)
        nb = wl.pool_blocks(w, lens)
        bm = BlockManager(nb, w.block_size, False, wl.free_order(w, nb))
        sc = wl.decode_script(w, lens)
        _play(bm, sc.setup)
        slots = _append_batch(bm, sc.step)
        cow = []
    tables, lens = bm.block_tables(sc.batch, max_blocks=max_blocks, pad=-1)
    pairs = np.array(cow, dtype=np.int64).reshape(-1, 2)
    return DecodeBatch(w, nb, tables, lens, slots.astype(np.int64), pairs, bm)
