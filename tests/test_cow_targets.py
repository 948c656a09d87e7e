"""pkv_cow_targets (host, native): copy-on-write pairs -> the per-sequence
(logical block, source) arrays of the fused launches' folded copy.

Pinned against the BlockManager's own copy-on-write: forked samples appending
into a shared partial block ("ans20xx day 31", fork and copy-on-write) produce
pairs whose dst sits in exactly one table, at the block the sample's append
went to.
"""
import numpy as np
import pytest

from paged_kv_cache_138_gb300 import workloads as wl


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def test_targets_of_the_block_managers_copy_on_write(ops):
    from paged_kv_cache_138_gb300.block_manager import BlockManager
    bm = BlockManager(64, 16, False, None)
    bm.allocate(0, list(range(21)))                 # 2 blocks, the second partial
    for k in range(1, 4):
        bm.fork(0, k)
    slots = [bm.append_slot(k, 100 + k) for k in range(4)]
    pairs = bm.take_cow_pairs()
    assert len(pairs) == 3                          # samples 0-2 copy, 3 writes in place
    tables, lens = bm.block_tables(list(range(4)), pad=-1)
    cb, cs = ops.cow_targets(pairs, tables)
    for k in range(4):
        if cb[k] >= 0:
            src, dst = next((s, d) for s, d in pairs if d == tables[k][cb[k]])
            assert cs[k] == src
            # the copy is the block the append wrote into
            assert slots[k] // 16 == tables[k][cb[k]]
    assert sorted(int(c) for c in cs if c >= 0) == sorted(int(s) for s, _ in pairs)
    assert (cb >= 0).sum() == 3


def test_no_pairs_and_errors(ops):
    from paged_kv_cache_138_gb300._lib import PagedKVError
    tables = np.array([[3, 4, -1], [5, 6, 7]], np.int32)
    cb, cs = ops.cow_targets(np.zeros((0, 2), np.int64), tables)
    assert (cb == -1).all() and (cs == -1).all()
    cb, cs = ops.cow_targets([[9, 6]], tables)
    assert list(cb) == [-1, 1] and list(cs) == [-1, 9]
    with pytest.raises(PagedKVError) as e:          # dst in no table
        ops.cow_targets([[9, 11]], tables)
    assert e.value.status == -5
    with pytest.raises(PagedKVError) as e:          # dst in two tables
        ops.cow_targets([[9, 4]], np.array([[3, 4], [4, 5]], np.int32))
    assert e.value.status == -5
    with pytest.raises(PagedKVError) as e:          # two copies for one sequence
        ops.cow_targets([[9, 6], [10, 7]], tables)
    assert e.value.status == -2


def test_prefix_sharing_workload_targets(ops):
    """The prefix-sharing workload's 120 pairs land one per forked sample,
    on the first block past the 2048-token prompt (logical block 128)."""
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    batch = prepare_batch(wl.WORKLOADS["prefix-sharing"])
    cb, cs = ops.cow_targets(batch.cow_pairs, batch.block_tables)
    assert (cb >= 0).sum() == 120 and set(cb[cb >= 0].tolist()) == {128}
    # sample 15 of each prompt wrote in place
    assert (cb.reshape(8, 16)[:, 15] == -1).all()
