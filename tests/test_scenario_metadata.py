"""Block tables, context lengths, slots and COW pairs of every workload: the
native BlockManager path must equal the oracle's, bit for bit (CPU only)."""
import numpy as np
import pytest

from parity_helpers import oracle_batch
from paged_kv_cache_138_gb300 import workloads as wl


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_native_batch_equals_oracle(native_lib, name):
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    w = wl.WORKLOADS[name]
    nat = prepare_batch(w)
    tables, lens, slots, cow, nb = oracle_batch(w)
    assert nat.num_blocks == nb
    assert np.array_equal(nat.context_lens, lens)
    assert np.array_equal(nat.block_tables, tables)
    assert np.array_equal(nat.slot_mapping, slots)
    assert np.array_equal(nat.cow_pairs, cow)
    nat.manager.check_invariants()


def test_workload_shapes():
    w = wl.WORKLOADS["tiny"]
    assert wl.context_lengths(w).tolist() == [7, 16, 31, 48, 63]
    assert sum(wl.blocks_for(L) for L in wl.context_lengths(w)) == 11
    w = wl.WORKLOADS["gqa-32-8"]
    assert wl.pool_blocks(w) == int(np.ceil(1.1 * 256 * 256))
    w = wl.WORKLOADS["llama2-7b-32layer"]
    assert wl.pool_blocks(w) == 16384
    w = wl.WORKLOADS["prefix-sharing"]
    p = wl.prefix_sharing_private_tokens(w)
    assert len(p) == 128 and p.min() >= 64 and p.max() <= 512
    L = wl.context_lengths(wl.WORKLOADS["llama2-13b-layer"])
    assert L.min() >= 1 and L.max() <= 4096 and len(L) == 64


def test_prefix_sharing_cow_count(native_lib):
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    b = prepare_batch(wl.WORKLOADS["prefix-sharing"])
    # 8 prompts x 15 samples copy the shared partial block; the 16th writes in place
    assert b.cow_pairs.shape == (120, 2)
    assert len(set(b.cow_pairs[:, 1].tolist())) == 120
    assert len(set(b.cow_pairs[:, 0].tolist())) == 8
    # all 16 samples of a prompt share its 128 prompt blocks
    t = b.block_tables
    for j in range(8):
        rows = t[j * 16:(j + 1) * 16, :128]
        assert (rows == rows[0]).all()
