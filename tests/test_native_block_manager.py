"""The native BlockManager (pkv_bm_*) against the pages' examples and the oracle."""
import random

import pytest

from bm_replay import replay
from conftest import load_golden
from oracle.block_manager import BlockManager as OracleBM
from oracle.block_manager import OutOfBlocks as OracleOOB


@pytest.fixture
def bm_mod(native_lib):
    from paged_kv_cache_138_gb300 import block_manager
    return block_manager


class Ids:
    def __init__(self):
        self.ids = {}

    def __call__(self, name):
        return self.ids.setdefault(name, len(self.ids) + 100)


@pytest.mark.parametrize("name", [
    "blockmanager_example1.json",
    "blockmanager_example2.json",
    "blockmanager_example3.json",
    "blockmanager_eviction_trace.json",
    "blockmanager_duplicate_hash.json",
])
def test_golden_replay_native(bm_mod, name):
    fx = load_golden(name)
    bm = bm_mod.BlockManager(fx["num_blocks"], fx["block_size"], fx.get("enable_prefix_cache", True))
    replay(fx, bm, bm_mod.OutOfBlocks, seq_id=Ids(), check=lambda b: b.check_invariants())


def test_allocate_requests_native(bm_mod):
    fx = load_golden("allocate_requests.json")
    bm = bm_mod.BlockManager(64, fx["block_size"], enable_prefix_cache=False)
    tables = [bm.allocate(i, list(range(L))) for i, L in enumerate(fx["lengths"])]
    assert tables == fx["tables"]
    t, lens = bm.block_tables(range(5), pad=-1)
    assert lens.tolist() == fx["lengths"]
    assert int((t >= 0).sum()) == fx["physical_blocks"]


def test_fork_cow_native(bm_mod):
    bm = bm_mod.BlockManager(16, 4, True)
    bm.allocate(1, [1, 2, 3, 4, 5, 6])
    bm.fork(1, 2)
    assert bm.append_slot(2, 7) == 10
    assert bm.take_cow_pairs() == [(1, 2)]
    assert bm.append_slot(1, 8) == 6 and bm.take_cow_pairs() == []
    bm.check_invariants()


def _apply(bm, oob, op, *args):
    try:
        return ("ok", getattr(bm, op)(*args))
    except oob:
        return ("oob", None)


def test_differential_against_oracle(bm_mod):
    """Random operation streams: native and oracle managers must agree exactly."""
    rnd = random.Random(1234)
    for trial in range(40):
        bs = rnd.choice([2, 4, 16])
        nb = rnd.randint(3, 48)
        prefix = rnd.random() < 0.8
        order = list(range(nb))
        rnd.shuffle(order)
        nat = bm_mod.BlockManager(nb, bs, prefix, initial_free_order=order)
        ora = OracleBM(nb, bs, prefix, initial_free_order=order)
        live, next_id = [], 0
        vocab = rnd.choice([2, 5, 1000])
        for _ in range(250):
            r = rnd.random()
            if r < 0.25 or not live:
                toks = [rnd.randrange(vocab) for _ in range(rnd.randint(0, 5 * bs))]
                a = _apply(nat, bm_mod.OutOfBlocks, "allocate", next_id, toks)
                b = _apply(ora, OracleOOB, "allocate", next_id, toks)
                assert a == b
                if a[0] == "ok":
                    assert nat.num_cached_tokens(next_id) == ora.num_cached_tokens(next_id)
                    live.append(next_id)
                    next_id += 1
            elif r < 0.7:
                seq, tok = rnd.choice(live), rnd.randrange(vocab)
                assert _apply(nat, bm_mod.OutOfBlocks, "append_slot", seq, tok) == \
                    _apply(ora, OracleOOB, "append_slot", seq, tok)
            elif r < 0.8:
                parent = rnd.choice(live)
                nat.fork(parent, next_id)
                ora.fork(parent, next_id)
                live.append(next_id)
                next_id += 1
            else:
                seq = rnd.choice(live)
                nat.free(seq)
                ora.free(seq)
                live.remove(seq)
            assert nat.take_cow_pairs() == ora.take_cow_pairs()
            assert nat.num_free_blocks == ora.num_free_blocks
            assert nat.free_list() == list(ora.free_blocks)
            assert nat.evictable_list() == list(ora.evictable)
            assert nat.ref_counts() == ora.ref
            for s in live:
                assert nat.block_table(s) == ora.block_table(s)
            nat.check_invariants()
            assert nat.can_allocate(bs + 1) == ora.can_allocate(bs + 1)


def test_bad_arguments_native(bm_mod):
    from paged_kv_cache_138_gb300._lib import PagedKVError
    with pytest.raises(ValueError):
        bm_mod.BlockManager(4, 2, True, initial_free_order=[0, 1, 1, 2])
    bm = bm_mod.BlockManager(4, 2, True)
    bm.allocate(1, [1, 2])
    with pytest.raises(PagedKVError):
        bm.allocate(1, [3])            # id in use
    with pytest.raises(PagedKVError):
        bm.append_slot(99, 1)          # unknown sequence
    with pytest.raises(PagedKVError):
        bm.slot(1, 2)                  # position past the table
    bm.free(99)                        # unknown id: ignored
    bm.check_invariants()


def test_utilization_follows_the_allocator_formula(bm_mod):
    """1 - free / num_blocks ("qaqbuyan: vLLM PagedAttention", the block
    allocator), with evictable cached blocks counted as free: an empty pool
    is 0, allocating k of n blocks gives k / n, freeing returns it to 0
    whether the freed blocks are cached (evictable) or not."""
    for cache in (True, False):
        bm = bm_mod.BlockManager(10, 4, enable_prefix_cache=cache)
        assert bm.utilization == 0.0
        bm.allocate(1, list(range(9)))           # 3 blocks
        assert bm.utilization == pytest.approx(0.3)
        bm.allocate(2, list(range(100, 117)))    # 5 blocks
        assert bm.utilization == pytest.approx(0.8)
        bm.free(1)
        assert bm.utilization == pytest.approx(0.5)
        bm.free(2)
        assert bm.utilization == 0.0


def test_negative_capacity_copies_nothing(bm_mod):
    """The C ABI's copy-out calls take a capacity; a negative one copies
    nothing (the count is still returned)."""
    import ctypes
    import numpy as np
    from paged_kv_cache_138_gb300._lib import lib
    bm = bm_mod.BlockManager(8, 2, True)
    bm.allocate(1, [1, 2, 3, 4, 5])
    out = np.full(8, -7, dtype=np.int32)
    p = out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert lib().pkv_bm_block_table(bm._h, 1, p, -1) == 3
    assert lib().pkv_bm_ref_counts(bm._h, p, -5) == 8
    assert (out == -7).all()
    assert lib().pkv_bm_block_table(bm._h, 1, p, 2) == 3
    assert list(out[:3]) == list(bm.block_table(1)[:2]) + [-7]
