"""Pins the oracle BlockManager to the pages' worked examples and invariants."""
import copy
import random

import pytest

from bm_replay import OracleAdapter, replay
from conftest import load_golden
from oracle.block_manager import BlockManager, OutOfBlocks


def make(fx):
    return OracleAdapter(BlockManager(fx["num_blocks"], fx["block_size"],
                                      fx.get("enable_prefix_cache", True)))


@pytest.mark.parametrize("name", [
    "blockmanager_example1.json",
    "blockmanager_example2.json",
    "blockmanager_example3.json",
    "blockmanager_eviction_trace.json",
    "blockmanager_duplicate_hash.json",
])
def test_golden_replay(name):
    fx = load_golden(name)
    bm = make(fx)
    replay(fx, bm, OutOfBlocks, check=lambda b: b.bm.check_invariants())


def test_key_questions():
    fx = load_golden("blockmanager_key_questions.json")
    bs = fx["block_size"]
    for case in fx["cases"]:
        n = case["tokens"]
        bm = BlockManager(16, bs, True)
        toks = list(range(100, 100 + n))
        assert len(bm._chain(toks)) == case["full_blocks"]
        table = bm.allocate("p", toks)
        assert len(table) == case["blocks"]
        bm.free("p")
        # re-allocating the same prompt hits at most (n - 1) // bs blocks
        bm.allocate("q", toks)
        assert bm.num_cached_tokens("q") == case["matchable"] * bs
        if "cached_if_all_hit" in case:
            assert bm.num_cached_tokens("q") == case["cached_if_all_hit"]
        bm.check_invariants()


def test_chain_hash_depends_on_prefix():
    # "two blocks both [7, 8], one after [1, 2], one after [5, 6]: same hash? no"
    bm = BlockManager(8, 2, True)
    assert bm._chain([1, 2, 7, 8])[1] != bm._chain([5, 6, 7, 8])[1]
    bm.allocate("a", [1, 2, 7, 8, 9])
    bm.allocate("b", [5, 6, 7, 8, 9])
    assert bm.num_cached_tokens("b") == 0
    bm.check_invariants()


def test_allocate_requests_tables():
    fx = load_golden("allocate_requests.json")
    bs = fx["block_size"]
    bm = BlockManager(64, bs, enable_prefix_cache=False)
    tables = [bm.allocate(i, list(range(L))) for i, L in enumerate(fx["lengths"])]
    assert tables == fx["tables"]
    assert sum(len(t) for t in tables) == fx["physical_blocks"]
    waste = sum(len(t) * bs - L for t, L in zip(tables, fx["lengths"]))
    assert waste == fx["tail_waste_tokens"]
    bm.check_invariants()


def test_self_check_shared_block_free_twice():
    # share a block between two sequences, free one, then the other: the first
    # free returns only the blocks that were not shared
    bm = BlockManager(8, 2, True)
    bm.allocate("a", [1, 2, 3, 4, 5])          # [0, 1, 2]
    bm.allocate("b", [1, 2, 3, 4, 6])          # [0, 1, 3], shares 0 and 1
    before = bm.num_free_blocks
    bm.free("a")
    assert bm.num_free_blocks == before + 1    # only block 2 was private
    bm.check_invariants()
    bm.free("b")
    assert bm.num_free_blocks == 8
    bm.check_invariants()


def test_last_token_never_hits_and_full_prompt():
    bm = BlockManager(8, 4, True)
    bm.allocate("a", list(range(8)))
    bm.free("a")
    bm.allocate("b", list(range(8)))
    assert bm.num_cached_tokens("b") == 4       # (8-1)//4 = 1 block, never all
    bm.check_invariants()


def test_prefix_cache_off_never_caches():
    bm = BlockManager(8, 2, enable_prefix_cache=False)
    bm.allocate("a", [1, 2, 3, 4])
    bm.free("a")
    assert list(bm.evictable) == [] and len(bm.free_blocks) == 8
    bm.allocate("b", [1, 2, 3, 4, 5])
    assert bm.num_cached_tokens("b") == 0
    bm.check_invariants()


def test_append_filled_block_is_cached_then_hit():
    bm = BlockManager(8, 2, True)
    bm.allocate("a", [7, 8, 9])
    bm.append_slot("a", 10)
    bm.free("a")
    bm.allocate("b", [7, 8, 9, 10, 11])
    assert bm.num_cached_tokens("b") == 4
    bm.check_invariants()


def test_append_out_of_blocks_is_atomic():
    bm = BlockManager(2, 2, True)
    bm.allocate("a", [1, 2, 3, 4])
    state = copy.deepcopy(bm.__dict__)
    with pytest.raises(OutOfBlocks):
        bm.append_slot("a", 5)
    assert bm.__dict__ == state


def test_fork_and_copy_on_write():
    # ans20xx day 31: a fork shares every block; a write into the shared partial
    # last block takes a private copy, the last holder writes in place
    bm = BlockManager(16, 4, True)
    bm.allocate("p", [1, 2, 3, 4, 5, 6])      # [0, 1], block 1 partial
    bm.fork("p", "c")
    assert bm.ref[0] == 2 and bm.ref[1] == 2
    bm.check_invariants()
    s = bm.append_slot("c", 7)
    assert bm.block_table("c") == [0, 2] and s == 2 * 4 + 2
    assert bm.take_cow_pairs() == [(1, 2)]
    assert bm.ref[1] == 1 and bm.ref[2] == 1
    s = bm.append_slot("p", 8)                 # ref 1 now: in place, no copy
    assert s == 1 * 4 + 2 and bm.take_cow_pairs() == []
    bm.check_invariants()
    # a fork at a block boundary never copies: the next token opens a new block
    bm.append_slot("p", 9)                     # block 1 full
    bm.fork("p", "d")
    bm.append_slot("d", 10)
    assert bm.take_cow_pairs() == [] and bm.block_table("d")[:2] == [0, 1]
    bm.check_invariants()
    for seq in ("p", "c", "d"):
        bm.free(seq)
    bm.check_invariants()
    assert bm.num_free_blocks == 16


def test_cow_out_of_blocks_is_atomic():
    bm = BlockManager(2, 4, True)
    bm.allocate("p", [1, 2, 3, 4, 5])          # [0, 1]
    bm.fork("p", "c")
    state = copy.deepcopy(bm.__dict__)
    with pytest.raises(OutOfBlocks):
        bm.append_slot("c", 6)
    assert bm.__dict__ == state


def test_random_ops_keep_invariants():
    rnd = random.Random(7)
    for trial in range(30):
        bs = rnd.choice([2, 4, 16])
        bm = BlockManager(rnd.randint(4, 40), bs, rnd.random() < 0.8,
                          initial_free_order=None)
        live, next_id = [], 0
        vocab = rnd.choice([3, 50])
        for _ in range(200):
            r = rnd.random()
            try:
                if r < 0.3 or not live:
                    n = rnd.randint(0, 4 * bs)
                    toks = [rnd.randrange(vocab) for _ in range(n)]
                    bm.allocate(next_id, toks)
                    live.append(next_id)
                    next_id += 1
                elif r < 0.65:
                    bm.append_slot(rnd.choice(live), rnd.randrange(vocab))
                elif r < 0.75:
                    bm.fork(rnd.choice(live), next_id)
                    live.append(next_id)
                    next_id += 1
                else:
                    seq = rnd.choice(live)
                    bm.free(seq)
                    live.remove(seq)
            except OutOfBlocks:
                pass
            bm.check_invariants()
        for seq in live:
            bm.free(seq)
        bm.check_invariants()
