"""The multi-step continuous-batching driver against the oracle, every step.

A small serving trace (shared system prompts, so prefix-cache hits; a pool too
small for the batch, so preemption and eviction) runs until every request has
finished.  After each step every decoded row is compared with the fp64 oracle's
attention over that request's full token history, whose K/V and queries come
from the same content-keyed generator.  The BlockManager operations the driver
made are then replayed on the oracle BlockManager, which must return the same
tables, slots, cache hits and OutOfBlocks outcomes.
"""
import numpy as np
import pytest

from oracle import attention as oa
from oracle.block_manager import BlockManager as OracleBM
from oracle.block_manager import OutOfBlocks as OracleOOB
from parity_helpers import assert_matches_oracle
from paged_kv_cache_138_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
SEED, HQ, HKV, BS, D = 5, 4, 2, 16, 128


def oracle_row(tokens, rid, pos):
    toks = tokens[:pos + 1]
    k, v = wl.token_kv_host(wl.prefix_keys(toks, SEED), HKV, D)
    n = len(toks)
    nb = -(-n // BS)
    kc = np.zeros((nb * BS, HKV, D), np.float16)
    vc = np.zeros_like(kc)
    kc[:n], vc[:n] = k, v
    q = wl.step_query_host(SEED, rid, pos, HQ, D)[None]
    return oa.paged_attention_decode(q, kc.reshape(nb, BS, HKV, D), vc.reshape(nb, BS, HKV, D),
                                     np.arange(nb, dtype=np.int32)[None],
                                     np.array([n], np.int32), 1 / np.sqrt(D))[0]


def replay_on_oracle(log, num_blocks, order):
    bm = OracleBM(num_blocks, BS, True, order)
    for e in log:
        if e[0] == "allocate":
            _, rid, toks, cached = e
            try:
                bm.allocate(rid, list(toks))
                assert cached is not None and bm.num_cached_tokens(rid) == cached, e[:2]
            except OracleOOB:
                assert cached is None, e[:2]
        elif e[0] == "append":
            _, rid, tok, slot = e
            try:
                assert bm.append_slot(rid, tok) == slot, e
            except OracleOOB:
                assert slot is None, e
        elif e[0] == "free":
            bm.free(e[1])
        elif e[0] == "cow":
            assert [tuple(p) for p in bm.take_cow_pairs()] == list(e[1])
        bm.check_invariants()
    return bm


@pytest.mark.parametrize("preemption,grouped", [("recompute", False), ("swap", False),
                                                 ("recompute", True)])
def test_driver_matches_oracle_every_step(native_lib, preemption, grouped):
    from paged_kv_cache_138_gb300.driver import ContinuousBatchDriver, HostSources
    reqs = wl.serving_requests(SEED, num_requests=18, num_system_prompts=3,
                               system_prompt_len=40, suffix_max=12, new_min=3, new_max=60)
    nb = 22
    order = np.random.default_rng(9).permutation(nb).astype(np.int32)
    drv = ContinuousBatchDriver(nb, HQ, HKV, max_batch=6, max_blocks_per_seq=8,
                                sources=HostSources(SEED, HQ, HKV, D), free_order=order,
                                record_ops=True, preemption=preemption, host_blocks=64,
                                grouped=grouped)
    for r in reqs:
        drv.add_request(r.rid, r.prompt, r.max_new_tokens)
    got_rows, ref_rows, steps = [], [], 0
    cached = preempted = shared_rows = 0
    while not drv.idle:
        res = drv.step()
        steps += 1
        assert steps < 400
        cached += res.cached_tokens
        shared_rows += res.shared_tokens
        preempted += len(res.preempted)
        if not res.rids:
            continue
        out = res.out.cpu().numpy().astype(np.float64)
        for i, (rid, pos) in enumerate(zip(res.rids, res.positions)):
            got_rows.append(out[i])
            ref_rows.append(oracle_row(drv.requests[rid].tokens, rid, pos))
    drv.check_errors()
    rows = len(got_rows)
    assert_matches_oracle(np.stack(got_rows), np.stack(ref_rows))
    assert all(r.done for r in drv.requests.values())
    assert rows == sum(r.max_new_tokens for r in reqs)   # every token decoded once
    assert cached > 0, "the trace should hit the prefix cache"
    assert preempted > 0, "the pool is sized to force preemption"
    if grouped:
        assert shared_rows > 0, "requests on one system prompt should be grouped"
    if preemption == "swap":
        assert drv.swapped_out_blocks > 0 and drv.swapped_in_blocks > 0
        assert len(drv.host_free) == 64
    bm = replay_on_oracle(drv.ops_log, nb, order)
    assert bm.num_free_blocks == nb
