"""The native continuous-batching scheduler's host logic, step by step against a
plain Python statement of the same policy running on the oracle BlockManager
(CPU only: no kernel is launched)."""
import ctypes
from collections import deque

import numpy as np
import pytest

from oracle.block_manager import BlockManager as OracleBM
from oracle.block_manager import OutOfBlocks
from paged_kv_cache_138_gb300 import workloads as wl

MASK64 = (1 << 64) - 1


def mix64(z):
    z = (z + 0x9E3779B97F4A7C15) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def sample(seed, rid, pos, vocab=32000):
    return mix64(seed ^ mix64((rid * 0x100000001B3 + pos) & MASK64)) % vocab


class RefScheduler:
    """Finish -> admit FCFS -> one append per running request; on OutOfBlocks
    preempt the not-yet-decoded request with the most generated tokens
    (recompute, or swap into FIFO host blocks)."""

    def __init__(self, bm, max_batch, bs, swap, host_blocks, seed):
        self.bm, self.max_batch, self.bs, self.swap, self.seed = bm, max_batch, bs, swap, seed
        self.reqs, self.waiting, self.running = {}, deque(), []
        self.host_free = deque(range(host_blocks))

    def add(self, rid, prompt, max_new):
        self.reqs[rid] = {"tokens": list(prompt), "max_new": max_new, "gen": 0, "host": None}
        self.waiting.append(rid)

    def step(self):
        out = {"finished": 0, "admitted": 0, "preempted": 0, "prefill": [], "swap_in": [],
               "swap_out": [], "batch": [], "cached": 0}
        for rid in [r for r in self.running if self.reqs[r]["gen"] >= self.reqs[r]["max_new"]]:
            self.bm.free(rid)
            self.running.remove(rid)
            out["finished"] += 1
        while self.waiting and len(self.running) < self.max_batch:
            rid = self.waiting[0]
            r = self.reqs[rid]
            try:
                table = self.bm.allocate(rid, r["tokens"])
            except OutOfBlocks:
                break
            self.waiting.popleft()
            cached = self.bm.num_cached_tokens(rid)
            out["cached"] += cached
            if r["host"] is not None:
                for i in range(cached // self.bs, len(r["host"])):
                    out["swap_in"].append((r["host"][i], table[i]))
                self.host_free.extend(r["host"])
                r["host"] = None
            else:
                for pos in range(cached, len(r["tokens"])):
                    out["prefill"].append((rid, pos, table[pos // self.bs] * self.bs + pos % self.bs))
            self.running.append(rid)
            out["admitted"] += 1
        pending, done = list(self.running), set()
        i = 0
        while i < len(pending):
            rid = pending[i]
            r = self.reqs[rid]
            pos = len(r["tokens"])
            tok = sample(self.seed, rid, pos)
            try:
                slot = self.bm.append_slot(rid, tok)
            except OutOfBlocks:
                cands = [x for x in self.running if x not in done]
                victim = max(cands, key=lambda x: self.reqs[x]["gen"])  # first max wins
                v = self.reqs[victim]
                if self.swap:
                    table = self.bm.block_table(victim)
                    used = -(-len(v["tokens"]) // self.bs)
                    if len(self.host_free) >= used:
                        v["host"] = [self.host_free.popleft() for _ in range(used)]
                        out["swap_out"].extend(zip(table[:used], v["host"]))
                self.bm.free(victim)
                self.running.remove(victim)
                self.waiting.appendleft(victim)
                out["preempted"] += 1
                if victim == rid:
                    i += 1
                else:
                    pending.remove(victim)
                continue
            r["tokens"].append(tok)
            r["gen"] += 1
            out["batch"].append((rid, pos, tok, slot))
            done.add(rid)
            i += 1
        return out


@pytest.mark.parametrize("swap", [False, True])
def test_native_scheduler_matches_reference_policy(native_lib, swap):
    from paged_kv_cache_138_gb300._lib import lib
    from paged_kv_cache_138_gb300.block_manager import BlockManager
    from paged_kv_cache_138_gb300.serving import _StepOut
    seed, bs, nb, B, mb = 9, 16, 22, 6, 8
    order = np.random.default_rng(9).permutation(nb)
    bm = BlockManager(nb, bs, True, order)
    h = lib().pkv_sched_create(bm._h, B, mb, bs, 1 if swap else 0, 64, ctypes.c_uint64(seed),
                               32000)
    ref = RefScheduler(OracleBM(nb, bs, True, order), B, bs, swap, 64, seed)
    reqs = wl.serving_requests(seed, num_requests=18, num_system_prompts=3,
                               system_prompt_len=40, suffix_max=12, new_min=3, new_max=60)
    for r in reqs:
        p = np.array(r.prompt, np.int32)
        assert lib().pkv_sched_add_request(h, r.rid, p.ctypes.data_as(ctypes.c_void_p), len(p),
                                           r.max_new_tokens) == 0
        ref.add(r.rid, r.prompt, r.max_new_tokens)
    arrs = {
        "batch_rids": np.zeros(B, np.int64), "positions": np.zeros(B, np.int32),
        "tokens": np.zeros(B, np.int32), "slots": np.zeros(B, np.int64),
        "block_tables": np.zeros((B, mb), np.int32), "context_lens": np.zeros(B, np.int32),
        "prefill_rids": np.zeros(B * mb * bs, np.int64),
        "prefill_positions": np.zeros(B * mb * bs, np.int32),
        "prefill_slots": np.zeros(B * mb * bs, np.int64),
        "swap_in_pairs": np.zeros((B * mb, 2), np.int64),
        "swap_out_pairs": np.zeros((B * mb, 2), np.int64),
        "cow_pairs": np.zeros((B, 2), np.int64),
    }
    o = _StepOut()
    for k, a in arrs.items():
        setattr(o, k, a.ctypes.data_as(ctypes.c_void_p))
    o.prefill_cap, o.swap_cap, o.cow_cap, o.group_limit = B * mb * bs, B * mb, B, 0
    steps = preempted = 0
    while lib().pkv_sched_num_unfinished(h) > 0:
        assert lib().pkv_sched_step(h, ctypes.byref(o)) == 0
        exp = ref.step()
        steps += 1
        assert steps < 500
        assert (o.num_finished, o.num_admitted, o.num_preempted, o.cached_tokens) == \
            (exp["finished"], exp["admitted"], exp["preempted"], exp["cached"])
        n = o.num_prefill
        got_pf = list(zip(arrs["prefill_rids"][:n].tolist(), arrs["prefill_positions"][:n].tolist(),
                          arrs["prefill_slots"][:n].tolist()))
        assert got_pf == exp["prefill"]
        assert [tuple(x) for x in arrs["swap_in_pairs"][:o.num_swap_in].tolist()] == exp["swap_in"]
        assert [tuple(x) for x in arrs["swap_out_pairs"][:o.num_swap_out].tolist()] == \
            exp["swap_out"]
        Bn = o.num_batch
        got = list(zip(arrs["batch_rids"][:Bn].tolist(), arrs["positions"][:Bn].tolist(),
                       arrs["tokens"][:Bn].tolist(), arrs["slots"][:Bn].tolist()))
        assert got == exp["batch"]
        for b, (rid, pos, _, _) in enumerate(exp["batch"]):
            assert arrs["context_lens"][b] == pos + 1
            t = ref.bm.block_table(rid)
            assert arrs["block_tables"][b, :len(t)].tolist() == t
        preempted += o.num_preempted
        bm.check_invariants()
    assert preempted > 0
    assert bm.num_free_blocks == nb
    lib().pkv_sched_destroy(h)


def test_request_tokens_negative_capacity_copies_nothing(native_lib):
    from paged_kv_cache_138_gb300._lib import lib
    from paged_kv_cache_138_gb300.block_manager import BlockManager
    bm = BlockManager(8, 16, True)
    h = lib().pkv_sched_create(bm._h, 2, 4, 16, 0, 0, ctypes.c_uint64(1), 100)
    try:
        p = np.array([5, 6, 7], np.int32)
        assert lib().pkv_sched_add_request(h, 3, p.ctypes.data_as(ctypes.c_void_p), 3, 2) == 0
        out = np.full(4, -7, np.int32)
        q = out.ctypes.data_as(ctypes.c_void_p)
        assert lib().pkv_sched_request_tokens(h, 3, q, -1) == 3
        assert (out == -7).all()
        assert lib().pkv_sched_request_tokens(h, 3, q, 2) == 3
        assert list(out) == [5, 6, -7, -7]
    finally:
        lib().pkv_sched_destroy(h)
