"""Multi-step decode over a changing batch: continuous batching without a model.

What a step does follows "qaqbuyan: vLLM PagedAttention" (continuous batching
timeline and `ContinuousBatchingScheduler.step`) and the scheduling paragraph
of "ans20xx day 31":

1. requests that produced their last token release their blocks (reverse-order
   free; hashed full blocks stay in the LRU pool and can be hit again);
2. waiting requests are admitted first-come first-served while the
   BlockManager can allocate them; prefix-cache hits skip part of the prompt
   and the KV of the remaining prompt tokens is written (reshape_and_cache);
3. every running request decodes one token: `append_slot` (a new block at a
   block boundary, a private copy when the partial block is shared), then
   copy_blocks for the copy-on-write pairs, reshape_and_cache of the new
   token's K/V and paged decode attention over the whole batch.

When `append_slot` finds no block, a running request is preempted: of those
that have not yet decoded in this step, the one with the most generated tokens
(p1 `_preempt_request` picks by that count).  Its blocks are freed and it goes
back to the front of the queue with all its tokens.  With preemption="recompute"
its prompt is prefilled again on re-admission (the prefix cache often still
holds most of it); with preemption="swap" its blocks are first copied to pinned
host memory (swap_blocks) and copied back into its new blocks on re-admission.

There is no model: next tokens, queries and K/V come from ``sources``, which
must give the same K/V for the same token prefix (as a model would).  Every
device operation goes through the C ABI; the host side is the native
BlockManager.
"""
from collections import deque
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

from . import ops
from .block_manager import BlockManager, OutOfBlocks


@dataclass(eq=False)
class Request:
    rid: int
    tokens: List[int]
    max_new_tokens: int
    generated: int = 0
    preemptions: int = 0
    swapped: Optional[List[int]] = None   # host blocks holding its KV while swapped out

    @property
    def done(self):
        return self.generated >= self.max_new_tokens


@dataclass
class StepResult:
    rids: List[int]
    positions: List[int]           # position of the token decoded for each rid
    out: torch.Tensor              # fp16 [B, Hq, D] (device; valid until the next step)
    admitted: List[int] = field(default_factory=list)
    finished: List[int] = field(default_factory=list)
    preempted: List[int] = field(default_factory=list)
    prefill_tokens: int = 0
    cached_tokens: int = 0
    kv_tokens: int = 0             # tokens attended over this step
    groups: int = 0                # grouped launches: groups planned this step
    shared_tokens: int = 0         # tokens read through a group's shared prefix


class ContinuousBatchDriver:
    def __init__(self, num_blocks, num_q_heads, num_kv_heads, max_batch, max_blocks_per_seq,
                 sources, device="cuda", block_size=16, head_dim=128, enable_prefix_cache=True,
                 free_order=None, record_ops=False, preemption="recompute", host_blocks=0,
                 grouped=False):
        """sources: object with
             next_token(req) -> int
             kv(req, positions) -> (k, v) fp16 CUDA tensors [n, Hkv, D] for the
                                   prefixes req.tokens[:p + 1]
             query(req, pos) -> fp16 CUDA tensor [Hq, D]
        """
        self.dev = torch.device(device)
        self.bs, self.D = block_size, head_dim
        self.Hq, self.Hkv = num_q_heads, num_kv_heads
        self.max_batch, self.max_blocks = max_batch, max_blocks_per_seq
        self.src = sources
        self.bm = BlockManager(num_blocks, block_size, enable_prefix_cache, free_order)
        self.k_cache = torch.zeros((num_blocks, block_size, num_kv_heads, head_dim),
                                   dtype=torch.float16, device=self.dev)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.out = torch.empty((max_batch, num_q_heads, head_dim), dtype=torch.float16,
                               device=self.dev)
        self.q = torch.empty_like(self.out)
        self.k_new = torch.empty((max_batch, num_kv_heads, head_dim), dtype=torch.float16,
                                 device=self.dev)
        self.v_new = torch.empty_like(self.k_new)
        self.workspace = ops.alloc_workspace(max_batch, num_q_heads, max_blocks_per_seq, self.dev,
                                             block_size)
        self.dev_err = ops.new_error_word(self.dev)
        if num_blocks < max_blocks_per_seq:
            raise ValueError("the pool must hold at least one full-length sequence")
        if preemption not in ("recompute", "swap"):
            raise ValueError("preemption is 'recompute' or 'swap'")
        self.preemption = preemption
        # grouped attention: requests whose tables start with the same blocks
        # (prefix-cache hits on a shared prompt) stream those blocks once
        self.grouped = bool(grouped)
        self.gws = None
        # swap space: pinned host pools for K and V and a FIFO of their free blocks
        self.host_k = self.host_v = None
        self.host_free = deque(range(host_blocks))
        if preemption == "swap":
            shape = (host_blocks,) + tuple(self.k_cache.shape[1:])
            self.host_k = torch.empty(shape, dtype=torch.float16, pin_memory=True)
            self.host_v = torch.empty(shape, dtype=torch.float16, pin_memory=True)
        self.swapped_out_blocks = 0
        self.swapped_in_blocks = 0
        self.waiting = deque()
        self.running: List[Request] = []
        self.requests = {}
        self.ops_log = [] if record_ops else None
        self.steps = 0

    # ---- queue -----------------------------------------------------------------
    def add_request(self, rid, prompt, max_new_tokens):
        if not prompt:
            raise ValueError("a request needs at least one prompt token")
        req = Request(int(rid), [int(t) for t in prompt], int(max_new_tokens))
        self.requests[req.rid] = req
        self.waiting.append(req)

    @property
    def idle(self):
        return not self.waiting and not self.running

    def _log(self, *entry):
        if self.ops_log is not None:
            self.ops_log.append(entry)

    # ---- device writes -------------------------------------------------------------
    def _to_device(self, arr):
        """Host array -> device through a pinned staging tensor (asynchronous)."""
        t = torch.from_numpy(np.ascontiguousarray(arr))
        if self.dev.type == "cuda":
            t = t.pin_memory()
        return t.to(self.dev, non_blocking=True)

    def _write_kv(self, k, v, slots):
        slot_t = self._to_device(np.asarray(slots, dtype=np.int64))
        ops.reshape_and_cache(k, v, slot_t, self.k_cache, self.v_cache, dev_err=self.dev_err)

    def _prefill(self, req, cached):
        n = len(req.tokens)
        if cached >= n:
            return 0
        positions = np.arange(cached, n)
        table = np.asarray(self.bm.block_table(req.rid), dtype=np.int64)
        slots = table[positions // self.bs] * self.bs + positions % self.bs
        k, v = self.src.kv(req, positions.tolist())
        self._write_kv(k, v, slots)
        return len(positions)

    def _next_tokens(self, reqs):
        if hasattr(self.src, "next_tokens"):
            return [int(t) for t in self.src.next_tokens(reqs)]
        return [int(self.src.next_token(r)) for r in reqs]

    def _swap(self, pairs, out):
        pairs_d = torch.tensor(pairs, dtype=torch.int64, device=self.dev)
        if out:
            ops.swap_blocks([self.k_cache, self.v_cache], [self.host_k, self.host_v], pairs_d,
                            dev_err=self.dev_err)
        else:
            ops.swap_blocks([self.host_k, self.host_v], [self.k_cache, self.v_cache], pairs_d,
                            dev_err=self.dev_err)

    def _preempt(self, res, batch):
        # p1 preempts the request with the most generated tokens.  Requests that
        # already appended this step are not candidates: their new block may
        # already carry a registered hash whose K/V row is written later in the
        # step, so freeing them now could leave a cached block with a hole.
        victim = max((r for r in self.running if r not in batch), key=lambda r: r.generated)
        table = self.bm.block_table(victim.rid)
        victim.swapped = None
        if self.preemption == "swap" and len(self.host_free) >= len(table):
            # swap-out: the blocks holding its tokens go to host memory before the
            # device blocks are freed (stream order keeps later writes after the copy)
            n_used = -(-len(victim.tokens) // self.bs)
            host = [self.host_free.popleft() for _ in range(n_used)]
            if n_used:
                self._swap([(table[i], host[i]) for i in range(n_used)], out=True)
            victim.swapped = host
            self.swapped_out_blocks += n_used
        self.bm.free(victim.rid)
        self._log("free", victim.rid)
        self.running.remove(victim)
        victim.preemptions += 1
        self.waiting.appendleft(victim)
        res.preempted.append(victim.rid)
        return victim

    # ---- one step --------------------------------------------------------------------
    def step(self) -> StepResult:
        res = StepResult([], [], self.out[:0])
        # 1. release finished requests
        for r in [r for r in self.running if r.done]:
            self.bm.free(r.rid)
            self._log("free", r.rid)
            self.running.remove(r)
            res.finished.append(r.rid)
        # 2. admit FCFS while blocks last
        while self.waiting and len(self.running) < self.max_batch:
            r = self.waiting[0]
            if -(-(len(r.tokens) + 1) // self.bs) > self.max_blocks:
                raise ValueError("request %d does not fit max_blocks_per_seq" % r.rid)
            try:
                self.bm.allocate(r.rid, r.tokens)
            except OutOfBlocks:
                self._log("allocate", r.rid, tuple(r.tokens), None)
                break
            cached = self.bm.num_cached_tokens(r.rid)
            self._log("allocate", r.rid, tuple(r.tokens), cached)
            self.waiting.popleft()
            host = getattr(r, "swapped", None)
            if host is not None:
                # swap-in: blocks past the prefix-cache hits come back from host memory
                table = self.bm.block_table(r.rid)
                first = cached // self.bs
                pairs = [(host[i], table[i]) for i in range(first, len(host))]
                if pairs:
                    self._swap(pairs, out=False)
                self.swapped_in_blocks += len(pairs)
                self.host_free.extend(host)
                r.swapped = None
            else:
                res.prefill_tokens += self._prefill(r, cached)
            res.cached_tokens += cached
            self.running.append(r)
            res.admitted.append(r.rid)
        # 3. one decode token per running request: one native call appends for the
        # whole batch; an OutOfBlocks stops it at the failing request, which is
        # handled (preemption) before the call resumes from there
        batch, slots = [], []
        pending = list(self.running)
        for r in pending:
            if len(r.tokens) + 1 > self.max_blocks * self.bs:
                raise ValueError("request %d outgrew max_blocks_per_seq" % r.rid)
        toks = self._next_tokens(pending)
        i = 0
        while i < len(pending):
            got, done, rc = self.bm.append_slots_partial([r.rid for r in pending[i:]], toks[i:])
            for j in range(done):
                r, tok, slot = pending[i + j], int(toks[i + j]), int(got[j])
                self._log("append", r.rid, tok, slot)
                r.tokens.append(tok)
                r.generated += 1
                batch.append(r)
                slots.append(slot)
            i += done
            if rc == 0:
                break
            if rc != -4:
                raise RuntimeError("append_slot failed with status %d" % rc)
            r = pending[i]
            self._log("append", r.rid, int(toks[i]), None)
            victim = self._preempt(res, batch)
            if victim is r:
                i += 1
            else:
                k = pending.index(victim)      # not yet appended: after i
                del pending[k]
                del toks[k]
        pairs = self.bm.take_cow_pairs()
        if pairs:
            self._log("cow", tuple(map(tuple, pairs)))
            ops.copy_blocks(self.k_cache, self.v_cache,
                            torch.tensor(pairs, dtype=torch.int64, device=self.dev),
                            dev_err=self.dev_err)
        B = len(batch)
        self.steps += 1
        if B == 0:
            return res
        tables, lens = self.bm.block_tables([r.rid for r in batch], max_blocks=self.max_blocks)
        if self.grouped:
            # members of a group must be adjacent: order the batch by first block
            order = np.argsort(tables[:, 0], kind="stable")
            batch = [batch[j] for j in order]
            slots = [slots[j] for j in order]
            tables, lens = tables[order], lens[order]
        # new tokens' K/V and queries
        if hasattr(self.src, "decode_batch"):
            k, v, q = self.src.decode_batch(batch)
            self.k_new[:B].copy_(k)
            self.v_new[:B].copy_(v)
            self.q[:B].copy_(q)
        else:
            for i, r in enumerate(batch):
                pos = len(r.tokens) - 1
                k, v = self.src.kv(r, [pos])
                self.k_new[i].copy_(k[0])
                self.v_new[i].copy_(v[0])
                self.q[i].copy_(self.src.query(r, pos))
        self._write_kv(self.k_new[:B], self.v_new[:B], slots)
        scale = 1.0 / float(np.sqrt(self.D))
        groups = None
        if self.grouped:
            gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, self.bs,
                                                          16 // (self.Hq // self.Hkv))
            if mx > 0:
                groups = (gf, sg, gs, mx, mo)
        tables_d = self._to_device(tables)
        lens_d = self._to_device(lens)
        if groups is not None:
            gf, sg, gs, mx, mo = groups
            need = ops.grouped_workspace_bytes(B, self.Hq, self.max_blocks, mx, self.bs, self.D)
            if self.gws is None or self.gws.numel() < need:
                self.gws = torch.empty(max(need, 1), dtype=torch.uint8, device=self.dev)
            meta = self._to_device(np.concatenate([gf, sg, gs]).astype(np.int32))
            n_g = len(gs)
            ops.paged_attention_decode_grouped(self.out[:B], self.q[:B], self.k_cache,
                                               self.v_cache, tables_d, lens_d, meta[:n_g + 1],
                                               meta[n_g + 1:n_g + 1 + B],
                                               meta[n_g + 1 + B:], mx, mo, scale,
                                               workspace=self.gws, dev_err=self.dev_err)
            res.groups = len(gs)
            res.shared_tokens = int(gs[sg].sum())
        else:
            ops.paged_attention_decode(self.out[:B], self.q[:B], self.k_cache, self.v_cache,
                                       tables_d, lens_d, scale, workspace=self.workspace,
                                       dev_err=self.dev_err)
        res.rids = [r.rid for r in batch]
        res.positions = [len(r.tokens) - 1 for r in batch]
        res.out = self.out[:B]
        res.kv_tokens = int(lens.sum())
        return res

    def check_errors(self):
        code = ops.read_error_word(self.dev_err)
        if code:
            raise RuntimeError("device reported error code %d" % code)


class HostSources:
    """Content-keyed synthetic values computed on the host (small runs, tests)."""

    def __init__(self, seed, num_q_heads, num_kv_heads, head_dim=128, device="cuda"):
        from . import workloads as wl
        self.wl, self.seed = wl, seed
        self.Hq, self.Hkv, self.D, self.dev = num_q_heads, num_kv_heads, head_dim, device

    def next_token(self, req):
        return self.wl.next_token_host(self.seed, req.rid, len(req.tokens))

    def kv(self, req, positions):
        keys = self.wl.prefix_keys(req.tokens[:max(positions) + 1], self.seed)
        k, v = self.wl.token_kv_host([keys[p] for p in positions], self.Hkv, self.D)
        return torch.from_numpy(k).to(self.dev), torch.from_numpy(v).to(self.dev)

    def query(self, req, pos):
        return torch.from_numpy(self.wl.step_query_host(self.seed, req.rid, pos, self.Hq,
                                                        self.D)).to(self.dev)


class DeviceSources:
    """Values drawn on the device (large runs, benchmarks).  K/V depend on the
    request and position, so blocks reused through the prefix cache keep the
    values the first prefill wrote (the driver never rewrites cached tokens)."""

    def __init__(self, seed, num_q_heads, num_kv_heads, head_dim=128, device="cuda"):
        self.seed, self.Hq, self.Hkv, self.D = seed, num_q_heads, num_kv_heads, head_dim
        self.dev = torch.device(device)
        self.gen = torch.Generator(device=self.dev)
        self.gen.manual_seed(seed)
        self.rng = np.random.default_rng(seed)

    def next_token(self, req):
        return int(self.rng.integers(0, 32000))

    def kv(self, req, positions):
        n = len(positions)
        k = torch.randn((n, self.Hkv, self.D), generator=self.gen, device=self.dev).half()
        v = torch.randn((n, self.Hkv, self.D), generator=self.gen, device=self.dev).half()
        return k, v

    def query(self, req, pos):
        return torch.randn((self.Hq, self.D), generator=self.gen, device=self.dev).half()

    def next_tokens(self, reqs):
        return self.rng.integers(0, 32000, size=len(reqs)).tolist()

    def decode_batch(self, batch):
        B = len(batch)
        x = torch.randn((B, 2 * self.Hkv + self.Hq, self.D), generator=self.gen,
                        device=self.dev).half()
        return x[:, :self.Hkv], x[:, self.Hkv:2 * self.Hkv], x[:, 2 * self.Hkv:]
