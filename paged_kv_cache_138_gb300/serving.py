"""Continuous batching with the native scheduler (pkv_sched_*) in the loop.

Each step is one native call that plans everything on the host (finish, admit
with prefix-cache hits, append a sampled token per running request, preempt by
recompute or swap, copy-on-write, tables, shared-prefix groups), followed by
the device work it returns, in order: swap-ins and prefill writes, swap-outs,
copy_blocks, then one fused launch that writes the new tokens' K/V and runs
paged attention over the batch (grouped when the step formed groups), and the
merge.  The step's metadata and prefill slots are copied on a side stream
while the previous step's kernels run; the decode stream waits only for that
copy.  Python only marshals the arrays and launches.

Values (K/V of prefill and decoded tokens, queries) come from a source object:
``DeviceRandomValues`` draws them on the device (benchmarks);
``ContentKeyedValues`` derives them from each request's token prefix on the
host (tests: a block found again through the prefix cache then holds what a
fresh prefill would write, and the oracle can recompute every row).
"""
import ctypes

import numpy as np
import torch

from . import ops
from . import workloads as wl
from ._lib import PKV_OK, PagedKVError, lib
from .block_manager import BlockManager


class _StepOut(ctypes.Structure):
    _fields_ = [
        ("batch_rids", ctypes.c_void_p), ("positions", ctypes.c_void_p),
        ("tokens", ctypes.c_void_p), ("slots", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
        ("prefill_rids", ctypes.c_void_p), ("prefill_positions", ctypes.c_void_p),
        ("prefill_slots", ctypes.c_void_p), ("prefill_cap", ctypes.c_int64),
        ("swap_in_pairs", ctypes.c_void_p), ("swap_out_pairs", ctypes.c_void_p),
        ("swap_cap", ctypes.c_int64),
        ("cow_pairs", ctypes.c_void_p), ("cow_cap", ctypes.c_int64),
        ("group_limit", ctypes.c_int32), ("group_first", ctypes.c_void_p),
        ("seq_group", ctypes.c_void_p), ("group_shared", ctypes.c_void_p),
        ("num_groups", ctypes.c_int32), ("max_shared_tokens", ctypes.c_int32),
        ("max_own_tokens", ctypes.c_int32),
        ("num_batch", ctypes.c_int32), ("num_prefill", ctypes.c_int32),
        ("num_swap_in", ctypes.c_int32), ("num_swap_out", ctypes.c_int32),
        ("num_cow", ctypes.c_int32), ("num_admitted", ctypes.c_int32),
        ("num_finished", ctypes.c_int32), ("num_preempted", ctypes.c_int32),
        ("cached_tokens", ctypes.c_int64),
    ]


class _DecodeLaunch(ctypes.Structure):
    _fields_ = [
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
        ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("meta", ctypes.c_void_p), ("meta_bytes", ctypes.c_size_t),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("scale", ctypes.c_float), ("dev_err", ctypes.c_void_p), ("meta_staged", ctypes.c_int32),
    ]


class NativeServingDriver:
    """Continuous batching without a model: the native scheduler plans each
    step on a BlockManager (admissions with prefix-cache hits, one sampled
    token per running request, preemption by recompute or swap, copy-on-write,
    shared-prefix groups) and step() launches the device work it returns.
    K/V and q values come from ``values`` (DeviceRandomValues or
    ContentKeyedValues)."""

    def __init__(self, num_blocks, num_q_heads, num_kv_heads, max_batch, max_blocks_per_seq,
                 values, device="cuda", block_size=16, head_dim=128, enable_prefix_cache=True,
                 free_order=None, preemption="recompute", host_blocks=0, seed=0, grouped=False):
        if preemption not in ("recompute", "swap"):
            raise ValueError("preemption is 'recompute' or 'swap'")
        if num_blocks < max_blocks_per_seq:
            raise ValueError("the pool must hold at least one full-length sequence")
        self.dev = torch.device(device)
        self.bs, self.D, self.Hq, self.Hkv = block_size, head_dim, num_q_heads, num_kv_heads
        self.max_batch, self.max_blocks = max_batch, max_blocks_per_seq
        self.values = values
        self.bm = BlockManager(num_blocks, block_size, enable_prefix_cache, free_order)
        self._h = lib().pkv_sched_create(self.bm._h, max_batch, max_blocks_per_seq, block_size,
                                         1 if preemption == "swap" else 0, int(host_blocks),
                                         ctypes.c_uint64(seed), 32000)
        if not self._h:
            raise ValueError("pkv_sched_create rejected its arguments")
        shape = (num_blocks, block_size, num_kv_heads, head_dim)
        self.k_cache = torch.zeros(shape, dtype=torch.float16, device=self.dev)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.host_k = self.host_v = None
        if preemption == "swap" and host_blocks:
            hs = (host_blocks,) + shape[1:]
            self.host_k = torch.empty(hs, dtype=torch.float16, pin_memory=True)
            self.host_v = torch.empty(hs, dtype=torch.float16, pin_memory=True)
        B, mb = max_batch, max_blocks_per_seq
        # Two sets of step arrays in pinned host memory, used alternately: the
        # scheduler writes set k % 2 while the device may still be copying set
        # (k - 1) % 2; set reuse waits on the event recorded after its copies.
        pin = self.dev.type == "cuda"
        spec = {
            "batch_rids": ((B,), torch.int64), "positions": ((B,), torch.int32),
            "tokens": ((B,), torch.int32), "slots": ((B,), torch.int64),
            "block_tables": ((B, mb), torch.int32), "context_lens": ((B,), torch.int32),
            "prefill_rids": ((B * mb * block_size,), torch.int64),
            "prefill_positions": ((B * mb * block_size,), torch.int32),
            "prefill_slots": ((B * mb * block_size,), torch.int64),
            "swap_in_pairs": ((B * mb, 2), torch.int64),
            "swap_out_pairs": ((B * mb, 2), torch.int64),
            "cow_pairs": ((B, 2), torch.int64),
            "groups": ((3 * B + 1,), torch.int32),   # group_first | seq_group | group_shared
        }
        # block tables, context lengths and groups sit in one pinned buffer in
        # the layout of the device staging area, so the decode launch moves
        # them with one copy
        packed = ("block_tables", "context_lens", "groups")
        self.sets = []
        for _ in range(2):
            t = {n: torch.zeros(shape, dtype=dt, pin_memory=pin) for n, (shape, dt) in spec.items()
                 if n not in packed}
            meta_host = torch.zeros(B * mb + B + 3 * B + 1, dtype=torch.int32, pin_memory=pin)
            t["block_tables"] = meta_host[:B * mb].view(B, mb)
            t["context_lens"] = meta_host[B * mb:B * mb + B]
            t["groups"] = meta_host[B * mb + B:]
            o = _StepOut()
            for name, ten in t.items():
                if name != "groups":
                    setattr(o, name, ctypes.c_void_p(ten.data_ptr()))
            g = t["groups"]
            o.group_first = ctypes.c_void_p(g.data_ptr())
            o.seq_group = ctypes.c_void_p(g[B + 1:].data_ptr())
            o.group_shared = ctypes.c_void_p(g[2 * B + 1:].data_ptr())
            o.group_limit = 16 // (num_q_heads // num_kv_heads) if grouped else 0
            o.prefill_cap = B * mb * block_size
            o.swap_cap = B * mb
            o.cow_cap = B
            ev = torch.cuda.Event() if pin else None
            self.sets.append({"t": t, "a": {n: x.numpy() for n, x in t.items()}, "out": o,
                              "event": ev, "used": False})
        self.out = torch.empty((B, num_q_heads, head_dim), dtype=torch.float16, device=self.dev)
        # the step's q, k_new and v_new: views of one buffer (one generator
        # launch fills all three)
        nq, nk = B * num_q_heads * head_dim, B * num_kv_heads * head_dim
        self.qkv = torch.empty(nq + 2 * nk, dtype=torch.float16, device=self.dev)
        self.q = self.qkv[:nq].view(B, num_q_heads, head_dim)
        self.k_new = self.qkv[nq:nq + nk].view(B, num_kv_heads, head_dim)
        self.v_new = self.qkv[nq + nk:].view(B, num_kv_heads, head_dim)
        self.grouped = bool(grouped)
        if self.grouped:
            # steps without a shared prefix run the plain entry point on the same buffer
            n = max(ops.grouped_workspace_bytes(B, num_q_heads, mb, mb * block_size, block_size,
                                                head_dim),
                    ops.workspace_bytes(B, num_q_heads, mb, block_size, head_dim))
            self.workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=self.dev)
        else:
            self.workspace = ops.alloc_workspace(B, num_q_heads, mb, self.dev, block_size)
        self.dev_err = ops.new_error_word(self.dev)
        self.scale = 1.0 / float(np.sqrt(head_dim))
        self.steps = 0
        # the decode launch: one native call per step (cache write, plain or
        # grouped attention).  Each set of step arrays has its own device
        # staging for the step's metadata, copied on a side stream while the
        # previous step's kernels run (pkv_sched_stage_decode); the decode
        # stream waits for that copy only.
        meta_bytes = int(lib().pkv_sched_meta_bytes(self._h))
        ws = self.workspace
        self.copy_stream = torch.cuda.Stream(self.dev) if pin else None
        for st in self.sets:
            st["meta"] = torch.empty(meta_bytes, dtype=torch.uint8, device=self.dev)
            dl = _DecodeLaunch()
            dl.k_cache, dl.v_cache = self.k_cache.data_ptr(), self.v_cache.data_ptr()
            dl.num_blocks = num_blocks
            dl.num_q_heads, dl.num_kv_heads, dl.head_dim = num_q_heads, num_kv_heads, head_dim
            dl.q, dl.k_new, dl.v_new = (self.q.data_ptr(), self.k_new.data_ptr(),
                                        self.v_new.data_ptr())
            dl.out = self.out.data_ptr()
            dl.meta, dl.meta_bytes = st["meta"].data_ptr(), meta_bytes
            dl.workspace = ws.data_ptr() if ws is not None else None
            dl.workspace_bytes = ws.numel() if ws is not None else 0
            dl.scale = self.scale
            dl.dev_err = self.dev_err.data_ptr()
            dl.meta_staged = 1 if pin else 0
            st["launch"] = dl
            st["staged"] = torch.cuda.Event() if pin else None
            # device copy of the set's prefill slots (staged with the metadata)
            st["prefill_slots_dev"] = torch.empty(B * mb * block_size, dtype=torch.int64,
                                                  device=self.dev)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().pkv_sched_destroy(h)
            self._h = None

    def add_request(self, rid, prompt, max_new_tokens):
        """Queue a request: prompt token ids, tokens to generate."""
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        rc = lib().pkv_sched_add_request(self._h, int(rid), p.ctypes.data_as(ctypes.c_void_p),
                                         len(p), int(max_new_tokens))
        if rc != PKV_OK:
            raise PagedKVError(rc, "add_request")

    @property
    def idle(self):
        """True when no request is waiting or running."""
        return lib().pkv_sched_num_unfinished(self._h) == 0

    def request_tokens(self, rid):
        """A request's tokens so far (prompt + generated), int32."""
        n = lib().pkv_sched_request_tokens(self._h, int(rid), None, 0)
        if n < 0:
            raise PagedKVError(int(n), "request_tokens")
        out = np.empty(max(n, 1), np.int32)
        lib().pkv_sched_request_tokens(self._h, int(rid), out.ctypes.data_as(ctypes.c_void_p), n)
        return out[:n]

    def _to_device(self, arr):
        t = torch.from_numpy(np.ascontiguousarray(arr))
        if self.dev.type == "cuda":
            t = t.pin_memory()
        return t.to(self.dev, non_blocking=True)

    def _h2d(self, t):
        return t.to(self.dev, non_blocking=True)

    def step(self):
        """Plan and launch one step.  Returns a dict with the decode batch's ids,
        positions, the output rows (device, valid until the next step) and
        counters."""
        st = self.sets[self.steps % 2]
        if st["used"] and st["event"] is not None:
            st["event"].synchronize()           # its copies from two steps ago are done
        o, t, a = st["out"], st["t"], st["a"]
        rc = lib().pkv_sched_step(self._h, ctypes.byref(o))
        if rc != PKV_OK:
            raise PagedKVError(rc, "sched_step")
        cuda = self.dev.type == "cuda"
        # one stream for the whole step, looked up once
        stream = torch.cuda.current_stream(self.dev) if cuda else None
        staged = st["staged"] is not None and (o.num_batch or o.num_prefill)
        if staged:
            # this set's staging was last read by the step two back, which the
            # event above has seen finish; the copies run beside this step's
            # first launches and the previous step's kernels
            cs = self.copy_stream
            if o.num_prefill:
                with torch.cuda.stream(cs):
                    st["prefill_slots_dev"][:o.num_prefill].copy_(
                        t["prefill_slots"][:o.num_prefill], non_blocking=True)
            if o.num_batch:
                rc = lib().pkv_sched_stage_decode(self._h, ctypes.byref(o),
                                                  ctypes.byref(st["launch"]),
                                                  ctypes.c_void_p(cs.cuda_stream))
                if rc != PKV_OK:
                    raise PagedKVError(rc, "sched_stage_decode")
            st["staged"].record(cs)
        caches = ([self.k_cache, self.v_cache], [self.host_k, self.host_v])
        if o.num_swap_in:
            ops.swap_blocks(caches[1], caches[0], self._h2d(t["swap_in_pairs"][:o.num_swap_in]),
                            dev_err=self.dev_err, stream=stream)
        if o.num_prefill:
            n = o.num_prefill
            k, v = self.values.prefill(self, a["prefill_rids"][:n], a["prefill_positions"][:n],
                                       stream=stream)
            if staged:
                stream.wait_event(st["staged"])
                slots = st["prefill_slots_dev"][:n]
            else:
                slots = self._h2d(t["prefill_slots"][:n])
            ops.reshape_and_cache(k, v, slots, self.k_cache, self.v_cache, dev_err=self.dev_err,
                                  stream=stream)
        if o.num_swap_out:
            ops.swap_blocks(caches[0], caches[1], self._h2d(t["swap_out_pairs"][:o.num_swap_out]),
                            dev_err=self.dev_err, stream=stream)
        if o.num_cow:
            ops.copy_blocks(self.k_cache, self.v_cache, self._h2d(t["cow_pairs"][:o.num_cow]),
                            dev_err=self.dev_err, stream=stream)
        B = o.num_batch
        res = {"rids": a["batch_rids"][:B].copy(), "positions": a["positions"][:B].copy(),
               "out": self.out[:B], "admitted": o.num_admitted, "finished": o.num_finished,
               "preempted": o.num_preempted, "prefill": o.num_prefill,
               "cached": int(o.cached_tokens), "swap_in": o.num_swap_in,
               "swap_out": o.num_swap_out, "kv_tokens": int(a["context_lens"][:B].sum()),
               "groups": 0, "shared_tokens": 0}
        if B:
            if staged:   # before the fill, so the fill and the decode launch stay adjacent
                stream.wait_event(st["staged"])
            self.values.decode_into(self, res["rids"], res["positions"], B, stream=stream)
            rc = lib().pkv_sched_launch_decode(
                self._h, ctypes.byref(o), ctypes.byref(st["launch"]),
                ctypes.c_void_p(stream.cuda_stream) if cuda else None)
            if rc != PKV_OK:
                raise PagedKVError(rc, "sched_launch_decode")
            if o.num_groups and o.max_shared_tokens > 0:
                g = a["groups"]
                res["groups"] = o.num_groups
                res["shared_tokens"] = int(g[2 * self.max_batch + 1:][
                    g[self.max_batch + 1:self.max_batch + 1 + B]].sum())
        if st["event"] is not None:
            st["event"].record(stream)
        st["used"] = True
        self.steps += 1
        return res

    def check_errors(self):
        """Synchronise and raise if a kernel reported a device error code."""
        code = ops.read_error_word(self.dev_err)
        if code:
            raise RuntimeError("device reported error code %d" % code)


class DeviceRandomValues:
    """K/V/q drawn on the device from one counter-based stream
    (``ops.fill_normal``): one launch for a step's q, k_new and v_new, one for
    a step's prefill rows."""

    def __init__(self, seed, num_q_heads, num_kv_heads, head_dim=128, device="cuda"):
        self.Hq, self.Hkv, self.D = num_q_heads, num_kv_heads, head_dim
        self.seed, self.offset = int(seed), 0
        self.dev = device

    def prefill(self, drv, rids, positions, stream=None):
        x = torch.empty((2, len(rids), self.Hkv, self.D), dtype=torch.float16, device=self.dev)
        self.offset = ops.fill_normal(x, self.seed, self.offset, stream)
        return x[0], x[1]

    def decode_into(self, drv, rids, positions, num_rows, stream=None):
        """Fill rows 0 .. num_rows - 1 of the driver's q, k_new and v_new (the
        three share one buffer, so the whole buffer is drawn in one launch)."""
        self.offset = ops.fill_normal(drv.qkv, self.seed, self.offset, stream)


class ContentKeyedValues:
    """K/V of a token = a function of the request's token prefix; q of a decode
    step = a function of (request, position).  Host-side, for tests."""

    def __init__(self, seed, num_q_heads, num_kv_heads, head_dim=128, device="cuda"):
        self.seed, self.Hq, self.Hkv, self.D, self.dev = seed, num_q_heads, num_kv_heads, \
            head_dim, device

    def _kv(self, drv, rids, positions):
        ks, vs, cache = [], [], {}
        for rid, pos in zip(rids.tolist(), positions.tolist()):
            if rid not in cache:
                cache[rid] = wl.prefix_keys(drv.request_tokens(rid), self.seed)
            k, v = wl.token_kv_host([cache[rid][pos]], self.Hkv, self.D)
            ks.append(k[0])
            vs.append(v[0])
        return (torch.from_numpy(np.stack(ks)).to(self.dev),
                torch.from_numpy(np.stack(vs)).to(self.dev))

    def prefill(self, drv, rids, positions, stream=None):
        return self._kv(drv, rids, positions)

    def decode_into(self, drv, rids, positions, num_rows, stream=None):
        k, v = self._kv(drv, rids, positions)
        q = np.stack([wl.step_query_host(self.seed, r, p, self.Hq, self.D)
                      for r, p in zip(rids.tolist(), positions.tolist())])
        drv.k_new[:num_rows].copy_(k)
        drv.v_new[:num_rows].copy_(v)
        drv.q[:num_rows].copy_(torch.from_numpy(q))
