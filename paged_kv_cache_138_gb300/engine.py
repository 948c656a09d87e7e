"""Device state and the decode step: per layer, reshape_and_cache then attention.

``DecodeStep`` owns the KV cache of every layer ([layers, num_blocks, 16, Hkv,
128] fp16 for K and for V), the step's inputs (q, the new token's k/v, slot
mapping, block tables, context lengths), the output and the attention
workspace, all resident in HBM.  ``run()`` enqueues one decode step through
the C ABI; ``run_from_host()`` is the same step fed from pinned host buffers,
with the host->device copies of the inputs and the device->host copy of the
output inside it.
"""
import torch

from . import ops
from . import workloads as wl
from ._lib import PKV_ERR_UNSUPPORTED, PagedKVError
from .scenario import DecodeBatch


class DecodeStep:
    """One decode batch resident in HBM (caches of every layer, the step's
    inputs, output and workspace) and the launches of one step over it:
    eager (prepared launches), from a CUDA graph, or fed from pinned host
    buffers (sequential or pipelined)."""

    def __init__(self, batch: DecodeBatch, device=None, num_layers=None, host_values=None,
                 fused=False, grouped=False, fold_cow=True):
        """host_values: None draws q/K/V on the device (torch generator seeded by
        the workload); otherwise the tuple of ``workloads.host_tensors`` (numpy).
        fused: each layer is one launch of the fused cache-write + attention
        kernel instead of reshape_and_cache followed by attention.
        grouped: sequences sharing leading blocks (forked samples) are planned
        into groups whose shared prefix is streamed once (with fused: one
        launch writing the new tokens and attending).
        fold_cow: with fused, the batch's copy-on-write copies are made inside
        each layer's attention launch instead of by copy_blocks."""
        self.fused = bool(fused)
        w = batch.workload
        self.batch = batch
        self.device = torch.device(device or "cuda")
        L = num_layers or w.num_layers
        S, Hq, Hkv, D, bs = batch.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
        self.num_layers, self.scale = L, w.scale
        dev = self.device
        if host_values is None:
            self.k_cache = torch.empty((L, batch.num_blocks, bs, Hkv, D), dtype=torch.float16,
                                       device=dev)
            self.v_cache = torch.empty_like(self.k_cache)
            self.q = torch.empty((L, S, Hq, D), dtype=torch.float16, device=dev)
            self.k_new = torch.empty((L, S, Hkv, D), dtype=torch.float16, device=dev)
            self.v_new = torch.empty_like(self.k_new)
            for i, t in enumerate((self.k_cache, self.v_cache, self.q, self.k_new, self.v_new)):
                wl.device_normal_fp16_(t, w.seed * 16 + i)
        else:
            q, k_new, v_new, k_cache, v_cache = host_values
            self.q = torch.from_numpy(q).to(dev)
            self.k_new = torch.from_numpy(k_new).to(dev)
            self.v_new = torch.from_numpy(v_new).to(dev)
            self.k_cache = torch.from_numpy(k_cache).to(dev)
            self.v_cache = torch.from_numpy(v_cache).to(dev)
        self.block_tables = torch.from_numpy(batch.block_tables).to(dev)
        self.context_lens = torch.from_numpy(batch.context_lens).to(dev)
        self.slot_mapping = torch.from_numpy(batch.slot_mapping).to(dev)
        self.cow_pairs = torch.from_numpy(batch.cow_pairs).to(dev)
        # fused steps make the copy-on-write copies inside each layer's
        # attention launch (one copy per sequence); others, or a sequence
        # needing two copies in one step, use copy_blocks
        self.cow = None
        if self.fused and batch.cow_pairs.shape[0] and fold_cow:
            try:
                cb, cs = ops.cow_targets(batch.cow_pairs, batch.block_tables)
                self.cow = (torch.from_numpy(cb).to(dev), torch.from_numpy(cs).to(dev))
            except PagedKVError as e:
                if e.status != PKV_ERR_UNSUPPORTED:
                    raise
        self.out = torch.empty((L, S, Hq, D), dtype=torch.float16, device=dev)
        self.groups = None
        if grouped:
            gf, sg, gs, mx, mo = ops.shared_prefix_groups(batch.block_tables, batch.context_lens,
                                                          bs, 16 // (Hq // Hkv))
            if mx > 0:
                self.groups = (torch.from_numpy(gf).to(dev), torch.from_numpy(sg).to(dev),
                               torch.from_numpy(gs).to(dev), mx, mo)
        if self.groups is not None:
            n = ops.grouped_workspace_bytes(S, Hq, batch.max_blocks, self.groups[3], bs)
            self.workspace = torch.empty(n, dtype=torch.uint8, device=dev) if n else None
        else:
            self.workspace = ops.alloc_workspace(S, Hq, batch.max_blocks, dev, bs)
        self.dev_err = ops.new_error_word(dev)
        self._host = None
        self._launches = {}   # prepared launches by (kind, layer, stream, buffer set)

    # ---- device-resident step ---------------------------------------------------
    def apply_cow(self, stream=None):
        """copy_blocks for the batch's copy-on-write pairs, every layer (nothing
        when the attention launches make the copies)."""
        if self.cow_pairs.shape[0] == 0 or self.cow is not None:
            return
        ops.copy_blocks([self.k_cache[i] for i in range(self.num_layers)],
                        [self.v_cache[i] for i in range(self.num_layers)],
                        self.cow_pairs, dev_err=self.dev_err, stream=stream)

    def run_layer(self, i, stream=None, bufs=None):
        """Layer i of one step.  bufs: the step's input/output tensors (q, k_new,
        v_new, slot_mapping, block_tables, context_lens, out); default self."""
        if not self.fused:
            self.cache_write(i, stream, bufs)
        self.attend(i, stream, bufs)

    def _prepared(self, kind, i, stream, bufs, make):
        """The launch `kind` of layer i on (stream, bufs), marshalled once."""
        key = (kind, i, ops._stream_handle(stream).value, id(bufs))
        launch = self._launches.get(key)
        if launch is None:
            launch = self._launches[key] = make()
        return launch

    def cache_write(self, i, stream=None, bufs=None):
        """reshape_and_cache of layer i's new tokens (unfused steps)."""
        b = self if bufs is None else bufs
        self._prepared("write", i, stream, b, lambda: ops.reshape_and_cache(
            b.k_new[i], b.v_new[i], b.slot_mapping, self.k_cache[i], self.v_cache[i],
            dev_err=self.dev_err, stream=stream, prepare=True))()

    def attend(self, i, stream=None, bufs=None):
        """Layer i's attention launch (with the cache write when fused)."""
        b = self if bufs is None else bufs

        def make():
            if self.groups is not None:
                gf, sg, gs, mx, mo = self.groups
                if self.fused:
                    return ops.paged_attention_decode_grouped_fused(
                        b.out[i], b.q[i], b.k_new[i], b.v_new[i], self.k_cache[i],
                        self.v_cache[i], b.block_tables, b.context_lens, gf, sg, gs, mx, mo,
                        self.scale, workspace=self.workspace, dev_err=self.dev_err,
                        stream=stream, prepare=True, cow=self.cow)
                return ops.paged_attention_decode_grouped(
                    b.out[i], b.q[i], self.k_cache[i], self.v_cache[i], b.block_tables,
                    b.context_lens, gf, sg, gs, mx, mo, self.scale, workspace=self.workspace,
                    dev_err=self.dev_err, stream=stream, prepare=True)
            if self.fused:
                return ops.paged_attention_decode_fused(
                    b.out[i], b.q[i], b.k_new[i], b.v_new[i], self.k_cache[i], self.v_cache[i],
                    b.block_tables, b.context_lens, self.scale, workspace=self.workspace,
                    dev_err=self.dev_err, stream=stream, prepare=True, cow=self.cow)
            return ops.paged_attention_decode(
                b.out[i], b.q[i], self.k_cache[i], self.v_cache[i], b.block_tables,
                b.context_lens, self.scale, workspace=self.workspace, dev_err=self.dev_err,
                stream=stream, prepare=True)

        self._prepared("attend", i, stream, b, make)()

    def run(self, stream=None, bufs=None):
        """Every layer of one step (without the COW copies: apply_cow)."""
        for i in range(self.num_layers):
            self.run_layer(i, stream, bufs)
        return self.out if bufs is None else bufs.out

    # ---- CUDA graph of one step ---------------------------------------------------
    def capture_graph(self):
        """Record one decode step (COW copies, then every layer) into a CUDA
        graph; ``replay()`` then launches it with one call.  The step allocates
        nothing, so the captured kernels reuse the buffers above."""
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):          # warm-up outside capture (one-time set-up)
            self.apply_cow(s)
            self.run(s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.apply_cow(s)
            self.run(s)
        torch.cuda.current_stream(self.device).wait_stream(s)
        self.graph = g
        return g

    def replay(self):
        """Launch the captured step (capture_graph) with one call."""
        self.graph.replay()
        return self.out

    def cow_launches_per_step(self):
        """copy_blocks launches of one step (apply_cow): 0 when folded."""
        return 1 if self.cow_pairs.shape[0] and self.cow is None else 0

    def kernel_launches_per_step(self):
        """Kernels of this library one run() launches (COW copies excluded)."""
        merge = 1 if ops.workspace_bytes(self.batch.num_seqs, self.q.shape[2],
                                         self.batch.max_blocks,
                                         self.batch.workload.block_size) else 0
        if self.groups is not None:         # (cache write,) shared + own tiles, merge
            return self.num_layers * (2 if self.fused else 3)
        return self.num_layers * ((1 if self.fused else 2) + merge)

    def split_tokens(self):
        """Tokens per split unit of this batch's attention launches."""
        w = self.batch.workload
        return ops.split_tokens(self.batch.num_seqs, w.num_kv_heads, self.batch.max_blocks,
                                w.block_size)

    def check_errors(self):
        """Synchronise and raise if a kernel reported a device error code."""
        code = ops.read_error_word(self.dev_err)
        if code:
            raise RuntimeError("device reported error code %d" % code)

    # ---- end to end from host buffers -------------------------------------------
    def host_buffers(self):
        """Pinned host copies of the step inputs and an output buffer."""
        if self._host is None:
            pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
            self._host = {
                "q": pin(self.q), "k_new": pin(self.k_new), "v_new": pin(self.v_new),
                "slot_mapping": pin(self.slot_mapping), "block_tables": pin(self.block_tables),
                "context_lens": pin(self.context_lens),
                "out": torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True),
            }
        return self._host

    def host_bytes_per_step(self):
        """(host-to-device, device-to-host) bytes of one step fed from host."""
        h = self.host_buffers()
        up = sum(h[k].numel() * h[k].element_size()
                 for k in ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens"))
        return up, h["out"].numel() * h["out"].element_size()

    def run_from_host(self, stream=None):
        """One step whose inputs come from pinned host buffers and whose output
        goes back to one (the copies on the step's stream)."""
        h = self.host_buffers()
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            for name in ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens"):
                getattr(self, name).copy_(h[name], non_blocking=True)
            self.run(stream=s)
            h["out"].copy_(self.out, non_blocking=True)
        return h["out"]

    # ---- end to end, pipelined: copies of step i+1 overlap the kernels of step i --
    _INPUTS = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")

    def _pipeline(self):
        if getattr(self, "_pipe", None) is None:
            from types import SimpleNamespace
            sets = []
            for _ in range(2):
                b = SimpleNamespace(**{n: torch.empty_like(getattr(self, n))
                                       for n in self._INPUTS + ("out",)})
                sets.append(b)
            ev = lambda: torch.cuda.Event()
            self._pipe = SimpleNamespace(
                sets=sets, copy=torch.cuda.Stream(self.device),
                inputs_ready=[ev(), ev()], compute_done=[ev(), ev()], started=[False, False])
        return self._pipe

    def run_from_host_pipelined(self, host_inputs, host_outputs, stream=None):
        """Steps k = 0 .. n-1 fed from pinned host buffers: host_inputs[k] is a
        dict of the input tensors (names as host_buffers()), host_outputs[k] the
        pinned output of step k.  Two device buffer sets alternate: the
        host->device copies of step k+1 and the device->host copy of step k's
        output run on a copy stream while step k's kernels run.  Returns after
        enqueueing; synchronise before reading host_outputs."""
        P = self._pipeline()
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        n = len(host_inputs)

        def upload(k):
            j = k % 2
            b = P.sets[j]
            with torch.cuda.stream(P.copy):
                if P.started[j]:
                    P.copy.wait_event(P.compute_done[j])  # step k-2 no longer reads set j
                for name in self._INPUTS:
                    getattr(b, name).copy_(host_inputs[k][name], non_blocking=True)
                P.inputs_ready[j].record(P.copy)

        if n:
            upload(0)
        for k in range(n):
            j = k % 2
            b = P.sets[j]
            if k + 1 < n:
                upload(k + 1)
            # the copy stream runs in order and took step k's inputs after step
            # k-2's output copy (uploads of k+1 are enqueued after the output
            # copy of k-1), so this one wait also covers set j's out buffer
            s.wait_event(P.inputs_ready[j])
            self.apply_cow(s)
            self.run(s, bufs=b)
            P.compute_done[j].record(s)
            P.started[j] = True
            with torch.cuda.stream(P.copy):
                P.copy.wait_event(P.compute_done[j])
                host_outputs[k].copy_(b.out, non_blocking=True)
        return host_outputs
