#!/usr/bin/env python
"""Decode-step benchmark of the paged KV-cache hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

A step is one decode step of the workload: (copy_blocks for pending
copy-on-write pairs,) then per layer reshape_and_cache of the new token and
paged decode attention over every sequence (one fused launch per layer by
default).  Inputs are synthetic and resident in HBM before timing starts.  The
default workload is the full Llama-2-7B decode step at batch 64 x 4096-token
contexts: 32 layers x 32 heads MHA, head_dim 128, block_size 16, blocks
scattered over a 128 GiB K+V pool (137 GB of KV read per step, far larger than
the 129 MB L2, so no flush is needed between steps).  A workload whose step
would fit in 4x the L2 size (the 5-sequence tiny case) is timed step by step
instead, each step between its own events and L2 flushed by a buffer write
after each.

Prints one JSON line.  `value` is KV bytes read per step / device time per step
(GB/s, whole job over all ranks); `e2e` is the same metric through the same
public API with the step inputs copied from pinned host memory and the output
copied back inside the timed region; `roofline` times the attention launch
alone in a loop of its own.  `--impl reference` times the CPU fp64 oracle on
the host cores instead, on bounded samples of the same workload whose inputs
it draws itself (no GPU code runs in that arm).  Under torchrun each rank runs
its own copy of the batch (weak scaling, no collective on the data path).
"""
import argparse
import dataclasses
import datetime
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "llama2-7b-32layer"
DECODE_WORKLOADS = ("tiny", "llama2-13b-layer", "gqa-32-8", "prefix-sharing",
                    "llama2-7b-32layer", "llama2-7b-layer")
# end-to-end windows: fixed sizes, whatever --steps is, so that the one
# unoverlapped upload at a window's start and download at its end are spread
# over enough pipelined steps
E2E_WINDOWS = 5
E2E_STEPS_PER_WINDOW = 50
# the attention launch alone: this many back-to-back launches between two events
ROOFLINE_LAUNCHES = 200
CLOCK_PERIOD_MS = 50
# sequences per sample of the oracle arm (one layer, every head of each)
REFERENCE_SAMPLE_SEQS = 8
METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and seq-steps/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=list(DECODE_WORKLOADS) + ["serving", "swap"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None,
                    help="pipelined steps per end-to-end window (default %d)"
                         % E2E_STEPS_PER_WINDOW)
    ap.add_argument("--unfused", action="store_true",
                    help="separate reshape_and_cache and attention launches per layer")
    ap.add_argument("--driver", choices=["native", "python"], default="native",
                    help="serving workload: native scheduler or the Python reference driver")
    ap.add_argument("--grouped", choices=["auto", "on", "off"], default="auto",
                    help="shared-prefix grouped attention (auto: on for prefix-sharing)")
    ap.add_argument("--block-size", type=int, default=16,
                    help="tokens per KV block: 8, 16, 32 or 64")
    ap.add_argument("--cow-kernel", action="store_true",
                    help="copy-on-write copies by copy_blocks, not inside the fused launches")
    return ap.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


TRAFFIC_SOURCES = ("attention_kernel.cuh", "paged_attention.cu", "pkv_device.cuh")


def kernel_source_digest():
    """sha256 (16 hex digits) of the attention kernels and their launch code."""
    import hashlib
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_138_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel_key):
    """dram bytes per launch from the committed ncu summary, if it still
    describes the current kernel and launch source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
        if rec and rec.get("source_sha256_16") == kernel_source_digest():
            return rec
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, each stamped with
    nvidia-smi's own wall-clock timestamp, so that the samples taken inside a
    timed region can be picked out afterwards (the tool's pipe output arrives
    in bursts, so arrival times say nothing)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index, period_ms=CLOCK_PERIOD_MS):
        self.idx, self.period_ms = gpu_index, period_ms
        self.proc, self.samples, self.t_start = None, [], None
        self._lines, self._reader = [], None

    def start(self):
        self.t_start = time.time()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self._lines.append(line)

    def ready(self, settle_s=0.6):
        """Wait until the tool has been sampling for settle_s."""
        if self.proc is not None:
            time.sleep(max(0.0, self.t_start + settle_s - time.time()))

    def stop(self):
        if self.proc is not None:
            time.sleep(2.0 * self.period_ms / 1e3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self._reader is not None:
                self._reader.join(timeout=5)
        self.samples = []
        for line in self._lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            reasons = {n for n, v in zip(self.REASONS, f[6:10]) if v.lower().startswith("active")}
            self.samples.append((ts, sm, mx, reasons))

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and the throttle reasons seen, over the
        samples stamped in [t0, t1] (all samples when no window is given)."""
        sel = [s for s in self.samples
               if (t0 is None or s[0] >= t0) and (t1 is None or s[0] <= t1)]
        sm = [s[1] for s in sel]
        reasons = set().union(*[s[3] for s in sel]) if sel else set()
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": sel[-1][2] if sel else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "period_ms": self.period_ms}


def workload_config(w, tables, lens, num_blocks, l2_bytes):
    """The `config` object of the JSON line: the workload's shape and sizes,
    from host metadata only (both arms print the same one)."""
    from paged_kv_cache_138_gb300 import accounting
    kv = accounting.step_kv_bytes(lens, w.num_kv_heads, w.head_dim, layers=w.num_layers)
    unique = None
    if w.name == "prefix-sharing":
        unique = accounting.unique_kv_bytes(tables, lens, w.block_size, w.num_kv_heads,
                                            w.head_dim)
    step_bytes = unique if unique is not None else kv / w.num_layers
    alloc = sum(-(-int(L) // w.block_size) * w.block_size for L in lens)
    cfg = {"workload": w.name, "description": w.description,
           "num_seqs": int(len(lens)), "num_q_heads": w.num_q_heads,
           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
           "block_size": w.block_size, "layers": w.num_layers,
           "tokens": int(sum(int(L) for L in lens)), "kv_bytes_per_step": kv,
           "unique_kv_bytes_per_step": unique, "pool_blocks": int(num_blocks),
           "tail_waste_pct": 100.0 * (alloc - sum(int(L) for L in lens)) / alloc}
    if l2_bytes is None:
        cfg["l2"] = "unknown L2 size (no GPU)"
    elif step_bytes < 4 * l2_bytes:
        cfg["l2"] = ("L2 flushed between timed steps (%d MiB write, outside the per-step "
                     "events)" % (max(4 * l2_bytes, 512 << 20) >> 20))
    else:
        cfg["l2"] = ("inputs larger than L2 (%.0f MB per layer-step vs %.0f MB L2); no flush"
                     % (step_bytes / 1e6, l2_bytes / 1e6))
    return cfg, kv, unique


def device_l2_bytes():
    import torch
    if not torch.cuda.is_available():
        return None
    return torch.cuda.get_device_properties(0).L2_cache_size


def bench_workload(args, rank=0):
    from paged_kv_cache_138_gb300 import dist as pd
    from paged_kv_cache_138_gb300 import workloads as wl
    w = pd.replica(wl.WORKLOADS[args.workload], rank)
    if args.block_size != w.block_size:
        if args.workload == "prefix-sharing":
            raise SystemExit("the prefix-sharing workload is defined for block size 16")
        w = dataclasses.replace(w, block_size=args.block_size)
    return w


class OracleSampler:
    """Times the fp64 C oracle -- reshape_and_cache of the new token, then
    attention over every head of one layer -- on a few sequences of the
    workload.  Its inputs are drawn here on the host (seeded N(0, 1) fp16 for
    q, the new K/V and the K/V of the sequences' blocks, compacted into a small
    pool), from the oracle's own batch metadata: nothing of the GPU path is
    used.  Timing depends on the shapes and lengths only, not on the values."""

    def __init__(self, w, tables, lens, max_seqs, seed):
        import numpy as np

        from paged_kv_cache_138_gb300 import workloads as wl
        self.w, self.tables, self.lens = w, tables, lens
        bs = w.block_size
        per_seq = sorted(-(-int(L) // bs) for L in lens)
        cap = max(1, sum(per_seq[-max_seqs:]))
        rng = np.random.default_rng([seed, 99])
        shape = (cap, bs, w.num_kv_heads, w.head_dim)
        self.kc = wl.host_normal_fp16(rng, shape)
        self.vc = wl.host_normal_fp16(rng, shape)
        self.q = wl.host_normal_fp16(rng, (max_seqs, w.num_q_heads, w.head_dim))
        self.k_new = wl.host_normal_fp16(rng, (max_seqs, w.num_kv_heads, w.head_dim))
        self.v_new = wl.host_normal_fp16(rng, (max_seqs, w.num_kv_heads, w.head_dim))

    def time(self, seqs, min_seconds=0.0, threads=None):
        """(seconds, KV bytes attended over in that time, threads used): the
        sample repeated until at least min_seconds of oracle time."""
        import numpy as np

        from oracle import attention as oa
        from oracle import cache_ops as oc
        from paged_kv_cache_138_gb300 import accounting
        w, bs = self.w, self.w.block_size
        lens = np.ascontiguousarray(self.lens[seqs], dtype=np.int32)
        remap = {}
        rows = []
        for s, L in zip(seqs, lens):
            ids = [int(b) for b in self.tables[s][:-(-int(L) // bs)]]
            rows.append([remap.setdefault(b, len(remap)) for b in ids])
        t2 = np.full((len(seqs), max(len(r) for r in rows)), -1, dtype=np.int32)
        for i, r in enumerate(rows):
            t2[i, :len(r)] = r
        # the new token of each sequence sits at position L - 1 (the slot rule)
        slots = np.array([oc.slot(t2[i], int(L) - 1, bs) for i, L in enumerate(lens)],
                         dtype=np.int64)
        n = len(seqs)
        q, kn, vn = self.q[:n], self.k_new[:n], self.v_new[:n]
        si = np.repeat(np.arange(n, dtype=np.int32), w.num_q_heads)
        hi = np.tile(np.arange(w.num_q_heads, dtype=np.int32), n)
        kv_once = accounting.step_kv_bytes(lens, w.num_kv_heads, w.head_dim)
        dt, kv = 0.0, 0.0
        all_threads = oa.num_threads()
        if threads is not None:
            oa.set_num_threads(threads)
        try:
            while True:
                t0 = time.perf_counter()
                oc.reshape_and_cache(kn, vn, slots, self.kc, self.vc)
                oa.paged_attention_decode_rows(q, self.kc, self.vc, t2, lens, w.scale, si, hi)
                dt += time.perf_counter() - t0
                kv += kv_once
                if dt >= min_seconds:
                    return dt, kv, oa.num_threads()
        finally:
            oa.set_num_threads(all_threads)


def oracle_metadata(w):
    """The oracle's own batch (tables, lengths, slots, COW pairs, pool size)."""
    from oracle.batch import oracle_batch
    return oracle_batch(w)


def cpu_baseline(w, tables, lens):
    """The oracle on the host cores: 8 random sequences x every head of layer 0
    for ~10 s with every core, and 2 of them on one core for ~3 s."""
    import numpy as np
    from oracle.build import build_oracle
    build_oracle()
    S = len(lens)
    seqs = sorted(np.random.default_rng(3).choice(S, size=min(S, REFERENCE_SAMPLE_SEQS),
                                                  replace=False).tolist())
    smp = OracleSampler(w, tables, lens, len(seqs), seed=w.seed)
    tot_t, tot_kv, threads = smp.time(seqs, min_seconds=10.0)
    cpu = {"value": tot_kv / tot_t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": "%d random of %d sequences x all %d heads of layer 0 (reshape_and_cache "
                     "+ attention), repeated for %.1f s (fp64 C oracle, OpenMP; host-drawn "
                     "inputs)" % (len(seqs), S, w.num_q_heads, tot_t)}
    t1, kv1, _ = smp.time(seqs[:2], min_seconds=3.0, threads=1)
    cpu["single_thread"] = {"value": kv1 / t1 / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": "%d sequences x all %d heads, repeated for %.1f s" % (
                                min(2, len(seqs)), w.num_q_heads, t1)}
    return cpu


def run_reference(args):
    """The reference arm: the CPU fp64 oracle, timed on this host's cores, on
    bounded samples of the same workload.  It loads no GPU code of this
    repository: metadata from the oracle's BlockManager, values drawn on the
    host, the oracle's C library."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    if args.workload not in DECODE_WORKLOADS:
        print(json.dumps({"impl": "reference", "unavailable":
                          "no oracle arm for the %s workload" % args.workload}))
        return 0
    l2 = device_l2_bytes()
    if l2 is None:
        print(json.dumps({"impl": "reference",
                          "unavailable": "no CUDA device: the workload's L2 rule needs it"}))
        return 0
    import numpy as np
    from oracle.build import build_oracle
    build_oracle()
    w = bench_workload(args)
    tables, lens, _, _, nb = oracle_metadata(w)
    cfg, kv_step, _ = workload_config(w, tables, lens, nb, l2)
    S = len(lens)
    n = min(S, REFERENCE_SAMPLE_SEQS)
    smp = OracleSampler(w, tables, lens, n, seed=w.seed)
    rng = np.random.default_rng(5)
    times, kvs, threads = [], [], 1
    for i in range(args.warmup + args.steps):
        seqs = sorted(rng.choice(S, size=n, replace=False).tolist())
        dt, kv, threads = smp.time(seqs)
        if i >= args.warmup:
            times.append(dt)
            kvs.append(kv)
    value = sum(kvs) / sum(times) / 1e9
    sample = ("%d steps, each %d random of %d sequences x all %d heads of one layer "
              "(fp64 oracle; host-drawn inputs)" % (args.steps, n, S, w.num_q_heads))
    ms_full = 1e3 * kv_step / (value * 1e9)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_full, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "ms_per_step_note": "a full step of the workload (%d layers x %d sequences) at "
                                "the sampled rate; each timed sample took %.2f ms on average"
                                % (w.num_layers, S, 1e3 * sum(times) / len(times)),
            "seq_steps_per_s": world * S / (ms_full / 1e3),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def setup(args, device, rank=0):
    from paged_kv_cache_138_gb300.engine import DecodeStep
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    w = bench_workload(args, rank)
    batch = prepare_batch(w)
    grouped = {"on": True, "off": False}.get(getattr(args, "grouped", "auto"),
                                              args.workload == "prefix-sharing")
    step = DecodeStep(batch, device=device, fused=not getattr(args, "unfused", False),
                      grouped=grouped, fold_cow=not getattr(args, "cow_kernel", False))
    return w, batch, step


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from paged_kv_cache_138_gb300 import build as nb
    if rank == 0:
        nb.build()
    if world > 1:
        torch.distributed.barrier()
    w, batch, step = setup(args, device, rank)
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size
    cfg, kv_bytes, unique_kv = workload_config(w, batch.block_tables, batch.context_lens,
                                               batch.num_blocks, l2_bytes)
    stream = torch.cuda.current_stream(device)
    # a step whose bytes L2 could hold across steps gets L2 flushed between
    # timed steps (a write of a buffer 4x the L2 size); each step is then timed
    # by its own event pair so the flush stays outside the measured time
    step_bytes = unique_kv if unique_kv is not None else kv_bytes / w.num_layers
    flush_buf = (torch.empty(max(4 * l2_bytes, 512 << 20), dtype=torch.uint8, device=device)
                 if step_bytes < 4 * l2_bytes else None)

    def flush_l2():
        if flush_buf is not None:
            flush_buf.zero_()

    def per_step_timed(n, body):
        """n steps of body(), each between its own events, L2 flushed after each;
        returns the per-step device times (ms)."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            a.record(stream)
            body()
            b.record(stream)
            flush_l2()
        torch.cuda.synchronize(device)
        return [a.elapsed_time(b) for a, b in ev]

    def one_step():
        step.apply_cow(stream)
        step.run(stream)

    clocks = ClockSampler(device.index).start()
    for _ in range(max(args.warmup, 3)):
        one_step()
    torch.cuda.synchronize(device)
    step.check_errors()

    # ---- device-resident timed region: exactly --steps steps -------------------------
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.ready()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    t_host0 = time.time()
    if flush_buf is None:
        start.record(stream)
        for _ in range(args.steps):
            one_step()
        stop.record(stream)
        torch.cuda.synchronize(device)
    else:
        step_ms = per_step_timed(args.steps, one_step)
    t_host1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = start.elapsed_time(stop) if flush_buf is None else sum(step_ms)
    step.check_errors()
    if world > 1:
        t = torch.tensor([elapsed_ms], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    ms_per_step = elapsed_ms / args.steps
    value = world * kv_bytes / (ms_per_step / 1e3) / 1e9

    # ---- the attention launch alone: ROOFLINE_LAUNCHES back to back between two
    # events (layer after layer), each launch waiting on nothing but the previous one
    n_attn = max(ROOFLINE_LAUNCHES, step.num_layers)
    for i in range(step.num_layers):
        step.attend(i, stream)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    t_attn0 = time.time()
    a0.record(stream)
    for j in range(n_attn):
        step.attend(j % step.num_layers, stream)
    a1.record(stream)
    torch.cuda.synchronize(device)
    t_attn1 = time.time()
    attn_ms = a0.elapsed_time(a1) / n_attn
    step.check_errors()

    # ---- end to end through the public API from pinned host buffers ----------------
    # every step copies its inputs (q, new K/V, slots, block tables, context
    # lengths) from pinned host memory and its output back; the copies of step
    # k+1 and k-1 run on a copy stream beside step k's kernels
    per_window = args.e2e_steps or E2E_STEPS_PER_WINDOW
    h2d, d2h = step.host_bytes_per_step()
    host = step.host_buffers()
    step.run_from_host_pipelined([host] * 3, [host["out"]] * 3, stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    # E2E_WINDOWS back-to-back windows, each with its own warm start; the median
    # window is reported (one host stall -- a page fault, another process --
    # would otherwise be spread over every step of a single window)
    import gc
    windows = []
    gc.disable()
    try:
        for _ in range(E2E_WINDOWS):
            if flush_buf is not None:
                # L2 flushed between steps: no overlap of neighbouring steps
                windows.append(sum(per_step_timed(per_window, lambda: step.run_from_host(stream)))
                               / per_window)
                continue
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step.run_from_host_pipelined([host] * per_window, [host["out"]] * per_window,
                                         stream)
            stream.wait_stream(step._pipe.copy)
            e1.record(stream)
            torch.cuda.synchronize(device)
            windows.append(e0.elapsed_time(e1) / per_window)
    finally:
        gc.enable()
    e2e_ms = sorted(windows)[len(windows) // 2]
    e2e_mean_ms = sum(windows) / len(windows)
    if world > 1:
        t = torch.tensor([e2e_ms], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_value = world * kv_bytes / (e2e_ms / 1e3) / 1e9

    # ---- the same step replayed from a CUDA graph (one launch call per step) ---------
    step.capture_graph()
    for _ in range(3):
        step.replay()
    torch.cuda.synchronize(device)
    if flush_buf is None:
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            step.replay()
        g1.record(stream)
        torch.cuda.synchronize(device)
        graph_ms = g0.elapsed_time(g1) / args.steps
    else:
        graph_ms = sum(per_step_timed(args.steps, step.replay)) / args.steps
    step.check_errors()

    # ---- a step that L2 could partly keep between steps (under 8x its size):
    # also timed step by step with L2 flushed after each (besides the main
    # figure, which runs back to back on inputs larger than L2)
    flushed = None
    if flush_buf is None and step_bytes < 8 * l2_bytes:
        flush_buf = torch.empty(max(4 * l2_bytes, 512 << 20), dtype=torch.uint8, device=device)
        n_fl = min(max(args.steps, 50), 500)
        fl_ms = sum(per_step_timed(n_fl, one_step)) / n_fl
        flushed = {"ms_per_step": fl_ms, "value": world * kv_bytes / (fl_ms / 1e3) / 1e9,
                   "unit": "GB/s", "steps": n_fl,
                   "note": "each step between its own events, L2 flushed by a %d MiB write "
                           "after each" % (flush_buf.numel() >> 20)}
        flush_buf = None
        step.check_errors()
    clocks.stop()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak, peak_kind = hbm_peak()
    # forked samples share prompt blocks: the roofline counts each distinct
    # (block, row) once -- what HBM must deliver at minimum
    layer_kv = unique_kv if unique_kv is not None else kv_bytes / w.num_layers
    achieved = layer_kv / (attn_ms / 1e3) / 1e9
    tr = traffic_record(("fused/" if step.fused else "") + "paged_attention_decode/" +
                        args.workload + ("" if w.block_size == 16 else "/bs%d" % w.block_size))
    share = attn_ms * step.num_layers / ms_per_step
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "algorithmic_bytes_per_launch": layer_kv,
                "launch_ms": attn_ms, "launches": n_attn,
                "timing": "CUDA events around %d back-to-back attention launches (layers in "
                          "turn), independent of --steps; launch_ms = elapsed / launches"
                          % n_attn,
                "launches_x_layers_over_step": share,
                "consistency": ("the launch alone takes %.1f %% of the step per layer: the "
                                "rest of the step is %s" % (100 * share, "the copy-on-write "
                                "copy" if step.cow_launches_per_step() else
                                "stream gaps between launches") if share <= 1.0 else
                                "the launch alone is slower than its share of the step"),
                "kernel": ("paged_attention_decode_grouped%s (%sshared-prefix + own-tile "
                           "units, then the LSE merge kernel)"
                           % (("_fused", "cache write + ") if step.fused else ("", ""))
                           if step.groups is not None else
                           "paged_attention_decode_fused (cache write + split kernel, then "
                           "the LSE merge kernel)" if step.fused else
                           "paged_attention_decode (split kernel, then the LSE merge kernel)"),
                "clocks": clocks.summary(t_attn0, t_attn1),
                "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS}
    cpu = None
    if not args.no_cpu_baseline:
        o_tables, o_lens, _, _, _ = oracle_metadata(w)
        cpu = cpu_baseline(w, o_tables, o_lens)
    launches = step.kernel_launches_per_step() + step.cow_launches_per_step()
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 (fp32 accumulate)",
        "data": "synthetic",
        "config": cfg,
        "impl_config": {"fused_cache_write": step.fused,
                        "grouped_shared_prefix": step.groups is not None,
                        "cow_copies": ("inside the attention launches" if step.cow is not None
                                       else "copy_blocks" if batch.cow_pairs.shape[0]
                                       else None),
                        "split_tokens": step.split_tokens()},
        "seq_steps_per_s": world * batch.num_seqs / (ms_per_step / 1e3),
        "pct_of_hbm_peak": {"measured": 100 * value / world / peak if peak_kind == "measured"
                            else None, "nominal_8tbs": 100 * value / world / NOMINAL_HBM_GBS},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "mean_ms_per_step": e2e_mean_ms, "windows": len(windows),
                "steps_per_window": per_window,
                "timing": "median of %d windows of %d pipelined steps" % (len(windows),
                                                                           per_window)},
        "l2_flushed": flushed,
        "graph": {"ms_per_step": graph_ms, "value": world * kv_bytes / (graph_ms / 1e3) / 1e9,
                  "unit": "GB/s", "note": "same step replayed from a CUDA graph"},
        "gpu_launches": launches * args.steps,
        "clocks": dict(clocks.summary(t_host0, t_host1),
                       window_s=round(t_host1 - t_host0, 4),
                       note="samples stamped inside the timed region"),
        "clocks_whole_run": clocks.summary(),
    }
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_serving(args):
    """Steady-state continuous batching (host BlockManager in the loop): a trace
    of requests sharing 4 system prompts of 1024 tokens plus private suffixes,
    64..512 new tokens each, decoded at batch <= 64 on the Llama-2-13B layer
    shape.  Time covers whole steps: admissions, prefill writes, appends,
    metadata copies, reshape_and_cache and attention."""
    import torch

    from paged_kv_cache_138_gb300 import workloads as wl
    from paged_kv_cache_138_gb300.driver import ContinuousBatchDriver, DeviceSources
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    Hq = Hkv = 40
    reqs = wl.serving_requests(2024, num_requests=4096, num_system_prompts=4,
                               system_prompt_len=1024, suffix_max=512, new_min=64, new_max=512)
    nb = 64 * 110
    grouped = args.grouped == "on"
    native = args.driver == "native"
    if native:
        from paged_kv_cache_138_gb300.serving import DeviceRandomValues, NativeServingDriver
        grouped = args.grouped != "off"
        drv = NativeServingDriver(nb, Hq, Hkv, max_batch=64, max_blocks_per_seq=160,
                                  values=DeviceRandomValues(7, Hq, Hkv, device=device),
                                  device=device, seed=7, grouped=grouped)
    else:
        drv = ContinuousBatchDriver(nb, Hq, Hkv, max_batch=64, max_blocks_per_seq=160,
                                    sources=DeviceSources(7, Hq, Hkv), device=device,
                                    grouped=grouped)
    for r in reqs:
        drv.add_request(r.rid, r.prompt, r.max_new_tokens)
    import gc
    gc.collect()
    gc.freeze()     # the trace's token lists are long-lived: keep them out of GC scans
    stats = {"seq_steps": 0, "kv_tokens": 0, "preempted": 0, "admitted": 0, "cached": 0,
             "prefill": 0, "shared_tokens": 0}
    for _ in range(max(args.warmup, 3) * 20):
        drv.step()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    steps = min(args.steps, 2000)
    for _ in range(steps):
        res = drv.step()
        if native:
            stats["shared_tokens"] += res["shared_tokens"]
            stats["seq_steps"] += len(res["rids"])
            stats["kv_tokens"] += res["kv_tokens"]
            stats["preempted"] += res["preempted"]
            stats["admitted"] += res["admitted"]
            stats["cached"] += res["cached"]
            stats["prefill"] += res["prefill"]
            continue
        stats["seq_steps"] += len(res.rids)
        stats["kv_tokens"] += res.kv_tokens
        stats["preempted"] += len(res.preempted)
        stats["admitted"] += len(res.admitted)
        stats["cached"] += res.cached_tokens
        stats["prefill"] += res.prefill_tokens
        stats["shared_tokens"] += res.shared_tokens
    e1.record()
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    drv.check_errors()
    kv_bytes = stats["kv_tokens"] * 2 * Hkv * 128 * 2
    line = {"metric": METRIC, "value": kv_bytes / wall / 1e9, "unit": "GB/s", "n_gpus": 1,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": "serving", "description": " ".join(
                run_serving.__doc__.split(".")[0].split()),
                       "max_batch": 64, "pool_blocks": nb, "heads": Hq,
                       "grouped_shared_prefix": grouped,
                       "scheduler": "native (pkv_sched_step)" if native else "python"},
            "seq_steps_per_s": stats["seq_steps"] / wall,
            "device_ms_per_step": e0.elapsed_time(e1) / steps, "stats": stats}
    print(json.dumps(line))
    return 0


def run_swap(args):
    """swap_blocks bandwidth over the host link: device pool -> pinned host pool
    (swap-out) and back (swap-in), 1024 random blocks of K and V of the
    Llama-2-7B shape (32 KV heads: 128 KiB per block per cache), against a
    plain contiguous cudaMemcpy of the same bytes."""
    import numpy as np
    import torch

    from paged_kv_cache_138_gb300 import ops
    device = torch.device("cuda", 0)
    nb, hb, n = 4096, 2048, 1024
    shape = (16, 32, 128)
    k = torch.randn((nb,) + shape, device=device).half()
    v = torch.randn((nb,) + shape, device=device).half()
    hk = torch.empty((hb,) + shape, dtype=torch.float16, pin_memory=True)
    hv = torch.empty_like(hk).pin_memory()
    rng = np.random.default_rng(1)
    out_pairs = torch.from_numpy(np.stack([rng.choice(nb, n, replace=False),
                                           rng.choice(hb, n, replace=False)], 1)).to(device)
    in_pairs = out_pairs[:, [1, 0]].contiguous()
    err = ops.new_error_word(device)
    nbytes = 2 * n * k[0].numel() * 2

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / reps / 1e3

    reps = max(3, min(args.steps, 20))
    t_out = timed(lambda: ops.swap_blocks([k, v], [hk, hv], out_pairs, dev_err=err), reps)
    t_in = timed(lambda: ops.swap_blocks([hk, hv], [k, v], in_pairs, dev_err=err), reps)
    flat_d = torch.empty(nbytes // 2, dtype=torch.float16, device=device)
    flat_h = torch.empty(nbytes // 2, dtype=torch.float16, pin_memory=True)
    t_ref_out = timed(lambda: flat_h.copy_(flat_d, non_blocking=True), reps)
    t_ref_in = timed(lambda: flat_d.copy_(flat_h, non_blocking=True), reps)
    assert ops.read_error_word(err) == 0
    line = {"metric": "swap_blocks GB/s (device <-> pinned host)", "value": nbytes / t_out / 1e9,
            "unit": "GB/s", "n_gpus": 1, "steps": reps, "warmup": 3,
            "ms_per_step": t_out * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bytes", "data": "synthetic",
            "config": {"workload": "swap", "blocks": n, "bytes_per_direction": nbytes},
            "swap_out_gbs": nbytes / t_out / 1e9, "swap_in_gbs": nbytes / t_in / 1e9,
            "contiguous_memcpy_d2h_gbs": nbytes / t_ref_out / 1e9,
            "contiguous_memcpy_h2d_gbs": nbytes / t_ref_in / 1e9}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "serving":
        return run_serving(args)
    if args.workload == "swap":
        return run_swap(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
