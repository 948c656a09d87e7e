"""Every benchmark workload at its full size, run through DecodeStep as
bench.py runs it (copy_blocks for COW pairs, then per layer reshape_and_cache
and paged attention; the prefix-sharing step also in the benchmark's fused,
grouped form with the copies inside the launch), checked against the oracle.

The oracle gets host copies of the caches taken BEFORE the step and applies its
own copy_blocks and reshape_and_cache; nothing the GPU wrote is an oracle input.
Small workloads are compared on every output row, large ones on seeded samples
of rows the oracle evaluates one by one.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import cache_ops as oc
from parity_helpers import assert_matches_oracle, attention_tolerance, oracle_batch
from paged_kv_cache_138_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
TOL = attention_tolerance()


def run_and_check(name, layers_checked, rows_per_layer, all_rows=False, fused=False,
                  grouped=False, whole_cache=False):
    from paged_kv_cache_138_gb300.engine import DecodeStep
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    w = wl.WORKLOADS[name]
    batch = prepare_batch(w)
    tables, lens, slots, pairs, nb = oracle_batch(w)
    assert np.array_equal(batch.block_tables, tables) and np.array_equal(batch.slot_mapping, slots)
    step = DecodeStep(batch, fused=fused, grouped=grouped)
    before = {i: (step.k_cache[i].cpu().numpy(), step.v_cache[i].cpu().numpy())
              for i in layers_checked}
    step.apply_cow()
    out = step.run()
    step.check_errors()
    torch.cuda.synchronize()
    rng = np.random.default_rng(77)
    S, Hq = batch.num_seqs, w.num_q_heads
    worst = 0.0
    for i in layers_checked:
        kc, vc = before[i]
        oc.copy_blocks([kc], [vc], pairs)
        oc.reshape_and_cache(step.k_new[i].cpu().numpy(), step.v_new[i].cpu().numpy(), slots,
                             kc, vc)
        q = step.q[i].cpu().numpy()
        gpu = out[i].cpu().numpy().astype(np.float64)
        if all_rows:
            ref = oa.paged_attention_decode(q, kc, vc, tables, lens, w.scale)
            part = gpu
        else:
            si = rng.integers(0, S, size=rows_per_layer).astype(np.int32)
            hi = rng.integers(0, Hq, size=rows_per_layer).astype(np.int32)
            si[:2] = [int(np.argmax(lens)), int(np.argmin(lens))]   # longest and shortest
            ref = oa.paged_attention_decode_rows(q, kc, vc, tables, lens, w.scale, si, hi)
            part = gpu[si, hi]
        assert np.isfinite(gpu).all()
        worst = max(worst, float(np.abs(part - ref).max()))
        assert_matches_oracle(part, ref, (name, i))
        if whole_cache:
            # every block: copies, new tokens and untouched blocks, bit for bit
            assert np.array_equal(step.k_cache[i].cpu().numpy().view(np.uint16),
                                  kc.view(np.uint16))
            assert np.array_equal(step.v_cache[i].cpu().numpy().view(np.uint16),
                                  vc.view(np.uint16))
        # the new token's K/V landed at its slot, bit for bit
        bs = w.block_size
        for s in rng.integers(0, S, size=8):
            b, o = divmod(int(slots[s]), bs)
            assert np.array_equal(step.k_cache[i, b, o].cpu().numpy().view(np.uint16),
                                  kc[b, o].view(np.uint16))
    report = os.environ.get("PKV_PARITY_REPORT")
    if report:
        with open(report, "a") as f:
            f.write(json.dumps({"workload": name, "max_abs_err": worst, "tol": TOL,
                                "rows": "all" if all_rows else rows_per_layer,
                                "layers": list(layers_checked)}) + "\n")
    assert worst <= TOL, "max abs error %.3g" % worst
    return worst


def test_llama2_13b_layer_full_size(native_lib):
    run_and_check("llama2-13b-layer", [0], 0, all_rows=True)


def test_gqa_32_8_full_size(native_lib):
    run_and_check("gqa-32-8", [0], 256)


def test_prefix_sharing_full_size(native_lib):
    run_and_check("prefix-sharing", [0], 0, all_rows=True)


def test_prefix_sharing_full_size_as_benchmarked(native_lib):
    """The benchmark's form of the step: one fused grouped launch that also
    makes the 120 copy-on-write copies; the whole cache must equal the
    oracle's copy_blocks + reshape_and_cache, every output row the oracle's."""
    run_and_check("prefix-sharing", [0], 0, all_rows=True, fused=True, grouped=True,
                  whole_cache=True)


def test_llama2_7b_32_layer_full_size(native_lib):
    run_and_check("llama2-7b-32layer", [0, 31], 96)


def test_llama2_7b_single_layer_full_size(native_lib):
    run_and_check("llama2-7b-layer", [0], 128)


def test_llama2_7b_every_layer_sampled(native_lib):
    """All 32 layers of the 7B step.  Per layer a few sequences are drawn and
    only their blocks are copied to the host before the step (compacted,
    tables renumbered); the oracle applies its own cache write of those
    sequences' new tokens and evaluates every query head of them."""
    from paged_kv_cache_138_gb300.engine import DecodeStep
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    w = wl.WORKLOADS["llama2-7b-32layer"]
    batch = prepare_batch(w)
    tables, lens, slots, pairs, nb = oracle_batch(w)
    assert len(pairs) == 0
    step = DecodeStep(batch)
    rng = np.random.default_rng(79)
    S, Hq, bs = batch.num_seqs, w.num_q_heads, w.block_size
    picked = {}
    for i in range(step.num_layers):
        seqs = np.sort(rng.choice(S, size=3, replace=False))
        blocks = sorted({int(b) for s in seqs for b in tables[s][:-(-int(lens[s]) // bs)]})
        idx = torch.tensor(blocks, dtype=torch.long, device=step.k_cache.device)
        picked[i] = (seqs, blocks, step.k_cache[i].index_select(0, idx).cpu().numpy(),
                     step.v_cache[i].index_select(0, idx).cpu().numpy())
    out = step.run()
    step.check_errors()
    torch.cuda.synchronize()
    worst = 0.0
    for i, (seqs, blocks, kc, vc) in picked.items():
        remap = {b: j for j, b in enumerate(blocks)}
        t2 = np.array([[remap.get(int(b), -1) if b >= 0 else -1 for b in tables[s]]
                       for s in seqs], dtype=np.int32)
        s2 = np.array([remap[int(slots[s]) // bs] * bs + int(slots[s]) % bs for s in seqs],
                      dtype=np.int64)
        oc.reshape_and_cache(step.k_new[i].cpu().numpy()[seqs], step.v_new[i].cpu().numpy()[seqs],
                             s2, kc, vc)
        q = step.q[i].cpu().numpy()[seqs]
        si = np.repeat(np.arange(len(seqs), dtype=np.int32), Hq)
        hi = np.tile(np.arange(Hq, dtype=np.int32), len(seqs))
        ref = oa.paged_attention_decode_rows(q, kc, vc, t2, lens[seqs], w.scale, si, hi)
        gpu = out[i].cpu().numpy().astype(np.float64)[seqs[si], hi]
        assert_matches_oracle(gpu, ref, ("layer", i))
        worst = max(worst, float(np.abs(gpu - ref).max()))
    assert worst <= TOL, "max abs error %.3g" % worst


def test_graph_replay_matches_eager(native_lib):
    """One decode step captured in a CUDA graph gives the eager step's bits."""
    from paged_kv_cache_138_gb300.engine import DecodeStep
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    w = wl.WORKLOADS["prefix-sharing"]
    step = DecodeStep(prepare_batch(w))
    step.apply_cow()
    eager = step.run().clone()
    step.capture_graph()
    step.out.zero_()
    step.replay()
    torch.cuda.synchronize()
    step.check_errors()
    assert torch.equal(step.out.view(torch.int16), eager.view(torch.int16))


def test_pipelined_host_steps_match_sequential(native_lib):
    """Double-buffered end-to-end steps (copies overlapping kernels) produce the
    same outputs as one-at-a-time steps, for inputs that differ per step."""
    from paged_kv_cache_138_gb300.engine import DecodeStep
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    w = wl.WORKLOADS["llama2-13b-layer"]
    step = DecodeStep(prepare_batch(w))
    base = step.host_buffers()
    g = torch.Generator().manual_seed(5)
    inputs, outs_seq, outs_pipe = [], [], []
    for k in range(5):
        d = {n: base[n].clone().pin_memory() for n in step._INPUTS}
        d["q"].copy_(torch.randn(d["q"].shape, generator=g).half())
        d["k_new"].copy_(torch.randn(d["k_new"].shape, generator=g).half())
        d["v_new"].copy_(torch.randn(d["v_new"].shape, generator=g).half())
        inputs.append(d)
        outs_pipe.append(torch.empty_like(base["out"]).pin_memory())
    for d in inputs:                       # reference: one step at a time
        for n in step._INPUTS:
            getattr(step, n).copy_(d[n])
        step.run()
        outs_seq.append(step.out.cpu())
    step.run_from_host_pipelined(inputs, outs_pipe)
    torch.cuda.synchronize()
    step.check_errors()
    for a, b in zip(outs_seq, outs_pipe):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(outs_seq[0], outs_seq[1])
