"""Paged decode attention on the GPU against the fp64 oracle, element by element.

Tolerance: max |out_gpu - out_oracle| <= 2e-3 on fp16 outputs (fp16 inputs,
fp32 accumulation on the GPU, one fp16 rounding of the result).  Calls go
through the C ABI (ops -> libpagedkv.so).
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
D = 128


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def case(seed, lengths, Hq, Hkv, extra=5, pad=-1):
    rng = np.random.default_rng(seed)
    need = [wl.blocks_for(L) for L in lengths]
    nb = sum(need) + extra
    order = rng.permutation(nb).astype(np.int32)
    tables = wl.handout_tables(lengths, order, pad=pad)
    q = wl.host_normal_fp16(rng, (len(lengths), Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    return q, kc, vc, tables, np.array(lengths, dtype=np.int32)


def run_gpu(ops, q, kc, vc, tables, lens, scale, err=None):
    out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
    e = ops.new_error_word() if err is None else err
    ops.paged_attention_decode(out, torch.from_numpy(q).cuda(), torch.from_numpy(kc).cuda(),
                               torch.from_numpy(vc).cuda(), torch.from_numpy(tables).cuda(),
                               torch.from_numpy(lens).cuda(), scale, dev_err=e)
    code = ops.read_error_word(e)
    return out.cpu().numpy(), code


def assert_close(gpu, ref):
    assert_matches_oracle(gpu, ref)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (32, 8), (16, 2), (40, 40)])
@pytest.mark.parametrize("lengths", [
    [7, 16, 31, 48, 63],
    [1, 15, 16, 17, 33],
    [511, 512, 513, 1000, 2049, 4096],
])
def test_attention_matches_oracle(ops, Hq, Hkv, lengths):
    q, kc, vc, tables, lens = case(sum(lengths) + Hq, lengths, Hq, Hkv)
    scale = 1.0 / np.sqrt(D)
    gpu, code = run_gpu(ops, q, kc, vc, tables, lens, scale)
    assert code == 0
    assert_close(gpu, oa.paged_attention_decode(q, kc, vc, tables, lens, scale))


def test_zero_length_rows_are_zero(ops):
    q, kc, vc, tables, lens = case(3, [0, 20, 0, 600], 8, 2)
    gpu, code = run_gpu(ops, q, kc, vc, tables, lens, 0.0883883)
    assert code == 0
    assert (gpu[0] == 0).all() and (gpu[2] == 0).all()
    assert_close(gpu, oa.paged_attention_decode(q, kc, vc, tables, lens, 0.0883883))


def test_nan_poison_past_context_never_read(ops):
    lengths = [5, 16, 33, 700]
    q, kc, vc, tables, lens = case(4, lengths, 16, 4, extra=9)
    used = np.zeros(kc.shape[:2], dtype=bool)
    for s, L in enumerate(lengths):
        for t in range(L):
            used[tables[s][t // 16], t % 16] = True
    kc[~used] = np.float16(np.nan)
    vc[~used] = np.float16(np.nan)
    scale = 1.0 / np.sqrt(D)
    gpu, code = run_gpu(ops, q, kc, vc, tables, lens, scale)
    assert code == 0
    assert_close(gpu, oa.paged_attention_decode(q, kc, vc, tables, lens, scale))


def test_permutation_of_placement_is_bit_exact(ops):
    q, kc, vc, tables, lens = case(5, [100, 1500, 37], 8, 2)
    rng = np.random.default_rng(50)
    nb = kc.shape[0]
    pi = rng.permutation(nb)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    t2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1).astype(np.int32)
    a, _ = run_gpu(ops, q, kc, vc, tables, lens, 0.1)
    b, _ = run_gpu(ops, q, kc2, vc2, t2, lens, 0.1)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def split_tiles(ops, S, Hkv, max_blocks, bs=16):
    """The split length (16-token tiles) the launch picks for these sizes."""
    return ops.split_tokens(S, Hkv, max_blocks, bs) // 16


@pytest.mark.parametrize("S,Hkv,G,T", [(256, 4, 2, 128), (32, 8, 4, 64), (8, 8, 1, 32)])
@pytest.mark.parametrize("fused", [False, True])
def test_every_split_length_matches_oracle(ops, S, Hkv, G, T, fused):
    """Splits of 2048, 1024 and 512 tokens: a few long contexts (cut at every
    kind of boundary) among many short ones, plain and with the fused write."""
    rng = np.random.default_rng(S + T)
    lengths = rng.integers(1, 120, size=S)
    lengths[:6] = [4096, 2049, 2048, 1025, 513, 3000]
    lengths = lengths.tolist()
    q, kc, vc, tables, lens = case(S * 7 + T, lengths, Hkv * G, Hkv)
    assert split_tiles(ops, S, Hkv, tables.shape[1]) == T
    scale = 1 / np.sqrt(D)
    out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    err = ops.new_error_word()
    if fused:
        rng2 = np.random.default_rng(T)
        k_new = wl.host_normal_fp16(rng2, (S, Hkv, D))
        v_new = wl.host_normal_fp16(rng2, (S, Hkv, D))
        ops.paged_attention_decode_fused(out, torch.from_numpy(q).cuda(),
                                         torch.from_numpy(k_new).cuda(),
                                         torch.from_numpy(v_new).cuda(), dk, dv,
                                         torch.from_numpy(tables).cuda(),
                                         torch.from_numpy(lens).cuda(), scale, dev_err=err)
        slots = np.array([oc.slot(tables[s], int(L) - 1, 16) for s, L in enumerate(lengths)],
                         np.int64)
        oc.reshape_and_cache(k_new, v_new, slots, kc, vc)
    else:
        ops.paged_attention_decode(out, torch.from_numpy(q).cuda(), dk, dv,
                                   torch.from_numpy(tables).cuda(),
                                   torch.from_numpy(lens).cuda(), scale, dev_err=err)
    assert ops.read_error_word(err) == 0
    assert_close(out.cpu().numpy(), oa.paged_attention_decode(q, kc, vc, tables, lens, scale))
    if fused:
        assert np.array_equal(dk.cpu().numpy().view(np.uint16), kc.view(np.uint16))


def test_batch_order_does_not_change_any_bit(ops):
    """A sequence's splits depend on its own length only, so reordering the
    batch (sorted by length, then longest first) permutes the output rows bit
    for bit, whichever grid row each sequence lands on."""
    rng = np.random.default_rng(14)
    lengths = rng.integers(1, 3000, size=24).tolist()
    q, kc, vc, tables, lens = case(15, lengths, 32, 8)
    a, code = run_gpu(ops, q, kc, vc, tables, lens, 0.1)
    assert code == 0
    for order in (np.argsort(lens), np.argsort(lens)[::-1].copy()):
        b, code = run_gpu(ops, q[order], kc, vc, tables[order], lens[order], 0.1)
        assert code == 0
        assert np.array_equal(b.view(np.uint16), a[order].view(np.uint16))


def test_identity_table_equals_contiguous_layout(ops):
    # one sequence whose blocks are 0..n-1 in order: the paged kernel must give
    # what torch's dense attention gives on the same contiguous K/V
    L, Hq, Hkv = 777, 8, 8
    q, kc, vc, _, _ = case(6, [L], Hq, Hkv, extra=0)
    tables = np.arange(wl.blocks_for(L), dtype=np.int32)[None]
    gpu, _ = run_gpu(ops, q, kc, vc, tables, np.array([L], np.int32), 1.0 / np.sqrt(D))
    K = torch.from_numpy(kc.reshape(-1, Hkv, D)[:L].astype(np.float64)).permute(1, 0, 2)
    V = torch.from_numpy(vc.reshape(-1, Hkv, D)[:L].astype(np.float64)).permute(1, 0, 2)
    Q = torch.from_numpy(q[0].astype(np.float64))[:, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=1.0 / np.sqrt(D))
    assert_close(gpu[0], ref[:, 0].numpy())


def test_bad_metadata_is_reported_not_trapped(ops):
    q, kc, vc, tables, lens = case(7, [40, 40, 40], 8, 8)
    tables[1, 1] = kc.shape[0] + 100          # block id outside the pool
    gpu, code = run_gpu(ops, q, kc, vc, tables, lens, 0.1)
    assert code == 1                           # PKV_DEV_BAD_BLOCK_ID
    ref = oa.paged_attention_decode(q[[0, 2]], kc, vc, tables[[0, 2]], lens[[0, 2]], 0.1)
    assert_close(gpu[[0, 2]], ref)             # other sequences unaffected
    lens2 = lens.copy()
    lens2[2] = 16 * tables.shape[1] + 1        # longer than its table
    _, code = run_gpu(ops, q, kc, vc, np.where(tables < kc.shape[0], tables, 0).astype(np.int32),
                      lens2, 0.1)
    assert code == 2                           # PKV_DEV_BAD_CONTEXT_LEN


def test_tiny_workload_full_step(ops):
    """The whole hot path on the tiny workload: BlockManager -> slots ->
    reshape_and_cache -> paged attention, against the oracle's own chain."""
    from paged_kv_cache_138_gb300.engine import DecodeStep
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    w = wl.WORKLOADS["tiny"]
    batch = prepare_batch(w)
    hv = wl.host_tensors(w, batch.num_blocks)
    step = DecodeStep(batch, host_values=hv)
    out = step.run()
    step.check_errors()
    tables, lens, slots, _, _ = oracle_batch(w)
    q, k_new, v_new, kc, vc = [a.copy() for a in hv]
    oc.reshape_and_cache(k_new[0], v_new[0], slots, kc[0], vc[0])
    ref = oa.paged_attention_decode(q[0], kc[0], vc[0], tables, lens, w.scale)
    report = os.environ.get("PKV_PARITY_REPORT")
    if report:
        err = float(np.abs(out[0].cpu().numpy().astype(np.float64) - ref).max())
        with open(report, "a") as f:
            f.write(json.dumps({"workload": "tiny", "max_abs_err": err, "tol": TOL,
                                "rows": "all", "layers": [0]}) + "\n")
    assert_close(out[0].cpu().numpy(), ref)
    # the cache now holds each new token at its slot
    assert np.array_equal(step.k_cache.cpu().numpy().view(np.uint16), kc.view(np.uint16))


def test_long_context_and_many_sequences(ops):
    """Maximum-size edges: one 65,536-token context (128 splits of 512) next to
    short ones, and a batch of 4,096 short sequences in one launch."""
    lengths = [65536, 1, 4097, 16]
    q, kc, vc, tables, lens = case(11, lengths, 8, 2, extra=1)
    gpu, code = run_gpu(ops, q, kc, vc, tables, lens, 1 / np.sqrt(D))
    assert code == 0
    assert_close(gpu, oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D)))
    rng = np.random.default_rng(12)
    lengths = rng.integers(1, 64, size=4096).tolist()
    q, kc, vc, tables, lens = case(13, lengths, 4, 4, extra=0)
    gpu, code = run_gpu(ops, q, kc, vc, tables, lens, 0.1)
    assert code == 0
    assert_close(gpu, oa.paged_attention_decode(q, kc, vc, tables, lens, 0.1))
