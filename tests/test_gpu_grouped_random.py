"""Seeded random sweep of grouped (shared-prefix) attention against the fp64 oracle.

Each case draws the query/KV head ratio, KV heads, block size, a set of groups
(1..16/G members each) sharing a prefix of 0..2048 tokens (a multiple of the
block size and of 16), per-member private lengths (an empty row among them in
plain launches) and plain or fused launch.
The batch goes through the host planner and the grouped entry point; the
output is compared element by element with the oracle's plain attention over
the same tables and, for fused launches, the cache bytes with the oracle's
cache write.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import cache_ops as oc
from parity_helpers import assert_matches_oracle
from paged_kv_cache_138_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def draw_case(seed):
    rng = np.random.default_rng(7000 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([8, 16, 32, 64]))
    fused = bool(seed % 2)
    unit = max(16, bs)
    rows = []            # per sequence: its block ids before they are scattered over the pool
    lens = []
    next_block = 0
    for _ in range(int(rng.integers(1, 9))):
        members = int(rng.integers(1, 16 // G + 1))
        prefix = unit * int(rng.integers(0, 2048 // unit + 1))
        pb = prefix // bs
        shared = list(range(next_block, next_block + pb))
        next_block += pb
        for _ in range(members):
            own = int(rng.integers(1 if fused else 0, 700))
            L = prefix + own
            extra = wl.blocks_for(L, bs) - pb
            rows.append(shared + list(range(next_block, next_block + extra)))
            next_block += extra
            lens.append(L)
    if not fused:                                     # an empty row among the groups
        at = int(rng.integers(0, len(rows) + 1))
        rows.insert(at, [])
        lens.insert(at, 0)
    nb = next_block + 2
    perm = rng.permutation(nb).astype(np.int32)       # scatter the blocks over the pool
    mb = max(1, max(len(r) for r in rows))
    tables = np.full((len(rows), mb), -1, np.int32)
    for i, r in enumerate(rows):
        tables[i, :len(r)] = perm[r]
    return rng, G * Hkv, Hkv, bs, tables, np.array(lens, np.int32), nb, fused


@pytest.mark.parametrize("seed", range(16))
def test_random_grouped_case_matches_oracle(ops, seed):
    rng, Hq, Hkv, bs, tables, lens, nb, fused = draw_case(seed)
    S = len(lens)
    q = wl.host_normal_fp16(rng, (S, Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, bs, 16 // (Hq // Hkv))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    dk, dv = dev(kc), dev(vc)
    err = ops.new_error_word()
    scale = 1 / np.sqrt(D)
    if fused:
        k_new = wl.host_normal_fp16(rng, (S, Hkv, D))
        v_new = wl.host_normal_fp16(rng, (S, Hkv, D))
        ops.paged_attention_decode_grouped_fused(out, dev(q), dev(k_new), dev(v_new), dk, dv,
                                                 dev(tables), dev(lens), dev(gf), dev(sg),
                                                 dev(gs), mx, mo, scale, dev_err=err)
        slots = np.array([oc.slot(tables[s], int(L) - 1, bs) for s, L in enumerate(lens)],
                         np.int64)
        oc.reshape_and_cache(k_new, v_new, slots, kc, vc)
    else:
        ops.paged_attention_decode_grouped(out, dev(q), dk, dv, dev(tables), dev(lens), dev(gf),
                                           dev(sg), dev(gs), mx, mo, scale, dev_err=err)
    assert ops.read_error_word(err) == 0
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    assert_matches_oracle(out.cpu().numpy(), ref, (S, Hq, Hkv, bs, fused, list(gs)))
    if fused:
        assert np.array_equal(dk.cpu().numpy().view(np.uint16), kc.view(np.uint16))
        assert np.array_equal(dv.cpu().numpy().view(np.uint16), vc.view(np.uint16))
