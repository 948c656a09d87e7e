"""Seeded random sweep of paged attention against the fp64 oracle.

Each case draws the batch size, head counts (G in 1, 2, 4, 8), block size,
a length mix (uniform, ragged with empty rows, or lengths on block and split
boundaries) and plain or fused launch, so the launch picks every split length
and both kinds of grid row order; the output is compared element by element
(max |GPU - oracle| <= 2e-3, and in fp16 units of each row's largest value
a mean of at most 0.25 and a maximum of at most 3) and, for fused launches,
the cache bytes too.
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
    rng = np.random.default_rng(9000 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 4, 8, 16]))
    bs = int(rng.choice([8, 16, 32, 64]))
    S = int(rng.integers(1, 160))
    kind = seed % 3
    if kind == 0:
        lengths = np.full(S, int(rng.integers(1, 3000)))
    elif kind == 1:
        lengths = rng.integers(0, 4500, size=S)
    else:
        edges = [1, bs - 1, bs, bs + 1, 511, 512, 513, 1024, 1025, 2047, 2048, 2049]
        lengths = rng.choice(edges, size=S)
    while int(np.sum(lengths)) * Hkv * 512 > 300e6:      # keep each case under 300 MB of KV
        lengths = lengths // 2
    return rng, S, Hkv * G, Hkv, bs, [int(x) for x in lengths], bool(seed % 2)


@pytest.mark.parametrize("seed", range(24))
def test_random_case_matches_oracle(ops, seed):
    rng, S, Hq, Hkv, bs, lengths, fused = draw_case(seed)
    nb = sum(wl.blocks_for(L, bs) for L in lengths) + 3
    tables = wl.handout_tables(lengths, rng.permutation(nb).astype(np.int32), block_size=bs)
    q = wl.host_normal_fp16(rng, (S, Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.empty((S, Hq, D), dtype=torch.float16, device="cuda")
    dk, dv = dev(kc), dev(vc)
    err = ops.new_error_word()
    scale = 1 / np.sqrt(D)
    lens = np.array(lengths, np.int32)
    if fused:
        k_new = wl.host_normal_fp16(rng, (S, Hkv, D))
        v_new = wl.host_normal_fp16(rng, (S, Hkv, D))
        ops.paged_attention_decode_fused(out, dev(q), dev(k_new), dev(v_new), dk, dv, dev(tables),
                                         dev(lens), scale, dev_err=err)
        live = [s for s, L in enumerate(lengths) if L > 0]
        slots = np.array([oc.slot(tables[s], lengths[s] - 1, bs) for s in live], np.int64)
        if live:
            oc.reshape_and_cache(k_new[live], v_new[live], slots, kc, vc)
    else:
        ops.paged_attention_decode(out, dev(q), dk, dv, dev(tables), dev(lens), scale,
                                   dev_err=err)
    assert ops.read_error_word(err) == 0
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    assert_matches_oracle(out.cpu().numpy(), ref, (S, Hq, Hkv, bs, fused))
    if fused:
        assert np.array_equal(dk.cpu().numpy().view(np.uint16), kc.view(np.uint16))
        assert np.array_equal(dv.cpu().numpy().view(np.uint16), vc.view(np.uint16))
