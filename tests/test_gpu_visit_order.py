"""The order in which a launch visits the sequences of a batch.

In batches of at most 128 sequences whose last split can be at least half a
split long (by the table width), the last split plane is visited in an order
computed on the device from the context lengths (longest, shortest, second
longest, ...); other planes and other batches take a fixed stride order
(grouped launches keep the batch order for their own units).  The order must change which
CTA runs a sequence and nothing else: every sequence visited exactly once
(outputs start as NaN), every output equal to the oracle's within the 2e-3
bound, and a permuted batch giving the permuted outputs bit for bit.
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
MAX_RANKED = 128


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def batch(seed, lengths, Hq, Hkv):
    rng = np.random.default_rng(seed)
    need = [wl.blocks_for(int(L)) for L in lengths]
    nb = sum(need) + 3
    tables = wl.handout_tables(lengths, rng.permutation(nb).astype(np.int32))
    S = len(lengths)
    q = wl.host_normal_fp16(rng, (S, Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    kn = wl.host_normal_fp16(rng, (S, Hkv, D))
    vn = wl.host_normal_fp16(rng, (S, Hkv, D))
    return q, kc, vc, kn, vn, tables, np.asarray(lengths, np.int32)


def ranked(ops, S, Hkv, tables):
    """Whether a launch of these sizes visits its last split plane in the
    length-ranked order (block size 16: one tile per block)."""
    split_tiles = ops.split_tokens(S, Hkv, tables.shape[1]) // 16
    table_tiles = tables.shape[1]
    planes = -(-table_tiles // split_tiles)
    last = table_tiles - (planes - 1) * split_tiles
    return S <= MAX_RANKED and 2 * last >= split_tiles


def run(ops, q, kc, vc, tables, lens, fused=False, kn=None, vn=None):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    e = ops.new_error_word()
    kcd, vcd = dev(kc), dev(vc)
    if fused:
        ops.paged_attention_decode_fused(out, dev(q), dev(kn), dev(vn), kcd, vcd, dev(tables),
                                         dev(lens), 1 / np.sqrt(D), dev_err=e)
    else:
        ops.paged_attention_decode(out, dev(q), kcd, vcd, dev(tables), dev(lens), 1 / np.sqrt(D),
                                   dev_err=e)
    return out.cpu().numpy(), ops.read_error_word(e), kcd.cpu().numpy(), vcd.cpu().numpy()


def lengths_with_ties(seed, S, hi):
    """Lengths 1..hi with many equal values (ties are broken by batch index),
    including 1, tile and block boundaries and the longest allowed."""
    rng = np.random.default_rng(seed)
    pool = np.array(sorted({1, 15, 16, 17, 31, 33, hi // 3, hi // 2, hi - 1, hi}), np.int64)
    lens = rng.choice(pool, size=S)
    lens[rng.integers(0, S)] = hi
    return lens.astype(np.int32)


CASES = [
    # S, Hq, Hkv, longest context.  Ranked: the 24- to 128-sequence batches
    # (one split per sequence) and 64 x 4096 (two splits: the second plane).
    # Not ranked: 5 sequences (units far shorter than a split), 129 sequences.
    (5, 8, 8, 63),
    (24, 24, 24, 512),
    (64, 32, 16, 1024),
    (127, 32, 16, 2048),
    (128, 32, 8, 2048),
    (129, 32, 8, 2048),
    (64, 8, 8, 4096),
]


@pytest.mark.parametrize("S,Hq,Hkv,hi", CASES)
@pytest.mark.parametrize("fused", [False, True])
def test_every_sequence_visited_once(ops, S, Hq, Hkv, hi, fused):
    lens = lengths_with_ties(S * 7 + hi, S, hi)
    q, kc, vc, kn, vn, tables, lens = batch(S + hi, lens, Hq, Hkv)
    expect_ranked = (S, hi) in {(24, 512), (64, 1024), (127, 2048), (128, 2048), (64, 4096)}
    assert ranked(ops, S, Hkv, tables) == expect_ranked
    got, code, kc_gpu, vc_gpu = run(ops, q, kc, vc, tables, lens, fused, kn, vn)
    assert code == 0
    assert np.isfinite(got).all()
    if fused:
        slots = np.array([tables[s, (L - 1) // 16] * 16 + (L - 1) % 16
                          for s, L in enumerate(lens)], np.int64)
        oc.reshape_and_cache(kn, vn, slots, kc, vc)
        assert np.array_equal(kc_gpu, kc) and np.array_equal(vc_gpu, vc)
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D))
    assert_matches_oracle(got, ref)


def test_all_lengths_equal_and_empty_rows(ops):
    """Every length tied (the order is then the batch order) and rows of
    length 0 among them, in a ranked batch."""
    S, Hq, Hkv = 128, 32, 8
    lens = np.full(S, 1500, np.int32)
    lens[[0, 17, 127]] = 0
    q, kc, vc, _, _, tables, lens = batch(91, lens, Hq, Hkv)
    assert ranked(ops, S, Hkv, tables)
    got, code, _, _ = run(ops, q, kc, vc, tables, lens)
    assert code == 0
    assert (got[[0, 17, 127]] == 0).all()
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D))
    assert_matches_oracle(got, ref)


@pytest.mark.parametrize("S,Hq,Hkv,hi", [(128, 32, 8, 2048), (64, 40, 40, 4096), (200, 8, 8, 600)])
def test_permuted_batch_permutes_outputs_bitwise(ops, S, Hq, Hkv, hi):
    rng = np.random.default_rng(S + hi)
    lens = rng.integers(1, hi, S, endpoint=True).astype(np.int32)
    q, kc, vc, _, _, tables, lens = batch(5 + S, lens, Hq, Hkv)
    perm = rng.permutation(S)
    got, code, _, _ = run(ops, q, kc, vc, tables, lens)
    got_p, code_p, _, _ = run(ops, q[perm], kc, vc, tables[perm], lens[perm])
    assert code == 0 and code_p == 0
    assert np.array_equal(got_p.view(np.uint16), got[perm].view(np.uint16))


def test_bad_length_in_a_ranked_batch_is_reported(ops):
    """A negative and an oversized context length among ranked sequences: the
    error word says so and every other sequence is still right."""
    S, Hq, Hkv = 64, 16, 16
    lens = np.random.default_rng(4).integers(1, 2048, S, endpoint=True).astype(np.int32)
    lens[0] = 2048
    q, kc, vc, _, _, tables, lens = batch(44, lens, Hq, Hkv)
    assert ranked(ops, S, Hkv, tables)
    bad = lens.copy()
    bad[3] = -5
    bad[40] = tables.shape[1] * 16 + 1
    tables[40][tables[40] < 0] = 0             # its (clamped) length reads whole-table blocks
    got, code, _, _ = run(ops, q, kc, vc, tables, bad)
    assert code == 2                           # PKV_DEV_BAD_CONTEXT_LEN
    keep = [s for s in range(S) if s not in (3, 40)]
    ref = oa.paged_attention_decode(q[keep], kc, vc, tables[keep], lens[keep], 1 / np.sqrt(D))
    assert_matches_oracle(got[keep], ref)
