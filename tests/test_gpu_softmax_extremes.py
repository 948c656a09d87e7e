"""Paged decode attention against the fp64 oracle on inputs where the softmax
bookkeeping decides the result (built by ``softmax_cases``):

  * logits that climb (or fall, or dip and climb) through the whole context,
    so that the kernels' lazy rescale runs on many tiles of every warp and
    neighbouring splits' maxima lie more than 100 log2 units apart (the LSE
    merge's exp2 underflows for the low splits);
  * one or two dominant keys placed at the first and last token of a context,
    inside a tile, on both sides of a block (and tile, and warp) boundary and
    on both sides of every boundary a split can have;

for the plain, fused (cache write inside the launch) and grouped shared-prefix
launches.  A mistake in the rescale, in the cross-warp or cross-split merge or
in the row a token is read from moves an output by O(|V|) here, not by the
O(1e-3) it would on N(0, 1) data.  Tolerance 2e-3 absolute, as everywhere.
The fused cases poison the new token's slot with NaN before the launch, so the
kernel must use the row it writes.
"""
import numpy as np
import pytest
import torch

import softmax_cases as sc
from oracle import attention as oa
from oracle import cache_ops as oc
from parity_helpers import assert_matches_oracle

pytestmark = pytest.mark.gpu
D = sc.D
SCALE = 1.0 / np.sqrt(D)
FACTORS = [1.0, -1.0, 0.5, 2.0, -2.0, 1.5]


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def new_token_rows(kc, vc, tables, lens, bs=16):
    """The K/V rows at position L - 1 of every sequence (the fused launches'
    k_new / v_new) and their slots."""
    slots = np.array([oc.slot(tables[s], int(L) - 1, bs) for s, L in enumerate(lens)], np.int64)
    k_new = np.stack([kc[sl // bs, sl % bs] for sl in slots])
    v_new = np.stack([vc[sl // bs, sl % bs] for sl in slots])
    return k_new, v_new, slots


def run_split(ops, q, kc, vc, tables, lens, fused):
    """One plain or fused launch; returns (out, error code, cache K/V after)."""
    dk, dv = dev(kc), dev(vc)
    err = ops.new_error_word()
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    if fused:
        k_new, v_new, slots = new_token_rows(kc, vc, tables, lens)
        blk, off = torch.from_numpy(slots // 16).cuda(), torch.from_numpy(slots % 16).cuda()
        dk[blk, off] = float("nan")                 # the kernel must write these rows
        dv[blk, off] = float("nan")
        ops.paged_attention_decode_fused(out, dev(q), dev(k_new), dev(v_new), dk, dv,
                                         dev(tables), dev(lens), SCALE, dev_err=err)
    else:
        ops.paged_attention_decode(out, dev(q), dk, dv, dev(tables), dev(lens), SCALE,
                                   dev_err=err)
    return out.cpu().numpy(), ops.read_error_word(err), dk.cpu().numpy(), dv.cpu().numpy()


def check(got, kc, vc, q, tables, lens, code, dk=None, dv=None):
    assert code == 0
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, SCALE)
    assert np.isfinite(got).all()
    assert_matches_oracle(got, ref)
    # the outputs are O(1): an O(|V|) mistake would not hide under the tolerance
    assert np.abs(ref).max() > 0.5
    if dk is not None:
        assert np.array_equal(dk.view(np.uint16), kc.view(np.uint16))
        assert np.array_equal(dv.view(np.uint16), vc.view(np.uint16))


@pytest.mark.parametrize("S,Hkv,G", [(256, 4, 2), (32, 8, 4), (8, 8, 1)])
@pytest.mark.parametrize("fused", [False, True])
def test_climbing_falling_and_dipping_logits(ops, S, Hkv, G, fused):
    """Ramps, valleys and steep short ramps, at every split length a launch
    picks (2048, 1024, 512 tokens for these shapes)."""
    rng = np.random.default_rng(S + G)
    lengths = rng.integers(1, 120, size=S)
    lengths[:6] = [4096, 4097, 2049, 3000, 513, 17]
    tables, lens, nb = sc.plain_tables(S + 1, lengths.tolist())
    T = ops.split_tokens(S, Hkv, tables.shape[1])
    slope = {512: 0.25, 1024: 0.125}.get(T, 0.1)    # > 100 log2 units per split
    profiles = [sc.ramp(slope), sc.ramp(slope), sc.valley(slope), sc.valley(slope, 0.3),
                sc.ramp(1.0), sc.ramp(1.0)]
    profiles += [sc.ramp(1.0) if s % 2 else sc.valley(0.5) for s in range(6, S)]
    factors = [FACTORS[s % len(FACTORS)] for s in range(S)]
    q, kc, vc = sc.build(S + 2, tables, lens, profiles, Hq=Hkv * G, Hkv=Hkv, nb=nb,
                         seq_factor=factors)
    # the inputs reach the rescale branch at this launch's split length
    x = sc.logits_log2(q, kc, tables, lens, SCALE, 0, 0)
    rescales, maxima = sc.tile_loop_rescales(x, T)
    assert rescales >= 4 * len(maxima) and np.diff(maxima)[0] > 100
    got, code, dk, dv = run_split(ops, q, kc, vc, tables, lens, fused)
    check(got, kc, vc, q, tables, lens, code, *((dk, dv) if fused else ()))


def spike_specs(lengths):
    """(L, [(position, height), ...]) per sequence: one dominant key at the
    first, a middle and the last token; two near-equal keys across a tile
    boundary (two warps) and across every multiple of 512 tokens (the
    boundaries of 512-, 1024- and 2048-token splits); one key on each side of
    those boundaries alone."""
    specs = []
    for L in lengths:
        specs += [(L, [(L - 1, 24.0)]), (L, [(0, 24.0)]), (L, [(8, 24.0)]),
                  (L, [(15, 24.0), (16, 24.5)])]
        for b in range(512, L, 512):
            specs += [(L, [(b - 1, 24.0), (b, 23.5)]), (L, [(b - 1, 24.0)]), (L, [(b, 24.0)])]
    return specs


@pytest.mark.parametrize("Hkv,G,v_scale", [(8, 4, 0.4), (2, 4, 0.4), (4, 1, 0.4), (4, 2, 1.0)])
@pytest.mark.parametrize("fused", [False, True])
def test_dominant_keys_at_every_boundary(ops, Hkv, G, v_scale, fused):
    """v_scale 1.0: V rows up to ~4.5 in magnitude, where one dominant token's
    output must be its V row to within the fp16 output rounding."""
    specs = spike_specs([17, 513, 2049, 4097])
    lengths = [L for L, _ in specs]
    tables, lens, nb = sc.plain_tables(40 + Hkv, lengths)
    q, kc, vc = sc.build(41 + Hkv, tables, lens, [sc.spikes(p) for _, p in specs],
                         Hq=Hkv * G, Hkv=Hkv, nb=nb, gain_kind="positive", v_scale=v_scale)
    got, code, dk, dv = run_split(ops, q, kc, vc, tables, lens, fused)
    check(got, kc, vc, q, tables, lens, code, *((dk, dv) if fused else ()))


def run_grouped(ops, q, kc, vc, tables, lens, fused):
    G = q.shape[1] // kc.shape[2]
    gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, 16, 16 // G)
    assert mx > 0
    dk, dv = dev(kc), dev(vc)
    err = ops.new_error_word()
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    meta = (dev(tables), dev(lens), dev(gf), dev(sg), dev(gs), mx, mo, SCALE)
    if fused:
        k_new, v_new, slots = new_token_rows(kc, vc, tables, lens)
        blk, off = torch.from_numpy(slots // 16).cuda(), torch.from_numpy(slots % 16).cuda()
        dk[blk, off] = float("nan")
        dv[blk, off] = float("nan")
        ops.paged_attention_decode_grouped_fused(out, dev(q), dev(k_new), dev(v_new), dk, dv,
                                                 *meta, dev_err=err)
    else:
        ops.paged_attention_decode_grouped(out, dev(q), dk, dv, *meta, dev_err=err)
    return out.cpu().numpy(), ops.read_error_word(err), dk.cpu().numpy(), dv.cpu().numpy()


@pytest.mark.parametrize("Hq,Hkv,groups", [(4, 4, [16, 5, 1]), (16, 4, [4, 2, 1])])
@pytest.mark.parametrize("prefix", [1024, 2048])
@pytest.mark.parametrize("kind", ["ramp", "spikes"])
@pytest.mark.parametrize("fused", [False, True])
def test_grouped_shared_prefix_extremes(ops, Hq, Hkv, groups, prefix, kind, fused):
    """Forked samples: the shared prefix is streamed once for all members (the
    16 MMA rows hold every member's heads), each member with its own gain, so
    one member's logits climb through the prefix while another's fall; own
    tiles continue the profile.  Spikes sit at the prefix's split boundaries
    and in the own tiles."""
    n = sum(groups)
    rng = np.random.default_rng(prefix + Hq + n)
    own = rng.integers(1, 700, size=n)
    tables, lens, nb = sc.forked_tables(prefix + n, groups, prefix, own)
    if kind == "ramp":
        profiles = [sc.ramp(0.1)] * n
        factors = [FACTORS[s % len(FACTORS)] for s in range(n)]
        gain_kind = "mixed"
    else:
        profiles = [sc.spikes([(511, 24.0), (512, 23.5), (prefix - 1, 24.5), (prefix, 25.0),
                               (-1, 24.0 + (s % 3))]) for s in range(n)]
        factors, gain_kind = None, "positive"
    q, kc, vc = sc.build(prefix + n + 1, tables, lens, profiles, Hq=Hq, Hkv=Hkv, nb=nb,
                         seq_factor=factors, gain_kind=gain_kind)
    got, code, dk, dv = run_grouped(ops, q, kc, vc, tables, lens, fused)
    check(got, kc, vc, q, tables, lens, code, *((dk, dv) if fused else ()))
