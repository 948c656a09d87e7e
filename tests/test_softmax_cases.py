"""The extreme-softmax inputs of the GPU parity tests, checked on the CPU.

Before those inputs can stand for "the rescale branch and the split merge are
tested", three things must hold, and none needs a GPU:
  * the tile-schedule emulation counts what it claims to (a hand-worked case);
  * on the ramp inputs the running maximum of every rising row moves many
    times after a warp's first tile (the branch runs), for every split length
    a launch can pick, and consecutive splits' maxima lie more than 100 log2
    units apart (the merge's exp2 of a split underflows);
  * the oracle, on such inputs, gives the closed form: one dominant key returns
    that key's V row.
"""
import numpy as np
import pytest

import softmax_cases as sc
from oracle import attention as oa

SCALE = 1.0 / np.sqrt(sc.D)


def test_emulation_counts_a_hand_worked_schedule():
    # logits rise by 9 per tile: a warp's next tile lies 4 tiles (36) higher,
    # so every tile of a warp after its first moves the maximum
    x = np.repeat(np.arange(64) * 9.0, 16)            # 64 tiles, one split of 64
    r, maxima = sc.tile_loop_rescales(x, split_tokens=1024)
    assert r == 4 * (16 - 1) and maxima == [63 * 9.0]
    # a rise of 1 per tile is 4 per warp tile: the maximum set by a warp's
    # first tile (k = 0) is beaten by more than 8 at its tiles k = 3 and k = 6
    x = np.repeat(np.arange(32) * 1.0, 16)
    r, maxima = sc.tile_loop_rescales(x, split_tokens=512)
    assert r == 4 * 2
    # falling logits: the first tile holds every warp's maximum
    r, _ = sc.tile_loop_rescales(-x, split_tokens=512)
    assert r == 0
    # two splits: the maxima are reported per split, the tail split is ragged
    x = np.arange(700, dtype=np.float64)
    _, maxima = sc.tile_loop_rescales(x, split_tokens=512)
    assert maxima == [511.0, 699.0]


@pytest.mark.parametrize("split_tokens,slope", [(512, 0.2), (1024, 0.1), (2048, 0.1)])
def test_ramp_inputs_reach_the_rescale_branch_and_far_apart_splits(split_tokens, slope):
    lengths = [4096, 4097, 3000]
    tables, lens, nb = sc.plain_tables(1, lengths)
    profiles = [sc.ramp(slope)] * len(lengths)
    q, kc, vc = sc.build(2, tables, lens, profiles, Hq=4, Hkv=1, nb=nb)
    gains = sc.gains_for(4)
    for s in range(len(lengths)):
        for h in range(4):
            x = sc.logits_log2(q, kc, tables, lens, SCALE, s, h)
            r, maxima = sc.tile_loop_rescales(x, split_tokens)
            # neighbouring full splits' maxima lie |gain| * slope * split apart
            gaps = np.diff(maxima)[:-1] * np.sign(gains[h])
            assert (gaps >= 0.9 * abs(gains[h]) * slope * split_tokens).all(), (s, h, gaps)
            if abs(gains[h]) >= 1:
                assert (gaps > 100).all()
            if gains[h] >= 0.5:
                # rising rows: the branch runs many times in every split
                assert r >= 4 * len(maxima), (s, h, r)
            else:
                # falling rows: the first tile keeps every warp's maximum,
                # later splits lie far below the first
                assert r == 0
                assert maxima[0] - maxima[-1] > 100


def test_short_steep_ramps_rescale_on_every_warp_tile():
    tables, lens, nb = sc.plain_tables(3, [17, 100, 513])
    q, kc, vc = sc.build(4, tables, lens, [sc.ramp(1.0)] * 3, Hq=1, Hkv=1, nb=nb)
    for s, L in enumerate(lens):
        x = sc.logits_log2(q, kc, tables, lens, SCALE, s, 0)
        r, _ = sc.tile_loop_rescales(x, 512)
        tiles = -(-int(L) // 16)
        # a warp's tiles are 64 tokens (64 log2 units) apart
        assert r >= max(0, tiles - 4) - 2, (L, r)


def test_spikes_dominate_and_oracle_returns_the_dominant_row():
    lengths = [17, 513, 2049]
    tables, lens, nb = sc.plain_tables(5, lengths)
    pos = [16, 0, 1024]
    profiles = [sc.spikes([(p, 24.0)]) for p in pos]
    q, kc, vc = sc.build(6, tables, lens, profiles, Hq=8, Hkv=2, nb=nb, gain_kind="positive")
    out = oa.paged_attention_decode(q, kc, vc, tables, lens, SCALE)
    for s, p in enumerate(pos):
        blk, off = tables[s][p // 16], p % 16
        for h in range(8):
            x = sc.logits_log2(q, kc, tables, lens, SCALE, s, h)
            others = np.delete(x, p)
            assert x[p] - others.max() >= 15
            v = vc[blk, off, h // 4].astype(np.float64)
            # the other tokens weigh at most L * 2^-15 relative
            assert np.abs(out[s, h] - v).max() <= 2.0 * lengths[s] * 2.0 ** -15


def test_forked_builder_shares_the_prefix_profile():
    tables, lens, nb = sc.forked_tables(7, [3, 1], 256, [40, 0, 90, 17])
    prof = [sc.ramp(0.5)] * 4
    q, kc, vc = sc.build(8, tables, lens, prof, Hq=2, Hkv=1, nb=nb,
                         seq_factor=[1.0, -1.0, 2.0, 1.0])
    # members 0-2 read the same first 16 blocks
    assert (tables[0, :16] == tables[1, :16]).all() and (tables[1, :16] == tables[2, :16]).all()
    x0 = sc.logits_log2(q, kc, tables, lens, SCALE, 0, 0)[:256]
    x1 = sc.logits_log2(q, kc, tables, lens, SCALE, 1, 0)[:256]
    assert np.allclose(x1, -x0, atol=0.05)          # same keys, opposite gain
    # every slot a sequence reads is finite; the unread rest is NaN
    for s, L in enumerate(lens):
        t = np.arange(L)
        assert np.isfinite(kc[tables[s][t // 16], t % 16]).all()


MISTAKES = ["no_l_rescale", "no_o_rescale", "merge_first_max", "drop_last_split",
            "drop_last_token", "row_shift"]


@pytest.mark.parametrize("split_tokens,slope", [(512, 0.25), (1024, 0.125), (2048, 0.1)])
def test_planted_kernel_mistakes_fail_on_these_inputs(split_tokens, slope):
    """The fp64 model of the kernels' combination (per-warp lazy rescale,
    cross-warp and cross-split merges) matches the oracle on the ramp and
    spike inputs; each planted mistake misses the oracle by far more than the
    2e-3 tolerance on at least one of them (on N(0, 1) inputs most of these
    mistakes stay under it)."""
    lengths = [4097, 3000, 2049, 2049, 4097]
    tables, lens, nb = sc.plain_tables(11, lengths)
    b = split_tokens
    profiles = [sc.ramp(slope), sc.valley(slope), sc.spikes([(b - 1, 24.0), (b, 23.5)]),
                sc.spikes([(2048, 24.0)]), sc.ramp(-slope)]
    q, kc, vc = sc.build(12, tables, lens, profiles, Hq=2, Hkv=1, nb=nb,
                         seq_factor=[1.0, 1.0, 1.0, 1.0, 1.0], gain_kind="positive")
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, SCALE)
    worst = {m: 0.0 for m in MISTAKES}
    for s, L in enumerate(lengths):
        t = np.arange(L)
        v = vc[tables[s][t // 16], t % 16, 0].astype(np.float64)
        for h in range(2):
            x = sc.logits_log2(q, kc, tables, lens, SCALE, s, h)
            assert np.abs(sc.emulated_row(x, v, split_tokens) - ref[s, h]).max() < 1e-6
            for m in MISTAKES:
                got = sc.emulated_row(x, v, split_tokens, m)
                err = np.abs(got - ref[s, h]).max() if np.isfinite(got).all() else np.inf
                worst[m] = max(worst[m], err)
    for m, e in worst.items():
        assert e > 0.05, (m, e)
