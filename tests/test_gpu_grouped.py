"""Grouped (shared-prefix) attention: the same result as plain paged attention,
with each group's shared prefix streamed once for all its members."""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import cache_ops as oc
from parity_helpers import assert_matches_oracle, oracle_batch
from paged_kv_cache_138_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def forked_case(seed, groups, Hq, Hkv, bs, prefix_tokens, own_max=700, own_min=0):
    """groups: members per group.  Each group's members share prefix_tokens of
    blocks, then hold private blocks of own_min..own_max further tokens."""
    rng = np.random.default_rng(seed)
    lens, rows = [], []
    next_block = 0
    pb = prefix_tokens // bs
    for members in groups:
        prefix = list(range(next_block, next_block + pb))
        next_block += pb
        for _ in range(members):
            own = int(rng.integers(own_min, own_max + 1))
            L = prefix_tokens + own
            extra = -(-L // bs) - pb
            rows.append(prefix + list(range(next_block, next_block + extra)))
            next_block += extra
            lens.append(L)
    nb = next_block + 2
    perm = rng.permutation(nb).astype(np.int32)        # scatter the blocks
    mb = max(len(r) for r in rows)
    tables = np.full((len(rows), mb), -1, np.int32)
    for i, r in enumerate(rows):
        tables[i, :len(r)] = perm[r]
    q = wl.host_normal_fp16(rng, (len(rows), Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    return q, kc, vc, tables, np.array(lens, np.int32)


def run_grouped(ops, q, kc, vc, tables, lens, bs, err=None):
    gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, bs,
                                                  16 // (q.shape[1] // kc.shape[2]))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    e = ops.new_error_word() if err is None else err
    ops.paged_attention_decode_grouped(out, dev(q), dev(kc), dev(vc), dev(tables), dev(lens),
                                       dev(gf), dev(sg), dev(gs), mx, mo, 1 / np.sqrt(D),
                                       dev_err=e)
    return out.cpu().numpy().astype(np.float64), ops.read_error_word(e), gs


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv,groups", [(8, 8, [16, 3, 1, 5]), (32, 8, [4, 4, 2, 1]),
                                           (16, 8, [8, 1, 7])])
@pytest.mark.parametrize("prefix", [512, 1024 + 512])
def test_grouped_matches_oracle(ops, bs, Hq, Hkv, groups, prefix):
    q, kc, vc, tables, lens = forked_case(bs + Hq + prefix, groups, Hq, Hkv, bs, prefix)
    got, code, gs = run_grouped(ops, q, kc, vc, tables, lens, bs)
    assert code == 0
    assert (gs > 0).sum() == sum(1 for m in groups if m > 1)
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D))
    assert np.isfinite(got).all()
    assert_matches_oracle(got, ref)


def test_grouped_prefix_sharing_workload(ops):
    """The prefix-sharing workload at full size (8 groups of 16 forked samples
    sharing 2048 tokens), after its copy-on-write step."""
    w = wl.WORKLOADS["prefix-sharing"]
    tables, lens, slots, pairs, nb = oracle_batch(w)
    q, k_new, v_new, kc, vc = wl.host_tensors(w, nb)
    q, k_new, v_new, kc, vc = q[0], k_new[0], v_new[0], kc[0], vc[0]
    oc.copy_blocks([kc], [vc], pairs)
    oc.reshape_and_cache(k_new, v_new, slots, kc, vc)
    got, code, gs = run_grouped(ops, q, kc, vc, tables, lens, 16)
    assert code == 0 and list(gs) == [2048] * 8
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, w.scale)
    assert_matches_oracle(got, ref)


def test_bad_group_is_reported(ops):
    q, kc, vc, tables, lens = forked_case(3, [4], 8, 8, 16, 512)
    gf = np.array([0, 4], np.int32)
    sg = np.zeros(4, np.int32)
    gs = np.array([512], np.int32)
    tables = tables.copy()
    tables[2, 3] = (tables[2, 3] + 1) % kc.shape[0]      # member 2 no longer shares block 3
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
    err = ops.new_error_word()
    ops.paged_attention_decode_grouped(out, dev(q), dev(kc), dev(vc), dev(tables), dev(lens),
                                       dev(gf), dev(sg), dev(gs), 512, 700, 0.1, dev_err=err)
    assert ops.read_error_word(err) == 6      # PKV_DEV_BAD_GROUP


@pytest.mark.parametrize("case", ["group_id_out_of_range", "group_past_batch",
                                  "member_of_other_group", "shared_longer_than_reserved"])
def test_malformed_groups_are_reported(ops, case):
    """Group metadata the kernels cannot trust is reported (BAD_GROUP) and
    every access stays inside the buffers: a sequence naming no group, a
    group running past the batch, a member whose group id names another
    group, a shared prefix longer than the launch reserved workspace for."""
    prefix = 1024 if case == "shared_longer_than_reserved" else 512
    q, kc, vc, tables, lens = forked_case(5, [4], 8, 8, 16, prefix)
    gf = np.array([0, 4], np.int32)
    sg = np.zeros(4, np.int32)
    gs = np.array([prefix], np.int32)
    mx = prefix
    if case == "group_id_out_of_range":
        sg[2] = 7
    elif case == "group_past_batch":
        gf[1] = 9
    elif case == "member_of_other_group":
        gf, gs = np.array([0, 4, 4], np.int32), np.array([prefix, 0], np.int32)
        sg[2] = 1
    else:
        mx = 512                      # the launch reserves one 512-token shared split
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
    err = ops.new_error_word()
    ops.paged_attention_decode_grouped(out, dev(q), dev(kc), dev(vc), dev(tables), dev(lens),
                                       dev(gf), dev(sg), dev(gs), mx, 700, 0.1, dev_err=err)
    assert ops.read_error_word(err) == 6      # PKV_DEV_BAD_GROUP


def test_own_tokens_beyond_the_stated_bound_are_reported(ops):
    q, kc, vc, tables, lens = forked_case(4, [3, 2], 8, 8, 16, 512, own_max=900)
    gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, 16, 16)
    assert mo > 600
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
    err = ops.new_error_word()
    ops.paged_attention_decode_grouped(out, dev(q), dev(kc), dev(vc), dev(tables), dev(lens),
                                       dev(gf), dev(sg), dev(gs), mx, 100, 0.1, dev_err=err)
    assert ops.read_error_word(err) == 6      # PKV_DEV_BAD_GROUP


def grouped_fused(ops, q, kc, vc, tables, lens, bs, k_new, v_new, err):
    gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, bs,
                                                  16 // (q.shape[1] // kc.shape[2]))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    dk, dv = dev(kc), dev(vc)
    ops.paged_attention_decode_grouped_fused(out, dev(q), dev(k_new), dev(v_new), dk, dv,
                                             dev(tables), dev(lens), dev(gf), dev(sg), dev(gs),
                                             mx, mo, 1 / np.sqrt(D), dev_err=err)
    return out, dk, dv, gs


@pytest.mark.parametrize("bs", [8, 16, 64])
@pytest.mark.parametrize("Hq,Hkv,groups", [(8, 8, [16, 3, 1, 5]), (32, 8, [4, 4, 2, 1])])
def test_grouped_fused_cache_write_and_attention(ops, bs, Hq, Hkv, groups):
    """One launch writes every member's new token (in its own blocks) and
    attends with the shared prefix streamed once: the oracle's cache write
    then plain attention, and the cache bytes, must agree."""
    q, kc, vc, tables, lens = forked_case(bs * 3 + Hq, groups, Hq, Hkv, bs, 1024, own_min=1)
    rng = np.random.default_rng(bs + Hkv)
    k_new = wl.host_normal_fp16(rng, (len(lens), Hkv, D))
    v_new = wl.host_normal_fp16(rng, (len(lens), Hkv, D))
    err = ops.new_error_word()
    out, dk, dv, gs = grouped_fused(ops, q, kc, vc, tables, lens, bs, k_new, v_new, err)
    assert ops.read_error_word(err) == 0
    assert (gs > 0).sum() == sum(1 for m in groups if m > 1)
    slots = np.array([oc.slot(tables[s], int(L) - 1, bs) for s, L in enumerate(lens)], np.int64)
    oc.reshape_and_cache(k_new, v_new, slots, kc, vc)
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D))
    got = out.cpu().numpy().astype(np.float64)
    assert_matches_oracle(got, ref)
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), kc.view(np.uint16))
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), vc.view(np.uint16))


def test_grouped_fused_equals_cache_write_then_grouped_bitwise(ops):
    q, kc, vc, tables, lens = forked_case(77, [8, 5, 1], 32, 8, 16, 1536, own_min=1)
    rng = np.random.default_rng(78)
    k_new = wl.host_normal_fp16(rng, (len(lens), 8, D))
    v_new = wl.host_normal_fp16(rng, (len(lens), 8, D))
    err = ops.new_error_word()
    fused, dk, dv, _ = grouped_fused(ops, q, kc, vc, tables, lens, 16, k_new, v_new, err)
    slots = np.array([oc.slot(tables[s], int(L) - 1, 16) for s, L in enumerate(lens)], np.int64)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    k2, v2 = dev(kc), dev(vc)
    ops.reshape_and_cache(dev(k_new), dev(v_new), dev(slots), k2, v2)
    gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, 16, 4)
    two = torch.empty_like(fused)
    ops.paged_attention_decode_grouped(two, dev(q), k2, v2, dev(tables), dev(lens), dev(gf),
                                       dev(sg), dev(gs), mx, mo, 1 / np.sqrt(D), dev_err=err)
    assert ops.read_error_word(err) == 0
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16))
    assert torch.equal(dk.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(dv.view(torch.int16), v2.view(torch.int16))


def test_grouped_fused_new_token_inside_the_shared_prefix_is_reported(ops):
    """A member whose context ends exactly at the shared prefix would have its
    new token in a block the group shares: reported, not written there."""
    q, kc, vc, tables, lens = forked_case(5, [3], 8, 8, 16, 512, own_max=40, own_min=1)
    lens = lens.copy()
    lens[1] = 512                                  # member 1 holds only the prefix
    rng = np.random.default_rng(6)
    k_new = wl.host_normal_fp16(rng, (3, 8, D))
    v_new = wl.host_normal_fp16(rng, (3, 8, D))
    err = ops.new_error_word()
    _, dk, _, gs = grouped_fused(ops, q, kc, vc, tables, lens, 16, k_new, v_new, err)
    assert list(gs) == [512]
    assert ops.read_error_word(err) == 6           # PKV_DEV_BAD_GROUP
    last = tables[1][511 // 16]
    assert np.array_equal(dk[last].cpu().numpy().view(np.uint16), kc[last].view(np.uint16))
