"""Block sizes 8, 32 and 64 and the fused cache-write + attention kernel,
against the oracle (which takes any block size)."""
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


def case(seed, lengths, Hq, Hkv, bs, extra=3):
    rng = np.random.default_rng(seed)
    nb = sum(wl.blocks_for(L, bs) for L in lengths) + extra
    tables = wl.handout_tables(lengths, rng.permutation(nb).astype(np.int32), block_size=bs)
    q = wl.host_normal_fp16(rng, (len(lengths), Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    k_new = wl.host_normal_fp16(rng, (len(lengths), Hkv, D))
    v_new = wl.host_normal_fp16(rng, (len(lengths), Hkv, D))
    return q, kc, vc, tables, np.array(lengths, np.int32), k_new, v_new


def used_mask(tables, lengths, nb, bs):
    used = np.zeros((nb, bs), bool)
    for s, L in enumerate(lengths):
        for t in range(L):
            used[tables[s][t // bs], t % bs] = True
    return used


LENGTHS = [1, 7, 8, 9, 16, 17, 100, 511, 512, 513, 1500, 2049]


@pytest.mark.parametrize("bs", [8, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8)])
def test_block_sizes_match_oracle(ops, bs, Hq, Hkv):
    q, kc, vc, tables, lens, _, _ = case(bs * 7 + Hq, LENGTHS, Hq, Hkv, bs)
    used = used_mask(tables, LENGTHS, kc.shape[0], bs)
    kc[~used] = np.float16(np.nan)            # anything read past a context shows up
    vc[~used] = np.float16(np.nan)
    scale = 1 / np.sqrt(D)
    out = torch.empty((len(LENGTHS), Hq, D), dtype=torch.float16, device="cuda")
    err = ops.new_error_word()
    ops.paged_attention_decode(out, torch.from_numpy(q).cuda(), torch.from_numpy(kc).cuda(),
                               torch.from_numpy(vc).cuda(), torch.from_numpy(tables).cuda(),
                               torch.from_numpy(lens).cuda(), scale, dev_err=err)
    assert ops.read_error_word(err) == 0
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    assert_matches_oracle(out.cpu().numpy(), ref, (bs, Hq, Hkv))


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4), (40, 40)])
def test_fused_cache_write_and_attention(ops, bs, Hq, Hkv):
    lengths = [1, 8, 9, 16, 17, 33, 64, 65, 700, 1025]
    q, kc, vc, tables, lens, k_new, v_new = case(bs + Hq * 3, lengths, Hq, Hkv, bs)
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    out = torch.empty((len(lengths), Hq, D), dtype=torch.float16, device="cuda")
    err = ops.new_error_word()
    ops.paged_attention_decode_fused(out, torch.from_numpy(q).cuda(),
                                     torch.from_numpy(k_new).cuda(),
                                     torch.from_numpy(v_new).cuda(), dk, dv,
                                     torch.from_numpy(tables).cuda(),
                                     torch.from_numpy(lens).cuda(), 1 / np.sqrt(D), dev_err=err)
    assert ops.read_error_word(err) == 0
    # oracle: the slot formula on the tables, reshape_and_cache, then attention
    slots = np.array([oc.slot(tables[s], int(L) - 1, bs) for s, L in enumerate(lengths)],
                     np.int64)
    oc.reshape_and_cache(k_new, v_new, slots, kc, vc)
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D))
    assert_matches_oracle(out.cpu().numpy(), ref, (bs, Hq, Hkv))
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), kc.view(np.uint16))
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), vc.view(np.uint16))


def test_fused_equals_unfused_step_bitwise(ops):
    """reshape_and_cache + attention and the fused launch agree bit for bit."""
    lengths = [5, 300, 4096, 17]
    q, kc, vc, tables, lens, k_new, v_new = case(3, lengths, 32, 8, 16)
    slots = np.array([oc.slot(tables[s], int(L) - 1, 16) for s, L in enumerate(lengths)],
                     np.int64)
    dev = lambda a: torch.from_numpy(a).cuda()
    a_k, a_v, b_k, b_v = dev(kc), dev(vc), dev(kc), dev(vc)
    out_a = torch.empty((4, 32, D), dtype=torch.float16, device="cuda")
    out_b = torch.empty_like(out_a)
    ops.reshape_and_cache(dev(k_new), dev(v_new), dev(slots), a_k, a_v)
    ops.paged_attention_decode(out_a, dev(q), a_k, a_v, dev(tables), dev(lens), 0.0883883)
    ops.paged_attention_decode_fused(out_b, dev(q), dev(k_new), dev(v_new), b_k, b_v,
                                     dev(tables), dev(lens), 0.0883883)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(a_k.view(torch.int16), b_k.view(torch.int16))
    assert torch.equal(a_v.view(torch.int16), b_v.view(torch.int16))
