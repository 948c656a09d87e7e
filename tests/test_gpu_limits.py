"""Attention at the largest sizes a launch accepts, against the fp64 oracle.

* 65,535 sequences: the most one launch takes (the grid's second dimension is
  the batch); 65,536 is refused with PKV_ERR_UNSUPPORTED before anything runs.
* One context of 2^20 + 7 tokens: a lone sequence gets 1024-token splits
  (the longest that still gives 1,024 CTAs), so its row is merged from 1,025
  partials (the merge's lanes loop over them 33 times), the last split
  holding 7 tokens.  Three tokens -- in the first
  split, a middle one and the last -- carry the same dominant key, so the
  output is close to the mean of their three V rows (O(1), not the ~1e-3
  average of a million N(0, 1) rows) and a dropped or misweighted split moves
  it by O(1).
* reshape_and_cache of 2^20 tokens filling every slot of a 2^16-block pool,
  and copy_blocks of 8,000 pairs in 4 layers, bit for bit.
* The empty cases: no sequences, no tokens, no pairs.
Tolerance: max |out_gpu - out_oracle| <= 2e-3 on fp16 outputs.
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
PKV_ERR_UNSUPPORTED = -2


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def many_sequences(seed, S, Hq, Hkv, max_len):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, max_len, S, endpoint=True).astype(np.int32)
    nb = sum(wl.blocks_for(int(L)) for L in lens) + 1
    tables = wl.handout_tables(lens, rng.permutation(nb).astype(np.int32))
    q = wl.host_normal_fp16(rng, (S, Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    kn = wl.host_normal_fp16(rng, (S, Hkv, D))
    vn = wl.host_normal_fp16(rng, (S, Hkv, D))
    return q, kc, vc, kn, vn, tables, lens


@pytest.mark.parametrize("fused", [False, True])
def test_largest_batch(ops, fused):
    S, Hq, Hkv = 65535, 8, 1
    q, kc, vc, kn, vn, tables, lens = many_sequences(65535, S, Hq, Hkv, 32)
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    e = ops.new_error_word()
    kcd, vcd = dev(kc), dev(vc)
    if fused:
        ops.paged_attention_decode_fused(out, dev(q), dev(kn), dev(vn), kcd, vcd, dev(tables),
                                         dev(lens), 1 / np.sqrt(D), dev_err=e)
        slots = (tables[np.arange(S), (lens - 1) // 16].astype(np.int64) * 16 + (lens - 1) % 16)
        oc.reshape_and_cache(kn, vn, slots, kc, vc)
        assert np.array_equal(kcd.cpu().numpy(), kc) and np.array_equal(vcd.cpu().numpy(), vc)
    else:
        ops.paged_attention_decode(out, dev(q), kcd, vcd, dev(tables), dev(lens), 1 / np.sqrt(D),
                                   dev_err=e)
    assert ops.read_error_word(e) == 0
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D))
    assert_matches_oracle(got, ref)


def test_one_sequence_too_many_is_refused(ops):
    from paged_kv_cache_138_gb300._lib import PagedKVError
    S, Hq, Hkv = 65536, 8, 1
    q = torch.zeros(S, Hq, D, dtype=torch.float16, device="cuda")
    kc = torch.zeros(4, 16, Hkv, D, dtype=torch.float16, device="cuda")
    tables = torch.zeros(S, 1, dtype=torch.int32, device="cuda")
    lens = torch.ones(S, dtype=torch.int32, device="cuda")
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    with pytest.raises(PagedKVError) as err:
        ops.paged_attention_decode(out, q, kc, kc.clone(), tables, lens, 0.1)
    assert err.value.status == PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.isnan(out).all()              # nothing was launched


@pytest.mark.parametrize("Hq", [1, 8])
def test_million_token_context(ops, Hq):
    L = (1 << 20) + 7
    Hkv = 1
    rng = np.random.default_rng(L + Hq)
    nb = wl.blocks_for(L) + 2
    tables = wl.handout_tables([L], rng.permutation(nb).astype(np.int32))
    lens = np.array([L], np.int32)
    q = wl.host_normal_fp16(rng, (1, Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    # the dominant key: 6 x the sum of the query rows (logit of head h about
    # 6 (|q_h|^2 + sum_j q_h.q_j) scale = 68 +- 16 against N(0, 1) for the rest)
    key = (6.0 * q[0].astype(np.float32).sum(axis=0)).astype(np.float16)
    spots = [5, L // 2 + 3, L - 3]
    for t in spots:
        kc[tables[0, t // 16], t % 16, 0] = key
    assert ops.split_tokens(1, Hkv, tables.shape[1]) == 1024
    out = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    e = ops.new_error_word()
    ops.paged_attention_decode(out, dev(q), dev(kc), dev(vc), dev(tables), dev(lens),
                               1 / np.sqrt(D), dev_err=e)
    assert ops.read_error_word(e) == 0
    got = out.cpu().numpy().astype(np.float64)
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D))
    assert np.isfinite(got).all()
    assert_matches_oracle(got, ref)
    mean3 = np.mean([vc[tables[0, t // 16], t % 16, 0].astype(np.float64) for t in spots], axis=0)
    assert np.abs(ref - mean3[None, None]).max() < 1e-3   # the three tokens dominate


def random_bits_fp16(rng, shape):
    """fp16 arrays of random bit patterns (NaNs and infinities included): the
    cache kernels move bits, and drawing bytes is far quicker on the host than
    drawing normals."""
    n = int(np.prod(shape))
    return np.frombuffer(rng.bytes(2 * n), dtype=np.float16).reshape(shape).copy()


def test_cache_write_of_a_million_tokens(ops):
    """reshape_and_cache of 2^20 tokens into a pool of exactly 2^16 blocks
    (every slot written once, in shuffled order, a few skipped with -1), bit
    for bit against the oracle's scatter."""
    T, Hkv, nb = 1 << 20, 1, 1 << 16
    rng = np.random.default_rng(20)
    k = random_bits_fp16(rng, (T, Hkv, D))
    v = random_bits_fp16(rng, (T, Hkv, D))
    slots = rng.permutation(nb * 16).astype(np.int64)
    slots[rng.choice(T, 5, replace=False)] = -1
    kc = np.zeros((nb, 16, Hkv, D), np.float16)
    vc = np.zeros_like(kc)
    kcd, vcd = dev(kc), dev(vc)
    e = ops.new_error_word()
    ops.reshape_and_cache(dev(k), dev(v), dev(slots), kcd, vcd, dev_err=e)
    assert ops.read_error_word(e) == 0
    oc.reshape_and_cache(k, v, slots, kc, vc)
    assert np.array_equal(kcd.cpu().numpy().view(np.uint16), kc.view(np.uint16))
    assert np.array_equal(vcd.cpu().numpy().view(np.uint16), vc.view(np.uint16))


def test_copy_of_eight_thousand_blocks_in_four_layers(ops):
    """copy_blocks of 8,000 (src, dst) pairs in each of 4 layers, bit for bit
    against the oracle (so every block outside the destinations unchanged)."""
    nb, Hkv, layers, P = 20000, 2, 4, 8000
    rng = np.random.default_rng(21)
    ids = rng.permutation(nb)
    pairs = np.stack([ids[:P], ids[P:2 * P]], axis=1).astype(np.int64)
    kcs = [random_bits_fp16(rng, (nb, 16, Hkv, D)) for _ in range(layers)]
    vcs = [random_bits_fp16(rng, (nb, 16, Hkv, D)) for _ in range(layers)]
    kd, vd = [dev(a) for a in kcs], [dev(a) for a in vcs]
    e = ops.new_error_word()
    ops.copy_blocks(kd, vd, dev(pairs), dev_err=e)
    assert ops.read_error_word(e) == 0
    oc.copy_blocks(kcs, vcs, pairs)
    for got, ref in zip(kd + vd, kcs + vcs):
        assert np.array_equal(got.cpu().numpy().view(np.uint16), ref.view(np.uint16))


def test_empty_calls_return_ok_and_touch_nothing(ops):
    """No sequences, no tokens, no pairs: every entry point returns OK,
    reports nothing and leaves the caches as they were."""
    Hq, Hkv, nb = 8, 2, 4
    kc = torch.randn(nb, 16, Hkv, D, device="cuda").half()
    vc = torch.randn(nb, 16, Hkv, D, device="cuda").half()
    k0, v0 = kc.clone(), vc.clone()
    q = torch.empty(0, Hq, D, dtype=torch.float16, device="cuda")
    kn = torch.empty(0, Hkv, D, dtype=torch.float16, device="cuda")
    out = torch.empty(0, Hq, D, dtype=torch.float16, device="cuda")
    tables = torch.empty(0, 3, dtype=torch.int32, device="cuda")
    lens = torch.empty(0, dtype=torch.int32, device="cuda")
    e = ops.new_error_word()
    ops.paged_attention_decode(out, q, kc, vc, tables, lens, 0.1, dev_err=e)
    ops.paged_attention_decode_fused(out, q, kn, kn.clone(), kc, vc, tables, lens, 0.1, dev_err=e)
    ops.reshape_and_cache(kn, kn.clone(), torch.empty(0, dtype=torch.int64, device="cuda"), kc, vc,
                          dev_err=e)
    ops.copy_blocks(kc, vc, torch.empty(0, 2, dtype=torch.int64, device="cuda"), dev_err=e)
    torch.cuda.synchronize()
    assert ops.read_error_word(e) == 0
    assert torch.equal(kc, k0) and torch.equal(vc, v0)
