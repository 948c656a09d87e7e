"""Pins the fp64 attention oracle to things other than itself.

* binary16 widening == NumPy's float16 -> float64 on all 65536 bit patterns
* identity block table == contiguous attention computed by torch's own
  scaled_dot_product_attention in float64 (GQA through repeat_interleave)
* the C oracle == the NumPy gather-and-concatenate form on tiny inputs (1e-12)
* permutation of physical block placement leaves the output bit-identical
* closed forms: L = 1 gives v; q = 0 or equal keys give the mean of V; one
  dominant key selects its value row; L = 0 gives zeros
* NaN poison in every slot past the context length never reaches the output
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa

D = 128


def rand_case(seed, S, Hq, Hkv, lengths, bs=16, extra_blocks=3, D=D):
    rng = np.random.default_rng(seed)
    need = [-(-L // bs) for L in lengths]
    nb = sum(need) + extra_blocks
    order = rng.permutation(nb)
    mb = max(need + [1])
    tables = np.full((S, mb), -1, dtype=np.int32)
    cur = 0
    for s, n in enumerate(need):
        tables[s, :n] = order[cur:cur + n]
        cur += n
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    kc = rng.standard_normal((nb, bs, Hkv, D)).astype(np.float16)
    vc = rng.standard_normal((nb, bs, Hkv, D)).astype(np.float16)
    return q, kc, vc, tables, np.array(lengths, dtype=np.int32)


def test_half_widening_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oa.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 3)])
def test_identity_table_matches_torch_sdpa(Hq, Hkv):
    rng = np.random.default_rng(11)
    bs, L = 16, 45
    nb = -(-L // bs)
    kc = rng.standard_normal((nb, bs, Hkv, D)).astype(np.float16)
    vc = rng.standard_normal((nb, bs, Hkv, D)).astype(np.float16)
    q = rng.standard_normal((1, Hq, D)).astype(np.float16)
    table = np.arange(nb, dtype=np.int32)[None]
    scale = 1.0 / np.sqrt(D)
    got = oa.paged_attention_decode(q, kc, vc, table, np.array([L], np.int32), scale)
    # contiguous K/V of the first L tokens, one query, heads grouped h // (Hq/Hkv)
    K = torch.from_numpy(kc.astype(np.float64).reshape(nb * bs, Hkv, D)[:L])
    V = torch.from_numpy(vc.astype(np.float64).reshape(nb * bs, Hkv, D)[:L])
    K = K.permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)   # [Hq, L, D]
    V = V.permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
    Q = torch.from_numpy(q.astype(np.float64)[0])[:, None, :]     # [Hq, 1, D]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)
    np.testing.assert_allclose(got[0], ref[:, 0, :].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed,Hq,Hkv,lengths", [
    (1, 8, 8, [7, 16, 31, 48, 63]),
    (2, 4, 1, [1, 2, 17, 33]),
    (3, 8, 2, [0, 5, 64, 100]),
    (4, 2, 2, [16, 32]),
])
def test_c_oracle_matches_gather_concat(seed, Hq, Hkv, lengths):
    q, kc, vc, tables, lens = rand_case(seed, len(lengths), Hq, Hkv, lengths)
    scale = 1.0 / np.sqrt(D)
    a = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    b = oa.paged_attention_gather_concat(q, kc, vc, tables, lens, scale)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_rows_variant_matches_full():
    q, kc, vc, tables, lens = rand_case(5, 4, 8, 2, [3, 40, 77, 16])
    scale = 0.1
    full = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    si = np.array([3, 0, 2, 2], np.int32)
    hi = np.array([7, 1, 0, 5], np.int32)
    rows = oa.paged_attention_decode_rows(q, kc, vc, tables, lens, scale, si, hi)
    assert np.array_equal(rows, full[si, hi])


def test_permutation_invariance_bit_exact():
    q, kc, vc, tables, lens = rand_case(6, 3, 4, 4, [20, 50, 9])
    rng = np.random.default_rng(99)
    nb = kc.shape[0]
    pi = rng.permutation(nb)                       # block b moves to pi[b]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    t2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1).astype(np.int32)
    scale = 1.0 / np.sqrt(D)
    a = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    b = oa.paged_attention_decode(q, kc2, vc2, t2, lens, scale)
    assert np.array_equal(a, b)


def test_closed_forms():
    q, kc, vc, tables, lens = rand_case(7, 4, 4, 2, [1, 30, 30, 30])
    scale = 1.0 / np.sqrt(D)
    bs = kc.shape[1]
    # equal keys for sequence 2; q = 0 for sequence 3; dominant key for seq 1
    for t in range(30):
        b, o = tables[2][t // bs], t % bs
        kc[b, o] = kc[tables[2][0], 0]
    q[3] = 0
    b5, o5 = tables[1][5 // bs], 5 % bs
    kc[b5, o5, 0] = np.float16(8.0) * np.sign(q[1, 0].astype(np.float32)).astype(np.float16)
    out = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    # L = 1: the single value row
    b0 = tables[0][0]
    np.testing.assert_array_equal(out[0, :, :], vc[b0, 0][[0, 0, 1, 1]].astype(np.float64))
    for s in (2, 3):
        rows = np.stack([vc[tables[s][t // bs], t % bs] for t in range(30)]).astype(np.float64)
        mean = rows.mean(axis=0)                       # [Hkv, D]
        np.testing.assert_allclose(out[s], mean[[0, 0, 1, 1]], rtol=0, atol=1e-12)
    # dominant logit (scale * 8 * sum|q| >> others): output ~= that value row
    np.testing.assert_allclose(out[1, 0], vc[b5, o5, 0].astype(np.float64), atol=1e-6)


def test_zero_length_gives_zeros():
    q, kc, vc, tables, lens = rand_case(8, 2, 2, 2, [0, 3])
    out = oa.paged_attention_decode(q, kc, vc, tables, lens, 0.1)
    assert np.all(out[0] == 0) and np.all(np.isfinite(out[1]))


def test_nan_poison_past_context_is_never_read():
    q, kc, vc, tables, lens = rand_case(9, 3, 4, 4, [5, 16, 33])
    scale = 1.0 / np.sqrt(D)
    clean = oa.paged_attention_decode(q, kc, vc, tables, lens, scale)
    kp, vp = kc.copy(), vc.copy()
    used = set()
    bs = kc.shape[1]
    for s, L in enumerate(lens):
        for t in range(L):
            used.add((int(tables[s][t // bs]), t % bs))
    for b in range(kc.shape[0]):
        for o in range(bs):
            if (b, o) not in used:
                kp[b, o] = np.float16(np.nan)
                vp[b, o] = np.float16(np.nan)
    poisoned = oa.paged_attention_decode(q, kp, vp, tables, lens, scale)
    assert np.array_equal(clean, poisoned)


def test_bad_block_id_is_reported():
    q, kc, vc, tables, lens = rand_case(10, 1, 2, 2, [20])
    tables[0, 1] = kc.shape[0] + 5
    with pytest.raises(oa.OracleError):
        oa.paged_attention_decode(q, kc, vc, tables, lens, 0.1)
