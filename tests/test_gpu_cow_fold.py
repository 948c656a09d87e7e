"""Copy-on-write folded into the fused attention launch
(pkv_paged_attention_decode_fused_cow / _grouped_fused_cow) against the
oracle's copy_blocks, reshape_and_cache and attention, in that order.

Forked samples share a prompt whose last block is partial; a sample that
appends writes into its own copy of that block ("ans20xx day 31", fork and
copy-on-write).  The cases cover the copy being the block the new token goes
into (the copy must carry the token) and an earlier block, block sizes 8
(either half of a 16-row tile), 16, 32 and 64 (a block staged by 2 or 4
tiles, the rows past the context copied from the source), grouped and plain
launches; every copy destination holds NaN before the launch, so a row the
kernel fails to copy shows.  Caches are compared bit for bit, outputs with
the parity measure.
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
SCALE = 1.0 / np.sqrt(D)


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def forked_with_cow(seed, prompts, samples, prompt_len, bs, Hkv, own_max, earlier=False):
    """Tables after each sample's first write past the prompt.  The prompt's
    last block is partial and shared; sample k > 0 of a prompt holds a private
    copy (dst) of it, sample 0 keeps the shared block (reference count 1 once
    the others copied).  With earlier=True every sample then holds own_max
    more tokens, so the copied block is no longer the one the new token goes
    into; sample 0's run past the shared block, since a launch that copies a
    block must not also write another sequence's new token into that source
    at a row the copies take (the pages' order is copy, then write; a fork
    gives every sample one length, so their first writes share one row).
    Returns tables, lens, nb, pairs (src, dst)."""
    rng = np.random.default_rng(seed)
    pb = wl.blocks_for(prompt_len, bs)
    rows, lens, pairs, nxt = [], [], [], 0
    for _ in range(prompts):
        prompt = list(range(nxt, nxt + pb))
        nxt += pb
        for k in range(samples):
            row = list(prompt)
            if k > 0:                       # the copy of the shared partial block
                pairs.append((prompt[-1], nxt))
                row[-1] = nxt
                nxt += 1
            extra = int(rng.integers(1, own_max + 1)) if earlier else 1
            if earlier and k == 0:              # its new token past the shared block
                extra = max(extra, pb * bs - prompt_len + 1)
            L = prompt_len + extra
            need = wl.blocks_for(L, bs) - len(row)
            row += list(range(nxt, nxt + need))
            nxt += need
            rows.append(row)
            lens.append(L)
    nb = nxt + 3
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(rows), max(len(r) for r in rows)), -1, np.int32)
    for i, r in enumerate(rows):
        tables[i, :len(r)] = perm[r]
    pairs = np.array([[perm[a], perm[b]] for a, b in pairs], np.int64).reshape(-1, 2)
    return tables, np.array(lens, np.int32), nb, pairs


def run_case(ops, seed, Hq, Hkv, bs, prompts, samples, prompt_len, earlier, grouped):
    tables, lens, nb, pairs = forked_with_cow(seed, prompts, samples, prompt_len, bs, Hkv, 300,
                                              earlier)
    rng = np.random.default_rng(seed + 1)
    S = len(lens)
    q = wl.host_normal_fp16(rng, (S, Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, bs, Hkv, D))
    k_new = wl.host_normal_fp16(rng, (S, Hkv, D))
    v_new = wl.host_normal_fp16(rng, (S, Hkv, D))
    kc[pairs[:, 1]] = np.float16(np.nan)            # destinations: nothing valid yet
    vc[pairs[:, 1]] = np.float16(np.nan)
    cb, cs = ops.cow_targets(pairs, tables)
    assert (cb >= 0).sum() == len(pairs)
    dk, dv = dev(kc), dev(vc)
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.float16, device="cuda")
    err = ops.new_error_word()
    if grouped:
        gf, sg, gs, mx, mo = ops.shared_prefix_groups(tables, lens, bs, 16 // (Hq // Hkv))
        assert mx > 0
        ops.paged_attention_decode_grouped_fused(
            out, dev(q), dev(k_new), dev(v_new), dk, dv, dev(tables), dev(lens), dev(gf),
            dev(sg), dev(gs), mx, mo, SCALE, dev_err=err, cow=(dev(cb), dev(cs)))
    else:
        ops.paged_attention_decode_fused(out, dev(q), dev(k_new), dev(v_new), dk, dv,
                                         dev(tables), dev(lens), SCALE, dev_err=err,
                                         cow=(dev(cb), dev(cs)))
    assert ops.read_error_word(err) == 0
    # the oracle: copy, then write the new tokens, then attend
    oc.copy_blocks([kc], [vc], pairs)
    slots = np.array([oc.slot(tables[s], int(L) - 1, bs) for s, L in enumerate(lens)], np.int64)
    oc.reshape_and_cache(k_new, v_new, slots, kc, vc)
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), kc.view(np.uint16))
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), vc.view(np.uint16))
    ref = oa.paged_attention_decode(q, kc, vc, tables, lens, SCALE)
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    assert_matches_oracle(got, ref)
    return cb, tables, lens


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4)])
@pytest.mark.parametrize("earlier", [False, True])
@pytest.mark.parametrize("grouped", [False, True])
def test_folded_copy_matches_copy_blocks_then_attention(ops, bs, Hq, Hkv, earlier, grouped):
    samples = 16 // (Hq // Hkv)
    # prompt lengths whose last block is partial, at both halves of a tile
    # and (block sizes 32, 64) in the block's first, middle and last tile
    lens = (1000 + 3, 1000 + 11) if bs <= 16 else (1024 + 3, 1024 + 20, 1024 + bs - 5)
    for prompt_len in lens:
        cb, tables, lens = run_case(ops, prompt_len + bs + Hq, Hq, Hkv, bs, 3, samples,
                                    prompt_len, earlier, grouped)
        new_block = (lens - 1) // bs
        copied = cb >= 0
        if earlier:
            assert (cb[copied] < new_block[copied]).any()
        else:
            assert (cb[copied] == new_block[copied]).all()


def test_folded_copy_in_a_long_split_context(ops):
    """Copies far into 4096-token contexts (the copied block in a later split
    than the first), plain launch."""
    run_case(ops, 77, 32, 8, 16, 4, 4, 3000 + 5, earlier=True, grouped=False)


def test_bad_copy_metadata_is_reported(ops):
    tables, lens, nb, pairs = forked_with_cow(5, 1, 4, 200 + 3, 16, 8, 10)
    rng = np.random.default_rng(6)
    S = len(lens)
    q = dev(wl.host_normal_fp16(rng, (S, 8, D)))
    kn = dev(wl.host_normal_fp16(rng, (S, 8, D)))
    kc = dev(wl.host_normal_fp16(rng, (nb, 16, 8, D)))
    out = torch.empty_like(q)
    cb, cs = ops.cow_targets(pairs, tables)
    for bad, code in (("past_context", 5), ("source_outside_pool", 1)):
        b, c = cb.copy(), cs.copy()
        s = int(np.argmax(b >= 0))
        if bad == "past_context":
            b[s] = (int(lens[s]) + 15) // 16          # a block past the last token
        else:
            c[s] = nb + 7
        err = ops.new_error_word()
        ops.paged_attention_decode_fused(out, q, kn, kn, kc, kc.clone(), dev(tables), dev(lens),
                                         SCALE, dev_err=err, cow=(dev(b), dev(c)))
        assert ops.read_error_word(err) == code, bad
