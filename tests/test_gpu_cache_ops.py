"""reshape_and_cache, slot mapping and copy_blocks on the GPU: bit-exact against
the oracle's definitions.  Calls go through the C ABI (ops -> libpagedkv.so)."""
import numpy as np
import pytest
import torch

from oracle import cache_ops as oc
from parity_helpers import oracle_batch
from paged_kv_cache_138_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops(native_lib):
    from paged_kv_cache_138_gb300 import ops as o
    return o


def bits(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("Hkv,nb,T", [(8, 64, 5), (40, 300, 64), (1, 7, 3), (32, 1000, 257)])
def test_reshape_and_cache_bit_exact(ops, Hkv, nb, T):
    rng = np.random.default_rng(Hkv * 1000 + T)
    bs, D = 16, 128
    kc = rng.standard_normal((nb, bs, Hkv, D)).astype(np.float16)
    vc = rng.standard_normal((nb, bs, Hkv, D)).astype(np.float16)
    k = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    v = rng.standard_normal((T, Hkv, D)).astype(np.float16)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::4] = -1                                   # skipped tokens
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    err = ops.new_error_word()
    ops.reshape_and_cache(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                          torch.from_numpy(slots).cuda(), dk, dv, dev_err=err)
    assert ops.read_error_word(err) == 0
    oc.reshape_and_cache(k, v, slots, kc, vc)
    assert np.array_equal(bits(dk), kc.view(np.uint16))
    assert np.array_equal(bits(dv), vc.view(np.uint16))


def test_reshape_and_cache_bad_slot_is_reported_and_skipped(ops):
    nb, bs, H, D = 4, 16, 2, 128
    kc = torch.zeros((nb, bs, H, D), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones((2, H, D), dtype=torch.float16, device="cuda")
    slots = torch.tensor([nb * bs, 3], dtype=torch.int64, device="cuda")
    err = ops.new_error_word()
    ops.reshape_and_cache(k, k, slots, kc, vc, dev_err=err)
    assert ops.read_error_word(err) == 3   # PKV_DEV_BAD_SLOT
    flat = kc.view(nb * bs, H, D)
    assert bool((flat[3] == 1).all()) and float(flat.sum()) == H * D


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_device_slot_mapping_matches_page_formula(ops, name):
    w = wl.WORKLOADS[name]
    tables, lens, slots, _, nb = oracle_batch(w)
    err = ops.new_error_word()
    got = ops.slot_mapping(torch.from_numpy(tables).cuda(), torch.from_numpy(lens - 1).cuda(), nb,
                           dev_err=err)
    assert ops.read_error_word(err) == 0
    assert np.array_equal(got.cpu().numpy(), slots)


def test_slot_mapping_edge_cases(ops):
    tables = torch.tensor([[5, 2], [1, -1], [9, 0]], dtype=torch.int32, device="cuda")
    pos = torch.tensor([17, -1, 3], dtype=torch.int32, device="cuda")
    err = ops.new_error_word()
    got = ops.slot_mapping(tables, pos, num_blocks=8, dev_err=err)
    assert got.cpu().tolist() == [2 * 16 + 1, -1, -1]
    assert ops.read_error_word(err) == 1     # block 9 is outside the pool of 8
    err = ops.new_error_word()
    ops.slot_mapping(tables, torch.tensor([40, 0, 0], dtype=torch.int32, device="cuda"), 16,
                     dev_err=err)
    assert ops.read_error_word(err) == 5     # position past the table


def test_copy_blocks_prefix_sharing_pairs(ops):
    w = wl.WORKLOADS["prefix-sharing"]
    _, _, _, pairs, nb = oracle_batch(w)
    assert pairs.shape == (120, 2)
    rng = np.random.default_rng(4)
    shape = (nb, 16, 32, 128)
    kc = rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    vc = rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    err = ops.new_error_word()
    ops.copy_blocks(dk, dv, torch.from_numpy(pairs).cuda(), dev_err=err)
    assert ops.read_error_word(err) == 0
    oc.copy_blocks([kc], [vc], pairs)
    assert np.array_equal(bits(dk), kc.view(np.uint16))
    assert np.array_equal(bits(dv), vc.view(np.uint16))


def test_copy_blocks_multi_layer_and_bad_pair(ops):
    rng = np.random.default_rng(5)
    layers = 3
    shape = (10, 16, 4, 128)
    ks = [rng.standard_normal(shape).astype(np.float16) for _ in range(layers)]
    vs = [rng.standard_normal(shape).astype(np.float16) for _ in range(layers)]
    dks = [torch.from_numpy(a).cuda() for a in ks]
    dvs = [torch.from_numpy(a).cuda() for a in vs]
    pairs = np.array([[1, 7], [3, 3], [12, 2], [4, 0]], dtype=np.int64)
    err = ops.new_error_word()
    ops.copy_blocks(dks, dvs, torch.from_numpy(pairs).cuda(), dev_err=err)
    assert ops.read_error_word(err) == 1      # pair (12, 2) names a block past the pool
    good = pairs[[0, 1, 3]]
    oc.copy_blocks(ks, vs, good)
    for a, d in zip(ks + vs, dks + dvs):
        assert np.array_equal(bits(d), a.view(np.uint16))


@pytest.mark.parametrize("Hkv", [12, 40])
def test_copy_blocks_partial_last_chunk(ops, Hkv):
    """A block copy is cut into 32 KB chunks: 12 KV heads make 48 KB blocks (a
    full chunk and half of one), 40 make 160 KB (five); every other block
    stays as it was."""
    rng = np.random.default_rng(Hkv)
    shape = (24, 16, Hkv, 128)
    kc = rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    vc = rng.standard_normal(shape, dtype=np.float32).astype(np.float16)
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    # destinations are fresh blocks, as copy-on-write makes them (no pair
    # writes a block another pair reads)
    pairs = np.array([[0, 23], [5, 6], [11, 11], [17, 1], [2, 20]], dtype=np.int64)
    err = ops.new_error_word()
    ops.copy_blocks(dk, dv, torch.from_numpy(pairs).cuda(), dev_err=err)
    assert ops.read_error_word(err) == 0
    oc.copy_blocks([kc], [vc], pairs)
    assert np.array_equal(bits(dk), kc.view(np.uint16))
    assert np.array_equal(bits(dv), vc.view(np.uint16))


def test_swap_blocks_device_host_round_trip(ops):
    """swap-out to pinned host memory and swap-in to other device blocks, bit-exact
    against the oracle's copy definition."""
    rng = np.random.default_rng(8)
    nb, hb = 40, 12
    shape = (nb, 16, 4, 128)
    kc = rng.standard_normal(shape).astype(np.float16)
    vc = rng.standard_normal(shape).astype(np.float16)
    dk, dv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    hk = torch.zeros((hb,) + shape[1:], dtype=torch.float16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = np.array([[3, 0], [17, 5], [39, 11], [8, 2]], dtype=np.int64)
    err = ops.new_error_word()
    ops.swap_blocks([dk, dv], [hk, hv], torch.from_numpy(out_pairs).cuda(), dev_err=err)
    assert ops.read_error_word(err) == 0
    for src, dst in out_pairs:
        assert np.array_equal(hk[dst].numpy().view(np.uint16), kc[src].view(np.uint16))
        assert np.array_equal(hv[dst].numpy().view(np.uint16), vc[src].view(np.uint16))
    in_pairs = np.array([[0, 20], [5, 21], [11, 3], [2, 39]], dtype=np.int64)
    ops.swap_blocks([hk, hv], [dk, dv], torch.from_numpy(in_pairs).cuda(), dev_err=err)
    assert ops.read_error_word(err) == 0
    # the oracle's own host pools after the swap-out, then the swap-in
    ek = np.zeros((hb,) + shape[1:], np.float16)
    ev = np.zeros_like(ek)
    for src, dst in out_pairs:
        ek[dst], ev[dst] = kc[src], vc[src]
    for src, dst in in_pairs:
        kc[dst], vc[dst] = ek[src], ev[src]
    assert np.array_equal(bits(dk), kc.view(np.uint16))
    assert np.array_equal(bits(dv), vc.view(np.uint16))
    bad = torch.tensor([[0, 1], [hb, 2]], dtype=torch.int64, device="cuda")
    ops.swap_blocks([hk], [dk], bad, dev_err=err)
    assert ops.read_error_word(err) == 1


def test_bounded_wait_gives_up_and_reports(ops):
    """A barrier nothing arrives on: the wait runs out after its limit, the
    kernel reports PKV_DEV_WAIT_TIMEOUT and returns; the GPU keeps working."""
    import ctypes
    import time
    from paged_kv_cache_138_gb300._lib import lib
    err = ops.new_error_word()
    landed = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    rc = lib().pkv_selftest_bounded_wait(ctypes.c_void_p(err.data_ptr()),
                                         ctypes.c_void_p(landed.data_ptr()), 50, stream)
    assert rc == 0
    assert ops.read_error_word(err) == 4          # PKV_DEV_WAIT_TIMEOUT
    assert int(landed.item()) == 0
    assert time.perf_counter() - t0 < 10
    # the context is still usable: a normal kernel runs and reports no error
    x = torch.randn((2, 16, 1, 16), device="cuda").half()
    err2 = ops.new_error_word()
    ops.copy_blocks(x, x.clone(), torch.tensor([[0, 1]], dtype=torch.int64, device="cuda"),
                    dev_err=err2)
    assert ops.read_error_word(err2) == 0 and torch.equal(x[0], x[1])
