"""Pins the slot / reshape_and_cache / copy_blocks oracle and the KV sizing arithmetic."""
import numpy as np
import pytest

from conftest import load_golden
from oracle import cache_ops


def test_slot_formula_example1():
    # P06 example 1: table [0, 1], bs 4 -> slot(x, 5) = 1 * 4 + 1 = 5; after the
    # third append the table is [0, 1, 2] and position 8 sits at slot 8
    assert cache_ops.slot([0, 1], 5, 4) == 5
    assert [cache_ops.slot([0, 1, 2], p, 4) for p in (6, 7, 8)] == [6, 7, 8]
    # a scattered table: position 17 of [9, 3] with bs 16 is row 1 of block 3
    assert cache_ops.slot([9, 3], 17, 16) == 3 * 16 + 1


def test_reshape_and_cache_reads_back():
    rng = np.random.default_rng(0)
    nb, bs, H, D, T = 6, 16, 2, 8, 5
    kc = rng.standard_normal((nb, bs, H, D)).astype(np.float16)
    vc = rng.standard_normal((nb, bs, H, D)).astype(np.float16)
    k = rng.standard_normal((T, H, D)).astype(np.float16)
    v = rng.standard_normal((T, H, D)).astype(np.float16)
    slots = np.array([0, 17, -1, 95, 40], dtype=np.int64)
    k0, v0 = kc.copy(), vc.copy()
    cache_ops.reshape_and_cache(k, v, slots, kc, vc)
    flat_k, flat_v = kc.reshape(nb * bs, H, D), vc.reshape(nb * bs, H, D)
    touched = set()
    for i, s in enumerate(slots):
        if s < 0:
            continue
        touched.add(int(s))
        assert flat_k[s].tobytes() == k[i].tobytes()
        assert flat_v[s].tobytes() == v[i].tobytes()
    for s in range(nb * bs):
        if s not in touched:
            assert flat_k[s].tobytes() == k0.reshape(nb * bs, H, D)[s].tobytes()
    with pytest.raises(IndexError):
        cache_ops.reshape_and_cache(k[:1], v[:1], np.array([nb * bs]), kc, vc)


def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(1)
    layers = [rng.standard_normal((8, 4, 2, 8)).astype(np.float16) for _ in range(6)]
    kcs, vcs = layers[:3], layers[3:]
    before = [c.copy() for c in layers]
    pairs = np.array([[1, 5], [2, 0]], dtype=np.int64)
    cache_ops.copy_blocks(kcs, vcs, pairs)
    for c, c0 in zip(layers, before):
        assert c[5].tobytes() == c0[1].tobytes()
        assert c[0].tobytes() == c0[2].tobytes()
        for b in (1, 2, 3, 4, 6, 7):
            assert c[b].tobytes() == c0[b].tobytes()


def test_kv_sizing_closed_forms():
    fx = load_golden("kv_sizing.json")
    from paged_kv_cache_138_gb300 import accounting
    for c in fx["cases"]:
        got = accounting.kv_cache_bytes(c["layers"], c["heads"], c["head_dim"], c["tokens"],
                                        c["bytes_per_elem"])
        assert got == c["bytes"]
        if "gib" in c:
            assert got / 2 ** 30 == c["gib"]
    # per-step accounting of a decode batch: valid tokens only
    assert accounting.step_kv_bytes([7, 16, 31, 48, 63], 8, 128) == 165 * 8 * 128 * 2 * 2


def test_prefix_sharing_savings_example():
    """The page's prefix-sharing arithmetic, in GiB as printed (rounded the
    page's way: 3.13, 1.53, 15.3), and the saving as the difference of the
    printed figures."""
    fx = load_golden("prefix_sharing_savings.json")
    from paged_kv_cache_138_gb300 import accounting
    gib = 2.0 ** 30
    page = fx["page"]
    full = accounting.kv_cache_bytes(fx["layers"], fx["heads"], fx["head_dim"], 4096,
                                     fx["bytes_per_elem"])
    assert abs(full / gib - page["cache_4096"]) < 0.006
    separate, shared = accounting.prefix_sharing_bytes(fx["num_requests"], fx["prefix_tokens"],
                                                       fx["layers"], fx["heads"],
                                                       fx["head_dim"], fx["bytes_per_elem"])
    assert abs(shared / gib - page["per_request"]) < 0.005
    assert shared == accounting.kv_cache_bytes(fx["layers"], fx["heads"], fx["head_dim"],
                                               fx["prefix_tokens"], fx["bytes_per_elem"])
    assert abs(shared / gib - page["shared"]) < 0.005
    assert abs(separate / gib - page["separate"]) < 0.05
    assert abs(round(separate / gib, 1) - round(shared / gib, 2) - page["saving"]) < 1e-9
    assert round(100 * (1 - shared / separate)) == page["saving_pct"]


def test_concurrent_requests_and_preallocation_examples():
    """The page's sizing of 10 concurrent 4096-token requests (in GiB, its
    weights in decimal GB, the total the sum of the printed figures) and its
    pre-allocation utilisations; paging's reservation for the same lengths
    (whole 16-token blocks) for contrast."""
    fx = load_golden("kv_sizing_examples.json")
    from paged_kv_cache_138_gb300 import accounting
    m, c = fx["model"], fx["concurrent"]
    one = accounting.kv_cache_bytes(m["layers"], m["heads"], m["head_dim"], c["tokens"],
                                    m["bytes_per_elem"])
    from decimal import ROUND_HALF_UP, Decimal
    # the page multiplies its per-request figure, rounded half-up to 3.13
    # (exactly 3.125 GiB), by the request count
    per = Decimal(one) / Decimal(2 ** 30)
    printed = float(per.quantize(Decimal("0.01"), rounding=ROUND_HALF_UP)) * c["requests"]
    assert abs(printed - c["cache_total"]) < 1e-9
    assert abs(c["requests"] * float(per) - c["cache_total"]) < 0.06     # exact: 31.25
    assert round(100 * printed / 80) == c["share_of_80"]
    weights = m["params"] * m["bytes_per_elem"] / 1e9
    assert weights == c["weights"]
    assert abs(printed + weights - c["total"]) < 1e-9
    pre = fx["preallocation"]
    for used, pct in pre["cases"]:
        assert round(100 * accounting.slot_utilization(used, pre["reserved"]), 1) == pct
        paged = accounting.slot_utilization(used, accounting.paged_reserved_tokens(used, 16))
        assert paged > 0.78 and accounting.paged_reserved_tokens(used, 16) - used < 16
