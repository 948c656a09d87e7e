"""The native continuous-batching scheduler driving the kernels, checked against
the oracle on every decoded row of every step (recompute and swap preemption)."""
import numpy as np
import pytest

from oracle import attention as oa
from parity_helpers import assert_matches_oracle
from paged_kv_cache_138_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
SEED, HQ, HKV, BS, D = 9, 4, 2, 16, 128


def oracle_row(tokens, rid, pos):
    toks = tokens[:pos + 1]
    k, v = wl.token_kv_host(wl.prefix_keys(toks, SEED), HKV, D)
    n = len(toks)
    nb = -(-n // BS)
    kc = np.zeros((nb * BS, HKV, D), np.float16)
    vc = np.zeros_like(kc)
    kc[:n], vc[:n] = k, v
    q = wl.step_query_host(SEED, rid, pos, HQ, D)[None]
    return oa.paged_attention_decode(q, kc.reshape(nb, BS, HKV, D), vc.reshape(nb, BS, HKV, D),
                                     np.arange(nb, dtype=np.int32)[None],
                                     np.array([n], np.int32), 1 / np.sqrt(D))[0]


@pytest.mark.parametrize("preemption,grouped", [("recompute", False), ("swap", False),
                                                 ("recompute", True), ("swap", True)])
def test_native_serving_matches_oracle_every_step(native_lib, preemption, grouped):
    from paged_kv_cache_138_gb300.serving import ContentKeyedValues, NativeServingDriver
    reqs = wl.serving_requests(SEED, num_requests=18, num_system_prompts=3,
                               system_prompt_len=40, suffix_max=12, new_min=3, new_max=60)
    nb = 22
    drv = NativeServingDriver(nb, HQ, HKV, max_batch=6, max_blocks_per_seq=8,
                              values=ContentKeyedValues(SEED, HQ, HKV, D),
                              free_order=np.random.default_rng(9).permutation(nb),
                              preemption=preemption, host_blocks=64, seed=SEED,
                              grouped=grouped)
    for r in reqs:
        drv.add_request(r.rid, r.prompt, r.max_new_tokens)
    got_rows, ref_rows, steps = [], [], 0
    stats = {"preempted": 0, "cached": 0, "swap_out": 0, "swap_in": 0, "shared_tokens": 0}
    while not drv.idle:
        res = drv.step()
        steps += 1
        assert steps < 500
        for k in stats:
            stats[k] += res[k]
        if len(res["rids"]) == 0:
            continue
        out = res["out"].cpu().numpy().astype(np.float64)
        for i, (rid, pos) in enumerate(zip(res["rids"].tolist(), res["positions"].tolist())):
            got_rows.append(out[i])
            ref_rows.append(oracle_row(drv.request_tokens(rid), rid, pos))
    drv.check_errors()
    assert_matches_oracle(np.stack(got_rows), np.stack(ref_rows))
    assert len(got_rows) == sum(r.max_new_tokens for r in reqs)
    assert stats["cached"] > 0 and stats["preempted"] > 0
    if preemption == "swap":
        assert stats["swap_out"] > 0 and stats["swap_in"] > 0
    if grouped:
        assert stats["shared_tokens"] > 0
    drv.bm.check_invariants()
    assert drv.bm.num_free_blocks == nb


@pytest.mark.parametrize("grouped", [False, True])
def test_native_serving_with_device_values_matches_oracle(native_lib, grouped):
    """The configuration the serving benchmark times (values drawn on the
    device, GQA, shared system prompts).  The oracle keeps its own copy of the
    cache, built from each step's inputs with its own reshape_and_cache
    (prefill rows, then after copy_blocks the new tokens, at the slots the
    step names) and copy_blocks; every few steps each decoded row is
    recomputed from that copy, the step's q rows and block tables.  At the end
    the device cache must equal the oracle's copy bit for bit."""
    import torch
    from oracle import cache_ops as oc
    from paged_kv_cache_138_gb300.serving import DeviceRandomValues, NativeServingDriver

    class Recorded(DeviceRandomValues):
        """Device draws, kept so the host can read them back after the step."""
        def prefill(self, drv, rids, positions, stream=None):
            k, v = super().prefill(drv, rids, positions, stream)
            self.prefill_kv = (k, v)
            return k, v

    hq, hkv = 8, 2
    reqs = wl.serving_requests(SEED + 1, num_requests=24, num_system_prompts=2,
                               system_prompt_len=48, suffix_max=12, new_min=3, new_max=40)
    nb, mb = 64, 8
    values = Recorded(3, hq, hkv, device="cuda")
    drv = NativeServingDriver(nb, hq, hkv, max_batch=8, max_blocks_per_seq=mb, values=values,
                              free_order=np.random.default_rng(4).permutation(nb), seed=SEED,
                              grouped=grouped)
    for r in reqs:
        drv.add_request(r.rid, r.prompt, r.max_new_tokens)
    kc = np.zeros(tuple(drv.k_cache.shape), np.float16)    # the driver's cache starts at 0
    vc = np.zeros_like(kc)
    got_rows, ref_rows, steps, shared = [], [], 0, 0
    while not drv.idle:
        values.prefill_kv = None
        res = drv.step()
        a = drv.sets[(drv.steps - 1) % 2]["a"]            # this step's arrays
        o = drv.sets[(drv.steps - 1) % 2]["out"]
        steps += 1
        assert steps < 500
        assert o.num_swap_in == 0 and o.num_swap_out == 0
        shared += res["shared_tokens"]
        torch.cuda.synchronize()
        if o.num_prefill:
            k, v = values.prefill_kv
            oc.reshape_and_cache(k.cpu().numpy(), v.cpu().numpy(),
                                 a["prefill_slots"][:o.num_prefill], kc, vc)
        if o.num_cow:
            oc.copy_blocks([kc], [vc], a["cow_pairs"][:o.num_cow])
        B = len(res["rids"])
        if B == 0:
            continue
        oc.reshape_and_cache(drv.k_new[:B].cpu().numpy(), drv.v_new[:B].cpu().numpy(),
                             a["slots"][:B], kc, vc)
        if steps % 3:
            continue
        out = res["out"].cpu().numpy().astype(np.float64)
        q = drv.q[:B].cpu().numpy()
        tables = np.ascontiguousarray(a["block_tables"][:B])
        lens = (res["positions"] + 1).astype(np.int32)
        assert (lens == a["context_lens"][:B]).all()
        got_rows.append(out)
        ref_rows.append(oa.paged_attention_decode(q, kc, vc, tables, lens, 1 / np.sqrt(D)))
    drv.check_errors()
    assert got_rows
    assert_matches_oracle(np.concatenate(got_rows), np.concatenate(ref_rows))
    assert np.array_equal(drv.k_cache.cpu().numpy().view(np.uint16), kc.view(np.uint16))
    assert np.array_equal(drv.v_cache.cpu().numpy().view(np.uint16), vc.view(np.uint16))
    if grouped:
        assert shared > 0
    drv.bm.check_invariants()
