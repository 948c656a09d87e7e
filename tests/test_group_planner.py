"""The native shared-prefix group planner against a plain Python restatement of
its rule, and on the workloads' own tables (CPU only)."""
import random

import numpy as np

from paged_kv_cache_138_gb300 import workloads as wl


def plan_reference(tables, lens, bs, limit):
    """Consecutive sequences with the same first block, at most `limit` per
    group; shared = common leading blocks with the first member, cut to a
    multiple of lcm(16, bs) and to the shortest member."""
    unit = int(np.lcm(16, bs))
    S = len(lens)
    first, seq_group, shared = [0], [0] * S, []
    s = 0
    while s < S:
        e = s + 1
        while e < S and e - s < limit and lens[s] > 0 and lens[e] > 0 and \
                tables[e][0] == tables[s][0]:
            e += 1
        tok = 0
        if e - s > 1:
            min_len = min(lens[s:e])
            lcp = -(-min_len // bs)
            for m in range(s + 1, e):
                k = 0
                while k < lcp and tables[m][k] == tables[s][k]:
                    k += 1
                lcp = k
            tok = min(lcp * bs, min_len)
            tok -= tok % unit
        for m in range(s, e):
            seq_group[m] = len(shared)
        shared.append(tok)
        first.append(e)
        s = e
    own = [lens[i] - shared[seq_group[i]] for i in range(S)]
    return first, seq_group, shared, max(shared), max(own)


def test_planner_matches_reference_on_random_tables(native_lib):
    from paged_kv_cache_138_gb300 import ops
    rnd = random.Random(3)
    for trial in range(200):
        bs = rnd.choice([8, 16, 32, 64])
        S = rnd.randint(1, 40)
        mb = rnd.randint(1, 12)
        prefixes = [[rnd.randrange(1000) for _ in range(mb)] for _ in range(3)]
        tables, lens = [], []
        for _ in range(S):
            base = list(rnd.choice(prefixes))
            cut = rnd.randint(0, mb)
            row = base[:cut] + [rnd.randrange(1000, 2000) for _ in range(mb - cut)]
            tables.append(row)
            lens.append(rnd.randint(0, mb * bs))
        tables = np.array(tables, np.int32)
        lens = np.array(lens, np.int32)
        limit = rnd.choice([1, 2, 4, 16])
        got = ops.shared_prefix_groups(tables, lens, bs, limit)
        ref = plan_reference(tables.tolist(), lens.tolist(), bs, limit)
        assert got[0].tolist() == ref[0]
        assert got[1].tolist() == ref[1]
        assert got[2].tolist() == ref[2]
        assert got[3:] == ref[3:]


def test_planner_on_prefix_sharing_workload(native_lib):
    from paged_kv_cache_138_gb300 import ops
    from paged_kv_cache_138_gb300.scenario import prepare_batch
    b = prepare_batch(wl.WORKLOADS["prefix-sharing"])
    first, seq_group, shared, mx, mo = ops.shared_prefix_groups(b.block_tables, b.context_lens)
    assert first.tolist() == list(range(0, 129, 16))
    assert shared.tolist() == [2048] * 8 and mx == 2048
    assert mo == int(b.context_lens.max()) - 2048
    b = prepare_batch(wl.WORKLOADS["llama2-13b-layer"])
    first, seq_group, shared, mx, mo = ops.shared_prefix_groups(b.block_tables, b.context_lens)
    assert len(shared) == 64 and mx == 0          # no sharing: one group per sequence
