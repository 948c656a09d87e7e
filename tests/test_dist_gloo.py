"""The N > 1 host path on CPU: two gloo ranks, as torchrun would launch them."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from paged_kv_cache_138_gb300 import dist as pd
        from paged_kv_cache_138_gb300 import workloads as wl
        from paged_kv_cache_138_gb300.scenario import prepare_batch
        w_, r_, _ = pd.env()
        assert (w_, r_) == (world, rank)
        w = pd.replica(wl.WORKLOADS["llama2-13b-layer"], rank)
        batch = prepare_batch(w)              # each rank's own batch, no exchange
        elapsed = 1.0 + rank                  # stand-in for a per-rank time
        pd.barrier()
        m = pd.max_over_ranks(elapsed)
        q.put((rank, m, int(batch.context_lens.sum()), batch.slot_mapping.tolist()[:4],
               pd.shard_bounds(64, world, rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(native_lib):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [2.0, 2.0]          # max over ranks
    assert res[0][2] != res[1][2] or res[0][3] != res[1][3]   # independent replicas
    assert res[0][4] == (0, 32) and res[1][4] == (32, 64)


def test_shard_bounds_cover_exactly():
    from paged_kv_cache_138_gb300.dist import shard_bounds
    for n in (0, 1, 5, 64, 257):
        for world in (1, 2, 3, 8):
            spans = [shard_bounds(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [e - s for s, e in spans]
            assert max(sizes) - min(sizes) <= 1
