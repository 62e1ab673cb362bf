"""Host logic of the N>1 bench path, as world_size-2 gloo ranks on CPU: the timed region's
max over ranks, the whole-job rate and each rank's own batch (no data exchange)."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 100.0 + 50.0 * rank                      # rank 1 is the slow one
    m = bench.max_over_ranks(ms)
    q.put((rank, m, bench.aggregate_rate(world, 8, m)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_rate_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, m, rate in res:
        assert m == 150.0
        assert abs(rate - 2 * 8 / 0.150) < 1e-9


def test_max_over_ranks_without_a_group_is_identity():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5


def _rank_batch(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch
    import bench
    from long_context_self_gb300 import synth
    w = bench.rank_workload(synth.WORKLOADS["tiny"], dist.get_rank())
    k, _, _ = synth.kv_cache(w, "cpu")
    gathered = [torch.zeros_like(k) for _ in range(world)]
    dist.all_gather(gathered, k)
    q.put((rank, w.seed, [bool(torch.equal(gathered[0], g)) for g in gathered]))
    dist.barrier()
    dist.destroy_process_group()


def test_each_rank_runs_its_own_batch():
    """Replicas draw distinct sequences: rank 0 keeps the workload's seed, rank 1's K cache
    differs from rank 0's (checked by gathering both over gloo)."""
    from long_context_self_gb300 import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_batch, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    base = synth.WORKLOADS["tiny"].seed
    assert [r[1] for r in res] == [base, base + 100]
    for _, _, same in res:
        assert same == [True, False]
