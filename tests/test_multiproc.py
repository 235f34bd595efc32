"""The N > 1 path on CPU: world_size-2 gloo ranks (no GPU).

bench.py runs N independent replicas (weak scaling, no data-path collective);
the only collective is the max of the per-rank timings.  These tests check
that host logic: each rank draws its own batch, the job throughput divides all
ranks' work by the slowest rank's time, and the reference arm's non-zero ranks
exit without work.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import fa_workloads as W
        w = bench.rank_workload(W.WORKLOADS["tiny"], rank)
        x = W.make_inputs(w, with_dout=False)
        # distinct batches per rank: gather a checksum of q from every rank
        cs = torch.tensor([float(x["q"].float().sum())])
        allcs = [torch.zeros(1) for _ in range(world)]
        dist.all_gather(allcs, cs)

        def reduce_max(v):
            t = torch.tensor([v], dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return float(t)

        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slowest
        value, slowest = bench.aggregate(local_ms, 1e12, world, reduce_max)
        ref_rc = None
        if rank != 0:
            ref_rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1",
                                 "--warmup", "0"])
        q.put((rank, [float(c) for c in allcs], value, slowest, ref_rc))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, cs0, v0, s0, _), (_, cs1, v1, s1, ref1) = results
    assert cs0 == cs1 and cs0[0] != cs0[1]  # each rank drew its own batch
    assert s0 == s1 == 15.0                  # max over ranks
    assert v0 == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
    assert ref1 == 0                         # reference arm: rank 1 exits, no work
