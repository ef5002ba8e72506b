"""The multi-GPU path of bench.py is replicas only: the layer shards by tokens
with no exchange, so N ranks run N independent replicas (weak scaling), each
on its own seeded batch, and only the timing is reduced (max over ranks).

These tests run that host logic as two gloo ranks on CPU processes, with the
oracle standing in for the GPU kernels: each rank's batch differs from the
other's, each rank's result is the layer applied to its own batch alone
(replicas share nothing), the max over ranks is the slowest rank's time on
every rank, and the whole-job rate counts every rank's tokens.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402




def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import moe_synth as ms
        import oracle

        wl = ms.WORKLOADS["tiny"]
        inp = bench.replica_layer(wl, rank)
        d = inp.dims
        r = oracle.forward(inp, nthreads=1)
        slow = bench.max_over_ranks(float(rank + 1), world)
        rate = bench.whole_job_rate(d.T, world, slow)
        gathered = [None] * world
        dist.all_gather_object(gathered, (inp.x.tobytes(), np.asarray(r[0]).tobytes()))
        results[rank] = dict(slow=slow, rate=rate, T=d.T, gathered=gathered)
    finally:
        dist.destroy_process_group()


def test_two_replicas_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(240)
        for p in procs:
            if p.is_alive():
                p.kill()
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(results)
    assert sorted(res) == [0, 1]
    # the slowest rank's time reaches every rank
    assert res[0]["slow"] == res[1]["slow"] == 2.0
    # whole-job rate: both ranks' tokens over the slowest time
    assert res[0]["rate"] == pytest.approx(2 * res[0]["T"] / 2.0)
    (x0, o0), (x1, o1) = res[0]["gathered"]
    assert x0 != x1  # each replica its own batch
    # replicas share nothing: rank r's output is the layer on rank r's batch alone
    import bench
    import moe_synth as ms
    import oracle
    for rank, o in ((0, o0), (1, o1)):
        r = oracle.forward(bench.replica_layer(ms.WORKLOADS["tiny"], rank), nthreads=1)
        assert np.asarray(r[0]).tobytes() == o
