"""The benchmark's multi-rank host logic on CPU: two gloo ranks (127.0.0.1) agree on the
slowest rank's time, pass the barrier, draw different batches, and the job's throughput
counts every rank's units over that time.  No GPU and no collective on the data path: the
ranks share nothing but the timing reduction."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    from gated_delta_rule_15_gb300 import inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w_, r_, l_ = bench.dist_setup()
    bench.barrier(world)
    ms = bench.max_over_ranks(1.0 + rank, world)
    d = inputs.chunk_inputs(1, 8, 2, 64, 64, gate="scalar", dtype="f32",
                            seed=bench.rank_seed(rank))
    q.put((rank, (w_, r_, l_), ms, float(d["q"].sum()),
           bench.job_throughput(1000, ms, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port, world = _free_port(), 2
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [(2, 0, 0), (2, 1, 1)]
    assert all(r[2] == 2.0 for r in res)            # the slowest rank's time
    assert res[0][3] != res[1][3]                   # independent batches
    assert all(r[4] == pytest.approx(2 * 1000 / 2e-3) for r in res)
