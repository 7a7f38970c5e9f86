"""The bench's N > 1 path on CPU: two gloo ranks on 127.0.0.1, no GPU.

The path shards by replicas only (query tokens are independent; there is no
collective on the data path), so what N > 1 adds is host logic: each rank
draws its own replica of the workload, the job's step time is the slowest
rank's, and the job rate counts every rank's units over that time."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench as b
        import synth
        slowest = b.max_over_ranks(0.001 * (rank + 1), world, "cpu")
        seed = b.replica_seed(0, rank)
        w = synth.make_workload(0, seed=seed, workers=1)
        q.put((rank, slowest, seed, w.q_bits.ravel()[:64].tolist()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # Every rank sees the slowest rank's time.
    assert all(abs(t - 0.002) < 1e-15 for _, t, _, _ in res)
    # Each replica has its own seed and so its own inputs.
    assert res[0][2] != res[1][2]
    assert not np.array_equal(res[0][3], res[1][3])


def test_single_process_helpers():
    assert bench.max_over_ranks(0.25, 1, "cpu") == 0.25
    assert bench.job_rate(2, 1e12, 0.5) == 4.0
    assert bench.job_rate(4, 2e9, 1.0, 1e9) == 8.0
    assert bench.replica_seed(2, 0) != bench.replica_seed(2, 1)
