"""Multi-rank host logic on CPU (gloo, world size 2): independent replicas
aggregate to the slowest rank's time and the tokens of all ranks; the
sequences are independent, so a rank's result does not depend on the others."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from linear_attention_recurrence_gb300.inputs import make_inputs

    local_ms = [3.0, 5.0][rank]
    ms, us, tps = bench.aggregate(local_ms, 1000, world)
    # each rank's replica: its own layer's inputs, run through the oracle
    x = make_inputs(8, seed=0, layer=rank, n_kh=2, n_vh=6, d=8, norm=False)
    o, s = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["S0"], nthreads=1)
    q.put((rank, ms, us, tps, float(np.abs(o).sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for rank, ms, us, tps, _ in res:
        assert ms == 5.0
        assert us == pytest.approx(5.0 * 1e3 / 2000)
        assert tps == pytest.approx(2000 / 5e-3)
    # replicas work on different inputs (layer = rank)
    assert res[0][4] != res[1][4]


def test_single_rank_aggregation_needs_no_group():
    import bench

    ms, us, tps = bench.aggregate(2.0, 500, 1)
    assert ms == 2.0 and us == pytest.approx(4.0) and tps == pytest.approx(250000.0)
