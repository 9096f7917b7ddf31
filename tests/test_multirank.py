"""Host logic of the multi-rank benchmark path, world size 2 on gloo (CPU).

Each rank runs an independent replica (no data-path collective); the ranks
only meet at barriers and in the max-over-ranks / sum-over-ranks reductions
that turn per-rank timings into the whole-job throughput.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    d = bench.Dist()
    d.init("gloo")
    try:
        d.barrier()
        flops = 1e12 * (rank + 1)          # rank r did (r+1) TFLOP
        ms = 100.0 * (rank + 1)            # in (r+1)*100 ms
        value, max_ms = bench.aggregate_throughput(d, flops, ms)
        out[rank] = (value, max_ms, d.max(float(rank)), d.sum(1.0))
    finally:
        d.done()


def test_two_rank_aggregation_on_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        value, max_ms, mx, sm = res[r]
        assert max_ms == 200.0                      # slowest rank's time
        assert abs(value - 3e12 / 0.2 / 1e12) < 1e-9  # all FLOPs / max time = 15 TFLOP/s
        assert mx == 1.0 and sm == 2.0


def test_single_rank_needs_no_process_group():
    import bench

    d = bench.Dist()
    assert d.world == int(os.environ.get("WORLD_SIZE", "1"))
    value, max_ms = bench.aggregate_throughput(d, 2e12, 500.0)
    assert max_ms == 500.0 and abs(value - 4.0) < 1e-12
