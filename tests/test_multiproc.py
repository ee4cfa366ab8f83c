"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas, no data-path collective).  The timing is the
slowest rank's (barrier + max over ranks), and the reference arm prints from rank 0 alone."""
import io
import contextlib
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


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, w, local = bench.dist_env()
        bench.barrier(w)
        ms = bench.max_over_ranks(1.5 + rank, w)   # rank 1 is the slow one
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            args = type("A", (), {"config": "tiny_decode", "steps": 1, "warmup": 3, "kv_cache": "fp16"})()
            if r != 0:
                bench.run_reference(args, r, w)   # rank 0 alone runs the oracle arm
        results[rank] = (r, w, local, ms, out.getvalue())
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_is_the_slowest_and_only_rank0_reports():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert sorted(res) == [0, 1]
    for rank, (r, w, local, ms, out) in res.items():
        assert (r, w, local) == (rank, 2, rank)
        assert ms == pytest.approx(2.5)
    assert res[1][4] == ""   # rank 1 printed nothing
