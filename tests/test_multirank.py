"""The multi-GPU host logic of bench.py with two ranks over gloo on the CPU: every rank ends with
the slowest rank's time, the whole-job rate counts every rank's units (weak scaling), only rank 0
reports, and the reference arm does no work on other ranks.  One process per rank, started with
'spawn', rendezvous on 127.0.0.1."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                        # rank r took 10 + 5 r ms
        slowest = bench.max_over_ranks(ms)
        rate = bench.job_rate(32 * 100, world, slowest)
        ref_rc = None
        if rank != 0:   # the reference arm returns at once on ranks other than 0
            sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"]
            ref_rc = bench.run_reference(bench.parse_args())
        results[rank] = (slowest, rate, ref_rc)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(results)
    slowest = 10.0 + 5.0 * (world - 1)
    for r in range(world):
        assert res[r][0] == slowest                      # every rank sees the slowest rank's time
        assert res[r][1] == pytest.approx(world * 3200 / (slowest / 1e3))
    assert res[1][2] == 0                                # reference arm: no work, exit 0, off rank 0


def test_one_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_rate(320, 1, 2.0) == pytest.approx(160000.0)
