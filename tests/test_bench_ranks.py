"""bench.py's multi-GPU bookkeeping on CPU: two gloo ranks (world size 2).

Each rank of `bench.py --gpus N` runs its own replica of the stack (the path
shards into independent problems, no collective on the data path); the line
reports the slowest rank's time and the whole job's bytes.  Checked here
without a GPU: the barrier, the max over ranks, the job throughput, and that
only rank 0 does the reference arm's work.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    try:
        bench.barrier(w)
        # rank 1 is the slow one: 30 ms for 10 steps against 20 ms
        ms_local = 20.0 if rank == 0 else 30.0
        ms_step, gbps = bench.job_throughput(1.0e9, ms_local, 10, w)
        results[rank] = (ms_step, gbps, bench.max_over_ranks(float(rank), w))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_rank_job_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        for r in range(world):
            ms_step, gbps, rmax = results[r]
            assert ms_step == pytest.approx(3.0)          # the slowest rank, per step
            assert gbps == pytest.approx(2 * 1.0e9 / 3.0e-3 / 1e9)
            assert rmax == 1.0


def test_single_rank_is_plain():
    import bench
    ms_step, gbps = bench.job_throughput(5.0e8, 40.0, 20, 1)
    assert ms_step == pytest.approx(2.0)
    assert gbps == pytest.approx(5.0e8 / 2.0e-3 / 1e9)


def test_reference_arm_other_ranks_do_no_work(capsys):
    """Under torchrun only rank 0 runs and prints the reference arm."""
    import bench

    class Args:
        pass

    bench.run_reference(Args(), 1, 2)
    assert capsys.readouterr().out == ""
