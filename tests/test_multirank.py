"""The multi-GPU path of bench.py on CPU: replicas only (every (b, h) pair is
independent, so each rank runs its own batch and no collective touches the
data).  Two gloo ranks check the one collective there is, the max of the
timed region over ranks behind the whole-job throughput, and the per-rank
batch seeds; the reference arm runs on rank 0 alone."""
import multiprocessing as mp
import socket
import types

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms_local, q):
    import os
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.job_throughput(ms_local, world, 1.0e12, 10, "cpu")))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ms = {0: 120.0, 1: 200.0}
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ms[r], q)) for r in (0, 1)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        ms_max, value = got[r]
        assert ms_max == 200.0  # the slower rank sets the job's time
        # 2 ranks x 10 steps x 1 TFLOP in 0.2 s
        assert abs(value - 100.0) < 1e-9


def test_one_rank_needs_no_collective():
    ms_max, value = bench.job_throughput(50.0, 1, 2.0e12, 5)
    assert ms_max == 50.0 and abs(value - 200.0) < 1e-9


def test_ranks_draw_distinct_batches():
    seeds = [bench.rank_seed(2, r) for r in range(8)]
    assert seeds[0] == 2 and len(set(seeds)) == 8


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(steps=1, warmup=0)
    assert bench.bench_reference(args, 2, 1) is None
