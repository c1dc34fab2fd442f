"""The multi-rank host logic of bench.py (rendezvous, barrier, max over ranks,
whole-job rate) on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    active = bench.init_dist(w, "gloo")
    bench.barrier(active)
    slow = bench.max_over_ranks(10.0 + rank, active)
    rate = bench.whole_job_rate(4096 * 20, w, slow)
    q.put((r, w, active, slow, rate))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for r, (rank, world, active, slow, rate) in enumerate(res):
        assert rank == r and world == 2 and active
        assert slow == 11.0                                  # the slowest rank's time
        assert rate == pytest.approx(4096 * 20 * 2 / 11.0)   # units of all ranks / max time


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, False) == 3.5
    assert bench.whole_job_rate(100, 1, 2.0) == 50.0


def _failing_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import time

    import bench
    _, w, _ = bench.dist_env()
    active = bench.init_dist(w, "gloo", timeout_s=5)
    bench.barrier(active)                     # both ranks reach the first barrier
    if rank == 1:
        q.put((rank, "left"))
        q.close()
        q.join_thread()
        os._exit(0)                           # rank 1 fails between steps
    t0 = time.time()
    try:
        bench.max_over_ranks(1.0, active)     # the next collective of rank 0
        q.put((rank, "no error"))
    except Exception as e:                    # noqa: BLE001 - any error is the detection
        q.put((rank, f"detected after {time.time() - t0:.1f}s: {type(e).__name__}"))
    q.close()
    q.join_thread()
    os._exit(0)


def test_a_rank_that_leaves_is_detected_by_the_others():
    """Host-side failure detection: rank 1 exits between steps; rank 0's next collective
    ends with an error within the process-group timeout instead of hanging."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_failing_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res[1] == "left"
    assert res[0].startswith("detected after"), res[0]
