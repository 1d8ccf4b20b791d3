"""The multi-GPU host logic of bench.py on CPU ranks (gloo, world size 2):
barrier, max-over-ranks of the timed duration, whole-job rate, and that each
rank draws its own sequences (weak scaling, no data-path collective)."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    try:
        w, r, _ = bench.dist_env()
        bench.dist_init(w, "gloo")
        bench.dist_barrier(w)
        ms_local = 100.0 + 50.0 * r                    # rank 1 is the slow one
        value, ms_step = bench.whole_job_rate(64, ms_local, 10, w, torch.device("cpu"))
        wl = W.workload_stack_decode()
        seed = wl.seed + 100 * r                       # the per-rank seed bench.py uses
        q.put((r, value, ms_step, seed))
        dist.destroy_process_group()
    except Exception as e:                             # report, never hang the parent
        q.put((rank, "error", repr(e), None))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for r, value, ms_step, seed in out:
        assert value != "error", ms_step
        assert ms_step == pytest.approx(15.0)          # max(100, 150) ms over 10 steps
        assert value == pytest.approx(2 * 64 / 0.015)   # both ranks' tokens over the slowest time
    assert out[0][3] != out[1][3]                      # different sequences per rank
