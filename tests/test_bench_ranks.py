"""Host-side multi-rank logic of bench.py on CPU with the gloo backend and
two ranks: the timed region's figure is the max over ranks, the job value
counts every rank's work, and ``bench.py --gpus 2`` outside a torchrun launch
starts two ranks itself (checked through the reference arm, which runs on the
CPU: both ranks join, rank 0 alone does the oracle work and prints)."""
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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    got = bench.max_over_ranks(local_ms, dist, "cpu")
    value = bench.job_tflops(2.0e12, 4, world, got)
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, got, value))


def test_two_gloo_ranks_take_the_max_and_count_all_work():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == 15.0
        # 2 ranks x 4 steps x 2e12 FLOP in 15 ms
        assert value == pytest.approx(2 * 4 * 2.0e12 / 15e-3 / 1e12)


def test_gpus_2_starts_two_ranks_itself():
    import json
    import subprocess
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    env["OMP_NUM_THREADS"] = "2"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--workload", "tiny_b1h1s128d64", "--steps", "2",
                        "--warmup", "1", "--ref-seconds", "1.5"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)
