"""The multi-process side of bench.py on the CPU: two gloo ranks run the
same helpers the GPU bench uses under torchrun (process-group set-up, the
barrier around the timed region, the max of the elapsed times over ranks),
and the reference arm runs on rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    w, r, local = bench.dist_setup(world)
    bench.barrier(w)
    # each rank's "elapsed time"; every rank must see the largest
    m = bench.max_over_ranks(0.5 + r, w)
    bench.barrier(w)
    q.put((r, w, local, m, dist.get_backend()))
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for r, w, local, m, backend in out:
        assert w == 2 and local == r and backend == "gloo"
        assert m == 1.5


def _bench(args, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, env=env,
                          capture_output=True, text=True, timeout=600, cwd=ROOT)


def test_reference_arm_runs_on_rank0_only():
    # rank 1 of 2: exits 0 without work or output
    r1 = _bench(["--impl", "reference", "--steps", "2", "--warmup", "3"],
                {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""


@pytest.mark.timeout(600)
def test_reference_arm_json_line():
    r0 = _bench(["--impl", "reference", "--steps", "2", "--warmup", "3",
                 "--reference-seconds", "2"], {"RANK": "0", "WORLD_SIZE": "1"})
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
