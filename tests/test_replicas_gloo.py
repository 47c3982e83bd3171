"""The multi-process path of bench.py, on the CPU with the gloo backend and
two ranks: every rank runs its own replica (the path has no exchange step),
the job's time is the slowest rank's, and only rank 0 reports."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local, pg = bench.dist_setup(False)
    assert (w, r, local) == (world, rank, rank) and pg is not None
    bench.barrier(pg, False)
    # rank r took (10 + r) ms for its 4 steps: the job is as slow as its slowest rank
    us, ms = bench.job_us_per_step(pg, 10.0 + rank, 4, world, False)
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as fh:
        json.dump({"us": us, "ms": ms}, fh)
    pg.destroy_process_group()


def test_two_gloo_ranks_time_the_slowest_replica(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        d = json.load(open(tmp_path / ("rank%d.json" % r)))
        assert d["ms"] == pytest.approx(11.0)
        # whole-job microseconds per step: 11 ms over 4 steps on each of 2 replicas
        assert d["us"] == pytest.approx(11.0e3 / (4 * world))


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    us, ms = bench.job_us_per_step(None, 8.0, 4, 1, False)
    assert (us, ms) == (2000.0, 8.0)


def test_reference_arm_under_torchrun_two_ranks():
    """bench.py --impl reference under torchrun: rank 0 alone times the oracle
    and prints one JSON line; the other rank exits 0 without output."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if '{"impl"' in l]
    assert len(lines) == 1, res.stdout[-2000:]
    d = json.loads(lines[0][lines[0].index("{"):])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
