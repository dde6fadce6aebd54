"""The benchmark's multi-process path on CPU: world size 2 over gloo.

The tree-verify path shards into independent replicas (one per GPU) with no
data-path exchange; the only collectives are the timing plumbing -- a barrier
around the timed region and a max over ranks of the elapsed time -- and the
whole-job value counts every rank's nodes against the slowest rank.  These
tests run that plumbing (and the reference arm under torchrun, where rank 0
alone works and prints) without a GPU.
"""
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
                      BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w = bench.init_dist()
    assert (r, w) == (rank, world)
    bench.barrier(w)
    ms = 10.0 + 5.0 * rank             # rank 1 is the slower one
    ms_max = bench.reduce_max(w, ms)
    value = bench.aggregate_value(w, 7, ms_max)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms_max": ms_max, "value": value}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_timing_collectives_world2_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    import bench
    for r in res:
        assert r["ms_max"] == 15.0                       # the max over ranks, seen by every rank
        # 2 ranks x 22 nodes x 64 layers x 7 steps in 15 ms
        assert r["value"] == pytest.approx(2 * bench.BUDGET * bench.N_LAYERS * 7 / 15e-3)


def test_reference_arm_under_torchrun_world2():
    port = _free_port()
    env = dict(os.environ, BENCH_BACKEND="gloo", PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                                   # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
