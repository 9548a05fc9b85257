"""The N > 1 host path of bench.py on CPU, world size 2 over gloo: process
group set-up, the barrier and the max-over-ranks timing reduction, and the
launch the contract uses (torch.distributed.run, 127.0.0.1) for the
reference arm, where rank 0 alone runs and prints and the other rank exits 0
without work.  The attention path shards (batch, head) units across ranks
with no data-path collective, so these host pieces are all of its
multi-process logic."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    world, r, local = bench._dist()
    res = {"world": world, "rank": r, "local": local, "backend": dist.get_backend()}
    bench._barrier(world)
    res["max"] = bench._max_over_ranks(1.5 + r, world)

    class A:
        steps, warmup, gpus = 1, 0, 2
    if r != 0:
        res["reference_rc"] = bench.run_reference(A, world, r)   # no work, no output
    bench._barrier(world)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as fh:
        json.dump(res, fh)


def test_gloo_world2_barrier_and_max_over_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, g in enumerate(got):
        assert (g["world"], g["rank"], g["local"]) == (2, r, r)
        assert g["backend"] == "gloo"
        assert g["max"] == 2.5                      # max over ranks of 1.5 + rank
    assert got[1]["reference_rc"] == 0


def test_torchrun_reference_arm_world2():
    """The driver's launch form with --nproc-per-node 2: one JSON line from
    rank 0 (the oracle's timed sample), exit 0 everywhere."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="4", CUDA_VISIBLE_DEVICES="")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
