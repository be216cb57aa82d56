"""The N>1 path of bench.py on CPU, world size 2 over gloo.

The hot path does not shard: N GPUs run N replicas with no collective on the
data path. What the multi-rank run adds is host logic: the timed region of
the slowest rank sets the step time (a MAX all-reduce), the whole-job rate
counts the bytes of every rank, and the reference arm under torchrun runs on
rank 0 alone (the other ranks exit 0 without work or output).
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rate_worker(rank, world, port, outdir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    # rank r timed 10 steps in (12 + 8 r) ms; each step streams 1e9 bytes per rank
    ms, gbs = bench.whole_job_rate(1e9, 12.0 + 8.0 * rank, 10, world, torch, torch.device("cpu"))
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "gbs": gbs}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_whole_job_rate_takes_the_slowest_rank(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rate_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        # slowest rank: 20 ms / 10 steps = 2 ms per step; 2 ranks x 1 GB / 2 ms
        assert got["ms"] == pytest.approx(2.0)
        assert got["gbs"] == pytest.approx(1000.0)


def test_single_rank_rate_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, gbs = bench.whole_job_rate(5e8, 30.0, 10, 1, torch, torch.device("cpu"))
    assert ms == pytest.approx(3.0) and gbs == pytest.approx(500e6 / 3e-3 / 1e9)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--ref-frac", "0.004"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
