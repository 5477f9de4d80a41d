"""The N > 1 path of the benchmark on CPU ranks (gloo, world size 2).

The workload partitions by sequence: every rank holds its own batch (same shapes, its own
seed) and the only exchange is the max-over-ranks of the timed interval, so what there is
to check is host logic: the process group comes up from the launcher's environment, each
rank's workload differs, the max reduction and the barrier work, and the reference arm
prints one line from rank 0 while the other rank exits quietly."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.dist_setup("gloo")
    cfg = bench.rank_config("llama7b", r)
    worst = bench.max_over_ranks(1.5 + r, ws)
    bench.barrier(ws)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"ws": ws, "rank": r, "local": local, "seed": cfg.seed, "batch": cfg.batch,
                   "heads": cfg.num_q_heads, "worst": worst}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_bench_helpers_on_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    mp.start_processes(_worker, args=(free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [g["ws"] for g in got] == [2, 2] and [g["rank"] for g in got] == [0, 1]
    assert got[0]["seed"] != got[1]["seed"]  # each rank its own sequences ...
    assert got[0]["batch"] == got[1]["batch"] and got[0]["heads"] == got[1]["heads"]  # ... of the same shape
    assert got[0]["worst"] == got[1]["worst"] == 2.5  # the slowest rank's time on every rank


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--config", "tiny"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
