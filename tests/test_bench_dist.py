"""bench.py's multi-process host logic on CPU with the gloo backend, world size 2:
the max-over-ranks timing reduction and barrier, and the reference arm under
torchrun (rank 0 alone runs the oracle and prints one JSON line)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.reduce_max(1.5 + rank, world)  # ranks report 1.5 and 2.5 ms
        # per-step times: rank 0 [1, 3, 2] (median 2, min 1), rank 1 [4, 0.5, 5] (median 4, min 0.5)
        stats = bench.step_stats([1.0, 3.0, 2.0] if rank == 0 else [4.0, 0.5, 5.0], world)
        out[rank] = (got, stats["ms_step_median"], stats["ms_step_min"])
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: (2.5, 4.0, 1.0), 1: (2.5, 4.0, 1.0)}  # the slowest rank's figures


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-total-seconds", "3",
           "--workload", "small_b1_h2_s256_d64"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["value"] > 0 and d["higher_is_better"] is True


def test_bench_rejects_too_few_warmup_steps():
    res = subprocess.run([sys.executable, "bench.py", "--warmup", "2", "--impl", "reference"],
                         cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert res.returncode != 0 and "warmup" in res.stderr


def test_reference_arm_times_a_window_with_dropout():
    """--window with --dropout is one combined call; the oracle arm times the same
    combination and the line's config names both."""
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "small_b1_h2_s256_d64",
                          "--window", "100", "--dropout", "0.1", "--steps", "1", "--warmup", "3",
                          "--ref-step-seconds", "1", "--ref-total-seconds", "10"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["config"]["elem_mask"]["window"] == 100 and line["config"]["dropout_p"] == 26 / 256
    assert line["value"] > 0 and line["cpu_baseline"]["cores"] >= 1
