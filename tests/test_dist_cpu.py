"""The multi-process glue of bench.py on CPU ranks (gloo, world size 2), launched the way a
multi-GPU run is: torch.distributed.run on 127.0.0.1.  The library's path shards by sequence
with no exchange, so the only cross-rank steps are the barriers around the timed region and the
max over ranks of the step time; the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=600):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=env)


def test_barrier_and_max_over_ranks_two_gloo_ranks(tmp_path):
    worker = tmp_path / "worker.py"
    worker.write_text(textwrap.dedent(f"""
        import os, sys
        sys.path.insert(0, {ROOT!r})
        import torch.distributed as dist
        import bench
        rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
        dist.init_process_group("gloo")
        bench.barrier(world)
        got = bench.max_over_ranks(1.5 + rank, world)
        assert got == 1.5 + (world - 1), got
        assert bench.max_over_ranks(7.0, 1) == 7.0          # one rank: no collective
        with open(os.path.join({str(tmp_path)!r}, f"rank{{rank}}.txt"), "w") as f:
            f.write(repr(got))
        dist.destroy_process_group()
    """))
    r = _torchrun([str(worker)])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert [(tmp_path / f"rank{i}.txt").read_text() for i in range(2)] == ["2.5", "2.5"]


def test_reference_arm_two_ranks_prints_one_line():
    """Rank 0 times the oracle and prints the one JSON line (n_gpus = 2); rank 1 exits 0 without work."""
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--workload", "single",
                   "--steps", "3", "--warmup", "3", "--cpu-seconds", "1"])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_our_arm_fails_loudly_without_a_gpu():
    """No CPU fallback: without CUDA the product path stops with an error instead of timing anything."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--workload", "single", "--steps", "3", "--warmup", "3",
                        "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode != 0
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
