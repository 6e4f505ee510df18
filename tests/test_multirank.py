"""The multi-GPU path on CPU: replicas with no data exchange, so what runs
across ranks is only the timing aggregation (the slowest rank's step time,
whole-job throughput = ranks x one rank's work / that time) and the
reference arm's rank-0-only rule.  Both run here as gloo process groups of
two ranks."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    b = _bench()
    step_ms = [0.25, 0.40][rank]          # rank 1 is the slow replica
    worst = b.max_over_ranks(step_ms, world, "cpu")
    value = b.whole_job_tflops(1e9, world, worst)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"worst": worst, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_sum_the_work(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["worst"] == 0.40
        assert abs(g["value"] - 2 * 1e9 / 0.40e-3 / 1e12) < 1e-12


def test_one_rank_is_unchanged():
    b = _bench()
    assert b.max_over_ranks(0.3, 1, "cpu") == 0.3
    assert b.whole_job_tflops(2e9, 1, 0.5) == pytest.approx(2e9 / 0.5e-3 / 1e12)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    """`bench.py --impl reference` launched as the driver launches it for
    N > 1: rank 0 alone runs the oracle and prints one JSON line; the other
    rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
