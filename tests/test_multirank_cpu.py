"""The multi-GPU form of the bench, on the CPU.

The layer-step does not shard: N GPUs run N independent replicas and the job
reports the tokens all ranks processed over the slowest rank's time.  These
tests run that aggregation over two gloo ranks, and the reference arm under
torchrun (rank 0 alone times the oracle; the other ranks exit without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist            # noqa: E402
import torch.multiprocessing as mp          # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench                                # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, totals, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.slowest_rank_ms(totals[rank], dist, "cpu")
        out[rank] = (got, bench.job_tokens_per_s(world, 7, 50, got))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_over_gloo():
    world, port = 2, _free_port()
    totals = [12.5, 14.75]          # ms: rank 1 is the slower replica
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, totals, out), nprocs=world, start_method="spawn")
        res = dict(out)
    for rank in range(world):
        got, value = res[rank]
        assert got == 14.75
        # 2 replicas x 7 tokens x 50 steps over the slowest rank's 14.75 ms
        assert value == pytest.approx(2 * 7 * 50 / 14.75e-3)


def test_single_process_needs_no_collective():
    assert bench.slowest_rank_ms(3.25) == 3.25
    assert bench.job_tokens_per_s(1, 7, 10, 2.0) == pytest.approx(35000.0)


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--experts", "16", "--hot", "12", "--tokens", "7", "--cpu-budget", "1"]
    env = dict(os.environ, OMP_NUM_THREADS=os.environ.get("OMP_NUM_THREADS", "4"))
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["single_core"]["cores"] == 1 and line["cpu_baseline"]["single_core"]["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
