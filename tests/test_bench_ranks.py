"""bench.py with several ranks, on the CPU (gloo): how ranks are folded into one line.

Decode requests are independent, so every rank runs the full workload with no
data-path collective (replicas only); the ranks meet only to agree on the
timed region.  These tests run that agreement as a real two-process gloo
group, and the reference arm under torchrun with two ranks.
"""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, outdir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    # rank r timed its steps at 10 + r ms and would have chosen 100 - 7 r steps
    step_ms = b.reduce_over_ranks([10.0 + rank, 2.0 * rank], "max", world)
    steps = b.reduce_over_ranks([100 - 7 * rank], "min", world)
    value = b.whole_job_tbs(world, 302e6, step_ms[0])
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
        json.dump({"step_ms": step_ms, "steps": steps, "value": value}, f)


def test_reduce_over_ranks_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["step_ms"] == [11.0, 2.0]        # the slowest rank's time, per entry
        assert r["steps"] == [93.0]               # the smallest step count
        assert r["value"] == pytest.approx(2 * 302e6 / 11e-3 / 1e12)
    assert res[0] == res[1]


def test_one_rank_is_the_identity():
    assert bench.reduce_over_ranks([3, 1.5], "max", 1) == [3.0, 1.5]
    assert bench.whole_job_tbs(1, 302e6, 100.0) == pytest.approx(302e6 / 0.1 / 1e12)


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 alone runs the oracle and prints one line; the other rank exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["gpu_launches"] == 0
