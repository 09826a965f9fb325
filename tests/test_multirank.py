"""The N > 1 launch of bench.py, on CPU with gloo (world size 2).

Decode attention has no collective: N GPUs run N independent replicas and
the reported time is the maximum over ranks.  These tests cover that host
logic without a GPU: the max-over-ranks reduction and barrier, and the
reference arm under torchrun (rank 0 alone runs and prints one line)."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    class Args:
        impl = "reference"  # gloo: the host-only arm

    w, r, _ = bench.dist_setup(Args)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + 5.0 * rank, w)  # per-rank step times
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    vals = [float((tmp_path / f"rank{r}.txt").read_text()) for r in range(world)]
    assert vals == [15.0, 15.0]  # every rank sees the slowest rank's time


def test_reference_arm_under_torchrun_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--config", "single"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
