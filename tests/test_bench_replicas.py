"""bench.py's multi-process path on CPU, two ranks over the gloo backend.

The hot path has no exchange step, so `bench.py --gpus N` runs N independent replicas
(one per GPU under torchrun): a barrier brackets the timed region, the elapsed time
is the maximum over ranks, and the whole-job value is all ranks' units over that
time.  Here the same helpers run as two gloo ranks (the process-group set-up picks
gloo when no GPU is visible), and the reference arm runs under torchrun with two
processes: rank 0 alone times the oracle and prints the one JSON line, the other rank
exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="exercises the CPU (gloo) set-up; with a GPU visible the ranks take NCCL")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    got_world, got_rank, _ = bench._dist()
    bench._barrier(got_world)
    elapsed = 1.0 + rank  # rank 1 is the slow one
    out = {"world": got_world, "rank": got_rank,
           "max": bench._max_over_ranks(elapsed, got_world),
           "rate": bench._job_rate(10, elapsed, got_world)}
    bench._barrier(got_world)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(out, f)
    torch.distributed.destroy_process_group()


def test_replica_time_is_the_slowest_rank_and_value_counts_all_ranks(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        with open(tmp_path / f"rank{rank}.json") as f:
            got = json.load(f)
        assert (got["world"], got["rank"]) == (2, rank)
        assert got["max"] == 2.0
        assert got["rate"] == 2 * 10 / 2.0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-tokens", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [line for line in p.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1, p.stdout
    got = json.loads(lines[0])
    assert got["impl"] == "reference" and got["n_gpus"] == 2 and got["value"] > 0
    assert got["cpu_baseline"]["kind"] == "oracle" and got["cpu_baseline"]["value"] == got["value"]
    assert got["e2e"] == {"value": got["value"], "unit": got["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
