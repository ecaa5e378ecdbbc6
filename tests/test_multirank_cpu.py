"""The multi-rank plumbing of bench.py on CPU (gloo, world size 2): the
max-over-ranks timing, the barrier, and the reference arm under torchrun
(rank 0 alone prints its JSON line; the other ranks exit 0 without work)."""
import json
import os
import socket
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    got = bench.max_over_ranks(10.0 * (rank + 1), w, "cpu")
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "max": got}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_two_gloo_ranks():
    import torch.multiprocessing as mp
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(world, _free_port(), d), nprocs=world, start_method="spawn")
        res = [json.load(open(os.path.join(d, f"rank{r}.json"))) for r in range(world)]
    assert [x["rank"] for x in res] == [0, 1]
    assert all(x["world"] == world and x["local"] == x["rank"] for x in res)
    assert all(x["max"] == 20.0 for x in res)          # every rank times the slowest


def _torchrun(*bench_args):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--gpus", "2", *bench_args]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


@pytest.mark.parametrize("workload", ["tiny", "trace"])
def test_reference_arm_prints_once_under_torchrun(workload):
    lines = _torchrun("--impl", "reference", "--workload", workload, "--steps", "1", "--warmup", "1")
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["n_gpus"] == 2 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] >= 1
