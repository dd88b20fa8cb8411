"""bench.py's multi-process host path, on the CPU: two ranks over gloo.

The path does not shard (replicas only: every rank runs the whole workload on its
own GPU and there is no data-path collective); the ranks only meet at barriers,
the timing is the maximum over ranks, and rank 0 alone prints.  Here two
processes set up the process group the way bench.py does under torchrun and
check the barrier and the max-over-ranks reduction, and the reference arm
(the CPU oracle) runs under torchrun with two ranks, printing one line.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bench_module():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank_main(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    bench = _bench_module()
    r, local, world = bench.dist_setup(2)
    bench.barrier(world)
    worst = bench.max_over_ranks(10.0 + r, world)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "local": local, "world": world, "max": worst, "backend": dist.get_backend()}, f)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_ranks_barrier_and_max_over_ranks_gloo(tmp_path):
    mp.spawn(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in (0, 1):
        got = json.load(open(tmp_path / f"rank{r}.json"))
        assert got == {"rank": r, "local": r, "world": 2, "max": 11.0, "backend": "gloo"}


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-seconds", "2"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [line for line in p.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["unit"] == "tok/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
