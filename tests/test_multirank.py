"""The N > 1 host path of bench.py on CPU ranks (gloo): rows are sharded by
giving each rank its own seeded batch of the same shape (weak scaling, no
data-path collective); timing takes the maximum over ranks; under torchrun
the reference arm runs on rank 0 alone and the other ranks exit 0."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        b.barrier(world)
        t = b.max_over_ranks(world, 1.5 + rank)       # per-rank step times
        layers = b.workload_layers("single", rank, None)
        x = layers[0].x
        got = torch.tensor([t, float(x.float().sum()), float(x.shape[0]), float(x.shape[1])], dtype=torch.float64)
        allv = [torch.zeros_like(got) for _ in range(world)]
        dist.all_gather(allv, got)
        if rank == 0:
            torch.save(torch.stack(allv), out)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_max_time_and_get_distinct_row_batches(tmp_path):
    out = str(tmp_path / "ranks.pt")
    mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
    r = torch.load(out)
    assert r[0, 0] == r[1, 0] == 2.5                   # max over ranks of 1.5 and 2.5
    assert r[0, 2] == r[1, 2] and r[0, 3] == r[1, 3]   # same shape per rank (weak scaling)
    assert r[0, 1] != r[1, 1]                          # a different seeded batch per rank


def test_reference_arm_under_torchrun_prints_once(tmp_path):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "single"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
