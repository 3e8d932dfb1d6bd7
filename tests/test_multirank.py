"""The N > 1 path of bench.py on CPU: replicas over a gloo process group.

The attention path does not shard (every GPU runs its own batch; no data
collective), so what runs across ranks is host logic: independent per-rank
batches, the barrier and the max over ranks of the timings, and rank 0 alone
printing the reference arm's line.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import workloads as wl
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.0 + rank)
        bench.barrier()
        w = wl.config(bench.DECODE_CFG, seed=bench.rank_seed(bench.DECODE_CFG, rank))
        np.save(os.path.join(out_dir, f"seq_lens_{rank}.npy"), w.seq_lens)
        with open(os.path.join(out_dir, f"max_{rank}.json"), "w") as f:
            json.dump({"max": got}, f)
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_max_and_independent_batches(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        assert json.load(open(tmp_path / f"max_{r}.json"))["max"] == float(world)
    a, b = (np.load(tmp_path / f"seq_lens_{r}.npy") for r in range(world))
    assert a.shape == b.shape and not np.array_equal(a, b)   # same shapes, independent draws
    import workloads as wl
    import bench
    assert np.array_equal(a, wl.config(bench.DECODE_CFG).seq_lens)  # rank 0 is the workload itself


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
