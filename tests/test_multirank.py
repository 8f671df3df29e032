"""The multi-GPU path of bench.py without a GPU: ranks are processes on the
gloo backend (127.0.0.1).  Each rank owns its own batch (weak scaling, no
collective on the data path); the step time is the maximum over ranks; only
rank 0 prints."""

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
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_tree_attn_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 3 * rank, world)
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    world = 2
    mp.spawn(_max_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    vals = [float(open(tmp_path / f"r{r}").read()) for r in range(world)]
    assert vals == [13.0, 13.0]


def test_rank_batches_are_distinct():
    w = W.WORKLOADS["b64_l1k_8k_n64_greedy"]
    assert bench.rank_workload(w, 0) is w
    w1 = bench.rank_workload(w, 1)
    assert (w1.B, w1.n_nodes, w1.prefix, w1.Hq) == (w.B, w.n_nodes, w.prefix, w.Hq)
    assert not (W.prefix_lengths(w1) == W.prefix_lengths(w)).all()


def test_reference_arm_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny_b1_f32", "--steps", "2", "--warmup", "0", "--gpus", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 2
