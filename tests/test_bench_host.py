"""Host-side checks of bench.py (no GPU): the reference arm's JSON line, and the
multi-replica logic -- per-rank seeds and the max-over-ranks reduction -- with two
gloo ranks on the CPU."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny_fp32"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True


def test_replicas_draw_different_batches():
    import bench
    a = bench.make_workload("bert_base_fp16", 0)
    b = bench.make_workload("bert_base_fp16", 1)
    assert not np.array_equal(a.wl["lengths"], b.wl["lengths"])
    assert a.wl["x_padded"].shape == b.wl["x_padded"].shape


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.reduce_max(1.0 + rank, world, torch.device("cpu"))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == 2.0 and out[1] == 2.0
