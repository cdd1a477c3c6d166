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


def test_single_thread_oracle_child_prints_its_rate():
    """The cpu_baseline's single-thread leg: bench.py in child mode with the BLAS pools
    capped at one thread prints the oracle's rate as one JSON line."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny_fp32", "--oracle-rate",
                        "0.2"], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["value"] > 0 and "sequences" in d["sample"]


def test_algorithmic_bytes_follow_the_method_steps():
    """Per-kernel work counts the method step's operands once in the storage type, never
    this design's fp32 intermediates: LayerNorm 2 T H e; proj / FC2 read A, W and the
    residual and write C; the step's list holds offsets + removal, seven steps per
    layer and the rebuild."""
    import bench
    wk = bench.make_workload("bert_large_bf16_x24", 0)
    T, H, F, e = wk.T, 1024, 4096, 2
    assert wk.work("layernorm1") == (0.0, 2 * e * T * H)
    assert wk.work("layernorm2") == (0.0, 2 * e * T * H)
    assert wk.work("gemm_proj") == (2.0 * T * H * H, e * (3 * T * H + H * H))
    assert wk.work("gemm_fc2") == (2.0 * T * F * H, e * (T * F + F * H + 2 * T * H))
    assert wk.work("attention")[1] == 4 * e * T * H
    steps = wk.method_steps()
    assert len(steps) == 2 + 7 * 24
    sw = bench.make_workload("swin_t_stage1_fp16", 0)
    assert len(sw.method_steps()) == 7
    assert sw.work("layernorm1") == (0.0, 2 * 2 * sw.T * 96)
