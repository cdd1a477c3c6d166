"""Benchmark: valid tokens/s per encoder layer on one GB300, with roofline fractions.

One step = one pass of the whole hot path over one batch of synthetic input.  The
default workload is the largest single-GPU configuration, the BERT-large-shaped bf16
stack (B=64, L=384, half the lengths U[32,128] and half U[256,384], H=1024, 16 heads,
FFN 4096, 24 layers): offsets + padding removal -> 24 encoder layers -> LayerNorm with
the padding rebuild, one C-ABI call (rpp_encoder_forward).  --workload picks another
configuration: bert_base_fp16, bert_large_int8, bert_large_int8_attn (the int8 config with
the attention's products on codes too), tiny_fp32, swin_t_stage1_fp16 (one
shifted-window block, rpp_swin_block_forward), swin_t_patch_merge_fp16.

Timing: W warm-up steps, then K steps, each bracketed by its own CUDA events on the
launch stream, with a 512 MiB write between timed steps to flush the 129 MB L2 (the
flush is outside the events).  The K-step loop is bracketed by a barrier and
torch.cuda.synchronize() on both sides and the per-rank time is max-reduced.  `value`
replays one captured CUDA graph of the step; the eager (direct C-ABI call) number is
reported next to it.  value = valid tokens per step x layers x ranks / time.

Extra keys: roofline (dominant kernel, timed live inside the step with the library's
launch-event hook; algorithmic bytes and flops per launch as the method steps define
them, never the design's own intermediates), layer_roofline (the step against the sum
of the method steps' ideal times), cpu_baseline (the CPU oracle on a bounded sample,
all host cores, with a single-thread run of the same oracle beside it),
e2e (the same metric through host buffers: pinned H2D of every step's inputs and D2H of
its output inside the timed region, the copies overlapping the neighbouring steps'
compute), gpu_launches, clocks (nvidia-smi sampled during the timed region), kernels
(per-kernel breakdown).  --impl reference times the CPU
oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import ctypes as C
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "valid tokens/sec per encoder layer at 1 GB300; % of tensor-core / HBM roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="bert_large_bf16_x24")
    p.add_argument("--oracle-rate", type=float, default=0.0, help=argparse.SUPPRESS)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return PEAKS_FALLBACK, "fallback"


def src_hash(rels):
    """Short hash of the sources a traffic figure was measured on (a path or a list)."""
    h = hashlib.sha256()
    for rel in ([rels] if isinstance(rels, str) else rels):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic():
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            return json.load(f)
    return {}


def threads_used():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count()])
    except Exception:
        return os.cpu_count()


def reduce_max(value, world, device):
    """Max over ranks of a per-rank time (the job is as slow as its slowest replica)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def oracle_single_thread(args, budget_s):
    """The oracle timed on ONE host thread: a child process of this script with every
    BLAS / OpenMP pool capped at one thread before numpy loads.  Returns the child's
    {value, sample, dt} or None if it could not run."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
              "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--workload", args.workload, "--oracle-rate", str(budget_s)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s * 10 + 120)
    except (OSError, subprocess.TimeoutExpired):
        return None
    for line in reversed(r.stdout.strip().splitlines()):
        try:
            return json.loads(line)
        except ValueError:
            continue
    return None


def measure_int8_peak(torch, dev):
    """Dense int8 GEMM rate of this GPU: torch._int_mm (cuBLASLt) on 8192^3, best of 10
    (CUDA events), in TOP/s.  None if the library call is not available here."""
    n = 8192
    try:
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
        for mat2 in (b, b.t().contiguous().t()):
            try:
                torch._int_mm(a, mat2)
            except RuntimeError:
                continue
            torch.cuda.synchronize()
            best = None
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch._int_mm(a, mat2)
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1)
                best = ms if best is None else min(best, ms)
            return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except (RuntimeError, AttributeError):
        return None
    return None


# ---------------------------------------------------------------- workloads
class BertWorkload:
    """BERT-shaped path: offsets + removal -> layers -> LN2 with padding rebuild."""
    ALL_INT8 = "bert_large_int8_attn"

    def __init__(self, cfg, rank, all_int8=False):
        from workloads import make_bert_workload
        self.cfg = cfg
        self.all_int8 = all_int8
        self.wl = make_bert_workload(cfg, seed=cfg.seed + 7919 * rank)   # each replica its own batch
        self.T = int(self.wl["lengths"].sum())
        self.sum_len2 = float((self.wl["lengths"].astype(np.float64) ** 2).sum())
        self.tokens_per_step = self.T * cfg.layers
        self.dtype = {"fp32": "f32", "fp16": "f16", "bf16": "bf16", "int8": "i8 GEMMs (exact), f16"}[cfg.dtype]
        if all_int8:
            self.dtype = "i8 GEMMs and attention products (exact), f16"

    def config(self):
        c = self.cfg
        lens = (f"50% U{list(c.bimodal[0])} + 50% U{list(c.bimodal[1])}" if c.bimodal
                else f"U[{c.len_lo},{c.len_hi or c.L}]")
        name = self.ALL_INT8 if self.all_int8 else c.name
        return {"workload": f"{name}: B={c.B} L={c.L} H={c.H} heads={c.nh}x{c.d} FFN={c.F} layers={c.layers} "
                            f"dtype={c.dtype}{' (attention on codes too)' if self.all_int8 else ''}, lengths {lens}, "
                            f"padding removed via offset mask",
                "global_batch": c.B, "seq_len": c.L, "valid_tokens": self.T}

    def setup(self, rpp, torch, dev):
        c, wl = self.cfg, self.wl
        B, L, H = c.B, c.L, c.H
        self.tdt = rpp.torch_dtype(c.storage_dtype)
        int8 = c.dtype == "int8"
        ecfg = rpp.encoder_cfg(c.H, c.nh, c.F, c.eps, c.storage_dtype, int8=(2 if self.all_int8 else int(int8)),
                               tokens_hint=self.T)
        self.layers = [rpp.EncoderLayer(ecfg, l, dev) for l in wl["layers"]]
        self.lengths = torch.as_tensor(wl["lengths"], device=dev)
        self.x = torch.as_tensor(wl["x_padded"].reshape(B * L, H)).to(dev, self.tdt)
        self.y = torch.empty_like(self.x)
        self.cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
        self.po = torch.zeros(B * L, dtype=torch.int32, device=dev)
        self.packed = torch.empty_like(self.x)
        self.ws = self.layers[0].workspace(B * L, dev)
        self.err = rpp.new_error_word(dev)
        self.scales = None
        if int8:   # per-tensor activation scales from the library's calibration pass (float layer)
            from workloads import make_calibration_batch
            cal = make_calibration_batch(c)
            fl = rpp.EncoderLayer(rpp.encoder_cfg(c.H, c.nh, c.F, c.eps, "fp16"), wl["layers"][0], dev)
            cl = torch.as_tensor(cal["lengths"], device=dev)
            ccu, cpo = rpp.build_offsets(cl, L)
            cx = rpp.remove_padding(torch.as_tensor(cal["x_padded"].reshape(B * L, H)).to(dev, self.tdt), cpo, ccu,
                                    B, L)
            self.scales = [rpp.encoder_layer_calibrate(fl, cx, ccu, B, L, workspace=self.ws) / 127.0
                           for _ in self.layers]
        self.rpp = rpp

    def step(self, x=None, lengths=None, y=None):
        self.rpp.encoder_forward(self.layers, self.lengths if lengths is None else lengths,
                                 self.x if x is None else x, self.cfg.L, act_scales=self.scales,
                                 y_padded=self.y if y is None else y, cu_seqlens=self.cu, padding_offset=self.po,
                                 packed=self.packed, workspace=self.ws, err=self.err)

    def host_io(self, torch):
        """(inputs: list of (pinned host, device) pairs, output: (device, pinned host), step):
        one set of host and device buffers of the step's input and output."""
        xh = torch.empty(self.x.shape, dtype=self.tdt, pin_memory=True)
        xh.copy_(self.x.cpu())
        lh = torch.empty(self.lengths.shape, dtype=torch.int32, pin_memory=True)
        lh.copy_(self.lengths.cpu())
        yh = torch.empty(self.y.shape, dtype=self.tdt, pin_memory=True)
        xd, ld, yd = torch.empty_like(self.x), torch.empty_like(self.lengths), torch.empty_like(self.y)
        return [(xh, xd), (lh, ld)], (yd, yh), lambda: self.step(xd, ld, yd)

    def work(self, label):
        """(flops, bytes) per launch: the algorithmic work of the method step(s) the kernel
        computes, over the packed batch (T valid tokens), with each operand read once and
        each result written once in the storage type e.  Intermediates of this design
        (the fp16 pre-LayerNorm sums, the fp16 residual copy, fp32 split-K slices) are not
        counted: they are traffic, not work.  The dense padded work that removal avoids is not counted either."""
        c, T = self.cfg, self.T
        H, F, B, L = c.H, c.F, c.B, c.L
        e = 4 if c.storage_dtype == "fp32" else 2
        lab = label.replace("_i8", "")
        if lab == "gemm_qkv":      # X and Wqkv in, Q|K|V out
            return 2.0 * T * H * 3 * H, e * (T * H + 3 * H * H + 3 * T * H)
        if lab == "gemm_proj":     # A and Wo in, C out, plus the residual read
            return 2.0 * T * H * H, e * (T * H + H * H + T * H + T * H)
        if lab == "gemm_fc1":
            return 2.0 * T * H * F, e * (T * H + F * H + T * F)
        if lab == "gemm_fc2":      # A and W2 in, C out, plus the residual read
            return 2.0 * T * F * H, e * (T * F + F * H + T * H + T * H)
        if lab == "attention":     # QK^T and PV over valid keys; Q, K, V read once, O written once
            return 4.0 * H * self.sum_len2, e * 4 * T * H
        if lab in ("layernorm1", "layernorm2"):   # row in, row out (+ the int8 code copy)
            return 0.0, 2 * e * T * H + (T * H if c.dtype == "int8" and lab == "layernorm1" else 0)
        if lab == "layernorm2_rebuild":   # valid rows in, every padded slot out (pads are zeros)
            return 0.0, e * T * H + e * B * L * H
        if lab == "offsets_remove":       # lengths in; cu, offsets out; valid rows gathered
            return 0.0, 4 * B + 4 * (B + 1) + 4 * T + 2 * e * T * H
        if lab in ("quantize_x", "quantize_attn"):
            return 0.0, e * T * H + T * H
        if lab == "build_offsets":
            return 0.0, 4 * (2 * B + 1 + T)
        if lab == "remove_padding":
            return 0.0, 2 * e * T * H + 4 * T
        if lab == "rebuild_padding":
            return 0.0, e * T * H + e * B * L * H
        return 0.0, 0.0

    def method_steps(self):
        """(flops, bytes) of every method step of one step of the path (offsets and
        removal, each layer's seven steps, the rebuild), for the layer-level roofline."""
        per_layer = [self.work(k) for k in ("gemm_qkv", "attention", "gemm_proj", "layernorm1", "gemm_fc1",
                                            "gemm_fc2", "layernorm2")]
        return [self.work("offsets_remove")] + per_layer * self.cfg.layers + [self.work("rebuild_padding")]

    def oracle_rate(self, budget_s):
        """The oracle, as it stands, over whole sequences of the batch for ~budget_s."""
        import oracle
        c, wl = self.cfg, self.wl
        lens = wl["lengths"]
        qlayers = scales = None
        if c.dtype == "int8":
            from workloads import make_calibration_batch
            cal = make_calibration_batch(c)
            scales = oracle.calibrate_int8(cal["x_padded"], cal["lengths"], wl["layers"][0], c.nh, c.eps)
            if self.all_int8:
                scales = np.concatenate([scales, oracle.calibrate_int8_qkv(cal["x_padded"], cal["lengths"],
                                                                           wl["layers"][0], c.nh)])
            qlayers = [oracle.prepare_int8_layer(l) for l in wl["layers"]]
        tokens = seqs = 0
        t0 = time.perf_counter()
        for b in range(c.B):
            n = int(lens[b])
            if n == 0:
                continue
            x = wl["x_padded"][b, :n].astype(np.float64)
            cu = np.array([0, n])
            if qlayers is not None:
                for q in qlayers:
                    x = oracle.bert_layer_int8(x, cu, q, scales, c.nh, c.eps)
            else:
                oracle.bert_forward(wl["x_padded"][b:b + 1, :n], lens[b:b + 1], wl["layers"], c.nh, c.eps)
            tokens += n * c.layers
            seqs += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        sample = f"{seqs} sequences ({tokens // c.layers} tokens) x {c.layers} layer(s) of the seeded batch, fp64 numpy"
        return tokens / dt, sample, dt


class SwinWorkload:
    """Pre-LN shifted-window block on B images (S1-S7)."""

    def __init__(self, cfg, rank):
        from workloads import make_swin_workload
        self.cfg = cfg
        self.wl = make_swin_workload(cfg, seed=cfg.seed + 7919 * rank)
        self.T = cfg.T
        self.tokens_per_step = self.T
        self.dtype = {"fp16": "f16", "bf16": "bf16"}[cfg.dtype]

    def config(self):
        c = self.cfg
        return {"workload": f"{c.name}: B={c.B} images {c.I}x{c.I} C={c.C} heads={c.nh}x{c.d} window {c.w}x{c.w} "
                            f"shift {c.s} MLP {c.F}, pre-LN, shift/partition/reverse fused into attention",
                "global_batch": c.B, "seq_len": c.I * c.I, "valid_tokens": self.T}

    def setup(self, rpp, torch, dev):
        c, wl = self.cfg, self.wl
        self.tdt = rpp.torch_dtype(c.dtype)
        scfg = rpp.swin_cfg(c.I, c.C, c.nh, c.w, c.s, c.F, c.eps, c.dtype)
        self.block = rpp.SwinBlock(scfg, wl["weights"], dev)
        self.x = torch.as_tensor(wl["x"].reshape(-1, c.C)).to(dev, self.tdt)
        self.y = torch.empty_like(self.x)
        self.ws = self.block.workspace(c.B, dev)
        self.err = rpp.new_error_word(dev)
        self.rpp = rpp

    def step(self, x=None, y=None):
        self.rpp.swin_block_forward(self.block, self.x if x is None else x, self.cfg.B,
                                    y=self.y if y is None else y, workspace=self.ws, err=self.err)

    def host_io(self, torch):
        xh = torch.empty(self.x.shape, dtype=self.tdt, pin_memory=True)
        xh.copy_(self.x.cpu())
        yh = torch.empty(self.y.shape, dtype=self.tdt, pin_memory=True)
        xd, yd = torch.empty_like(self.x), torch.empty_like(self.y)
        return [(xh, xd)], (yd, yh), lambda: self.step(xd, yd)

    def work(self, label):
        c, T = self.cfg, self.T
        C_, F = c.C, c.F
        e = 2
        if label in ("layernorm1", "layernorm2"):
            return 0.0, 2 * e * T * C_
        if label == "gemm_qkv":
            return 2.0 * T * C_ * 3 * C_, e * (T * C_ + 3 * C_ * C_ + 3 * T * C_)
        if label == "window_attention":   # QK^T and PV inside each window; qkv read once, out written once
            return 4.0 * T * (c.w * c.w) * C_, e * (3 * T * C_ + T * C_)
        if label == "gemm_proj":
            return 2.0 * T * C_ * C_, e * (T * C_ + C_ * C_ + 2 * T * C_)
        if label == "gemm_fc1":
            return 2.0 * T * C_ * F, e * (T * C_ + F * C_ + T * F)
        if label == "gemm_fc2":
            return 2.0 * T * F * C_, e * (T * F + F * C_ + 2 * T * C_)
        if label == "swin_mlp":   # FC1 + GELU + FC2 + residual, hidden layer on chip: h, y in, out
            return 4.0 * T * C_ * F, e * (3 * T * C_ + 2 * F * C_)
        return 0.0, 0.0

    def method_steps(self):
        """S1-S7 of the block, each with its own operands (FC1's output written and read
        once between the two MLP GEMMs, as the method states the step)."""
        return [self.work(k) for k in ("layernorm1", "gemm_qkv", "window_attention", "gemm_proj", "layernorm2",
                                       "gemm_fc1", "gemm_fc2")]

    def oracle_rate(self, budget_s):
        import oracle
        c, wl = self.cfg, self.wl
        imgs = 0
        t0 = time.perf_counter()
        for b in range(c.B):
            oracle.swin_block(wl["x"][b:b + 1], wl["weights"], c.I, c.w, c.s, c.nh, c.eps)
            imgs += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        return imgs * c.I * c.I / dt, f"{imgs} images ({imgs * c.I * c.I} tokens) of the seeded batch, fp64 numpy", dt


class MergeWorkload:
    """Swin stage downsampling (patch merge: 2x2 gather + LayerNorm over 4C, then the
    4C -> 2C GEMM) on the stage-1 output shape."""

    NAME = "swin_t_patch_merge_fp16"

    def __init__(self, cfg, rank):
        from workloads import make_patch_merge_workload
        self.cfg = cfg
        self.wl = make_patch_merge_workload(cfg, seed=cfg.seed + 300 + 7919 * rank)
        self.T = cfg.T                        # input tokens
        self.R = cfg.B * (cfg.I // 2) ** 2    # output tokens
        self.tokens_per_step = self.T
        self.dtype = {"fp16": "f16", "bf16": "bf16"}[cfg.dtype]

    def config(self):
        c = self.cfg
        return {"workload": f"{self.NAME}: B={c.B} images {c.I}x{c.I} C={c.C} -> {c.I // 2}x{c.I // 2} C={2 * c.C} "
                            f"(2x2 gather + LayerNorm(4C) + bias-free 4C->2C map); value counts input tokens",
                "global_batch": c.B, "seq_len": c.I * c.I, "valid_tokens": self.T}

    def setup(self, rpp, torch, dev):
        c, wl = self.cfg, self.wl
        self.tdt = rpp.torch_dtype(c.dtype)
        self.pm = rpp.PatchMerge(rpp.merge_cfg(c.I, c.C, c.eps, c.dtype), wl["gamma"], wl["beta"], wl["W"], dev)
        self.x = torch.as_tensor(wl["x"].reshape(-1, c.C)).to(dev, self.tdt)
        self.y = torch.empty(self.R, 2 * c.C, dtype=self.tdt, device=dev)
        self.ws = self.pm.workspace(c.B, dev)
        self.err = rpp.new_error_word(dev)
        self.rpp = rpp

    def step(self, x=None, y=None):
        self.rpp.patch_merge_forward(self.pm, self.x if x is None else x, self.cfg.B,
                                     y=self.y if y is None else y, workspace=self.ws, err=self.err)

    def host_io(self, torch):
        xh = torch.empty(self.x.shape, dtype=self.tdt, pin_memory=True)
        xh.copy_(self.x.cpu())
        yh = torch.empty(self.y.shape, dtype=self.tdt, pin_memory=True)
        xd, yd = torch.empty_like(self.x), torch.empty_like(self.y)
        return [(xh, xd)], (yd, yh), lambda: self.step(xd, yd)

    def work(self, label):
        C_, R, e = self.cfg.C, self.R, 2
        if label == "patch_merge_ln":      # every input token read once, the 4C rows written once
            return 0.0, e * (self.T * C_ + R * 4 * C_)
        if label == "gemm_reduction":
            return 2.0 * R * 4 * C_ * 2 * C_, e * (R * 4 * C_ + 8 * C_ * C_ + R * 2 * C_)
        return 0.0, 0.0

    def method_steps(self):
        return [self.work("patch_merge_ln"), self.work("gemm_reduction")]

    def oracle_rate(self, budget_s):
        import oracle
        c, wl = self.cfg, self.wl
        imgs = 0
        t0 = time.perf_counter()
        for b in range(c.B):
            oracle.patch_merge(wl["x"][b:b + 1], c.I, wl["gamma"], wl["beta"], wl["W"], c.eps)
            imgs += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        return imgs * c.I * c.I / dt, f"{imgs} images ({imgs * c.I * c.I} input tokens) of the seeded batch, fp64 numpy", dt


def make_workload(name, rank):
    from workloads import config_by_name
    if name == MergeWorkload.NAME:
        return MergeWorkload(config_by_name("swin_t_stage1_fp16"), rank)
    if name == BertWorkload.ALL_INT8:   # the int8 config with the attention on codes as well
        return BertWorkload(config_by_name("bert_large_int8"), rank, all_int8=True)
    cfg = config_by_name(name)
    return (SwinWorkload if cfg.kind == "swin" else BertWorkload)(cfg, rank)


# ---------------------------------------------------------------- clocks
def clocks_sampler_start(path):
    cmd = ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
           "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
           "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
           "--format=csv,noheader,nounits", "-lms", "200"]
    try:
        f = open(path, "w")
        return subprocess.Popen(cmd, stdout=f, stderr=subprocess.DEVNULL), f
    except (OSError, FileNotFoundError):
        return None, None


def clocks_sampler_stop(proc, f, path, gpu_index):
    if proc is None:
        return None
    proc.terminate()
    try:
        proc.wait(timeout=5)
    except subprocess.TimeoutExpired:
        proc.kill()
    f.close()
    sm, mx, reasons = [], 0.0, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    with open(path) as fh:
        for line in fh:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9 or parts[0] != str(gpu_index):
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- reference arm
def run_reference(args, wk, rank):
    if rank != 0:
        return
    for _ in range(max(0, args.warmup)):
        wk.oracle_rate(1.0)
    tot_tokens = tot_t = 0.0
    sample = ""
    for _ in range(args.steps):
        v, sample, dt = wk.oracle_rate(3.0)
        tot_tokens += v * dt
        tot_t += dt
    value = tot_tokens / tot_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wk.config(),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def main():
    args = parse()
    rank, world, local = dist_env()
    wk = make_workload(args.workload, rank)
    if args.oracle_rate > 0:   # child mode of the single-thread oracle leg (no GPU, no torch)
        v, sample, dt = wk.oracle_rate(args.oracle_rate)
        print(json.dumps({"value": v, "sample": sample, "dt": dt}), flush=True)
        return None
    if args.impl == "reference":
        return run_reference(args, wk, rank)

    import torch
    import remove_padding_prefix_gb300 as rpp
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    wk.setup(rpp, torch, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    for _ in range(max(args.warmup, 3)):
        wk.step()
    torch.cuda.synchronize()
    code = rpp.get_device_error(wk.err)
    if code:
        raise SystemExit(f"device error {code}")

    def timed(run_step):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            run_step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return reduce_max(sum(a.elapsed_time(b) for a, b in ev) / 1e3, world, dev)

    eager_s = timed(wk.step)
    y_eager = wk.y.clone()
    graph = None
    if not args.no_graph:   # one step captured into a CUDA graph (no allocation, no sync inside)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            wk.step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            wk.step()
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    import tempfile
    fd, clk_path = tempfile.mkstemp(prefix=f"rpp_clocks_rank{rank}_", suffix=".csv")
    os.close(fd)
    proc, fh = clocks_sampler_start(clk_path)
    time.sleep(0.3)
    total_s = timed(graph.replay if graph is not None else wk.step)
    clocks = clocks_sampler_stop(proc, fh, clk_path, local)
    try:
        os.unlink(clk_path)
    except OSError:
        pass
    code = rpp.get_device_error(wk.err)
    if code:
        raise SystemExit(f"device error {code}")
    if not torch.equal(wk.y, y_eager):
        raise SystemExit("graph replay output differs from the eager step")
    value = wk.tokens_per_step * args.steps * world / total_s
    value_eager = wk.tokens_per_step * args.steps * world / eager_s

    # ---- per-kernel durations inside the real step (launch-event hook).  With graphs
    # on, the hooked step is captured too (the event records become graph nodes) and
    # timed on replay, so host launch gaps stay out of the per-kernel times.
    lib = rpp.lib()
    cap = 4096
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(cap)]
    for e in evs:          # torch creates the CUDA event lazily, on first record
        e.record(stream)
    torch.cuda.synchronize()
    handles = (C.c_void_p * cap)(*[e.cuda_event for e in evs])
    if not all(handles):
        raise SystemExit("could not create CUDA events for the launch-event hook")
    reps = max(3, min(args.steps, 10))
    kernels, n_launch_step = {}, None
    hook_graph, start, start_inside = None, None, False
    if graph is not None:
        try:
            start = torch.cuda.Event(enable_timing=True, external=True)
            start_inside = True
        except TypeError:   # older torch: the start mark is recorded before each replay
            start = torch.cuda.Event(enable_timing=True)
        hook_graph = torch.cuda.CUDAGraph()
        lib.rpp_set_launch_events(handles, cap)
        try:
            with torch.cuda.graph(hook_graph):
                if start_inside:
                    start.record()
                wk.step()
        finally:
            n = lib.rpp_launch_event_count()
            labels = [lib.rpp_launch_event_label(i).decode() for i in range(n)]
            lib.rpp_set_launch_events(None, 0)
        torch.cuda.synchronize()
        hook_graph.replay()
        torch.cuda.synchronize()
    for r in range(reps):
        flush.fill_(float(r))
        if hook_graph is not None:
            if not start_inside:
                start.record(stream)
            hook_graph.replay()
        else:
            start = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            lib.rpp_set_launch_events(handles, cap)
            try:
                wk.step()
            finally:
                n = lib.rpp_launch_event_count()
                labels = [lib.rpp_launch_event_label(i).decode() for i in range(n)]
                lib.rpp_set_launch_events(None, 0)
        torch.cuda.synchronize()
        n_launch_step = n
        prev = start
        for i, lab in enumerate(labels):
            kernels.setdefault(lab, []).append(prev.elapsed_time(evs[i]))
            prev = evs[i]
    del hook_graph
    peaks, peak_kind = load_peaks()
    int8_peak = measure_int8_peak(torch, dev) if getattr(wk.cfg, "dtype", "") == "int8" else None
    per_launch = {}
    for lab, vals in kernels.items():
        cnt = len(vals) / reps
        ms = float(np.mean(vals))
        f_, b_ = wk.work(lab)
        t_tc = f_ / (peaks["bf16_tflops"] * 1e12) if f_ else 0.0
        t_hbm = b_ / (peaks["hbm_gbs"] * 1e9) if b_ else 0.0
        bound = "tensor" if (t_tc >= t_hbm and f_) else "hbm"
        if bound == "tensor":
            ach = f_ / (ms * 1e-3) / 1e12
            d = {"bound": "tensor", "achieved": ach, "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"]}
        else:
            ach = b_ / (ms * 1e-3) / 1e9
            d = {"bound": "hbm", "achieved": ach, "unit": "GB/s", "frac": ach / peaks["hbm_gbs"] if b_ else None}
        d.update({"launches_per_step": cnt, "ms_per_launch": ms, "ms_per_step": ms * cnt, "flops": f_, "bytes": b_})
        if lab.endswith("_i8") and f_ and int8_peak:   # the exact int8 GEMMs run on the bf16 pipe
            d["frac_of_int8_peak"] = f_ / (ms * 1e-3) / 1e12 / int8_peak
        per_launch[lab] = d
    dom = max(per_launch, key=lambda k: per_launch[k]["ms_per_step"])
    # The dominant kernel alone: events just before and after each of its launches
    # (the hook's label filter), so the rest of the step keeps its launch overlap and
    # only this kernel's boundaries carry event records.
    dom_ms = None
    if graph is not None:
        lib.rpp_set_launch_event_filter(dom.encode())
        lib.rpp_set_launch_events(handles, cap)
        g3 = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g3):
                wk.step()
        finally:
            n3 = lib.rpp_launch_event_count()
            lib.rpp_set_launch_events(None, 0)
            lib.rpp_set_launch_event_filter(None)
        torch.cuda.synchronize()
        g3.replay()
        torch.cuda.synchronize()
        vals = []
        for r in range(reps):
            flush.fill_(float(r))
            g3.replay()
            torch.cuda.synchronize()
            vals += [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(n3 // 2)]
        del g3
        if vals:
            dom_ms = float(np.mean(vals))
    dd = dict(per_launch[dom])
    if dom_ms is not None:
        f_, b_ = wk.work(dom)
        dd["ms_per_launch"] = dom_ms
        if dd["bound"] == "tensor":
            dd["achieved"] = f_ / (dom_ms * 1e-3) / 1e12
            dd["frac"] = dd["achieved"] / peaks["bf16_tflops"]
        else:
            dd["achieved"] = b_ / (dom_ms * 1e-3) / 1e9
            dd["frac"] = dd["achieved"] / peaks["hbm_gbs"] if b_ else None
    traffic = None
    ent = load_traffic().get(f"{wk.cfg.name}:{dom}")
    if ent and ent.get("src_sha") == src_hash(ent["srcs"]):
        traffic = ent["bytes_per_launch"]
    roof = {"kernel": dom, "bound": dd["bound"], "achieved": dd["achieved"],
            "peak": peaks["bf16_tflops"] if dd["bound"] == "tensor" else peaks["hbm_gbs"], "unit": dd["unit"],
            "frac": dd["frac"], "traffic": traffic,
            "peak_source": (f"{peak_kind} bf16 dense burst (fp16 runs at the same nominal rate)"
                            if dd["bound"] == "tensor" else f"{peak_kind} HBM copy bandwidth"),
            "work_per_launch": dd["flops"] if dd["bound"] == "tensor" else dd["bytes"],
            "ms_per_launch": dd["ms_per_launch"],
            "timing": ("CUDA events just before and after each launch of this kernel inside the captured step "
                       "(other launches unmarked), graph replays with L2 flushed between them"
                       if dom_ms is not None else "CUDA events after every launch of an eager step")}

    # ---- the whole step against the sum of its method steps' ideal times
    ideal_s = 0.0
    for f_, b_ in wk.method_steps():
        ideal_s += max(f_ / (peaks["bf16_tflops"] * 1e12), b_ / (peaks["hbm_gbs"] * 1e9))
    ideal_sus = 0.0
    for f_, b_ in wk.method_steps():
        ideal_sus += max(f_ / (peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * 1e12),
                         b_ / (peaks["hbm_gbs"] * 1e9))
    step_s = total_s / args.steps
    layer_roof = {"ideal_ms_per_step": ideal_s * 1e3, "ms_per_step": step_s * 1e3, "frac": ideal_s / step_s,
                  "frac_vs_sustained_bf16": ideal_sus / step_s,
                  "how": ("sum over the method steps of max(flops / bf16 dense peak, algorithmic bytes / HBM copy "
                          "bandwidth), measured peaks; divided by the graph-replayed step time")}

    # ---- end to end through host buffers (eager calls of the public API).  Every step
    # copies its input from pinned host memory and reads its output back; the copies run
    # on their own streams, so step i's compute overlaps the input copy of step i + 1 and
    # the output copy of step i - 1 (two sets of device buffers; a set is refilled only
    # once the output copy that last used it has finished).  One time over all K steps,
    # from the first input copy to the last output copy; no L2 flush (the weights and the
    # activations of a step are larger than L2).
    e2e = None
    if not args.no_e2e:
        sets = [wk.host_io(torch) for _ in range(2)]
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

        def pipeline(k):
            ready = [torch.cuda.Event() for _ in range(k)]
            computed = [torch.cuda.Event() for _ in range(k)]
            done = [torch.cuda.Event() for _ in range(k)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(h2d)
            for i in range(k):
                ins, (yd, yh), run = sets[i % 2]
                if i >= 2:
                    h2d.wait_event(done[i - 2])
                with torch.cuda.stream(h2d):
                    for hb, db in ins:
                        db.copy_(hb, non_blocking=True)
                ready[i].record(h2d)
                stream.wait_event(ready[i])
                run()
                computed[i].record(stream)
                d2h.wait_event(computed[i])
                with torch.cuda.stream(d2h):
                    yh.copy_(yd, non_blocking=True)
                done[i].record(d2h)
            d2h.wait_event(done[k - 1])
            t1.record(d2h)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / 1e3
        pipeline(3)

        def copy_gbs(to_device):   # this host link's rate on one step's buffers, outside the timed region
            ins, (yd, yh), _ = sets[0]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            nbytes = 0
            for hb, db in (ins if to_device else [(yh, yd)]):
                (db.copy_(hb, non_blocking=True) if to_device else hb.copy_(db, non_blocking=True))
                nbytes += hb.numel() * hb.element_size()
            e1.record(stream)
            torch.cuda.synchronize()
            return nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9
        link = {"h2d_gbs": round(copy_gbs(True), 1), "d2h_gbs": round(copy_gbs(False), 1)}
        if world > 1:
            torch.distributed.barrier()
        e2e_s = reduce_max(pipeline(args.steps), world, dev)
        ins0, (_, yh0), _ = sets[(args.steps - 1) % 2]
        e2e = {"value": wk.tokens_per_step * args.steps * world / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": int(sum(hb.numel() * hb.element_size() for hb, _ in ins0)),
               "d2h_bytes_per_step": int(yh0.numel() * yh0.element_size()),
               "copies": "on their own streams, overlapping the neighbouring steps' compute",
               "host_link": link}
        if not torch.equal(yh0.to(dev), wk.y):
            raise SystemExit("e2e output mismatch")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, sample, _ = wk.oracle_rate(12.0)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads_used(), "kind": "oracle", "sample": sample}
        one = oracle_single_thread(args, 12.0)
        if one is not None:
            cpu["single_thread"] = {"value": one["value"], "unit": "tokens/s", "cores": 1, "sample": one["sample"]}

    if world > 1:
        torch.distributed.barrier()
    if rank == 0:
        cfgd = wk.config()
        cfgd.update({"parallelism": "replicas (independent batches per GPU)",
                     "l2": "flushed between timed steps (512 MiB write)", "inputs": "seeded synthetic, resident in HBM",
                     "launch": "CUDA graph of one step" if graph is not None else "eager C-ABI calls"})
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": wk.dtype, "data": "synthetic", "config": cfgd,
                "roofline": roof, "layer_roofline": layer_roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": int(n_launch_step * args.steps) if n_launch_step else None, "clocks": clocks,
                "value_eager": value_eager, "ms_per_step_eager": 1e3 * eager_s / args.steps,
                "kernels": per_launch,
                "int8_peak_tops": int8_peak,
                "kernel_timing": ("CUDA events recorded as graph nodes after every launch, replayed after the timed "
                                  "region with the same L2 flush" if graph is not None else
                                  "CUDA events recorded after every launch of an eager step")}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
