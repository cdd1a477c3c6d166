"""Benchmark: valid tokens/s per encoder layer on one GB300, with roofline fractions.

One step = the whole hot path on one batch of synthetic input: offset builder ->
padding removal -> encoder layer(s) -> padding rebuild (one C-ABI call,
rpp_encoder_forward).  The default workload is the BERT-base-shaped fp16 layer
(B=32, L=128, lengths U[16,128], H=768, 12 heads, FFN 3072); --workload picks another
configuration of the same family for extra measurements.

Timing: W warm-up steps, then K steps, each bracketed by its own CUDA events on the
launch stream; between timed steps a 512 MiB buffer is written to flush the 129 MB
L2 (the flush is outside the events).  The K-step loop is bracketed by a barrier and
torch.cuda.synchronize() on both sides and the per-rank time is max-reduced.
value = (valid tokens per step x layers-equivalent 1) x ranks / time.

Extra keys: roofline (dominant kernel, timed live with the library's launch-event
hook), cpu_baseline (the CPU oracle on a bounded sample, host cores), e2e (the same
metric through host buffers: pinned H2D of the padded input and lengths, D2H of the
padded output inside the timed region), gpu_launches, clocks (nvidia-smi sampled
during the timed region).  --impl reference times the CPU oracle as the reference arm.
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

# ncu DRAM traffic per launch of the dominant kernels, with the sha256 of the source
# file the counters were taken on (reported only while that file is unchanged)
TRAFFIC = {}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="bert_base_fp16")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def src_hash(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_traffic():
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            return json.load(f)
    return {}


# ---------------------------------------------------------------- algorithmic work per kernel
def kernel_work(label, cfg, T, sum_len2):
    """(flops, bytes) per launch of an encoder-layer kernel: the algorithmic work of the
    packed batch (T valid tokens); the padded work that removal avoids is not counted."""
    H, F, B, L = cfg.H, cfg.F, cfg.B, cfg.L
    e = 4 if cfg.storage_dtype == "fp32" else 2
    res1 = 4 if cfg.storage_dtype == "bf16" else e     # FC2 residual: fp32 copy of LN1 out for bf16
    if label.startswith("gemm_qkv"):
        return 2.0 * T * H * 3 * H, e * (T * H + 3 * H * H + 3 * T * H)
    if label.startswith("gemm_proj"):   # reads attn, Wo, residual x; writes the fp32 pre-LN sum
        return 2.0 * T * H * H, e * (T * H + H * H + T * H) + 4 * T * H
    if label.startswith("gemm_fc1"):
        return 2.0 * T * H * F, e * (T * H + F * H + T * F)
    if label.startswith("gemm_fc2"):    # reads GELU out, W2, residual x1; writes the fp32 pre-LN sum
        return 2.0 * T * F * H, e * (T * F + F * H) + res1 * T * H + 4 * T * H
    if label == "attention":            # QK^T and PV over valid keys; Q, K, V read once, O written once
        return 4.0 * H * sum_len2, e * 4 * T * H
    if label == "layernorm1":           # fp32 sum in, activation out (+ fp32 copy for bf16)
        return 0.0, 4 * T * H + e * T * H + (4 * T * H if cfg.storage_dtype == "bf16" else 0)
    if label == "layernorm2":
        return 0.0, 4 * T * H + e * T * H
    if label == "remove_padding":
        return 0.0, 2 * e * T * H + 4 * T
    if label == "rebuild_padding":      # reads valid rows, writes the whole padded batch
        return 0.0, e * T * H + e * B * L * H + 4 * (B + 1)
    if label == "build_offsets":
        return 0.0, 4 * (B + (B + 1) + T)
    return 0.0, 0.0


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


# ---------------------------------------------------------------- CPU oracle (reference arm / baseline)
def oracle_tokens_per_s(cfg, wl, budget_s=12.0, max_passes=20):
    """Time the oracle, as it stands, on a bounded sample of the workload: whole
    sequences of the batch in order, repeated until ~budget_s of CPU work."""
    import oracle
    layers = wl["layers"]
    lens = wl["lengths"]
    tokens = 0
    seqs = 0
    t0 = time.perf_counter()
    passes = 0
    while passes < max_passes:
        for b in range(cfg.B):
            n = int(lens[b])
            if n == 0:
                continue
            x = wl["x_padded"][b:b + 1]
            oracle.bert_forward(x[:, :max(n, 1)], lens[b:b + 1], layers, cfg.nh, cfg.eps)
            tokens += n * len(layers)
            seqs += 1
            if time.perf_counter() - t0 > budget_s:
                break
        passes += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [os.cpu_count()])
    except Exception:
        cores = os.cpu_count()
    sample = f"{seqs} sequences ({tokens // len(layers)} tokens) x {len(layers)} layer(s) of the seeded batch, fp64 numpy"
    return tokens / dt, cores, sample, dt


def run_reference(args, cfg, wl, rank):
    if rank != 0:
        return
    vals = []
    for _ in range(max(0, args.warmup)):
        oracle_tokens_per_s(cfg, wl, budget_s=2.0, max_passes=1)
    tot_tokens, tot_t = 0.0, 0.0
    cores = os.cpu_count()
    sample = ""
    for _ in range(args.steps):
        v, cores, sample, dt = oracle_tokens_per_s(cfg, wl, budget_s=5.0, max_passes=1)
        vals.append(v)
        tot_tokens += v * dt
        tot_t += dt
    value = tot_tokens / tot_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(cfg):
    return {"workload": f"{cfg.name}: B={cfg.B} L={cfg.L} H={cfg.H} heads={cfg.nh}x{cfg.d} FFN={cfg.F} "
                        f"layers={cfg.layers} dtype={cfg.dtype}, lengths "
                        + (f"50% U{list(cfg.bimodal[0])} + 50% U{list(cfg.bimodal[1])}" if cfg.bimodal else
                           f"U[{cfg.len_lo},{cfg.len_hi or cfg.L}]")
                        + ", padding removed via offset mask",
            "global_batch": cfg.B, "seq_len": cfg.L, "parallelism": "replicas (independent batches per GPU)",
            "l2": "flushed between timed steps (512 MiB write)", "inputs": "seeded synthetic, resident in HBM"}


# ---------------------------------------------------------------- our arm
def main():
    args = parse()
    from workloads import config_by_name, make_bert_workload
    rank, world, local = dist_env()
    cfg = config_by_name(args.workload)
    if cfg.kind != "bert":
        raise SystemExit("bench.py times the BERT-shaped path; Swin is measured by its own workload flag")
    wl = make_bert_workload(cfg, seed=cfg.seed + 7919 * rank)   # each replica its own batch
    if args.impl == "reference":
        return run_reference(args, cfg, wl, rank)

    import torch
    import remove_padding_prefix_gb300 as rpp
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    tdt = rpp.torch_dtype(cfg.storage_dtype)
    int8 = cfg.dtype == "int8"
    T_host = int(wl["lengths"].sum())   # the caller knows its lengths: tile-shape hint
    ecfg = rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, cfg.storage_dtype, int8=int8, tokens_hint=T_host)
    layers = [rpp.EncoderLayer(ecfg, l, dev) for l in wl["layers"]]
    scales = None
    B, L, H = cfg.B, cfg.L, cfg.H
    lengths = torch.as_tensor(wl["lengths"], device=dev)
    x = torch.as_tensor(wl["x_padded"].reshape(B * L, H)).to(dev, tdt)
    y = torch.empty_like(x)
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    po = torch.zeros(B * L, dtype=torch.int32, device=dev)
    packed = torch.empty_like(x)
    ws = layers[0].workspace(B * L, dev)
    err = rpp.new_error_word(dev)
    if int8:   # per-tensor activation scales from the library's calibration pass (float layer)
        from workloads import make_calibration_batch
        cal = make_calibration_batch(cfg)
        fl = rpp.EncoderLayer(rpp.encoder_cfg(cfg.H, cfg.nh, cfg.F, cfg.eps, "fp16"), wl["layers"][0], dev)
        cl = torch.as_tensor(cal["lengths"], device=dev)
        ccu, cpo = rpp.build_offsets(cl, L)
        cx = rpp.remove_padding(torch.as_tensor(cal["x_padded"].reshape(B * L, H)).to(dev, tdt), cpo, ccu, B, L)
        scales = [rpp.encoder_layer_calibrate(fl, cx, ccu, B, L, workspace=ws) / 127.0 for _ in layers]
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step():
        rpp.encoder_forward(layers, lengths, x, L, act_scales=scales, y_padded=y, cu_seqlens=cu,
                            padding_offset=po, packed=packed, workspace=ws, err=err)

    T = int(wl["lengths"].sum())
    sum_len2 = float((wl["lengths"].astype(np.float64) ** 2).sum())
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if rpp.get_device_error(err):
        raise SystemExit(f"device error {rpp.get_device_error(err)}")

    # ---- timed region: K steps, each bracketed by its own events; L2 flushed between
    def timed(run_step, label):
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
        tot = sum(a.elapsed_time(b) for a, b in ev) / 1e3
        if world > 1:
            t = torch.tensor([tot], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            tot = float(t.item())
        return tot

    eager_s = timed(step, "eager")
    y_eager = y.clone()
    # one step captured into a CUDA graph (the calls allocate nothing and never sync)
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    clk_path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{rank}.csv") if os.path.isdir(
        os.path.join(ROOT, "gpurun_out")) else f"/tmp/rpp_clocks_{rank}.csv"
    proc, fh = clocks_sampler_start(clk_path)
    time.sleep(0.3)
    total_s = timed(graph.replay if graph is not None else step, "graph")
    clocks = clocks_sampler_stop(proc, fh, clk_path, local)
    code = rpp.get_device_error(err)
    if code:
        raise SystemExit(f"device error {code}")
    if not torch.equal(y, y_eager):
        raise SystemExit("graph replay output differs from the eager step")
    tokens_per_step = T * len(layers)   # valid tokens x layers: tokens/s per encoder layer
    value = tokens_per_step * args.steps * world / total_s
    value_eager = tokens_per_step * args.steps * world / eager_s

    # ---- per-kernel durations inside the real step (launch-event hook)
    lib = rpp.lib()
    n_launch_step = None
    kernels = {}
    reps = max(3, min(args.steps, 10))
    cap = 4096
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(cap)]
    for e in evs:          # torch creates the CUDA event lazily, on first record
        e.record(stream)
    torch.cuda.synchronize()
    handles = (C.c_void_p * cap)(*[e.cuda_event for e in evs])
    if not all(handles):
        raise SystemExit("could not create CUDA events for the launch-event hook")
    for r in range(reps):
        flush.fill_(float(r))
        start = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        lib.rpp_set_launch_events(handles, cap)
        try:
            step()
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
    # average duration per launch of each kernel label (a label may repeat per layer)
    per_launch = {}
    for lab, vals in kernels.items():
        cnt = len(vals) / reps
        per_launch[lab] = {"launches_per_step": cnt, "ms_per_launch": float(np.mean(vals)),
                           "ms_per_step": float(np.mean(vals) * cnt)}
    dom = max(per_launch, key=lambda k: per_launch[k]["ms_per_step"])
    peaks, peak_kind = load_peaks()
    flops, nbytes = kernel_work(dom, cfg, T, sum_len2)
    ms = per_launch[dom]["ms_per_launch"]
    traffic_db = load_traffic()
    traffic = None
    ent = traffic_db.get(f"{cfg.name}:{dom}")
    if ent and ent.get("src_sha") == src_hash(ent["src"]):
        traffic = ent["bytes_per_launch"]
    if flops > 0 and dom.startswith("gemm"):
        achieved = flops / (ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": f"{peak_kind} bf16 burst (fp16 = bf16 rate)",
                "work_per_launch": flops, "ms_per_launch": ms}
    else:
        achieved = nbytes / (ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "peak_source": f"{peak_kind} HBM copy",
                "work_per_launch": nbytes, "ms_per_launch": ms}
    for lab, d in per_launch.items():
        f_, b_ = kernel_work(lab, cfg, T, sum_len2)
        d["tflops"] = f_ / (d["ms_per_launch"] * 1e-3) / 1e12 if f_ else None
        d["gbs"] = b_ / (d["ms_per_launch"] * 1e-3) / 1e9 if b_ else None
        d["frac"] = (d["tflops"] / peaks["bf16_tflops"]) if (lab.startswith("gemm") and f_) else \
            ((d["gbs"] / peaks["hbm_gbs"]) if b_ else None)

    # ---- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        xh = torch.empty(x.shape, dtype=tdt, pin_memory=True)
        xh.copy_(x.cpu())
        lh = torch.empty(B, dtype=torch.int32, pin_memory=True)
        lh.copy_(lengths.cpu())
        yh = torch.empty(y.shape, dtype=tdt, pin_memory=True)
        xd = torch.empty_like(x)
        ld = torch.empty_like(lengths)

        def e2e_step():
            xd.copy_(xh, non_blocking=True)
            ld.copy_(lh, non_blocking=True)
            rpp.encoder_forward(layers, ld, xd, L, act_scales=scales, y_padded=y, cu_seqlens=cu,
                                padding_offset=po, packed=packed, workspace=ws, err=err)
            yh.copy_(y, non_blocking=True)
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(float(i))
            ee[i][0].record(stream)
            e2e_step()
            ee[i][1].record(stream)
        torch.cuda.synchronize()
        e2e_s = sum(a.elapsed_time(b) for a, b in ee) / 1e3
        if world > 1:
            t = torch.tensor([e2e_s], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            e2e_s = float(t.item())
        e2e = {"value": tokens_per_step * args.steps * world / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": int(xh.numel() * xh.element_size() + lh.numel() * 4),
               "d2h_bytes_per_step": int(yh.numel() * yh.element_size())}
        if not torch.equal(yh.to(dev), y):
            raise SystemExit("e2e output mismatch")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample, _ = oracle_tokens_per_s(cfg, wl, budget_s=12.0)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}

    if world > 1:
        torch.distributed.barrier()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": {"fp32": "f32", "fp16": "f16", "bf16": "bf16", "int8": "i8 GEMMs (exact), f16"}[cfg.dtype],
                "data": "synthetic", "config": workload_config(cfg), "roofline": roof, "cpu_baseline": cpu,
                "e2e": e2e, "gpu_launches": int(n_launch_step * args.steps) if n_launch_step else None,
                "clocks": clocks, "tokens_per_step": T, "layers": len(layers),
                "launch": "CUDA graph of one step" if graph is not None else "eager C-ABI calls",
                "value_eager": value_eager, "ms_per_step_eager": 1e3 * eager_s / args.steps,
                "kernels": per_launch}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
