"""Benchmark of the tensor-parallel MLP forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one forward (FC1 + GeLU, FC2 with the shard sum in its K-loop) and one full
backward (D, dB, dA, dX) of the tensor-parallel MLP block through the C ABI, on seeded
synthetic bf16 inputs of the workload's shape. Throughput is algorithmic FLOPs
(12 * n * d * m per step: six GEMMs of 2 * n * d * m) over device time.

One process per GPU; with N > 1 (torchrun) every rank runs an independent replica
(nothing in the path exchanges data), the timed region is bracketed by a barrier and a
device synchronise, and the slowest rank's time is used. Rank 0 prints one JSON line.

--impl reference times the float64 CPU oracle on the host cores instead (rank 0 only),
each step a bounded sample of token rows of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from tensor_transformer_mlp_gb300 import workloads as wl  # noqa: E402

METRIC = "TP-MLP fwd+bwd TFLOP/s (bf16) and fraction of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_LAUNCHES_PER_STEP = 6
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel, from the
# committed ncu summary named below; None until a capture of the current kernel exists.
DOMINANT_KERNEL_TRAFFIC = 7013003349  # average over the six GEMM launches of one step
DOMINANT_KERNEL_PROFILE = "profiles/gemm_bf16_wide_kernel_large_mlp_dram.md"


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def aggregate(elapsed_s: float, units: float, world: int, device=None):
    """Whole-job figures: (max elapsed over ranks, sum of units over ranks)."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist

    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.lines: list[str] = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.05)
        self.skip = len(self.lines)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [ln.split(", ") for ln in self.lines[self.skip:] if ln.count(",") >= 6]
        if not rows:
            rows = [ln.split(", ") for ln in self.lines if ln.count(",") >= 6]
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), r[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def gpu_id_for(device_index: int) -> str:
    import torch

    props = torch.cuda.get_device_properties(device_index)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        s = str(uuid)
        return s if s.startswith("GPU-") else "GPU-" + s
    return str(device_index)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- oracle (CPU)

def oracle_rows_flops(cfg, rows: int) -> int:
    return 12 * rows * cfg.d * cfg.m


def time_oracle(cfg, inp, rows: int, row0: int = 0) -> float:
    """Float64 oracle forward + backward on `rows` token rows (full weights); seconds."""
    from oracle import mlp as omlp

    sl = slice(row0, row0 + rows)
    t0 = time.perf_counter()
    omlp.forward(inp["X"][sl], inp["A"], inp["B"], cfg.gelu)
    omlp.backward(inp["X"][sl], inp["A"], inp["B"], inp["G"][sl], cfg.gelu)
    return time.perf_counter() - t0


def calibrate_rows(cfg, inp, target_s: float, max_rows: int) -> int:
    """Rows of oracle work that take about target_s. Doubles a probe until one run takes at
    least a quarter of the target, then scales linearly from it (the probe's fixed part, the
    oracle's float64 conversion of the full weights, makes this an underestimate)."""
    rows = 16
    while True:
        t = time_oracle(cfg, inp, rows)
        if t >= target_s / 4 or rows >= max_rows or rows >= cfg.n:
            break
        rows *= 2
    return max(16, min(int(rows * target_s / max(t, 1e-3)), max_rows, cfg.n))


def host_cpu() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo) and architecture, for the CPU-baseline record."""
    import platform
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        model = next((ln.split(":", 1)[1].strip() for ln in out.splitlines() if ln.startswith("Model name:")), "")
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                model = next((ln.split(":", 1)[1].strip() for ln in f if ln.startswith("model name")), "")
        except OSError:
            pass
    return f"{model or 'unknown'} ({platform.machine()})"


_ONE_THREAD_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                   "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")


def single_thread_oracle(timeout_s: float = 120.0):
    """The oracle's full forward + backward on the single MLP block (n512 d1024 m4096), timed in a
    child process whose BLAS runs on one thread (the thread count is fixed when numpy loads its
    BLAS, hence the child). Returns a small record, or None if the child fails."""
    env = dict(os.environ)
    env.update({k: "1" for k in _ONE_THREAD_ENV})
    code = ("import json, bench; from tensor_transformer_mlp_gb300 import workloads as wl; "
            "cfg = wl.SINGLE_BLOCK; inp = wl.mlp_inputs(cfg); bench.time_oracle(cfg, inp, 16); "
            "s = bench.time_oracle(cfg, inp, cfg.n); "
            "print(json.dumps({'workload': cfg.name, 'seconds': s, 'value': bench.oracle_rows_flops(cfg, cfg.n) / s / 1e12}))")
    try:
        out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=timeout_s,
                             cwd=os.path.dirname(os.path.abspath(__file__)))
        rec = json.loads(out.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None
    rec.update({"unit": UNIT, "threads": 1, "sample": "full forward + backward of every token row, float64"})
    return rec


def cpu_baseline(cfg, inp, target_s=15.0):
    rows = calibrate_rows(cfg, inp, target_s, 8192)
    secs = time_oracle(cfg, inp, rows)
    return {"value": oracle_rows_flops(cfg, rows) / secs / 1e12, "unit": UNIT, "cores": os.cpu_count(),
            "cpu": host_cpu(), "kind": "oracle", "single_thread": single_thread_oracle(),
            "sample": f"float64 numpy oracle, forward+backward of {rows} of {cfg.n} token rows with full "
                      f"A [{cfg.d}x{cfg.m}] and B [{cfg.m}x{cfg.d}] (12*rows*d*m FLOP), {secs:.1f} s, "
                      f"BLAS on all host threads"}


def run_reference(args, cfg):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = wl.mlp_inputs(cfg)
    # each step a bounded sample of token rows, so the whole run stays within a few minutes
    per_step = 90.0 / max(1, args.steps + args.warmup)
    rows = calibrate_rows(cfg, inp, per_step, 4096)
    for i in range(args.warmup):
        time_oracle(cfg, inp, rows, row0=(i * rows) % max(1, cfg.n - rows))
    total = 0.0
    for i in range(args.steps):
        total += time_oracle(cfg, inp, rows, row0=(i * rows) % max(1, cfg.n - rows))
    value = oracle_rows_flops(cfg, rows) * args.steps / total / 1e12
    sample = (f"float64 numpy oracle, each step forward+backward of {rows} of {cfg.n} token rows with full "
              f"weights (12*rows*d*m FLOP per step)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(cfg),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "cpu": host_cpu(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def l2_note(cfg) -> str:
    """Whether one step's operands exceed the 126 MiB L2 (no flush needed) or not."""
    mib = 2 * (2 * cfg.n * cfg.d + 2 * cfg.d * cfg.m) / 2**20
    if mib > 126:
        return f"inputs larger than L2 ({mib:.0f} MiB of X, A, B, G per step), no flush"
    return f"inputs ({mib:.0f} MiB) fit in L2; steps re-read them from L2"


def config_dict(cfg):
    return {"workload": cfg.name, "n": cfg.n, "d": cfg.d, "m": cfg.m, "t": cfg.t, "gelu": cfg.gelu,
            "inputs": f"seed {cfg.seed}, X~N(0,{cfg.x_std}), A,B~N(0,{cfg.w_std}), G~N(0,{cfg.g_std}) (std), "
                      f"rounded to {cfg.dtype}",
            "l2": l2_note(cfg),
            "parallelism": "replicas (t shards on one GPU per replica)"}


# ----------------------------------------------------------------------------- SP kernels

def measure_sp(dev, peaks, reps: int = 100, sets: int = 4):
    """Times the sequence-parallel block and each of its memory-bound kernels on the SP
    workload. Each kernel is launched `reps` times back to back, rotating over `sets` buffer
    sets so that the bytes touched between two uses of a set exceed the L2 cache."""
    import torch

    import tensor_transformer_mlp_gb300 as tp

    cfg = wl.SP_BLOCK
    b, s, h, m, t = cfg.b, cfg.s, cfg.h, cfg.m, cfg.t
    sl = s // t
    inp = wl.sp_inputs(cfg)
    bf = torch.bfloat16
    x0 = torch.from_numpy(wl.to_shards(inp["x"], t)).to(dev).to(bf)
    A = torch.from_numpy(inp["A"]).to(dev).to(bf)
    B = torch.from_numpy(inp["B"]).to(dev).to(bf)
    gamma = torch.from_numpy(inp["gamma"]).to(dev)
    beta = torch.from_numpy(inp["beta"]).to(dev)
    stream = torch.cuda.current_stream(dev)
    N = b * s * h
    elt = 2

    def timed(fn, launches):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(launches):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / launches / 1e3

    xs = [x0.clone() for _ in range(sets)]
    ys = [torch.empty_like(x0) for _ in range(sets)]
    full = [torch.empty((b, s, h), dtype=bf, device=dev) for _ in range(sets)]
    outs = [torch.empty_like(x0) for _ in range(sets)]
    masks = [torch.empty((N + 31) // 32, dtype=torch.int32, device=dev) for _ in range(sets)]
    res = {}
    hbm = float(peaks.get("hbm_gbs"))

    def entry(name, secs, nbytes, note):
        gbs = nbytes / secs / 1e9
        res[name] = {"us": secs * 1e6, "bytes": nbytes, "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "note": note}

    sec = timed(lambda i: tp.tpmlp_sp_layernorm(xs[i % sets], gamma, beta, cfg.eps, ys[i % sets], stream), reps)
    entry("layernorm", sec, 2 * N * elt, "read x + write LN(x), bf16")
    sec = timed(lambda i: tp.tpmlp_sp_gather(ys[i % sets], full[i % sets], stream), reps)
    entry("gather", sec, 2 * N * elt, "read shards + write token order, bf16")
    sec = timed(lambda i: tp.tpmlp_sp_dropout_residual(xs[i % sets], ys[i % sets], outs[i % sets], masks[i % sets],
                                                       cfg.p_drop, cfg.seed, stream), reps)
    entry("dropout_residual", sec, 3 * N * elt + N // 8, "read x, y + write out (bf16) + mask bits")
    sec = timed(lambda i: tp.tpmlp_rmsnorm(xs[i % sets], gamma, cfg.eps, ys[i % sets], stream), reps)
    entry("rmsnorm", sec, 2 * N * elt, "read x + write RMSNorm(x), bf16")
    dgs = [torch.empty(h, dtype=torch.float32, device=dev) for _ in range(sets)]
    wsr = [torch.empty(tp.tpmlp_rmsnorm_backward_workspace_size(b * s, h), dtype=torch.uint8, device=dev)
           for _ in range(sets)]
    sec = timed(lambda i: tp.tpmlp_rmsnorm_backward(xs[i % sets], gamma, cfg.eps, ys[i % sets],
                                                    outs[i % sets], dgs[i % sets], wsr[i % sets], stream), reps)
    entry("rmsnorm_backward", sec, 3 * N * elt, "read x, dy + write dx (bf16), with the fixed-order dgamma sum")
    wsl = [torch.empty(tp.tpmlp_sp_layernorm_backward_workspace_size(b * s, h), dtype=torch.uint8, device=dev)
           for _ in range(sets)]
    dbs = [torch.empty(h, dtype=torch.float32, device=dev) for _ in range(sets)]
    # the SP backward's last step: LayerNorm backward of the shards plus the residual gradient
    sec = timed(lambda i: tp.tpmlp_sp_layernorm_backward(xs[i % sets], gamma, cfg.eps, ys[i % sets], outs[(i + 1) % sets],
                                                         outs[i % sets], dgs[i % sets], dbs[i % sets], wsl[i % sets],
                                                         stream), reps)
    entry("layernorm_backward", sec, 4 * N * elt,
          "read x, dy, residual gradient + write dx (bf16), with the fixed-order dgamma / dbeta sums")
    # the SP backward's first step: dropout backward fused with the gather into token order, reading
    # the forward's mask bits (the masks written by the dropout + residual timing above) ...
    sec = timed(lambda i: tp.tpmlp_sp_dropout_grad_gather(xs[i % sets], full[i % sets], cfg.p_drop, cfg.seed, stream,
                                                          mask_bits=masks[i % sets]), reps)
    entry("dropout_grad_gather", sec, 2 * N * elt + N // 8,
          "read dout shards + mask bits + write token-order gradient (bf16)")
    # ... or recomputing the mask from the seed
    sec = timed(lambda i: tp.tpmlp_sp_dropout_grad_gather(xs[i % sets], full[i % sets], cfg.p_drop, cfg.seed, stream),
                reps)
    entry("dropout_grad_gather_recompute", sec, 2 * N * elt,
          "read dout shards + write token-order gradient (bf16); mask recomputed from the seed")
    del full, wsr, wsl
    parts = torch.randn((t, b * s, h), dtype=torch.float32, device=dev)  # 1 GiB > L2
    sec = timed(lambda i: tp.tpmlp_sp_reduce_scatter(parts, outs[i % sets], stream), max(10, reps // 4))
    entry("reduce_scatter_splitk", sec, t * N * 4 + N * elt, "read t fp32 partials + write shards (bf16)")
    del parts

    out = torch.empty_like(x0)
    mask = torch.empty((N + 31) // 32, dtype=torch.int32, device=dev)
    for rs in ("fused", "splitk"):
        ws = torch.empty(tp.tpmlp_sp_block_workspace_size(b, s, h, m, t, bf, rs), dtype=torch.uint8, device=dev)
        sec = timed(lambda i: tp.tpmlp_sp_block(x0, gamma, beta, cfg.eps, A, B, cfg.p_drop, cfg.seed, out, mask, t,
                                               cfg.gelu, rs, ws, stream), 10)
        res[f"sp_block_{rs}"] = {"ms": sec * 1e3, "mlp_tflops": cfg.flops_mlp_fwd / sec / 1e12,
                                 "note": "whole block; TFLOP/s counts the MLP's 4*n*h*m only"}
        del ws
    # backward of the block (activations saved by a forward with Z/Y outputs)
    Zs = torch.empty((b * s, m), dtype=bf, device=dev)
    Ys = torch.empty((b * s, m), dtype=bf, device=dev)
    ws = torch.empty(tp.tpmlp_sp_block_workspace_size(b, s, h, m, t, bf, "fused"), dtype=torch.uint8, device=dev)
    tp.tpmlp_sp_block(x0, gamma, beta, cfg.eps, A, B, cfg.p_drop, cfg.seed, out, mask, t, cfg.gelu, "fused", ws,
                      stream, Zs, Ys)
    del ws
    dout = torch.randn_like(x0)
    dx = torch.empty_like(x0)
    dgam = torch.empty(h, dtype=torch.float32, device=dev)
    dbet = torch.empty(h, dtype=torch.float32, device=dev)
    dA = torch.empty((h, m), dtype=torch.float32, device=dev)
    dB = torch.empty((m, h), dtype=torch.float32, device=dev)
    wsb = torch.empty(tp.tpmlp_sp_block_backward_workspace_size(b, s, h, m, t, bf), dtype=torch.uint8, device=dev)
    sec = timed(lambda i: tp.tpmlp_sp_block_backward(x0, gamma, beta, cfg.eps, A, B, cfg.p_drop, cfg.seed, Zs, Ys,
                                                     dout, dx, dgam, dbet, dA, dB, t, cfg.gelu, wsb, stream,
                                                     mask_bits=mask), 10)
    res["sp_block_backward"] = {"ms": sec * 1e3, "mlp_tflops": 2 * cfg.flops_mlp_fwd / sec / 1e12,
                                "note": "whole backward, dropout mask read from the forward's mask bits; TFLOP/s "
                                        "counts the four GEMMs' 8*n*h*m only"}
    tp.tpmlp_device_status(stream)
    return {"workload": cfg.name, "l2": f"{sets} rotating buffer sets per kernel (>= 3 x 128 MiB between reuses)",
            "kernels": res}


# ----------------------------------------------------------------------------- attention

def measure_attention(dev, peaks, reps: int = 10):
    """Times the tensor-parallel attention block (forward, backward) on the GPT-style shape;
    algorithmic FLOPs: forward 8*n*h^2 + 4*b*s^2*h, backward twice that."""
    import torch

    import tensor_transformer_mlp_gb300 as tp

    cfg = wl.GPT_ATTENTION
    inp = wl.attn_inputs(cfg)
    bf = torch.bfloat16
    X = torch.from_numpy(inp["X"]).to(dev).to(bf)
    Wqkv = torch.from_numpy(inp["Wqkv"]).to(dev).to(bf)
    Wo = torch.from_numpy(inp["Wo"]).to(dev).to(bf)
    G = torch.from_numpy(inp["G"]).to(dev).to(bf)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps / 1e3

    _, saves = tp.attention_forward(X, Wqkv, Wo, cfg.heads, cfg.t)
    fwd = timed(lambda: tp.attention_forward(X, Wqkv, Wo, cfg.heads, cfg.t))
    bwd = timed(lambda: tp.attention_backward(X, Wqkv, Wo, G, saves, cfg.heads, cfg.t))
    tp.tpmlp_device_status(stream)
    ff = cfg.flops_fwd
    return {"workload": cfg.name, "forward_ms": fwd * 1e3, "forward_tflops": ff / fwd / 1e12,
            "backward_ms": bwd * 1e3, "backward_tflops": 2 * ff / bwd / 1e12,
            "note": "P materialised and saved (Megatron's form); softmax in the epilogues of two passes of the "
                    "scores GEMM, dS in the dP GEMM's epilogue; includes allocation of outputs and workspace by "
                    "the convenience wrappers"}


# ----------------------------------------------------------------------------- GPU arm

def measure_library_gemms(X, A, B, G, Z, Y, stream, steps: int, warmup: int):
    """The step's six GEMMs by torch.matmul (cuBLAS), as a library reference point.

    Same shapes and operand layouts as the library's step (transposed operands are views,
    which cuBLAS reads in place); bf16 outputs and no GeLU / GeLU' epilogues, so it does
    strictly less work than the step. Z stands in for D (same shape and dtype). Timed
    back to back like the step, with CUDA events on the launching stream.
    """
    import torch

    n, d = X.shape
    m = A.shape[1]
    nm = torch.empty((n, m), dtype=X.dtype, device=X.device)
    nd = torch.empty((n, d), dtype=X.dtype, device=X.device)
    md = torch.empty((m, d), dtype=X.dtype, device=X.device)
    dm = torch.empty((d, m), dtype=X.dtype, device=X.device)

    def six():
        torch.matmul(X, A, out=nm)          # FC1
        torch.matmul(Y, B, out=nd)          # FC2
        torch.matmul(G, B.t(), out=nm)      # dgrad-1
        torch.matmul(Y.t(), G, out=md)      # wgrad dB
        torch.matmul(X.t(), Z, out=dm)      # wgrad dA
        torch.matmul(Z, A.t(), out=nd)      # dgrad-2

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            six()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            six()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del nm, nd, md, dm
    return ms


def run_ours(args, cfg):
    import torch

    import tensor_transformer_mlp_gb300 as tp

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    tp.load_library()
    variant = tuple(int(v) for v in args.gemm_variant.split(","))
    tp.tpmlp_set_gemm_variant(*variant)

    inp = wl.mlp_inputs(cfg)
    bf = torch.bfloat16
    X, A, B, G = (torch.from_numpy(inp[k]).to(dev).to(bf) for k in "XABG")
    n, d, m, t = cfg.n, cfg.d, cfg.m, cfg.t
    O = torch.empty((n, d), dtype=bf, device=dev)
    Z = torch.empty((n, m), dtype=bf, device=dev)
    Y = torch.empty((n, m), dtype=bf, device=dev)
    dX = torch.empty((n, d), dtype=bf, device=dev)
    dA = torch.empty((d, m), dtype=torch.float32, device=dev)
    dB = torch.empty((m, d), dtype=torch.float32, device=dev)
    ws = torch.empty(tp.tpmlp_backward_workspace_size(n, m, bf), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        tp.tpmlp_forward(X, A, B, O, Z, Y, t, cfg.gelu, stream)
        tp.tpmlp_backward(X, A, B, G, Z, Y, dX, dA, dB, t, cfg.gelu, ws, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    tp.tpmlp_device_status(stream)

    sampler = ClockSampler(gpu_id_for(local)) if rank == 0 else None
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        tp.tpmlp_forward(X, A, B, O, Z, Y, t, cfg.gelu, stream)
        ev[i][1].record(stream)
        tp.tpmlp_backward(X, A, B, G, Z, Y, dX, dA, dB, t, cfg.gelu, ws, stream)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    tp.tpmlp_device_status(stream)
    elapsed = t_start.elapsed_time(t_end) / 1e3
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in ev)
    flops_step = cfg.flops_fwd_bwd
    max_elapsed, total_flops = aggregate(elapsed, flops_step * args.steps, world, dev)

    # End to end through the public API with host buffers, two ways. "layer": what one MLP layer
    # of a training step moves, with its weights A, B and its fp32 gradient accumulators dA, dB
    # resident on the device (uploaded once, read by the optimizer there): each step uploads the
    # activations X and the upstream gradient G from pinned host memory and reads the output O
    # and the input gradient dX back. "all": every tensor crosses every step (X, A, B, G up;
    # O, dX, dA, dB down). In both, step k+1's uploads and step k-1's downloads overlap step k
    # (two device buffer sets, one stream each way, events ordering the reuse).
    def e2e_run(up_names, down_names, k_steps):
        dev_in = {"X": X, "A": A, "B": B, "G": G}
        dev_out = {"O": O, "dX": dX, "dA": dA, "dB": dB}
        host_in = {k: dev_in[k].cpu().pin_memory() for k in up_names}
        host_out = {k: torch.empty_like(dev_out[k], device="cpu").pin_memory() for k in down_names}
        ins = [dict(dev_in), {k: (torch.empty_like(v) if k in up_names else v) for k, v in dev_in.items()}]
        outs = [dict(dev_out), {k: (torch.empty_like(v) if k in down_names else v) for k, v in dev_out.items()}]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready, in_free = [ev(), ev()], [ev(), ev()]
        done, out_free = [ev(), ev()], [ev(), ev()]
        for e in in_free + out_free:
            e.record(stream)

        def steps(k_n):
            for k in range(k_n):
                j = k % 2
                xi, oi = ins[j], outs[j]
                with torch.cuda.stream(s_in):
                    s_in.wait_event(in_free[j])
                    for name in up_names:
                        xi[name].copy_(host_in[name], non_blocking=True)
                    in_ready[j].record(s_in)
                stream.wait_event(in_ready[j])
                stream.wait_event(out_free[j])
                tp.tpmlp_forward(xi["X"], xi["A"], xi["B"], oi["O"], Z, Y, t, cfg.gelu, stream)
                tp.tpmlp_backward(xi["X"], xi["A"], xi["B"], xi["G"], Z, Y, oi["dX"], oi["dA"], oi["dB"], t,
                                  cfg.gelu, ws, stream)
                done[j].record(stream)
                in_free[j].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done[j])
                    for name in down_names:
                        host_out[name].copy_(oi[name], non_blocking=True)
                    out_free[j].record(s_out)

        steps(2)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        stream.wait_event(e0)
        s_out.wait_event(e0)
        steps(k_steps)
        e1.record(s_out)  # the last step's results are on the host once s_out reaches here
        torch.cuda.synchronize()
        el, fl = aggregate(e0.elapsed_time(e1) / 1e3, flops_step * k_steps, world, dev)
        h2d = sum(host_in[k].numel() * host_in[k].element_size() for k in up_names)
        d2h = sum(host_out[k].numel() * host_out[k].element_size() for k in down_names)
        del ins, outs, host_in, host_out
        return fl / el / 1e12, h2d, d2h

    e2e_steps = max(4, args.steps)
    e2e_layer, h2d, d2h = e2e_run(("X", "G"), ("O", "dX"), e2e_steps)
    e2e_all, h2d_all, d2h_all = e2e_run(("X", "A", "B", "G"), ("O", "dX", "dA", "dB"), e2e_steps)

    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    value = total_flops / max_elapsed / 1e12
    # The dominant kernel is the tcgen05 GEMM: all six launches of a step are instances of it
    # and nothing else runs, so its average launch is (fwd + bwd time) / 6 with 2*n*d*m FLOP.
    gemm_ms_per_launch = (fwd_ms + bwd_ms) / (args.steps * GEMM_LAUNCHES_PER_STEP)
    achieved = 2 * n * d * m / (gemm_ms_per_launch / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_elapsed / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_dict(cfg), **({} if variant == (1, 1, 0) else {"gemm_variant": list(variant)})),
        "frac_of_peak": value / world / peak,
        "fwd_tflops": 4 * n * d * m * args.steps / (fwd_ms / 1e3) / 1e12,
        "bwd_tflops": 8 * n * d * m * args.steps / (bwd_ms / 1e3) / 1e12,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": DOMINANT_KERNEL_TRAFFIC if cfg is wl.LARGE_MLP else None,
                     "kernel": "gemm_bf16_wide_kernel (tcgen05 cta_group::2, 256x512 tiles on SM pairs; "
                               "6 launches per step, 2*n*d*m FLOP each)",
                     "peak_source": f"{peak_src} bf16_tflops_sustained (kernel timed inside a long step)",
                     "traffic_profile": DOMINANT_KERNEL_PROFILE if cfg is wl.LARGE_MLP else None},
        "e2e": {"value": e2e_layer, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "note": "one training layer's traffic: X, G up and O, dX down every step from/to pinned host "
                        "memory; weights A, B and fp32 gradient accumulators dA, dB resident on the device; "
                        "step k+1's uploads and step k-1's downloads overlap step k"},
        "e2e_all_tensors": {"value": e2e_all, "unit": UNIT, "h2d_bytes_per_step": h2d_all,
                            "d2h_bytes_per_step": d2h_all, "steps": e2e_steps,
                            "note": "every tensor crosses every step: X, A, B, G up; O, dX, dA, dB down"},
        "gpu_launches": GEMM_LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks,
    }
    if world == 1:
        lib_ms = measure_library_gemms(X, A, B, G, Z, Y, stream, args.steps, args.warmup)
        line["library_reference"] = {
            "what": "torch.matmul (cuBLAS) of the step's six GEMMs: same shapes and operand layouts, bf16 "
                    "outputs, no GeLU / GeLU' epilogues (less work than the step); run and timed after the "
                    "step, back to back, CUDA events",
            "ms_per_step": lib_ms, "tflops": flops_step / (lib_ms / 1e3) / 1e12,
            "ours_ms_per_step": max_elapsed / args.steps * 1e3}
    if not args.no_sp:
        line["sp"] = measure_sp(dev, peaks)
        line["attention"] = measure_attention(dev, peaks)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp)
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.LARGE_MLP.name,
                    choices=sorted(k for k, c in wl.MLP_CONFIGS.items() if c.dtype == "bf16"))
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the timed oracle sample")
    ap.add_argument("--no-sp", action="store_true", help="skip the sequence-parallel kernel measurements")
    ap.add_argument("--gemm-variant", default="1,1,0",
                    help="GEMM kernel choice, pacing and tile band passed to tpmlp_set_gemm_variant "
                         "(default 1,1,0: the library's own per-GEMM choice)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    cfg = wl.MLP_CONFIGS[args.workload]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
