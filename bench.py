"""Throughput of the fused LoRA / QLoRA projection, forward + backward.

Default workload: Llama-3-8B-shaped q_proj + k_proj with the RoPE epilogue,
M = 8192 tokens (1 x 8192), hidden 4096, q 32x128, k 8x128, r = 64,
alpha = 16, theta = 5e5, positions 0..8191, bf16 W.  One step = one
``lora_qk_rope_fwd`` + one ``lora_qk_rope_bwd`` over the batch; every other
workload of ``lora_inputs.WORKLOADS`` runs ``lora_linear_fwd`` +
``lora_linear_bwd`` per projection.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead (a bounded token sample per step) and prints the same line
with ``"impl": "reference"``.  Under torchrun every rank runs its own
replica on its own GPU (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lora_inputs import WORKLOADS, draw_workload  # noqa: E402

METRIC = "fused LoRA fwd+bwd tokens/s & TFLOP/s at 1 B300; % of bf16 tensor peak / HBM BW"
DEFAULT_WORKLOAD = "llama8b_qk_rope"
FLUSH_BYTES = 512 << 20          # > 126 MB L2, written between timed steps


# --------------------------------------------------------------------- flops
def step_flops(wl, M) -> float:
    """Algorithmic FLOPs of fwd+bwd for all projections (W frozen, no dW):
    4Mkn (x·Wᵀ, dY·W) + 2Mr(k+n) (x·Aᵀ, (s·v)·Bᵀ) + 2Mr(2n+3k) (dY·B, u·A,
    dA, recomputed x·Aᵀ, dB)."""
    r = wl.r
    f = 0.0
    for p in wl.projections:
        k, n = p.k, p.n
        f += 4.0 * M * k * n + 2.0 * M * r * (k + n) + 2.0 * M * r * (2 * n + 3 * k)
    return f


def fwd_kernel_flops(wl, M) -> float:
    """FLOPs of one fused forward launch (all projections of the launch)."""
    r = wl.r
    return sum(2.0 * M * p.k * p.n + 2.0 * M * r * p.k + 2.0 * M * r * p.n
               for p in wl.projections)


# ------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (timing of the slowest replica)."""
    if world == 1:
        return float(value)
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in loaded:
            for name, flag in zip(names, r[3]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


# ------------------------------------------------------------------ peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(os.listdir(os.path.join(ROOT, "lora_qlora_linear_fwd_b300", "csrc"))):
        h.update(open(os.path.join(ROOT, "lora_qlora_linear_fwd_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the fused forward kernel from the committed ncu
    summary, if it was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    return d.get("dram_bytes_per_launch") if d.get("source_hash") == kernel_source_hash() else None


# ------------------------------------------------------------- GPU replica
class Replica:
    """Device-resident inputs and outputs of one workload plus the calls of
    one step through the C ABI."""

    def __init__(self, name: str, device: str, seed: int = 0):
        import lora_qlora_linear_fwd_b300 as L
        self.L = L
        self.wl = wl = WORKLOADS[name]
        self.dev = device
        self.M = M = wl.M
        data = draw_workload(name, seed=seed)
        bf = dict(dtype=torch.bfloat16, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.keep = []
        self.projs = []
        for p in wl.projections:
            d = {k: v.to(device) for k, v in data[p.name].items()}
            if wl.nf4:   # quantise the drawn W on the GPU (setup, not timed)
                codes = torch.empty(p.n, p.k // 2, dtype=torch.uint8, device=device)
                absmax = torch.empty(p.n, p.k // 64, **bf)
                L.nf4_quantize(d["W"], codes, absmax)
                d["Wdesc"] = L.nf4_weight(codes, absmax)
                d["codes"], d["absmax"] = codes, absmax
                del d["W"]
            else:
                d["Wdesc"] = L.bf16_weight(d["W"])
            d["y"] = torch.empty(M, p.n, **bf)
            d["dx"] = torch.empty(M, p.k, **bf)
            d["dA"] = torch.empty(wl.r, p.k, **f32)
            d["dB"] = torch.empty(p.n, wl.r, **f32)
            self.projs.append((p, d))
        del data
        if wl.rope:
            (pq, dq), (pk, dk) = self.projs
            self.max_pos = M
            self.pos = torch.arange(M, dtype=torch.int32, device=device)
            self.cache = torch.empty(M, wl.head_dim, **f32)
            L.lora_rope_cache_build(self.cache, M, wl.head_dim, wl.rope_theta)
            n_tot = pq.n + pk.n
            self.ws_f = L.workspace(L.OP_QK_ROPE_FWD, M, pq.k, n_tot, wl.r, device=device)
            self.ws_b = L.workspace(L.OP_QK_ROPE_BWD, M, pq.k, n_tot, wl.r, device=device)
            self.dx = torch.empty(M, pq.k, **bf)
        else:
            self.ws = {}
            for p, d in self.projs:
                self.ws[p.name] = (L.workspace(L.OP_FWD, M, p.k, p.n, wl.r, device=device),
                                   L.workspace(L.OP_BWD, M, p.k, p.n, wl.r, device=device))
        torch.cuda.synchronize()

    def inputs(self):
        """Per-step inputs (activations and incoming gradients)."""
        if self.wl.rope:
            (_, dq), (_, dk) = self.projs
            return [dq["x"], dq["dY"], dk["dY"]]
        out = []
        for _, d in self.projs:
            out += [d["x"], d["dY"]]
        return out

    def outputs(self):
        if self.wl.rope:
            (_, dq), (_, dk) = self.projs
            return [dq["y"], dk["y"], self.dx, dq["dA"], dq["dB"], dk["dA"], dk["dB"]]
        out = []
        for _, d in self.projs:
            out += [d["y"], d["dx"], d["dA"], d["dB"]]
        return out

    def fwd(self):
        L, wl = self.L, self.wl
        if wl.rope:
            (_, q), (_, k) = self.projs
            L.lora_qk_rope_fwd(q["x"], q["Wdesc"], q["A"], q["B"], k["Wdesc"], k["A"], k["B"],
                               q["y"], k["y"], wl.alpha, wl.rope_theta, self.pos, self.cache,
                               self.max_pos, self.ws_f)
        else:
            for p, d in self.projs:
                L.lora_linear_fwd(d["x"], d["Wdesc"], d["A"], d["B"], d["y"], wl.alpha,
                                  self.ws[p.name][0])

    def bwd(self):
        L, wl = self.L, self.wl
        if wl.rope:
            (_, q), (_, k) = self.projs
            L.lora_qk_rope_bwd(q["x"], q["Wdesc"], q["A"], q["B"], k["Wdesc"], k["A"], k["B"],
                               q["dY"], k["dY"], self.dx, q["dA"], q["dB"], k["dA"], k["dB"],
                               wl.alpha, wl.rope_theta, self.pos, self.cache, self.max_pos,
                               self.ws_b)
        else:
            for p, d in self.projs:
                L.lora_linear_bwd(d["x"], d["Wdesc"], d["A"], d["B"], d["dY"], d["dx"], d["dA"],
                                  d["dB"], wl.alpha, self.ws[p.name][1])

    def step(self):
        self.fwd()
        self.bwd()

    def check_status(self):
        wss = [self.ws_f, self.ws_b] if self.wl.rope else [w for pair in self.ws.values()
                                                           for w in pair]
        for w in wss:
            s = self.L.lora_read_device_status(w)
            if s:
                raise RuntimeError(f"device status {s:#x}")


def run_gpu(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    rep = Replica(args.workload, dev)
    wl, M = rep.wl, rep.M
    L = rep.L
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        flush.zero_()
        rep.step()
    torch.cuda.synchronize()
    rep.check_status()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    launches0 = L.lora_kernel_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                      # L2 flush: not inside the step's events
        a, b, c = ev[i]
        a.record(stream)
        rep.fwd()
        b.record(stream)
        rep.bwd()
        c.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    launches = L.lora_kernel_launch_count() - launches0
    clocks = sampler.stop()
    rep.check_status()
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    ms_local = statistics.mean(step_ms)
    ms = max_over_ranks(ms_local, world)
    fwd_ms_mean = statistics.mean(fwd_ms)

    # end to end through the C ABI with host buffers (pinned), copies timed
    e2e = run_e2e(rep, args, stream)
    e2e_ms = max_over_ranks(e2e["ms"], world)

    flops = step_flops(wl, M)
    peaks = measured_peaks()
    tokens_per_s = world * M / (ms / 1e3)
    # dominant kernel: the fused forward GEMM (one launch per fwd call)
    fk = fwd_kernel_flops(wl, M) / len(wl.projections) if not wl.rope else fwd_kernel_flops(wl, M)
    fwd_launch_ms = fwd_ms_mean / (1 if wl.rope else len(wl.projections))
    achieved = fk / (fwd_launch_ms / 1e3) / 1e12
    fwd_name = ("lora_qk_rope_fwd" if wl.rope else "lora_linear_fwd") + \
        " (rank pass + fused GEMM, 2 launches)"
    roofline = {"kernel": fwd_name, "bound": "tensor",
                "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "peak_source": peaks["source"] + " (burst)",
                "traffic": profiled_traffic(args.workload),
                "launch_ms": round(fwd_launch_ms, 4)}
    line = {
        "metric": METRIC,
        "value": round(tokens_per_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded, Llama/Qwen-shaped; no weights or datasets)",
        "tflops": round(world * flops / (ms / 1e3) / 1e12, 1),
        "tflops_frac_of_peak": round(flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
        "fwd_ms": round(fwd_ms_mean, 4),
        "bwd_ms": round(ms_local - fwd_ms_mean, 4),
        "region_wall_s": round(wall, 4),
        "config": {"workload": args.workload, "description": wl.description, "M": M,
                   "r": wl.r, "alpha": wl.alpha, "nf4": wl.nf4,
                   "projections": [[p.name, p.k, p.n] for p in wl.projections],
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (512 MiB write, outside step events)"},
        "roofline": roofline,
        "e2e": {"value": round(world * M / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": int(launches),
        "gpu_launches_per_step": launches / args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_tokens)
    return line


def run_e2e(rep, args, stream):
    """Same step through the C ABI with the step's inputs on the host: every
    step copies its inputs from pinned host memory and reads back all its
    results (y, dX, dA, dB); copies are inside the timed region."""
    ins = rep.inputs()
    outs = rep.outputs()
    h_in = [t.cpu().pin_memory() for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    steps = max(3, min(args.steps, 10))

    def one():
        for d, h in zip(ins, h_in):
            d.copy_(h, non_blocking=True)
        rep.step()
        for h, d in zip(h_out, outs):
            h.copy_(d, non_blocking=True)

    one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    return {"ms": a.elapsed_time(b) / steps, "h2d": h2d, "d2h": d2h}


# ----------------------------------------------------------- CPU (oracle)
def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(n[0]) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


def oracle_step(name: str, data, M: int):
    import oracle as ref
    wl = WORKLOADS[name]
    f = lambda t: t.float().numpy().astype(np.float64)
    if wl.rope:
        q, k = data["q_proj"], data["k_proj"]
        pos = np.arange(M)
        ref.qk_rope_fwd(f(q["x"]), f(q["W"]), f(q["A"]), f(q["B"]), f(k["W"]), f(k["A"]),
                        f(k["B"]), wl.alpha, pos, wl.rope_theta, wl.head_dim)
        ref.qk_rope_bwd(f(q["x"]), f(q["W"]), f(q["A"]), f(q["B"]), f(k["W"]), f(k["A"]),
                        f(k["B"]), f(q["dY"]), f(k["dY"]), wl.alpha, pos, wl.rope_theta,
                        wl.head_dim)
    else:
        for p in wl.projections:
            d = data[p.name]
            W = d["Wq"] if "Wq" in d else f(d["W"])
            ref.lora_fwd(f(d["x"]), W, f(d["A"]), f(d["B"]), wl.alpha)
            ref.lora_bwd(f(d["x"]), W, f(d["A"]), f(d["B"]), f(d["dY"]), wl.alpha)


def _oracle_sample(name: str, tokens: int):
    import oracle as ref
    wl = WORKLOADS[name]
    data = draw_workload(name, seed=0, M=tokens)
    if wl.nf4:
        for p in wl.projections:
            d = data[p.name]
            codes, absmax = ref.nf4_quantize(d["W"].float().numpy())
            d["Wq"] = ref.nf4_dequant(codes, absmax)
    return data


def cpu_baseline(name: str, tokens: int):
    """The fp64 oracle as it stands, on the host cores, over a bounded token
    sample of the same workload; tokens/s = sample tokens / time."""
    data = _oracle_sample(name, tokens)
    t0 = time.perf_counter()
    oracle_step(name, data, tokens)
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 2), "unit": "tokens/s", "cores": _blas_threads(),
            "kind": "oracle", "sample": f"{tokens} of {WORKLOADS[name].M} tokens, all "
            f"projections, fwd+bwd in fp64 numpy ({dt:.1f} s)"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    wl = WORKLOADS[args.workload]
    tokens = args.cpu_tokens
    data = _oracle_sample(args.workload, tokens)
    for _ in range(args.warmup):
        oracle_step(args.workload, data, tokens)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(args.workload, data, tokens)
        times.append(time.perf_counter() - t0)
    per_token = statistics.mean(times) / tokens
    ms_full = per_token * wl.M * 1e3
    value = 1.0 / per_token
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_full, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "description": wl.description, "M": wl.M,
                   "sample_tokens_per_step": tokens},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "kind": "oracle",
                         "cores": _blas_threads(),
                         "sample": f"{tokens} tokens per step of {wl.M}, fwd+bwd, fp64"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------- standalone nf4_dequant
NF4_DEQUANT_SHAPES = [  # W [n, k] of the Llama-3-8B and Qwen1.5-32B QLoRA projections
    (4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336),
    (5120, 5120), (1024, 5120), (27392, 5120), (5120, 27392)]


def run_nf4_dequant(args):
    """HBM throughput of ``nf4_dequant`` on the QLoRA weight shapes: bytes =
    codes n·k/2 + absmax n·k/32 + bf16 output 2·n·k, CUDA-event time per call
    with a 512 MiB L2 flush between calls (outside the events)."""
    import lora_qlora_linear_fwd_b300 as L
    dev = "cuda:0"
    torch.cuda.set_device(0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak = measured_peaks()["hbm_gbs"]
    g = torch.Generator(device="cpu").manual_seed(0)
    rows = []
    for n, k in NF4_DEQUANT_SHAPES:
        W = (torch.randn(n, k, generator=g) / math.sqrt(k)).to(torch.bfloat16).to(dev)
        codes = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
        absmax = torch.empty(n, k // 64, dtype=torch.bfloat16, device=dev)
        L.nf4_quantize(W, codes, absmax)
        out = torch.empty(n, k, dtype=torch.bfloat16, device=dev)
        del W
        for _ in range(args.warmup):
            L.nf4_dequant(codes, absmax, out)
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            L.nf4_dequant(codes, absmax, out)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        t = statistics.median(ts)
        nbytes = n * k // 2 + n * k // 32 + 2 * n * k
        gbs = nbytes / (t * 1e-3) / 1e9
        rows.append({"n": n, "k": k, "us": round(t * 1e3, 2), "GBps": round(gbs, 1),
                     "frac_hbm": round(gbs / peak, 3)})
        del codes, absmax, out
    return {"component": "nf4_dequant", "unit": "GB/s", "peak_hbm_gbs": peak,
            "peak_source": measured_peaks()["source"], "steps": args.steps,
            "warmup": args.warmup, "l2": "flushed between calls (512 MiB write, outside events)",
            "data": "synthetic: NF4 codes of W ~ N(0, 1/k) quantised by nf4_quantize",
            "shapes": rows}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=128,
                    help="token sample for the oracle timing (CPU baseline / reference arm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--component", default="step", choices=["step", "nf4_dequant"],
                    help="step: the fwd+bwd step (default); nf4_dequant: the standalone "
                         "dequantisation on the QLoRA weight shapes (1 GPU)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.component == "nf4_dequant":
        print(json.dumps(run_nf4_dequant(args)), flush=True)
        return 0
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    init_dist(world, "nccl")
    line = run_gpu(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
