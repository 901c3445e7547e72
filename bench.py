"""Throughput of the fused LoRA / QLoRA projection, forward + backward.

Headline workload: the Qwen1.5-32B-shaped QLoRA step, all 7 projections
(q/o 5120->5120, k/v 5120->1024, gate/up 5120->27392, down 27392->5120), NF4
base weights (block 64, bf16 absmax), M = 8192 tokens (4 x 2048), r = 64,
alpha = 16.  One step = ``lora_linear_fwd`` + ``lora_linear_bwd`` per
projection; the Llama-3-8B q/k + RoPE workload runs ``lora_qk_rope_fwd`` +
``lora_qk_rope_bwd`` instead.

Prints ONE JSON line (rank 0) with:
  * value / ms_per_step: tokens per second of the headline step, timed with
    CUDA events on the launching stream, L2 flushed between steps;
  * peaks: HBM copy bandwidth and bf16 matmul throughput measured in this
    run (beside the pool's MEASURED_PEAKS.json figures);
  * kernels / roofline / hbm_rooflines: every launch of the same K steps run
    again inside a per-launch timing session (lora_profile_begin), grouped by
    kernel, each with its algorithmic FLOPs or bytes;
  * per_workload: the other configurations' steps (parity shapes excepted);
  * e2e: the same step with its inputs copied from pinned host memory and
    all results read back, copies inside the timed region;
  * cpu_baseline: the fp64 oracle on a bounded token sample (all cores, and
    one core on a smaller sample).
``--impl reference`` times the fp64 CPU oracle instead (a bounded token
sample per step) and prints the same line with ``"impl": "reference"``.
Under torchrun every rank runs its own replica on its own GPU (weak
scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import math
import multiprocessing as mp
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
DEFAULT_WORKLOAD = "qwen32b_qlora_all7"
# configurations timed beside the headline (the 256-token single linear is a
# parity case, not a bench line)
OTHER_WORKLOADS = ("llama8b_qk_rope", "llama8b_mlp", "llama8b_mlp_swiglu", "llama8b_qlora_all7")
FLUSH_BYTES = 512 << 20          # > 126 MB L2, written between timed steps


# --------------------------------------------------------------------- work
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


def call_phases(wl, M):
    """The library calls of one step, in order, each with the algorithmic work
    of its launches in launch order: (call, [(phase, flops, bytes), ...]).

    bytes count each operand and result once, as the phase needs it (NF4 W:
    codes k/2 + bf16 absmax k/32 bytes per row); u and v of the backward are
    fp32-equivalent (their bf16 hi + lo parts)."""
    r = wl.r
    out = []
    if wl.extra.get("swiglu"):
        (pg, pu, pd) = wl.projections
        k, n, rl = pg.k, pg.n, 2 * r
        rp = 16 if rl <= 16 else 32 if rl <= 32 else 64 if rl <= 64 else 128
        kd, nd = pd.k, pd.n
        out.append(("fwd:gate_up", [
            ("fwd_rank", 2.0 * M * k * rl, 2.0 * M * k + 2.0 * rl * k + 2.0 * M * rl),
            ("fwd_gemm", 2.0 * M * k * 2 * n + 2.0 * M * r * 2 * n,
             2.0 * M * k + 4.0 * n * k + 6.0 * M * n + 2.0 * M * rl + 4.0 * n * r)]))
        out.append(("fwd:down", [
            ("fwd_rank", 2.0 * M * kd * r, 2.0 * M * kd + 2.0 * r * kd + 2.0 * M * r),
            ("fwd_gemm", 2.0 * M * kd * nd + 2.0 * M * r * nd,
             2.0 * M * kd + 2.0 * nd * kd + 2.0 * M * nd + 2.0 * M * r + 2.0 * nd * r)]))
        rpd = 16 if r <= 16 else 32 if r <= 32 else 64
        out.append(("bwd:down", [
            ("bwd_prep", 0.0, 4.0 * nd * r),
            ("bwd_rank", 2.0 * M * r * (kd + nd),
             2.0 * M * (kd + nd) + 2.0 * r * (kd + nd) + 8.0 * rpd * M + 2.0 * M * r),
            ("dx_gemm", 2.0 * M * nd * kd + 2.0 * M * r * kd,
             2.0 * M * nd + 2.0 * nd * kd + 2.0 * M * kd + 2.0 * M * r + 2.0 * r * kd),
            ("bwd_grads", 2.0 * M * r * (kd + nd),
             2.0 * M * (kd + nd) + 8.0 * rpd * M + 4.0 * r * (kd + nd))]))
        out.append(("bwd:gate_up", [
            ("bwd_prep", 0.0, 10.0 * M * n + 4.0 * rl * k + 8.0 * n * rl),
            ("bwd_rank", 2.0 * M * rl * (k + 2 * n),
             2.0 * M * (k + 2 * n) + 2.0 * rl * (k + 2 * n) + 8.0 * rp * M + 2.0 * M * rl),
            ("dx_gemm", 2.0 * M * 2 * n * k + 2.0 * M * rl * k,
             4.0 * M * n + 4.0 * n * k + 2.0 * M * k + 2.0 * M * rl + 2.0 * rl * k),
            ("bwd_grads", 2.0 * M * rl * (k + 2 * n),
             2.0 * M * (k + 2 * n) + 8.0 * rp * M + 4.0 * rl * (k + 2 * n))]))
        return out
    if wl.rope:
        (pq, pk) = wl.projections
        k, n, rl = pq.k, pq.n + pk.n, 2 * r
        rp = 16 if rl <= 16 else 32 if rl <= 32 else 64 if rl <= 64 else 128
        wbytes = 2.0 * n * k
        out.append(("fwd", [
            ("fwd_rank", 2.0 * M * k * rl, 2.0 * M * k + 2.0 * rl * k + 2.0 * M * rl),
            ("fwd_gemm", 2.0 * M * k * n + 2.0 * M * r * n,
             2.0 * M * k + wbytes + 2.0 * M * n + 2.0 * M * rl + 2.0 * n * r)]))
        out.append(("bwd", [
            ("bwd_prep", 0.0, 4.0 * M * n + 4.0 * rl * k + 4.0 * n * rl),
            ("bwd_rank", 2.0 * M * rl * (k + n),
             2.0 * M * (k + n) + 2.0 * rl * (k + n) + 8.0 * rp * M + 2.0 * M * rl),
            ("dx_gemm", 2.0 * M * n * k + 2.0 * M * rl * k,
             2.0 * M * n + wbytes + 2.0 * M * k + 2.0 * M * rl + 2.0 * rl * k),
            ("bwd_grads", 2.0 * M * rl * (k + n),
             2.0 * M * (k + n) + 8.0 * rp * M + 4.0 * rl * (k + n))]))
        return out
    rp = 16 if r <= 16 else 32 if r <= 32 else 64
    for p in wl.projections:
        k, n = p.k, p.n
        wbytes = (n * k / 2.0 + n * k / 32.0) if wl.nf4 else 2.0 * n * k
        out.append(("fwd:" + p.name, [
            ("fwd_rank", 2.0 * M * k * r, 2.0 * M * k + 2.0 * r * k + 2.0 * M * r),
            ("fwd_gemm", 2.0 * M * k * n + 2.0 * M * r * n,
             2.0 * M * k + wbytes + 2.0 * M * n + 2.0 * M * r + 2.0 * n * r)]))
        out.append(("bwd:" + p.name, [
            ("bwd_prep", 0.0, 4.0 * n * r),
            ("bwd_rank", 2.0 * M * r * (k + n),
             2.0 * M * (k + n) + 2.0 * r * (k + n) + 8.0 * rp * M + 2.0 * M * r),
            ("dx_gemm", 2.0 * M * n * k + 2.0 * M * r * k,
             2.0 * M * n + wbytes + 2.0 * M * k + 2.0 * M * r + 2.0 * r * k),
            ("bwd_grads", 2.0 * M * r * (k + n),
             2.0 * M * (k + n) + 8.0 * rp * M + 4.0 * r * (k + n))]))
    return out


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
def pool_peaks():
    """The machine's measured peaks (MEASURED_PEAKS.json), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d["bf16_tflops_sustained"], "source": "measured (pool)"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def measure_peaks(dev, sustained_s: float = 4.0):
    """Peaks measured in this run the way the pool measures them: a copy_ of
    1 Gi bf16 elements (read + write bytes, best of 10) and a bf16 8192^3
    torch.matmul (best of 10 = burst; back to back for `sustained_s` seconds
    = sustained), CUDA events on the current stream."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    a = torch.empty(1 << 30, dtype=torch.bfloat16, device=dev).fill_(1.0)
    b = torch.empty_like(a)
    best = float("inf")
    for i in range(12):
        s, e = ev(), ev()
        s.record()
        b.copy_(a)
        e.record()
        torch.cuda.synchronize()
        if i >= 2:
            best = min(best, s.elapsed_time(e))
    hbm = 2.0 * a.numel() * 2 / (best * 1e-3) / 1e9
    del a, b
    N = 8192
    g = torch.Generator(device=dev).manual_seed(0)
    x = torch.randn(N, N, device=dev, dtype=torch.bfloat16, generator=g)
    y = torch.randn(N, N, device=dev, dtype=torch.bfloat16, generator=g)
    best = float("inf")
    for i in range(12):
        s, e = ev(), ev()
        s.record()
        torch.matmul(x, y)
        e.record()
        torch.cuda.synchronize()
        if i >= 2:
            best = min(best, s.elapsed_time(e))
    burst = 2.0 * N ** 3 / (best * 1e-3) / 1e12
    s, e = ev(), ev()
    count = 0
    t_end = time.perf_counter() + sustained_s
    s.record()
    while time.perf_counter() < t_end:
        for _ in range(20):
            torch.matmul(x, y)
        count += 20
        torch.cuda.synchronize()
    e.record()
    torch.cuda.synchronize()
    sustained = 2.0 * N ** 3 * count / (s.elapsed_time(e) * 1e-3) / 1e12
    del x, y
    torch.cuda.empty_cache()
    return {"hbm_gbs": round(hbm, 1), "bf16_tflops": round(burst, 1),
            "bf16_tflops_sustained": round(sustained, 1),
            "how": "copy_ of 1 Gi bf16 (best of 10); bf16 matmul 8192^3 best of 10 (burst) and "
                   f"back to back for {sustained_s:g} s (sustained); CUDA events"}


def _code_only(src: str) -> str:
    """C/C++/CUDA source without its comments and blank space, so that an
    edit of the comments alone does not count as a change of the kernels
    (string literals are kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the code (comments and spacing left out) of every file under
    csrc: the traffic record applies while it is unchanged."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "lora_qlora_linear_fwd_b300", "csrc")
    for f in sorted(os.listdir(d)):
        h.update(f.encode() + b"\0")
        h.update(_code_only(open(os.path.join(d, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """ncu DRAM bytes per launch, by kernel name, from the committed summary
    for `workload`, when it was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    if not os.path.exists(p):
        return {}
    d = json.load(open(p))
    if d.get("source_hash") != kernel_source_hash():
        return {}
    return d.get("dram_bytes_per_launch", {})


# ------------------------------------------------------------- GPU replica
class Replica:
    """Device-resident inputs and outputs of one workload plus the calls of
    one step through the C ABI."""

    def __init__(self, name: str, device: str, seed: int = 0, stage_nf4: bool = True):
        """stage_nf4: give NF4 calls room to stage W in bf16 (the library then
        dequantises once per call and runs the bf16 GEMMs at M >= 2048);
        False: workspaces of exactly lora_workspace_size (in-GEMM decode)."""
        import lora_qlora_linear_fwd_b300 as L
        self.L = L
        self.name = name
        self.wl = wl = WORKLOADS[name]
        self.dev = device
        self.M = M = wl.M
        data = draw_workload(name, seed=seed)
        bf = dict(dtype=torch.bfloat16, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.projs = []
        for p in wl.projections:
            d = {k: v.to(device) for k, v in data.pop(p.name).items()}
            if wl.nf4:   # quantise the drawn W on the GPU (setup, not timed)
                codes = torch.empty(p.n, p.k // 2, dtype=torch.uint8, device=device)
                absmax = torch.empty(p.n, p.k // 64, **bf)
                d["Wdesc"] = L.nf4_weight(codes, absmax)
                L.nf4_quantize(d["W"], d["Wdesc"])
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
        if wl.extra.get("swiglu"):
            (pg, dg), (pu, du), (pd, dd) = self.projs
            self.h = torch.empty(M, pg.n, **bf)
            self.g = torch.empty(M, pg.n, **bf)
            self.u = torch.empty(M, pg.n, **bf)
            self.dh = torch.empty(M, pg.n, **bf)
            self.ws_f = torch.zeros(max(L.workspace_size(L.OP_SWIGLU_FWD, M, pg.k, pg.n, wl.r),
                                        L.workspace_size(L.OP_FWD, M, pd.k, pd.n, wl.r)),
                                    dtype=torch.uint8, device=device)
            self.ws_b = torch.zeros(max(L.workspace_size(L.OP_SWIGLU_BWD, M, pg.k, pg.n, wl.r),
                                        L.workspace_size(L.OP_BWD, M, pd.k, pd.n, wl.r)),
                                    dtype=torch.uint8, device=device)
        elif wl.rope:
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
            # calls run one after another on one stream: one workspace per op
            # kind, sized for the largest projection (and its staged W)
            stage = (lambda p: L.lora_nf4_stage_bytes(p.n, p.k)) if (wl.nf4 and stage_nf4) \
                else (lambda p: 0)
            self.ws_f = torch.zeros(max(L.workspace_size(L.OP_FWD, M, p.k, p.n, wl.r) + stage(p)
                                        for p in wl.projections), dtype=torch.uint8, device=device)
            self.ws_b = torch.zeros(max(L.workspace_size(L.OP_BWD, M, p.k, p.n, wl.r) + stage(p)
                                        for p in wl.projections), dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

    def inputs(self):
        """Per-step inputs (activations and incoming gradients)."""
        if self.wl.extra.get("swiglu"):
            (_, dg), _, (_, dd) = self.projs
            return [dg["x"], dd["dY"]]
        if self.wl.rope:
            (_, dq), (_, dk) = self.projs
            return [dq["x"], dq["dY"], dk["dY"]]
        out = []
        for _, d in self.projs:
            out += [d["x"], d["dY"]]
        return out

    def outputs(self):
        if self.wl.extra.get("swiglu"):
            (_, dg), (_, du), (_, dd) = self.projs
            return [dd["y"], dg["dx"], dg["dA"], dg["dB"], du["dA"], du["dB"], dd["dA"],
                    dd["dB"]]
        if self.wl.rope:
            (_, dq), (_, dk) = self.projs
            return [dq["y"], dk["y"], self.dx, dq["dA"], dq["dB"], dk["dA"], dk["dB"]]
        out = []
        for _, d in self.projs:
            out += [d["y"], d["dx"], d["dA"], d["dB"]]
        return out

    def call_io(self):
        """For each call of calls(), in order: (the per-step inputs it reads,
        the per-step results it writes), drawn from inputs() and outputs()."""
        wl = self.wl
        if wl.extra.get("swiglu"):
            (_, g), (_, u), (_, d) = self.projs
            return [([g["x"]], []), ([], [d["y"]]), ([d["dY"]], [d["dA"], d["dB"]]),
                    ([g["x"]], [g["dx"], g["dA"], g["dB"], u["dA"], u["dB"]])]
        if wl.rope:
            (_, q), (_, k) = self.projs
            return [([q["x"]], [q["y"], k["y"]]),
                    ([q["x"], q["dY"], k["dY"]], [self.dx, q["dA"], q["dB"], k["dA"], k["dB"]])]
        fwd = [([d["x"]], [d["y"]]) for _, d in self.projs]
        bwd = [([d["x"], d["dY"]], [d["dx"], d["dA"], d["dB"]]) for _, d in self.projs]
        return fwd + bwd

    def calls(self):
        """The library calls of one step, in order: [(name, fn)]."""
        L, wl = self.L, self.wl
        if wl.extra.get("swiglu"):
            (_, g), (_, u), (_, d) = self.projs
            return [
                ("fwd:gate_up", lambda: L.lora_swiglu_fwd(
                    g["x"], g["Wdesc"], g["A"], g["B"], u["Wdesc"], u["A"], u["B"], self.h,
                    wl.alpha, self.ws_f, g=self.g, u=self.u)),
                ("fwd:down", lambda: L.lora_linear_fwd(
                    self.h, d["Wdesc"], d["A"], d["B"], d["y"], wl.alpha, self.ws_f)),
                ("bwd:down", lambda: L.lora_linear_bwd(
                    self.h, d["Wdesc"], d["A"], d["B"], d["dY"], self.dh, d["dA"], d["dB"],
                    wl.alpha, self.ws_b)),
                ("bwd:gate_up", lambda: L.lora_swiglu_bwd(
                    g["x"], g["Wdesc"], g["A"], g["B"], u["Wdesc"], u["A"], u["B"], self.g,
                    self.u, self.dh, g["dx"], g["dA"], g["dB"], u["dA"], u["dB"], wl.alpha,
                    self.ws_b))]
        if wl.rope:
            (_, q), (_, k) = self.projs
            return [
                ("fwd", lambda: L.lora_qk_rope_fwd(
                    q["x"], q["Wdesc"], q["A"], q["B"], k["Wdesc"], k["A"], k["B"], q["y"],
                    k["y"], wl.alpha, wl.rope_theta, self.pos, self.cache, self.max_pos,
                    self.ws_f)),
                ("bwd", lambda: L.lora_qk_rope_bwd(
                    q["x"], q["Wdesc"], q["A"], q["B"], k["Wdesc"], k["A"], k["B"], q["dY"],
                    k["dY"], self.dx, q["dA"], q["dB"], k["dA"], k["dB"], wl.alpha,
                    wl.rope_theta, self.pos, self.cache, self.max_pos, self.ws_b))]
        out = []
        for p, d in self.projs:
            out.append(("fwd:" + p.name, lambda d=d: L.lora_linear_fwd(
                d["x"], d["Wdesc"], d["A"], d["B"], d["y"], wl.alpha, self.ws_f)))
        for p, d in self.projs:
            out.append(("bwd:" + p.name, lambda d=d: L.lora_linear_bwd(
                d["x"], d["Wdesc"], d["A"], d["B"], d["dY"], d["dx"], d["dA"], d["dB"],
                wl.alpha, self.ws_b)))
        return out

    def fwd(self):
        for name, fn in self.calls():
            if name.startswith("fwd"):
                fn()

    def bwd(self):
        for name, fn in self.calls():
            if name.startswith("bwd"):
                fn()

    def step(self):
        for _, fn in self.calls():
            fn()

    def check_status(self):
        for w in (self.ws_f, self.ws_b):
            s = self.L.lora_read_device_status(w)
            if s:
                raise RuntimeError(f"device status {s:#x}")


def time_steps(rep, steps, flush, stream):
    """CUDA-event times (ms) of `steps` steps: (step, fwd part)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()                      # L2 flush: not inside the step's events
        a, b, c = ev[i]
        a.record(stream)
        rep.fwd()
        b.record(stream)
        rep.bwd()
        c.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(c) for a, _, c in ev], [a.elapsed_time(b) for a, b, _ in ev]


def profile_steps(rep, steps, flush):
    """The same steps inside a per-launch timing session: every launch with
    its kernel, phase and algorithmic work.  Launches are matched to the
    call's phases by kernel name: an NF4 weight staged in bf16 adds an
    nf4_dequant launch, and a forward that forms x·Aᵀ in its GEMM (`xa`)
    has no rank pass (its GEMM carries the rank pass's FLOPs)."""
    L = rep.L
    phases = {name: ph for name, ph in call_phases(rep.wl, rep.M)}
    calls = rep.calls()
    cap = steps * (sum(len(ph) for ph in phases.values()) + 2 * len(calls)) + 16
    counts = []   # (call, launches)
    L.lora_profile_begin(cap)
    try:
        for _ in range(steps):
            flush.zero_()
            for name, fn in calls:
                c0 = L.lora_kernel_launch_count()
                fn()
                counts.append((name, L.lora_kernel_launch_count() - c0))
    finally:
        timed = L.lora_profile_end(cap)
    if len(timed) != sum(n for _, n in counts):
        raise RuntimeError(f"profile: {len(timed)} timed launches for {sum(n for _, n in counts)}")
    rows, i = [], 0
    for name, n in counts:
        ph = dict((x[0], x) for x in phases[name])
        skinny = [x for x in phases[name] if x[0] in ("fwd_rank", "bwd_rank", "bwd_grads")]
        for kname, ms in timed[i:i + n]:
            if kname.startswith("nf4_dequant"):
                p_ = next(q for q in rep.wl.projections if name.endswith(q.name)) \
                    if not rep.wl.rope and not rep.wl.extra.get("swiglu") else None
                nk = (p_.n * p_.k) if p_ else 0
                work = ("nf4_stage", 0.0, nk * (0.5 + 1.0 / 32 + 2.0))
            elif kname.startswith("bwd_prep"):
                work = ph["bwd_prep"]
            elif kname.startswith("lora_skinny"):
                work = skinny.pop(0)
            elif kname.startswith("lora_gemm_pair_kernel<fwd"):
                work = ph["fwd_gemm"]
                if kname.endswith(",xa>") and "fwd_rank" in ph:
                    work = ("fwd_gemm", work[1] + ph["fwd_rank"][1], work[2])
            elif kname.startswith("lora_gemm_pair_kernel<dx"):
                work = ph["dx_gemm"]
            else:
                raise RuntimeError(f"{name}: unexpected launch {kname}")
            rows.append((kname, ms, name) + work)
        i += n
    return rows


def summarise_kernels(rows, steps, peaks, pool):
    """Per kernel name: launches per step, time per step, share, and the
    algorithmic throughput of its launches (FLOP/s for the GEMMs, B/s for the
    streaming passes)."""
    total = sum(r[1] for r in rows)
    by = {}
    for kname, ms, call, phase, fl, b in rows:
        e = by.setdefault(kname, {"launches": 0, "ms": 0.0, "flops": 0.0, "bytes": 0.0,
                                  "phases": set()})
        e["launches"] += 1
        e["ms"] += ms
        e["flops"] += fl
        e["bytes"] += b
        e["phases"].add(phase)
    out = []
    for kname, e in sorted(by.items(), key=lambda kv: -kv[1]["ms"]):
        gemm = kname.startswith("lora_gemm_pair_kernel")
        row = {"kernel": kname, "phases": sorted(e["phases"]),
               "launches_per_step": e["launches"] / steps,
               "ms_per_step": round(e["ms"] / steps, 4),
               "share": round(e["ms"] / total, 4),
               "avg_launch_us": round(1e3 * e["ms"] / e["launches"], 2)}
        if gemm:
            tf = e["flops"] / (e["ms"] * 1e-3) / 1e12
            row.update({"bound": "tensor", "tflops": round(tf, 1),
                        "frac": round(tf / peaks["bf16_tflops"], 4),
                        "frac_pool": round(tf / pool["bf16_tflops"], 4)})
        else:
            gbs = e["bytes"] / (e["ms"] * 1e-3) / 1e9
            row.update({"bound": "hbm", "gbs": round(gbs, 1),
                        "frac": round(gbs / peaks["hbm_gbs"], 4),
                        "frac_pool": round(gbs / pool["hbm_gbs"], 4)})
        out.append((row, e))
    return out, total / steps


def flush_clean(flush):
    """L2 flush for short kernels: write the 512 MiB buffer (evicts the
    working set), then read half of it, so the dirty lines the write leaves
    in L2 go back to HBM before the timed launch instead of during it."""
    flush.zero_()
    flush[: flush.numel() // 2].max()


def launch_floor_us(dev, flush, steps=20):
    """CUDA-event time of the smallest nf4_dequant launch (64 x 64): the
    fixed launch-to-completion cost that a short launch cannot go below."""
    import lora_qlora_linear_fwd_b300 as L
    codes = torch.zeros(64, 32, dtype=torch.uint8, device=dev)
    absmax = torch.ones(64, 1, dtype=torch.bfloat16, device=dev)
    out = torch.empty(64, 64, dtype=torch.bfloat16, device=dev)
    Wq = L.nf4_weight(codes, absmax)
    ts = []
    for i in range(steps + 3):
        flush_clean(flush)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        L.nf4_dequant(Wq, out)
        b.record()
        torch.cuda.synchronize()
        if i >= 3:
            ts.append(a.elapsed_time(b))
    return round(statistics.median(ts) * 1e3, 2)


def run_nf4_dequant_shapes(shapes, dev, flush, steps, warmup, peak):
    """HBM throughput of ``nf4_dequant`` on weight shapes [(n, k)]: bytes =
    codes n·k/2 + absmax n·k/32 + bf16 output 2·n·k, CUDA-event time per call
    with an L2 flush between calls (flush_clean, outside the events)."""
    import lora_qlora_linear_fwd_b300 as L
    g = torch.Generator(device="cpu").manual_seed(0)
    rows = []
    for n, k in shapes:
        W = (torch.randn(n, k, generator=g) / math.sqrt(k)).to(torch.bfloat16).to(dev)
        codes = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
        absmax = torch.empty(n, k // 64, dtype=torch.bfloat16, device=dev)
        Wq = L.nf4_weight(codes, absmax)
        L.nf4_quantize(W, Wq)
        out = torch.empty(n, k, dtype=torch.bfloat16, device=dev)
        del W
        for _ in range(warmup):
            L.nf4_dequant(Wq, out)
        ts = []
        for _ in range(steps):
            flush_clean(flush)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            L.nf4_dequant(Wq, out)
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        t = statistics.median(ts)
        nbytes = n * k // 2 + n * k // 32 + 2 * n * k
        gbs = nbytes / (t * 1e-3) / 1e9
        rows.append({"n": n, "k": k, "us": round(t * 1e3, 2), "GBps": round(gbs, 1),
                     "frac_hbm": round(gbs / peak, 3)})
        del codes, absmax, out
    return rows


def nf4_fused_vs_unfused(name, proj, dev, flush, steps, warmup):
    """The NF4 projection `proj` of workload `name`, forward and backward:
    fused (NF4 codes decoded inside the GEMMs) against the unfused composition
    the library also offers, nf4_dequant into a bf16 W followed by the bf16
    calls; CUDA-event median over `steps` calls, L2 flushed between calls."""
    import lora_qlora_linear_fwd_b300 as L
    wl = WORKLOADS[name]
    p = next(q for q in wl.projections if q.name == proj)
    M, r = wl.M, wl.r
    d = {k: v.to(dev) for k, v in draw_workload(name, seed=0, only=[proj])[proj].items()}
    bf = dict(dtype=torch.bfloat16, device=dev)
    codes = torch.empty(p.n, p.k // 2, dtype=torch.uint8, device=dev)
    absmax = torch.empty(p.n, p.k // 64, **bf)
    Wq = L.nf4_weight(codes, absmax)
    L.nf4_quantize(d["W"], Wq)
    Wb = torch.empty(p.n, p.k, **bf)
    y = torch.empty(M, p.n, **bf)
    dx = torch.empty(M, p.k, **bf)
    dA = torch.empty(r, p.k, dtype=torch.float32, device=dev)
    dB = torch.empty(p.n, r, dtype=torch.float32, device=dev)
    # exact-size workspaces: the NF4 calls decode inside the GEMMs
    wsf = L.workspace(L.OP_FWD, M, p.k, p.n, r, device=dev)
    wsb = L.workspace(L.OP_BWD, M, p.k, p.n, r, device=dev)
    calls = {
        "fwd_fused": lambda: L.lora_linear_fwd(d["x"], Wq, d["A"], d["B"], y, wl.alpha, wsf),
        "fwd_dequant_then_bf16": lambda: (L.nf4_dequant(Wq, Wb),
                                          L.lora_linear_fwd(d["x"], Wb, d["A"], d["B"], y,
                                                            wl.alpha, wsf)),
        "bwd_fused": lambda: L.lora_linear_bwd(d["x"], Wq, d["A"], d["B"], d["dY"], dx, dA, dB,
                                               wl.alpha, wsb),
        "bwd_dequant_then_bf16": lambda: (L.nf4_dequant(Wq, Wb),
                                          L.lora_linear_bwd(d["x"], Wb, d["A"], d["B"], d["dY"],
                                                            dx, dA, dB, wl.alpha, wsb)),
    }
    out = {"workload": name, "projection": [proj, p.k, p.n], "M": M, "steps": steps}
    for key, fn in calls.items():
        for _ in range(warmup):
            fn()
        ts = []
        for _ in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        out[key + "_ms"] = round(statistics.median(ts), 4)
    out["fwd_unfused_over_fused"] = round(out["fwd_dequant_then_bf16_ms"] / out["fwd_fused_ms"], 3)
    out["bwd_unfused_over_fused"] = round(out["bwd_dequant_then_bf16_ms"] / out["bwd_fused_ms"], 3)
    return out


def nf4_small_m_probe(wl, dev, flush, peak, ms=(16, 32, 64), steps=20):
    """Supplementary probe: the fused NF4 forward at a few tokens per call,
    where it is bound by the weight stream.  Per NF4 weight shape and M, the
    CUDA-event time of lora_linear_fwd (codes decoded in the GEMM) and its
    bytes: codes n·k/2 + absmax n·k/32 + x, y, A, B in bf16."""
    import lora_qlora_linear_fwd_b300 as L
    g = torch.Generator(device="cpu").manual_seed(0)
    r, rows = wl.r, []
    for n, k in sorted({(p.n, p.k) for p in wl.projections}):
        W = (torch.randn(n, k, generator=g) / math.sqrt(k)).to(torch.bfloat16).to(dev)
        codes = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
        absmax = torch.empty(n, k // 64, dtype=torch.bfloat16, device=dev)
        Wq = L.nf4_weight(codes, absmax)
        L.nf4_quantize(W, Wq)
        del W
        A = (torch.rand(r, k, generator=g) * 2 - 1).mul(1 / math.sqrt(k)).to(torch.bfloat16).to(dev)
        B = (torch.randn(n, r, generator=g) * math.sqrt(0.02)).to(torch.bfloat16).to(dev)
        for M in ms:
            x = torch.randn(M, k, generator=g).to(torch.bfloat16).to(dev)
            y = torch.empty(M, n, dtype=torch.bfloat16, device=dev)
            ws = L.workspace(L.OP_FWD, M, k, n, r, device=dev)
            ts = []
            for i in range(steps + 3):
                flush_clean(flush)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                L.lora_linear_fwd(x, Wq, A, B, y, wl.alpha, ws)
                b.record()
                torch.cuda.synchronize()
                if i >= 3:
                    ts.append(a.elapsed_time(b))
            if L.lora_read_device_status(ws):
                raise RuntimeError("device status after the small-M probe")
            t = statistics.median(ts)
            nbytes = n * k // 2 + n * k // 32 + 2 * (M * k + M * n + r * (k + n))
            gbs = nbytes / (t * 1e-3) / 1e9
            rows.append({"n": n, "k": k, "M": M, "us": round(t * 1e3, 2), "GBps": round(gbs, 1),
                         "frac_hbm": round(gbs / peak, 3)})
        del codes, absmax, Wq, A, B
        torch.cuda.empty_cache()
    return rows


def torch_unfused_step(name, dev, flush, steps=10, warmup=3):
    """Context, not a target: the same step as plain torch bf16 autograd
    (cuBLAS), the shape of a PEFT LoRA layer: y = x·Wᵀ + s·(x·Aᵀ)·Bᵀ, then
    backward from dY into x, A and B (W frozen).  For NF4 workloads the drawn
    bf16 W stands in for the dequantised weight (same shape; no dequantise
    is timed)."""
    import torch.nn.functional as F
    wl = WORKLOADS[name]
    if wl.rope or wl.extra.get("swiglu"):
        return None
    data = draw_workload(name, seed=0)
    s = wl.alpha / wl.r
    projs = []
    for p in wl.projections:
        d = {k: v.to(dev) for k, v in data.pop(p.name).items()}
        x = d["x"].requires_grad_(True)
        A = d["A"].clone().requires_grad_(True)
        B = d["B"].clone().requires_grad_(True)
        projs.append((x, d["W"], A, B, d["dY"]))
    del data

    def step():
        for x, W, A, B, dY in projs:
            y = F.linear(x, W) + s * F.linear(F.linear(x, A), B)
            y.backward(dY)

    for _ in range(warmup):
        flush.zero_()
        step()
    ts = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    del projs
    torch.cuda.empty_cache()
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(wl.M / (ms * 1e-3), 1),
            "tflops": round(step_flops(wl, wl.M) / (ms * 1e-3) / 1e12, 1),
            "what": "torch bf16 autograd per projection (F.linear, cuBLAS), unfused LoRA "
                    "branch, W frozen (bf16 W for NF4 workloads, no dequantise timed); "
                    f"median of {steps} steps, L2 flushed between steps"}


def workload_line(rep, steps, warmup, flush, stream, peaks, pool):
    """Step time of one workload (used for the configurations beside the
    headline)."""
    for _ in range(warmup):
        flush.zero_()
        rep.step()
    torch.cuda.synchronize()
    step_ms, fwd_ms = time_steps(rep, steps, flush, stream)
    rep.check_status()
    ms = statistics.mean(step_ms)
    fl = step_flops(rep.wl, rep.M)
    tf = fl / (ms * 1e-3) / 1e12
    return {"ms_per_step": round(ms, 4), "ms_median": round(statistics.median(step_ms), 4),
            "fwd_ms": round(statistics.mean(fwd_ms), 4),
            "tokens_per_s": round(rep.M / (ms * 1e-3), 1), "tflops": round(tf, 1),
            "frac_of_burst": round(tf / peaks["bf16_tflops"], 4),
            "frac_of_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
            "frac_of_pool_burst": round(tf / pool["bf16_tflops"], 4),
            "steps": steps, "M": rep.M, "description": rep.wl.description}


def run_gpu(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    import lora_qlora_linear_fwd_b300 as L
    pool = pool_peaks()
    peaks = measure_peaks(dev, args.sustained_s)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    rep = Replica(args.workload, dev)
    wl, M = rep.wl, rep.M
    for _ in range(args.warmup):
        flush.zero_()
        rep.step()
    torch.cuda.synchronize()
    rep.check_status()

    # ---- the headline timed region (no instrumentation)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    launches0 = L.lora_kernel_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    step_ms, fwd_ms = time_steps(rep, args.steps, flush, stream)
    barrier(world)
    wall = time.perf_counter() - t0
    launches = L.lora_kernel_launch_count() - launches0
    clocks = sampler.stop()
    rep.check_status()
    ms_local = statistics.mean(step_ms)
    ms = max_over_ranks(ms_local, world)
    fwd_ms_mean = statistics.mean(fwd_ms)

    # ---- the same steps again, each launch timed (per-kernel rooflines)
    rows = profile_steps(rep, args.steps, flush)
    rep.check_status()
    kern, prof_ms_per_step = summarise_kernels(rows, args.steps, peaks, pool)
    traffic = profiled_traffic(args.workload)
    top_row, top = kern[0]
    top_kind = "tensor" if top_row["bound"] == "tensor" else "hbm"
    achieved = top_row["tflops"] if top_kind == "tensor" else top_row["gbs"]
    peak = peaks["bf16_tflops"] if top_kind == "tensor" else peaks["hbm_gbs"]
    tr = traffic.get(top_row["kernel"])
    roofline = {
        "kernel": top_row["kernel"], "bound": top_kind, "achieved": achieved, "peak": peak,
        "unit": "TFLOP/s" if top_kind == "tensor" else "GB/s",
        "frac": round(achieved / peak, 4),
        "peak_source": "measured in this run (burst)",
        "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)
        if top_kind == "tensor" else None,
        "frac_of_pool": top_row["frac_pool"],
        "pool_peak": pool["bf16_tflops"] if top_kind == "tensor" else pool["hbm_gbs"],
        "traffic": tr,
        "algorithmic_per_launch": (top["flops"] if top_kind == "tensor" else top["bytes"])
        / top["launches"],
        "avg_launch_us": top_row["avg_launch_us"], "launches_per_step":
        top_row["launches_per_step"], "share": top_row["share"],
        "timing": "CUDA events around each launch on its stream (lora_profile_begin), over "
                  f"{args.steps} steps run right after the timed region"}
    hbm_lines = [dict(r, peak=peaks["hbm_gbs"]) for r, _ in kern if r["bound"] == "hbm"]
    # nf4_dequant on the headline's weight shapes
    if wl.nf4:
        shapes = sorted({(p.n, p.k) for p in wl.projections})
        dq = run_nf4_dequant_shapes(shapes, dev, flush, 20, 3, peaks["hbm_gbs"])
        floor = launch_floor_us(dev, flush)
        for row in dq:
            nbytes = row["GBps"] * row["us"] * 1e3
            # the best a launch of these bytes can do: the launch floor plus
            # the bytes at the measured HBM rate
            best_us = floor + nbytes / (peaks["hbm_gbs"] * 1e3)
            hbm_lines.append({"kernel": "nf4_dequant_kernel", "shape": [row["n"], row["k"]],
                              "bound": "hbm", "gbs": row["GBps"], "us": row["us"],
                              "frac": row["frac_hbm"], "peak": peaks["hbm_gbs"],
                              "frac_pool": round(row["GBps"] / pool["hbm_gbs"], 4),
                              "launch_floor_us": floor,
                              "frac_of_floor_bound": round(best_us / row["us"], 3)})

    # ---- end to end through the C ABI with host buffers (pinned), copies timed
    e2e = run_e2e(rep, args, stream)
    e2e_ms = max_over_ranks(e2e["ms"], world)

    flops = step_flops(wl, M)
    tokens_per_s = world * M / (ms / 1e3)
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
        "tflops_frac_of_sustained": round(
            flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"], 4),
        "tflops_frac_of_pool_peak": round(flops / (ms / 1e3) / 1e12 / pool["bf16_tflops"], 4),
        "fwd_ms": round(fwd_ms_mean, 4),
        "bwd_ms": round(ms_local - fwd_ms_mean, 4),
        "ms_median": round(statistics.median(step_ms), 4),
        "region_wall_s": round(wall, 4),
        "config": {"workload": args.workload, "description": wl.description, "M": M,
                   "r": wl.r, "alpha": wl.alpha, "nf4": wl.nf4,
                   "projections": [[p.name, p.k, p.n] for p in wl.projections],
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed between timed steps (512 MiB write, outside step events)"},
        "peaks": {"this_run": peaks, "pool": pool},
        "roofline": roofline,
        "hbm_rooflines": hbm_lines,
        "kernels": [r for r, _ in kern],
        "profiled_ms_per_step": round(prof_ms_per_step, 4),
        "e2e": {"value": round(world * M / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e_ms, 4),
                "how": "pinned host buffers; host-to-device copies of each call's inputs and "
                       "device-to-host reads of its results on two copy streams, overlapping "
                       "the compute stream; every byte copied every step"},
        "gpu_launches": int(launches),
        "gpu_launches_per_step": launches / args.steps,
        "clocks": clocks,
    }
    del rep
    torch.cuda.empty_cache()

    # ---- the other configurations (rank 0 only reports them)
    if not args.no_per_workload:
        per = {}
        for name in OTHER_WORKLOADS:
            if name == args.workload:
                continue
            r2 = Replica(name, dev)
            per[name] = workload_line(r2, args.steps, args.warmup, flush, stream, peaks, pool)
            del r2
            torch.cuda.empty_cache()
        per[args.workload] = {
            "ms_per_step": line["ms_per_step"], "tokens_per_s": line["value"] / world,
            "tflops": round(flops / (ms / 1e3) / 1e12, 1),
            "frac_of_burst": line["tflops_frac_of_peak"],
            "frac_of_sustained": line["tflops_frac_of_sustained"],
            "frac_of_pool_burst": line["tflops_frac_of_pool_peak"], "steps": args.steps,
            "M": M, "description": wl.description, "headline": True}
        line["per_workload"] = per
        if wl.nf4:   # the headline step with the NF4 codes decoded inside the GEMMs
            r2 = Replica(args.workload, dev, stage_nf4=False)
            per[args.workload + ":nf4_decoded_in_gemm"] = workload_line(
                r2, args.steps, args.warmup, flush, stream, peaks, pool)
            del r2
            torch.cuda.empty_cache()
        if wl.nf4:   # the fused NF4 GEMMs against dequantising first
            line["nf4_fused_vs_unfused"] = nf4_fused_vs_unfused(args.workload, "gate_proj", dev,
                                                                flush, 10, 3)
            torch.cuda.empty_cache()
            line["nf4_small_m_probe"] = nf4_small_m_probe(wl, dev, flush, peaks["hbm_gbs"])
        line["torch_unfused_bf16"] = torch_unfused_step(args.workload, dev, flush)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_tokens, args.cpu_tokens_1core)
    return line


def run_e2e(rep, args, stream):
    """Same step through the C ABI with the step's inputs on the host: every
    step copies its inputs from pinned host memory and reads back all its
    results (y, dX, dA, dB); copies are inside the timed region.

    The copies run on two copy streams beside the compute stream, in the
    order the calls need them: a call waits for the host-to-device copies of
    its inputs, each result's device-to-host copy starts when the call that
    writes it is done, and a buffer is refilled (next step) only after its
    last reader and read back only before its next writer, so inputs of later
    calls and results of earlier ones move while the GPU computes."""
    ins = rep.inputs()
    outs = rep.outputs()
    h_in = {id(t): t.cpu().pin_memory() for t in ins}
    h_out = {id(t): torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs}
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    steps = max(3, min(args.steps, 10))
    calls, io = rep.calls(), rep.call_io()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    last_read, read_back = {}, {}   # tensor id -> event (previous step)

    def one():
        loaded = set()
        for (_, fn), (reads, writes) in zip(calls, io):
            for t in reads:
                if id(t) in loaded:
                    continue
                if id(t) in last_read:
                    s_in.wait_event(last_read[id(t)])
                with torch.cuda.stream(s_in):
                    t.copy_(h_in[id(t)], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
                stream.wait_event(e)
                loaded.add(id(t))
            for t in writes:
                if id(t) in read_back:
                    stream.wait_event(read_back[id(t)])
            fn()
            done = torch.cuda.Event()
            done.record(stream)
            for t in reads:
                last_read[id(t)] = done
            if writes:
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    for t in writes:
                        h_out[id(t)].copy_(t, non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_out)
                for t in writes:
                    read_back[id(t)] = e

    one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    for _ in range(steps):
        one()
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    b.record(stream)
    torch.cuda.synchronize()
    return {"ms": a.elapsed_time(b) / steps, "h2d": h2d, "d2h": d2h}


# ----------------------------------------------------------- CPU (oracle)
def _blas_threads():
    """Threads numpy's BLAS uses (threadpoolctl when present, else the
    thread-count environment, else every core)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return os.cpu_count()


def oracle_step(name: str, data, M: int):
    import oracle as ref
    wl = WORKLOADS[name]
    f = lambda t: t.float().numpy().astype(np.float64)
    if wl.extra.get("swiglu"):
        g, u, d = data["gate_proj"], data["up_proj"], data["down_proj"]
        W = lambda t: t["Wq"] if "Wq" in t else f(t["W"])
        args = (f(g["x"]), W(g), f(g["A"]), f(g["B"]), W(u), f(u["A"]), f(u["B"]))
        h = ref.swiglu_fwd(*args, wl.alpha)[0]
        ref.lora_fwd(h, W(d), f(d["A"]), f(d["B"]), wl.alpha)
        dh = ref.lora_bwd(h, W(d), f(d["A"]), f(d["B"]), f(d["dY"]), wl.alpha)[0]
        ref.swiglu_bwd(*args, dh, wl.alpha)
        return
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


def _quantize_rows(w_rows):
    """Oracle NF4 quantisation of a block of W rows (rows are independent)."""
    import oracle as ref
    return ref.nf4_quantize(w_rows)


def _quantize_workload(data, wl):
    """Oracle NF4 codes and absmax of every projection's W, row blocks spread
    over a spawned process pool (rows quantise independently)."""
    import oracle  # noqa: F401  (the workers import it too)
    workers = max(1, min(os.cpu_count() or 1, 32))
    out = {}
    with cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex:
        for p in wl.projections:
            W = data[p.name]["W"].float().numpy()
            step = max(64, -(-W.shape[0] // workers))
            parts = list(ex.map(_quantize_rows, [W[i:i + step]
                                                 for i in range(0, W.shape[0], step)]))
            out[p.name] = (np.concatenate([c for c, _ in parts]),
                           np.concatenate([a for _, a in parts]))
    return out


def _oracle_sample(name: str, tokens: int, quantized=None):
    """The workload's tensors with `tokens` rows of x and dY; NF4 weights are
    the oracle's quantisation of the drawn W (preparation of the oracle's
    inputs, outside its timing).  Returns (data, quantized)."""
    import oracle as ref
    wl = WORKLOADS[name]
    data = draw_workload(name, seed=0, M=tokens)
    if wl.nf4:
        if quantized is None:
            quantized = _quantize_workload(data, wl)
        for p in wl.projections:
            data[p.name]["Wq"] = ref.nf4_dequant(*quantized[p.name])
    return data, quantized


def _time_oracle(name, data, tokens):
    t0 = time.perf_counter()
    oracle_step(name, data, tokens)
    return time.perf_counter() - t0


def _time_oracle_one_core(name, tokens, quantized):
    """Oracle step time on one BLAS thread: timed in a spawned interpreter
    whose BLAS libraries load with one thread (environment set before numpy
    is imported there)."""
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
            "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    try:
        for k in keys:
            os.environ[k] = "1"
        with cf.ProcessPoolExecutor(1, mp_context=mp.get_context("spawn")) as ex:
            return ex.submit(_one_core_child, name, tokens, quantized).result()
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _one_core_child(name, tokens, quantized):
    data, _ = _oracle_sample(name, tokens, quantized)
    return _time_oracle(name, data, tokens), _blas_threads()


def cpu_baseline(name: str, tokens: int, tokens_1core: int):
    """The fp64 oracle as it stands, on the host cores, over a bounded token
    sample of the same workload; tokens/s = sample tokens / time.  Also one
    BLAS thread on a smaller sample."""
    data, quantized = _oracle_sample(name, tokens)
    dt = _time_oracle(name, data, tokens)
    del data
    dt1, threads1 = _time_oracle_one_core(name, tokens_1core, quantized)
    return {"value": round(tokens / dt, 2), "unit": "tokens/s", "cores": _blas_threads(),
            "cpu_count": os.cpu_count(), "kind": "oracle",
            "sample": f"{tokens} of {WORKLOADS[name].M} tokens, all projections, fwd+bwd in "
                      f"fp64 numpy ({dt:.1f} s)",
            "one_core": {"value": round(tokens_1core / dt1, 2), "unit": "tokens/s",
                         "cores": threads1,
                         "sample": f"{tokens_1core} tokens, all projections, fwd+bwd, one BLAS "
                                   f"thread ({dt1:.1f} s)"}}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    wl = WORKLOADS[args.workload]
    tokens = args.ref_tokens
    data, _ = _oracle_sample(args.workload, tokens)
    for _ in range(args.warmup):
        oracle_step(args.workload, data, tokens)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(args.workload, data, tokens)
        times.append(time.perf_counter() - t0)
    per_token = statistics.mean(times) / tokens
    value = 1.0 / per_token
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(per_token * wl.M * 1e3, 2),
        "ms_per_step_basis": f"scaled linearly from {tokens}-token samples to {wl.M} tokens",
        "ms_per_sample_step": round(statistics.mean(times) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "description": wl.description, "M": wl.M,
                   "sample_tokens_per_step": tokens},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "kind": "oracle",
                         "cores": _blas_threads(), "cpu_count": os.cpu_count(),
                         "sample": f"{tokens} tokens per step of {wl.M}, fwd+bwd, fp64"},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------- standalone nf4_dequant
NF4_DEQUANT_SHAPES = [  # W [n, k] of the Llama-3-8B and Qwen1.5-32B QLoRA projections
    (4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336),
    (5120, 5120), (1024, 5120), (27392, 5120), (5120, 27392)]


def run_nf4_dequant(args):
    dev = "cuda:0"
    torch.cuda.set_device(0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    pool = pool_peaks()
    rows = run_nf4_dequant_shapes(NF4_DEQUANT_SHAPES, dev, flush, args.steps, args.warmup,
                                  pool["hbm_gbs"])
    return {"component": "nf4_dequant", "unit": "GB/s", "peak_hbm_gbs": pool["hbm_gbs"],
            "peak_source": pool["source"], "steps": args.steps,
            "warmup": args.warmup, "l2": "flushed between calls (512 MiB write, outside events)",
            "data": "synthetic: NF4 codes of W ~ N(0, 1/k) quantised by nf4_quantize",
            "shapes": rows}


def run_nf4_small_m(args):
    """The small-M NF4 forward probe alone (the step line carries it too)."""
    dev = "cuda:0"
    torch.cuda.set_device(0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    pool = pool_peaks()
    rows = nf4_small_m_probe(WORKLOADS[args.workload], dev, flush, pool["hbm_gbs"],
                             steps=args.steps)
    return {"component": "nf4_small_m", "workload": args.workload, "unit": "us",
            "peak_hbm_gbs": pool["hbm_gbs"], "peak_source": pool["source"],
            "steps": args.steps, "l2": "flushed between calls (512 MiB write, outside events)",
            "rows": rows}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=512,
                    help="token sample of the oracle timing on all cores (CPU baseline)")
    ap.add_argument("--cpu-tokens-1core", type=int, default=32,
                    help="token sample of the oracle timing on one BLAS thread")
    ap.add_argument("--ref-tokens", type=int, default=128,
                    help="token sample per step of the reference arm")
    ap.add_argument("--sustained-s", type=float, default=4.0,
                    help="seconds of back-to-back matmuls for the sustained peak")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the step lines of the other configurations")
    ap.add_argument("--component", default="step", choices=["step", "nf4_dequant", "nf4_small_m"],
                    help="step: the fwd+bwd step (default); nf4_dequant: the standalone "
                         "dequantisation on the QLoRA weight shapes; nf4_small_m: the fused "
                         "NF4 forward at 16-64 tokens on the workload's weight shapes (1 GPU)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.component == "nf4_dequant":
        print(json.dumps(run_nf4_dequant(args)), flush=True)
        return 0
    if args.component == "nf4_small_m":
        print(json.dumps(run_nf4_small_m(args)), flush=True)
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
