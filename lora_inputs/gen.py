"""Workload shapes and seeded random draws.

Workloads are synthetic stand-ins for the Llama-3-8B and Qwen1.5-32B
projection shapes the Unsloth pages train on (no weights, tokenizer or
dataset are used).  Value distributions, read as N(mean, variance):

* activations ``x ~ N(0, 1)``, incoming gradients ``dY ~ N(0, 1)``
* base weight ``W ~ N(0, 1/d_in)`` (std ``1/sqrt(d_in)``)
* adapter ``A ~ U(-1/sqrt(d_in), +1/sqrt(d_in))``, ``B ~ N(0, 0.02)``
  (std ``sqrt(0.02)``; B is non-zero so the adapter branch is exercised)

Every tensor is drawn in fp32 from one CPU ``torch.Generator`` in the order
x, W, A, B, dY and rounded to bf16 (round to nearest even), or to fp16 when
``dtype=torch.float16`` is asked for.  Projections
that share an activation (q and k of the RoPE workload) draw x once.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Projection", "Workload", "WORKLOADS", "draw_projection",
           "draw_workload", "draw_shared_x", "draw_tensor"]


@dataclass(frozen=True)
class Projection:
    name: str
    k: int          # d_in
    n: int          # d_out


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    r: int
    alpha: float
    nf4: bool
    projections: tuple
    rope: bool = False
    rope_theta: float = 0.0
    head_dim: int = 128
    description: str = ""
    blocksize: int = 64
    extra: dict = field(default_factory=dict)


_LLAMA8B = (Projection("q_proj", 4096, 4096), Projection("k_proj", 4096, 1024),
            Projection("v_proj", 4096, 1024), Projection("o_proj", 4096, 4096),
            Projection("gate_proj", 4096, 14336), Projection("up_proj", 4096, 14336),
            Projection("down_proj", 14336, 4096))
_QWEN32B = (Projection("q_proj", 5120, 5120), Projection("k_proj", 5120, 1024),
            Projection("v_proj", 5120, 1024), Projection("o_proj", 5120, 5120),
            Projection("gate_proj", 5120, 27392), Projection("up_proj", 5120, 27392),
            Projection("down_proj", 27392, 5120))

WORKLOADS = {
    "single_512": Workload(
        "single_512", M=256, r=8, alpha=16.0, nf4=False,
        projections=(Projection("linear", 512, 512),),
        description="single LoRA linear 512->512, M=256 tokens, r=8, alpha=16, bf16 W"),
    "llama8b_qk_rope": Workload(
        "llama8b_qk_rope", M=8192, r=64, alpha=16.0, nf4=False,
        projections=(Projection("q_proj", 4096, 4096), Projection("k_proj", 4096, 1024)),
        rope=True, rope_theta=500000.0, head_dim=128,
        description="Llama-3-8B q_proj+k_proj with RoPE, M=8192 (1x8192), r=64, alpha=16, "
                    "theta=5e5, positions 0..8191, bf16 W"),
    "llama8b_mlp": Workload(
        "llama8b_mlp", M=4096, r=16, alpha=16.0, nf4=False,
        projections=(Projection("gate_proj", 4096, 14336), Projection("up_proj", 4096, 14336),
                     Projection("down_proj", 14336, 4096)),
        description="Llama-3-8B MLP gate/up 4096->14336, down 14336->4096, M=4096, r=16, bf16 W"),
    "llama8b_mlp_swiglu": Workload(
        "llama8b_mlp_swiglu", M=4096, r=16, alpha=16.0, nf4=False,
        projections=(Projection("gate_proj", 4096, 14336), Projection("up_proj", 4096, 14336),
                     Projection("down_proj", 14336, 4096)),
        description="Llama-3-8B MLP block: gate/up 4096->14336 fused with SwiGLU, down "
                    "14336->4096 on its output, M=4096, r=16, bf16 W",
        extra={"swiglu": True}),
    "llama8b_qlora_all7": Workload(
        "llama8b_qlora_all7", M=4096, r=16, alpha=16.0, nf4=True, projections=_LLAMA8B,
        description="QLoRA Llama-3-8B all 7 projections, NF4 W (block 64, bf16 absmax), "
                    "M=4096, r=16, alpha=16"),
    "qwen32b_qlora_all7": Workload(
        "qwen32b_qlora_all7", M=8192, r=64, alpha=16.0, nf4=True, projections=_QWEN32B,
        description="QLoRA Qwen1.5-32B all 7 projections, NF4 W (block 64, bf16 absmax), "
                    "M=8192 (4x2048), r=64, alpha=16"),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw_tensor(g: torch.Generator, shape, kind: str, scale: float = 1.0,
                dtype=torch.bfloat16) -> torch.Tensor:
    """One 16-bit tensor: ``kind`` 'normal' (std ``scale``) or 'uniform'
    (in ``[-scale, scale)``)."""
    if kind == "normal":
        t = torch.randn(shape, generator=g, dtype=torch.float32) * scale
    elif kind == "uniform":
        t = (torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0) * scale
    else:
        raise ValueError(kind)
    return t.to(dtype)


def draw_shared_x(g: torch.Generator, M: int, k: int, dtype=torch.bfloat16) -> torch.Tensor:
    return draw_tensor(g, (M, k), "normal", 1.0, dtype)


def draw_projection(g: torch.Generator, M: int, k: int, n: int, r: int, x=None,
                    dtype=torch.bfloat16) -> dict:
    """Draw x (unless given), W, A, B, dY for one projection, in that order."""
    if x is None:
        x = draw_shared_x(g, M, k, dtype)
    W = draw_tensor(g, (n, k), "normal", 1.0 / math.sqrt(k), dtype)
    A = draw_tensor(g, (r, k), "uniform", 1.0 / math.sqrt(k), dtype)
    B = draw_tensor(g, (n, r), "normal", math.sqrt(0.02), dtype)
    dY = draw_tensor(g, (M, n), "normal", 1.0, dtype)
    return {"x": x, "W": W, "A": A, "B": B, "dY": dY}


def draw_workload(name: str, seed: int = 0, M: int | None = None, only=None) -> dict:
    """All projections of a workload: ``{proj_name: {x, W, A, B, dY}}``.

    ``M`` overrides the token count (bounded samples); ``only`` restricts the
    projections returned.  The RoPE workload draws everything from one
    stream seeded with ``seed`` (x shared by q and k); every other workload
    gives projection ``i`` its own stream seeded with ``seed*1000 + i``, so a
    projection's tensors do not depend on which others are drawn.
    """
    wl = WORKLOADS[name]
    M = wl.M if M is None else int(M)
    out = {}
    if wl.extra.get("swiglu"):
        # one stream: x shared by gate and up; down_proj's own x is drawn but
        # the step feeds it the SwiGLU output, and its dY is the block's
        # incoming gradient
        g = _gen(seed)
        gate, up, down = wl.projections
        x = draw_shared_x(g, M, gate.k)
        out[gate.name] = draw_projection(g, M, gate.k, gate.n, wl.r, x=x)
        out[up.name] = draw_projection(g, M, up.k, up.n, wl.r, x=x)
        out[down.name] = draw_projection(g, M, down.k, down.n, wl.r)
        if only is not None:
            out = {k_: v for k_, v in out.items() if k_ in only}
        return out
    if wl.rope:
        g = _gen(seed)
        x = draw_shared_x(g, M, wl.projections[0].k)
        for p in wl.projections:
            out[p.name] = draw_projection(g, M, p.k, p.n, wl.r, x=x)
        if only is not None:
            out = {k_: v for k_, v in out.items() if k_ in only}
        return out
    for i, p in enumerate(wl.projections):
        if only is not None and p.name not in only:
            continue
        g = _gen(seed * 1000 + i)
        out[p.name] = draw_projection(g, M, p.k, p.n, wl.r)
    return out
