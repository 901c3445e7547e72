"""fp64 reference definitions of the fused LoRA / QLoRA projection.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py``; never by the library.

Sources (web pages about Unsloth; cited by title and section):

* [P1] "UnSloth加速微调体验：在LoRA基础上再提速3倍的秘密" — sections
  算子融合 (operator fusion, eq. ``y = Wx + ΔWx = Wx + BAx``),
  反向传播优化 (backward with recomputation, gradient equations),
  RoPE缓存集成 (RoPE cache fused into the Q/K projection).
* [P2] "微调太慢？试试Unsloth：实测训练速度翻倍，显存占用减半" — §5.1
  (inference with the adapter merged into the weight).
* [P3] "Unsloth教程：本地微调大模型速度提升数倍，显存节省60%" — 底层内核优化
  (fused kernels are mathematically equivalent to the unfused ops) and
  显存优化策略 (QLoRA: 4-bit NormalFloat4 base weight, only the adapter
  trained; 4096x4096 at rank 16 -> about 1.3e5 trainable parameters).
* [P5] "Unsloth自动化优化：无需手动调参的实现原理" — §3.2 (fused kernel also
  described as ``A@B + original_weight``), §3.3/§5 (NF4 is the default).
* [P4] "Unsloth框架：高效LLM微调与LoRA优化实践" — §3.1 计算图重写引擎
  (adjacent linear layers merged with their activation function).
* [P5] also §1, 模型结构自识别 (the SwiGLU block is one of the modules it
  recognises and optimises).
* [SwiGLU] Shazeer 2020, "GLU Variants Improve Transformer", §2: the
  gated unit ``Swish_1(x·W)·(x·V)`` with ``Swish_1(t) = t·sigmoid(t)``
  (SiLU); the pages name SwiGLU but do not write it out.
* [Philox] Salmon, Moraes, Dror, Shaw 2011, "Parallel random numbers: as easy
  as 1, 2, 3", §4 (the Philox counter-based generator; 4x64 words, 10
  rounds): the generator the dropout mask is drawn from.
* [QLoRA] Dettmers et al. 2023, "QLoRA: Efficient Finetuning of Quantized
  LLMs", §3 "4-bit NormalFloat Quantization" and the NF4 table in its
  appendix: the pages name NF4 but do not give its levels; §3 "Double
  Quantization" (8-bit float second-level quantisation of the block scales,
  blocks of 256, mean subtracted), which the pages do not mention.
* [OCP FP8] "OCP 8-bit Floating Point Specification (OFP8)" rev. 1.0, E4M3:
  the 8-bit float format of the double-quantised block scales.
* [IEEE 754] binary16 (fp16): the second 16-bit type; the pages'
  usage example "UnSloth加速微调体验" passes ``dtype = torch.float16`` and
  "Unsloth自动化优化" §3.1 falls back to fp16 where bf16 is unsupported.

Conventions (row-vector form of [P1] 算子融合, which writes column vectors):
``x [M,k]``, ``W [n,k]`` (out x in), ``A [r,k]``, ``B [n,r]``,
``y, dY [M,n]``; the LoRA scale is ``s = alpha / r``.  The pages print the
forward without ``s`` and list ``lora_alpha`` and ``r`` only as API
arguments; the standard LoRA reading ``s = alpha/r`` is taken.

All arithmetic is numpy float64.  Inputs are expected to already hold the
values the GPU receives (bf16-rounded), so the upcast to fp64 is exact.
"""
from __future__ import annotations

import numpy as np
from scipy.stats import norm

__all__ = [
    "lora_scale", "lora_fwd", "lora_bwd", "lora_adapter_grads", "merged_weight",
    "lora_param_count",
    "bf16_round", "nf4_codebook", "nf4_quantize", "nf4_unpack", "nf4_dequant",
    "rope_inv_freq", "rope_cos_sin", "rope_apply", "rope_apply_inverse",
    "qk_rope_fwd", "qk_rope_bwd",
    "sigmoid", "silu", "swiglu_fwd", "swiglu_bwd",
    "unmerged_weight", "nf4_merge",
    "philox4x64", "dropout_keep", "dropout_keep_prob", "lora_fwd_dropout",
    "lora_bwd_dropout",
    "f16_round", "round16", "e4m3_values", "e4m3_round", "e4m3_encode", "dq_encode",
    "dq_decode", "nf4_quantize_dq", "nf4_dequant_dq",
]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------------------
# LoRA projection
# ---------------------------------------------------------------------------
def lora_scale(alpha: float, r: int) -> float:
    """LoRA branch scale ``s = alpha / r`` (reading: the pages pass
    ``lora_alpha`` and ``r`` to ``get_peft_model`` in [P1] and never write the
    formula)."""
    return float(alpha) / float(r)


def lora_fwd(x, W, A, B, alpha: float):
    """Forward of the LoRA projection, [P1] 算子融合, eq. ``y = Wx + BAx``.

    Row form: ``v = x·Aᵀ`` (the rank-r down-projection), then
    ``y = x·Wᵀ + s·v·Bᵀ``.  Returns ``y`` [M,n] in fp64.
    """
    x, W, A, B = _f64(x), _f64(W), _f64(A), _f64(B)
    s = lora_scale(alpha, A.shape[0])
    v = x @ A.T
    return x @ W.T + s * (v @ B.T)


def lora_bwd(x, W, A, B, dy, alpha: float):
    """Backward of :func:`lora_fwd`, [P1] 反向传播优化.

    The page prints ``∂L/∂A = ∂L/∂y·xᵀBᵀ`` and ``∂L/∂B = ∂L/∂y·A·xᵀ``; that
    operand order does not type-check and the scale is missing.  Derived
    from the forward instead (W is frozen: only the adapter trains, [P3]
    显存优化策略), with ``v = x·Aᵀ`` recomputed rather than cached as the
    section describes::

        u  = dY·B
        dX = dY·W + s·u·A
        dA = s·uᵀ·x
        dB = s·dYᵀ·v

    Returns ``(dX [M,k], dA [r,k], dB [n,r])`` in fp64.
    """
    x, W, A, B, dy = _f64(x), _f64(W), _f64(A), _f64(B), _f64(dy)
    s = lora_scale(alpha, A.shape[0])
    u = dy @ B
    dx = dy @ W + s * (u @ A)
    dA, dB = lora_adapter_grads(x, A, B, dy, alpha)
    return dx, dA, dB


def lora_adapter_grads(x, A, B, dy, alpha: float):
    """The adapter part of :func:`lora_bwd` alone (no dX):
    ``dA = s·(dY·B)ᵀ·x`` and ``dB = s·dYᵀ·(x·Aᵀ)`` with ``x·Aᵀ`` recomputed."""
    x, A, B, dy = _f64(x), _f64(A), _f64(B), _f64(dy)
    s = lora_scale(alpha, A.shape[0])
    u = dy @ B
    v = x @ A.T                      # recomputed, not taken from the forward
    return s * (u.T @ x), s * (dy.T @ v)


def merged_weight(W, A, B, alpha: float):
    """Adapter merged into the base weight, ``W' = W + s·B·A``
    ([P2] §5.1; [P5] §3.2 "A@B + original_weight")."""
    W, A, B = _f64(W), _f64(A), _f64(B)
    return W + lora_scale(alpha, A.shape[0]) * (B @ A)


def unmerged_weight(Wm, A, B, alpha: float):
    """The inverse of :func:`merged_weight`: ``W = W' − s·B·A`` (taking the
    adapter back out of a merged weight, so training can resume on W)."""
    Wm, A, B = _f64(Wm), _f64(A), _f64(B)
    return Wm - lora_scale(alpha, A.shape[0]) * (B @ A)


def lora_param_count(k: int, n: int, r: int) -> int:
    """Trainable adapter parameters ``r·(k+n)`` ([P3] 显存优化策略)."""
    return int(r) * (int(k) + int(n))


# ---------------------------------------------------------------------------
# bf16 rounding (for the NF4 block scale, which is stored as bf16)
# ---------------------------------------------------------------------------
def bf16_round(a):
    """Round fp64 values to the nearest bfloat16 (ties to even), in fp64.

    bfloat16 keeps 8 significant bits and fp32's exponent range, so the
    spacing of representable values around ``|a|`` is
    ``2**(max(floor(log2|a|), -126) - 7)``; ``np.rint`` rounds half to even.
    Values beyond the largest finite bf16 become ``inf``.
    """
    a = _f64(a)
    out = np.zeros_like(a)
    nz = (a != 0) & np.isfinite(a)
    e = np.floor(np.log2(np.abs(a[nz])))
    e = np.maximum(e, -126.0)
    q = np.exp2(e - 7.0)
    out[nz] = np.rint(a[nz] / q) * q
    out[~np.isfinite(a)] = a[~np.isfinite(a)]
    big = np.abs(out) > 3.3895313892515355e38   # largest finite bf16
    out[big] = np.sign(out[big]) * np.inf
    return out


def f16_round(a):
    """Round fp64 values to the nearest IEEE binary16 (ties to even), in fp64.

    binary16 keeps 11 significant bits with exponents down to -14 (below
    that, subnormals spaced 2**-24), so the spacing around ``|a|`` is
    ``2**(max(floor(log2|a|), -14) - 10)``.  Magnitudes that round past the
    largest finite value 65504 (from 65520 up) become ``inf``.
    """
    a = _f64(a)
    out = np.zeros_like(a)
    nz = (a != 0) & np.isfinite(a)
    e = np.floor(np.log2(np.abs(a[nz])))
    e = np.maximum(e, -14.0)
    q = np.exp2(e - 10.0)
    out[nz] = np.rint(a[nz] / q) * q
    out[~np.isfinite(a)] = a[~np.isfinite(a)]
    big = np.abs(out) > 65504.0
    out[big] = np.sign(out[big]) * np.inf
    return out


def round16(a, dtype: str):
    """Round to the call's 16-bit type: ``"bf16"`` or ``"fp16"``."""
    if dtype == "bf16":
        return bf16_round(a)
    if dtype == "fp16":
        return f16_round(a)
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# NF4 (QLoRA NormalFloat4) — [P3] 显存优化策略, [P5] §3.3/§5, [QLoRA] §3
# ---------------------------------------------------------------------------
def nf4_codebook():
    """The 16 NF4 levels, built as [QLoRA] §3 describes.

    Quantiles of N(0,1) are taken at equally spaced probabilities that stop
    short of the tails by ``delta = (1/32 + 1/30)/2``: 8 levels for the
    positive half (9 points from ``1-delta`` to 1/2, the 1/2 point dropped)
    and 7 for the negative half (8 points, 1/2 dropped), plus an exact zero;
    the set is sorted and divided by its maximum so it spans [-1, 1].
    """
    delta = 0.5 * (1.0 / 32.0 + 1.0 / 30.0)
    hi = 1.0 - delta
    pos = norm.ppf(np.linspace(hi, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(hi, 0.5, 8)[:-1])
    levels = np.sort(np.concatenate([neg, [0.0], pos]))
    return levels / levels.max()


def nf4_quantize(W, blocksize: int = 64, decision: str = "fp64", rows_per_pass=None):
    """Blockwise NF4 quantisation of a row-major ``W [n,k]``.

    Reading (the pages give only the name NormalFloat4): blocks are
    ``blocksize`` consecutive elements along k; the block scale is
    ``absmax = max|w|`` stored as bf16 (round to nearest even); each element
    takes the index of the nearest level of :func:`nf4_codebook` to
    ``w/absmax`` (clamped to [-1,1]; ties to the lower index; a block with
    ``absmax == 0`` is all code 7, the exact zero).  Byte ``j`` of a row
    holds element ``2j`` in its high nibble and ``2j+1`` in its low nibble.

    ``decision`` selects the precision of the nearest-level decision:
    ``"fp64"`` (plain definition) or ``"fp32"`` (IEEE single-precision
    division and distances, the precision a GPU quantiser uses).

    Rows are processed ``rows_per_pass`` at a time (default: about 4M
    elements) only to bound memory; each row's result does not depend on it.

    Returns ``(codes uint8 [n, k/2], absmax float64 [n, k/blocksize])``.
    """
    W = np.asarray(W)
    n, k = W.shape
    assert k % blocksize == 0 and blocksize % 2 == 0
    if decision not in ("fp64", "fp32"):
        raise ValueError(decision)
    levels = nf4_codebook()
    packed = np.empty((n, k // 2), dtype=np.uint8)
    absmax = np.empty((n, k // blocksize), dtype=np.float64)
    rows = rows_per_pass or max(1, (1 << 22) // k)   # bounds the distance array
    for r0 in range(0, n, rows):
        blocks = _f64(W[r0:r0 + rows]).reshape(-1, k // blocksize, blocksize)
        am = bf16_round(np.max(np.abs(blocks), axis=2))
        safe = np.where(am == 0.0, 1.0, am)[:, :, None]
        if decision == "fp64":
            ratio = np.clip(blocks / safe, -1.0, 1.0)
            dist = np.abs(ratio[..., None] - levels)
        else:
            ratio = blocks.astype(np.float32) / safe.astype(np.float32)
            ratio = np.clip(ratio, np.float32(-1.0), np.float32(1.0))
            dist = np.abs(ratio[..., None] - levels.astype(np.float32))
        code = np.argmin(dist, axis=-1).astype(np.uint8)     # first minimum wins
        code[am == 0.0] = 7
        code = code.reshape(-1, k)
        packed[r0:r0 + rows] = (code[:, 0::2] << 4) | code[:, 1::2]
        absmax[r0:r0 + rows] = am
    return packed, absmax


def nf4_unpack(codes):
    """Split packed bytes into 4-bit indices: high nibble first."""
    codes = np.asarray(codes, dtype=np.uint8)
    n, kh = codes.shape
    out = np.empty((n, 2 * kh), dtype=np.uint8)
    out[:, 0::2] = codes >> 4
    out[:, 1::2] = codes & 0xF
    return out


def nf4_dequant(codes, absmax, blocksize: int = 64):
    """``W[i,j] = c[code(i,j)] · absmax[i, j // blocksize]`` in fp64."""
    idx = nf4_unpack(codes)
    absmax = _f64(absmax)
    levels = nf4_codebook()
    scale = np.repeat(absmax, blocksize, axis=1)
    return levels[idx] * scale


# ---------------------------------------------------------------------------
# Double quantisation of the NF4 block scales — [QLoRA] §3, [OCP FP8] E4M3
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0
DQ_GROUP = 256


def e4m3_values():
    """Value of each of the 256 E4M3 codes ([OCP FP8]): sign bit 7, exponent
    bits 6..3 with bias 7, mantissa bits 2..0; exponent 0 is subnormal
    (``m · 2**-9``); exponent 15 with mantissa 7 is NaN (there is no inf), so
    the largest finite magnitude is ``1.75 · 2**8 = 448``."""
    v = np.empty(256, dtype=np.float64)
    for c in range(256):
        e, m = (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            mag = np.nan
        elif e == 0:
            mag = m * 2.0 ** -9
        else:
            mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
        v[c] = -mag if c & 0x80 else mag
    return v


def e4m3_round(a):
    """Nearest E4M3 value to ``a`` (ties to the even mantissa), saturating at
    ±448 (magnitudes from 448 up map to 448, the reading of a saturating
    conversion).  Spacing: ``2**(max(floor(log2|a|), -6) - 3)``."""
    a = _f64(a)
    out = np.zeros_like(a)
    nz = a != 0
    e = np.maximum(np.floor(np.log2(np.abs(a[nz]))), -6.0)
    q = np.exp2(e - 3.0)
    out[nz] = np.rint(a[nz] / q) * q
    return np.clip(out, -E4M3_MAX, E4M3_MAX)


def e4m3_encode(a):
    """E4M3 code (uint8) of :func:`e4m3_round` of ``a``; the sign bit follows
    the sign of ``a`` (a negative value that rounds to zero is code 0x80)."""
    a = _f64(a)
    r = e4m3_round(a)
    table = e4m3_values()
    pos = {float(table[c]): c for c in range(0x7F)}    # finite non-negative codes
    mag = np.vectorize(lambda t: pos[float(t)], otypes=[np.int64])(np.abs(r))
    sign = np.signbit(a).astype(np.int64) << 7
    return (mag | sign).astype(np.uint8)


def dq_encode(c1, group: int = DQ_GROUP):
    """Double quantisation of first-level constants ``c1`` (block order),
    [QLoRA] §3: subtract the mean, then quantise blockwise (``group``
    constants per block) to 8-bit floats, here E4M3.

    Reading of the steps the paper leaves open, in IEEE fp32 (the paper's
    second-level constants are fp32): ``offset = fp32(mean(c1))``;
    ``d = fp32(c1 - offset)``; per group ``scale = fp32(max|d| / 448)`` (448
    being the largest E4M3 magnitude, so the absmax element lands on it);
    ``code = E4M3(fp32(d / scale))`` (0 when ``scale`` is 0).

    Returns ``(codes uint8 [len(c1)], scale float32 [ceil(len/group)],
    offset float32)``.
    """
    c1 = np.asarray(c1, dtype=np.float32).reshape(-1)
    nb = c1.size
    ng = (nb + group - 1) // group
    offset = np.float32(np.mean(c1.astype(np.float64)))
    d = (c1 - offset).astype(np.float32)
    scale = np.empty(ng, dtype=np.float32)
    codes = np.zeros(nb, dtype=np.uint8)
    for g in range(ng):
        dg = d[g * group:(g + 1) * group]
        s = np.float32(np.max(np.abs(dg)) / np.float32(E4M3_MAX))
        scale[g] = s
        if s > 0:
            codes[g * group:(g + 1) * group] = e4m3_encode((dg / s).astype(np.float32))
    return codes, scale, offset


def dq_decode(codes, scale, offset, group: int = DQ_GROUP):
    """Block scales from double-quantised form: ``bf16(fp32(fp32(e4m3(code) ·
    scale[b // group]) + offset))`` (each fp32 operation rounded to nearest;
    the result is rounded to bf16, the type a single-level block scale is
    stored in).  Returned in fp64, same shape as ``codes``."""
    codes = np.asarray(codes, dtype=np.uint8)
    flat = codes.reshape(-1)
    v = e4m3_values()[flat].astype(np.float32)
    s = np.repeat(np.asarray(scale, dtype=np.float32), group)[:flat.size]
    a = (v * s).astype(np.float32) + np.float32(offset)
    return bf16_round(a.astype(np.float32).astype(np.float64)).reshape(codes.shape)


def nf4_quantize_dq(W, blocksize: int = 64, decision: str = "fp32", group: int = DQ_GROUP):
    """NF4 quantisation with double-quantised block scales ([QLoRA] §3).

    The first-level constants are ``c1 = max|w|`` per block (exact);
    :func:`dq_encode` compresses them; the element codes are then chosen as
    in :func:`nf4_quantize` but against the block scale the decoder will use,
    ``dq_decode(...)`` (reading: codes are fitted to the scale they are
    decoded with; w/scale is clamped to [-1, 1], a zero scale gives code 7).

    Returns ``(codes uint8 [n, k/2], absmax_codes uint8 [n, k/blocksize],
    scale float32 [ceil(n·k/blocksize/group)], offset float32)``.
    """
    W = _f64(W)
    n, k = W.shape
    assert k % blocksize == 0
    blocks = W.reshape(n, k // blocksize, blocksize)
    c1 = np.max(np.abs(blocks), axis=2)
    qc, scale, offset = dq_encode(c1, group)
    qc = qc.reshape(n, k // blocksize)
    am = dq_decode(qc, scale, offset, group)
    levels = nf4_codebook()
    safe = np.where(am == 0.0, 1.0, am)[:, :, None]
    if decision == "fp64":
        ratio = np.clip(blocks / safe, -1.0, 1.0)
        dist = np.abs(ratio[..., None] - levels)
    elif decision == "fp32":
        ratio = blocks.astype(np.float32) / safe.astype(np.float32)
        ratio = np.clip(ratio, np.float32(-1.0), np.float32(1.0))
        dist = np.abs(ratio[..., None] - levels.astype(np.float32))
    else:
        raise ValueError(decision)
    code = np.argmin(dist, axis=-1).astype(np.uint8)
    code[am == 0.0] = 7
    code = code.reshape(n, k)
    packed = (code[:, 0::2] << 4) | code[:, 1::2]
    return packed.astype(np.uint8), qc, scale, offset


def nf4_dequant_dq(codes, absmax_codes, scale, offset, blocksize: int = 64,
                   group: int = DQ_GROUP):
    """``W = level[code] · dq_decode(...)`` in fp64 (the decoded scale is
    already a bf16 value)."""
    return nf4_dequant(codes, dq_decode(absmax_codes, scale, offset, group), blocksize)


# ---------------------------------------------------------------------------
# RoPE — [P1] RoPE缓存集成
# ---------------------------------------------------------------------------
def rope_inv_freq(head_dim: int, theta: float):
    """``theta ** (-2i/D)`` for ``i = 0 .. D/2-1`` (reading: Llama/Qwen
    rotary embedding; the section does not state the frequencies)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return float(theta) ** (-2.0 * i / head_dim)


def rope_cos_sin(positions, head_dim: int, theta: float):
    """Per-position cos/sin table ``[len(positions), D/2]`` (the contiguous
    cache of the section), angles ``pos · theta**(-2i/D)`` in fp64."""
    pos = np.asarray(positions, dtype=np.float64)
    ang = pos[:, None] * rope_inv_freq(head_dim, theta)[None, :]
    return np.cos(ang), np.sin(ang)


def rope_apply(y, positions, head_dim: int, theta: float):
    """Rotate each ``head_dim``-wide head of ``y [M, H*D]`` by its row's
    position: pairs ``(i, i+D/2)`` (the rotate-half pairing of Llama/Qwen);
    ``y'[i] = y[i]cos − y[i+D/2]sin``, ``y'[i+D/2] = y[i+D/2]cos + y[i]sin``."""
    y = _f64(y)
    M, N = y.shape
    D, h = head_dim, head_dim // 2
    assert N % D == 0
    c, s = rope_cos_sin(positions, D, theta)
    yh = y.reshape(M, N // D, D)
    a, b = yh[:, :, :h], yh[:, :, h:]
    c, s = c[:, None, :], s[:, None, :]
    out = np.concatenate([a * c - b * s, b * c + a * s], axis=2)
    return out.reshape(M, N)


def rope_apply_inverse(y, positions, head_dim: int, theta: float):
    """Transpose (= inverse) of :func:`rope_apply`: rotation by the negative
    angle.  This is the backward of the rotation."""
    y = _f64(y)
    M, N = y.shape
    D, h = head_dim, head_dim // 2
    c, s = rope_cos_sin(positions, D, theta)
    yh = y.reshape(M, N // D, D)
    a, b = yh[:, :, :h], yh[:, :, h:]
    c, s = c[:, None, :], s[:, None, :]
    out = np.concatenate([a * c + b * s, b * c - a * s], axis=2)
    return out.reshape(M, N)


def qk_rope_fwd(x, Wq, Aq, Bq, Wk, Ak, Bk, alpha, positions, theta,
                head_dim: int = 128):
    """q/k projections with RoPE applied after the LoRA sum
    ([P1] RoPE缓存集成: the rotation happens while computing
    ``q_proj(x) + lora_q(x)``).  Returns ``(q, k)`` in fp64."""
    q = rope_apply(lora_fwd(x, Wq, Aq, Bq, alpha), positions, head_dim, theta)
    k = rope_apply(lora_fwd(x, Wk, Ak, Bk, alpha), positions, head_dim, theta)
    return q, k


def qk_rope_bwd(x, Wq, Aq, Bq, Wk, Ak, Bk, dq, dk, alpha, positions, theta,
                head_dim: int = 128):
    """Backward of :func:`qk_rope_fwd`: undo the rotation on the incoming
    gradients, then :func:`lora_bwd` per projection; dX is summed over q
    and k because both read the same x.

    Returns ``(dX, dAq, dBq, dAk, dBk)`` in fp64."""
    dq_pre = rope_apply_inverse(dq, positions, head_dim, theta)
    dk_pre = rope_apply_inverse(dk, positions, head_dim, theta)
    dxq, dAq, dBq = lora_bwd(x, Wq, Aq, Bq, dq_pre, alpha)
    dxk, dAk, dBk = lora_bwd(x, Wk, Ak, Bk, dk_pre, alpha)
    return dxq + dxk, dAq, dBq, dAk, dBk


# ---------------------------------------------------------------------------
# Gate/up projections with the SwiGLU activation — [P4] §3.1 计算图重写引擎
# (linear layers merged with the activation that follows them), [P5] §1
# 模型结构自识别 (SwiGLU), [SwiGLU] §2
# ---------------------------------------------------------------------------
def sigmoid(t):
    """``1 / (1 + e^{-t})``; for ``t < 0`` evaluated as ``e^t / (1 + e^t)``
    (the same value) so that ``e^{-t}`` never overflows and the small tail
    keeps its relative precision."""
    t = _f64(t)
    e = np.exp(-np.abs(t))                  # in (0, 1]: no overflow
    return np.where(t >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def silu(t):
    """SiLU (Swish_1), ``t·sigmoid(t)`` ([SwiGLU] §2)."""
    t = _f64(t)
    return t * sigmoid(t)


def swiglu_fwd(x, Wg, Ag, Bg, Wu, Au, Bu, alpha: float):
    """The MLP's gate and up LoRA projections of one x, joined by SwiGLU::

        g = x·Wgᵀ + s·(x·Agᵀ)·Bgᵀ      (gate_proj, :func:`lora_fwd`)
        u = x·Wuᵀ + s·(x·Auᵀ)·Buᵀ      (up_proj)
        h = silu(g)·u                  (elementwise; h feeds down_proj)

    Returns ``(h, g, u)`` [M,n] in fp64."""
    g = lora_fwd(x, Wg, Ag, Bg, alpha)
    u = lora_fwd(x, Wu, Au, Bu, alpha)
    return silu(g) * u, g, u


def swiglu_bwd(x, Wg, Ag, Bg, Wu, Au, Bu, dh, alpha: float):
    """Backward of :func:`swiglu_fwd` for an incoming ``dh``.  With
    ``σ = sigmoid(g)`` the chain rule through ``h = g·σ·u`` gives::

        dg = dh·u·σ·(1 + g·(1 − σ))     (d silu(g)/dg = σ + g·σ·(1 − σ))
        du = dh·silu(g)

    then :func:`lora_bwd` of each projection; dX is their sum (both read x).
    g and u are recomputed from the inputs.

    Returns ``(dX, dAg, dBg, dAu, dBu)`` in fp64."""
    g = lora_fwd(x, Wg, Ag, Bg, alpha)
    u = lora_fwd(x, Wu, Au, Bu, alpha)
    dh = _f64(dh)
    sg = sigmoid(g)
    dg = dh * u * sg * (1.0 + g * (1.0 - sg))
    du = dh * g * sg
    dxg, dAg, dBg = lora_bwd(x, Wg, Ag, Bg, dg, alpha)
    dxu, dAu, dBu = lora_bwd(x, Wu, Au, Bu, du, alpha)
    return dxg + dxu, dAg, dBg, dAu, dBu


# ---------------------------------------------------------------------------
# Merging the adapter into an NF4 base weight — [P2] §5.1, [P5] §3.2
# ---------------------------------------------------------------------------
def nf4_merge(codes, absmax, A, B, alpha: float, sign: float = 1.0):
    """NF4 weight with the adapter merged in (``sign`` = +1) or taken out
    (-1): dequantise, add ``sign·s·B·A``, quantise again (:func:`nf4_dequant`,
    :func:`merged_weight`, :func:`nf4_quantize`).  The page describes the
    merge for inference; the NF4 weight is re-quantised because the merged
    weight is no longer representable in the old codes.

    Returns ``(codes, absmax)`` as :func:`nf4_quantize` does."""
    W = nf4_dequant(codes, absmax)
    Wm = merged_weight(W, A, B, alpha) if sign > 0 else unmerged_weight(W, A, B, alpha)
    return nf4_quantize(Wm)


# ---------------------------------------------------------------------------
# LoRA dropout on the adapter input — [P2] §3.3 table (dropout 0.05), [P4]
# §2.2 example (lora_dropout=0.1); mask drawn from [Philox]
# ---------------------------------------------------------------------------
_PHILOX_M = (0xD2E7470EE14C6C93, 0xCA5A826395121157)   # round multipliers
_PHILOX_W = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)   # key increments (Weyl)
_U64 = (1 << 64) - 1


def _mulhilo64(a, b):
    """128-bit product of uint64 arrays a·b as (high, low) words, from 32-bit
    halves (numpy has no 128-bit integers)."""
    a = np.asarray(a, dtype=np.uint64)
    b = np.asarray(b, dtype=np.uint64)
    m32 = np.uint64(0xFFFFFFFF)
    s32 = np.uint64(32)
    a0, a1 = a & m32, a >> s32
    b0, b1 = b & m32, b >> s32
    p00, p01, p10, p11 = a0 * b0, a0 * b1, a1 * b0, a1 * b1   # each < 2^64
    mid = (p00 >> s32) + (p01 & m32) + (p10 & m32)              # < 3·2^32
    lo = (p00 & m32) | ((mid & m32) << s32)
    hi = p11 + (p01 >> s32) + (p10 >> s32) + (mid >> s32)
    return hi, lo


def philox4x64(counter, key, rounds: int = 10):
    """[Philox] Philox4x64-R: four 64-bit counter words and two key words in,
    four 64-bit words out.  Each round multiplies words 0 and 2 by the two
    round multipliers and mixes the halves of the products with words 1 and
    3 and the key (``c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)``); the key
    advances by the two Weyl constants between rounds.  ``counter`` is
    ``[..., 4]`` and ``key`` ``[2]`` (uint64); returns ``[..., 4]`` uint64."""
    c = np.array(counter, dtype=np.uint64, copy=True)
    k0, k1 = np.uint64(key[0]), np.uint64(key[1])
    with np.errstate(over="ignore"):
        for rnd in range(rounds):
            if rnd > 0:
                k0 = k0 + np.uint64(_PHILOX_W[0])
                k1 = k1 + np.uint64(_PHILOX_W[1])
            hi0, lo0 = _mulhilo64(np.uint64(_PHILOX_M[0]), c[..., 0])
            hi1, lo1 = _mulhilo64(np.uint64(_PHILOX_M[1]), c[..., 2])
            c = np.stack([hi1 ^ c[..., 1] ^ k0, lo1, hi0 ^ c[..., 3] ^ k1, lo0], axis=-1)
    return c


def dropout_keep_prob(p: float) -> float:
    """Keep probability of the mask for a dropout rate ``p``: the drop
    threshold is ``t = round(p·65536)`` on 16-bit uniforms, so an element
    is kept with probability ``q = 1 − t/65536``."""
    return 1.0 - round(float(p) * 65536.0) / 65536.0


def dropout_keep(M: int, k: int, p: float, seed: int, offset: int):
    """Keep mask ``[M, k]`` (bool) of LoRA dropout on x [M, k].

    Element ``e = i·k + j`` of x takes 16-bit uniform number ``e mod 16`` of
    the Philox4x64-10 block with counter ``(e // 16, offset, 0, 0)`` and key
    ``(seed, 0)`` (the four 64-bit words read as sixteen 16-bit numbers,
    low half first); it is kept iff that number is at least
    ``round(p·65536)``.  The same (seed, offset) gives the same mask in the
    backward: nothing is stored."""
    n = M * k
    blocks = (n + 15) // 16
    ctr = np.zeros((blocks, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(blocks, dtype=np.uint64)
    ctr[:, 1] = np.uint64(offset)
    words = philox4x64(ctr, (int(seed) & _U64, 0))                  # [blocks, 4]
    u16 = np.stack([(words >> np.uint64(16 * h)) & np.uint64(0xFFFF) for h in range(4)],
                   axis=-1).reshape(blocks * 16)[:n]                  # word w, half h -> 4w+h
    t = round(float(p) * 65536.0)
    return (u16 >= t).reshape(M, k)


def lora_fwd_dropout(x, W, A, B, alpha: float, p: float, seed: int, offset: int):
    """:func:`lora_fwd` with dropout on the adapter's input only (the base
    product sees x unchanged): ``x̃ = x ⊙ keep / q``,
    ``y = x·Wᵀ + s·(x̃·Aᵀ)·Bᵀ``."""
    x = _f64(x)
    keep = dropout_keep(x.shape[0], x.shape[1], p, seed, offset)
    xd = x * keep / dropout_keep_prob(p)
    s = lora_scale(alpha, _f64(A).shape[0])
    return x @ _f64(W).T + s * ((xd @ _f64(A).T) @ _f64(B).T)


def lora_bwd_dropout(x, W, A, B, dy, alpha: float, p: float, seed: int, offset: int):
    """Backward of :func:`lora_fwd_dropout` (mask regenerated from the seed):
    ``u = dY·B``; ``dX = dY·W + s·(u·A) ⊙ keep / q``; ``dA = s·uᵀ·x̃``;
    ``dB = s·dYᵀ·(x̃·Aᵀ)``.  Returns ``(dX, dA, dB)``."""
    x, W, A, B, dy = _f64(x), _f64(W), _f64(A), _f64(B), _f64(dy)
    keep = dropout_keep(x.shape[0], x.shape[1], p, seed, offset)
    q = dropout_keep_prob(p)
    xd = x * keep / q
    s = lora_scale(alpha, A.shape[0])
    u = dy @ B
    dx = dy @ W + s * (u @ A) * keep / q
    return dx, s * (u.T @ xd), s * (dy.T @ (xd @ A.T))

