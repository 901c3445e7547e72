"""GPU parity of the fp16 variants and of double-quantised NF4 block scales
against the fp64 oracle.

fp16: the pages' usage example ("UnSloth加速微调体验") passes
``dtype = torch.float16``, and "Unsloth自动化优化" §3.1 falls back to fp16
where bf16 is unsupported; every entry point takes the call's 16-bit type
from the weight descriptor.  Double quantisation: QLoRA §3 "Double
Quantization" (E4M3 codes of the block scales, one fp32 scale per 256
blocks, the mean subtracted).  Cases: dense / NF4 / NF4 with double
quantisation weights, the one-launch and the rank-pass forward, fused NF4
decode and staged NF4, q/k + RoPE, gate/up + SwiGLU, dropout, merges, the
standalone dequantise / quantise kernels, and one full-size Llama-3-8B
projection."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection, draw_shared_x, draw_tensor
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, np64, rel_err

pytestmark = pytest.mark.gpu

ALPHA = 16.0
F16 = torch.float16
# max|err| / max|ref| for fp16 outputs: one fp16 rounding of the output
# (2^-11 relative), fp16 intermediates s·v / s·u (2^-11 of the adapter
# term) and fp32 accumulation over up to 14336 terms stay well inside this;
# a wrong operand or a bf16 instead of fp16 decode of any input exceeds it
TOL_F16 = 4e-3


def _nf4(W, dtype, dq):
    """NF4 descriptor of the oracle's quantisation of W, the tensors to keep
    alive, and the dequantised weight in fp64."""
    W64 = np64(W)
    if dq:
        codes, qc, scale, off = ref.nf4_quantize_dq(W64)
        c, q = cuda(torch.from_numpy(codes)), cuda(torch.from_numpy(qc))
        s = cuda(torch.from_numpy(scale))
        o = cuda(torch.tensor([off], dtype=torch.float32))
        return (L.nf4_weight(c, q, dtype=dtype, absmax_scale=s, absmax_offset=o), [c, q, s, o],
                ref.nf4_dequant_dq(codes, qc, scale, off))
    codes, absmax = ref.nf4_quantize(W64)
    c = cuda(torch.from_numpy(codes))
    a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
    return L.nf4_weight(c, a, dtype=dtype), [c, a], ref.nf4_dequant(codes, absmax)


def _weight(W, kind, dtype=F16):
    if kind == "dense":
        Wd = cuda(W)
        return L.dense_weight(Wd), [Wd], np64(W)
    return _nf4(W, dtype, kind == "nf4dq")


def _profiled(fn):
    L.lora_profile_begin(64)
    fn()
    torch.cuda.synchronize()
    return [name for name, _ in L.lora_profile_end(64)]


def _flag(kind):
    return L.OP_FLAG_DQ if kind == "nf4dq" else 0


@pytest.mark.parametrize("M,k,n,r,kind", [
    (200, 512, 768, 16, "dense"),       # one wave: x·Aᵀ formed in the GEMM
    (1100, 512, 4096, 64, "dense"),     # rank pass, then the GEMM
    (300, 192, 320, 8, "dense"),        # ragged M and n tails
    (520, 512, 768, 32, "nf4"),         # fused decode
    (520, 512, 768, 32, "nf4dq"),       # fused decode of expanded DQ scales
    (1100, 1024, 512, 16, "nf4dq"),
])
def test_fp16_linear_forward_and_backward(M, k, n, r, kind):
    d = draw_projection(torch.Generator().manual_seed(M + n + r), M, k, n, r, dtype=F16)
    Wd, keep, W64 = _weight(d["W"], kind)
    x, A, B, dy = (cuda(d[t]) for t in ("x", "A", "B", "dY"))
    y = torch.full((M, n), float("nan"), dtype=F16, device="cuda")
    wsf = L.workspace(L.OP_FWD | _flag(kind), M, k, n, r)
    fn = _profiled(lambda: L.lora_linear_fwd(x, Wd, A, B, y, ALPHA, wsf))
    dx = torch.full((M, k), float("nan"), dtype=F16, device="cuda")
    dA = torch.empty(r, k, dtype=torch.float32, device="cuda")
    dB = torch.empty(n, r, dtype=torch.float32, device="cuda")
    wsb = L.workspace(L.OP_BWD | _flag(kind), M, k, n, r)
    bn = _profiled(lambda: L.lora_linear_bwd(x, Wd, A, B, dy, dx, dA, dB, ALPHA, wsb))
    assert L.lora_read_device_status(wsf) == 0 and L.lora_read_device_status(wsb) == 0
    # the fp16 kernels ran
    gemm = [nm for nm in fn + bn if nm.startswith("lora_gemm_pair_kernel")]
    assert gemm and all(("f16" in nm) for nm in gemm), fn + bn
    if kind == "nf4dq":
        assert fn[0] == "nf4_dq_expand_kernel" and bn[0] == "nf4_dq_expand_kernel", (fn, bn)
    x64, A64, B64, dy64 = (np64(d[t]) for t in ("x", "A", "B", "dY"))
    assert rel_err(np64(y), ref.lora_fwd(x64, W64, A64, B64, ALPHA)) <= TOL_F16
    want = ref.lora_bwd(x64, W64, A64, B64, dy64, ALPHA)
    assert rel_err(np64(dx), want[0]) <= TOL_F16
    assert rel_err(np64(dA), want[1]) <= TOL_F32
    assert rel_err(np64(dB), want[2]) <= TOL_F32


@pytest.mark.parametrize("kind,dtype", [("nf4", F16), ("nf4dq", F16), ("nf4dq", torch.bfloat16)])
def test_nf4_staged_in_16_bit(kind, dtype):
    """M >= 2048 with room for the staged copy: W dequantised (double-
    quantised scales decoded on the way) into the workspace, then the
    16-bit kernels."""
    M, k, n, r = 2048, 512, 768, 16
    d = draw_projection(torch.Generator().manual_seed(91), M, k, n, r, dtype=dtype)
    Wd, keep, W64 = _weight(d["W"], kind, dtype)
    x, A, B, dy = (cuda(d[t]) for t in ("x", "A", "B", "dY"))
    y = torch.empty(M, n, dtype=dtype, device="cuda")
    stage = L.lora_nf4_stage_bytes(n, k)
    wsf = L.workspace(L.OP_FWD | _flag(kind), M, k, n, r, extra=stage)
    fn = _profiled(lambda: L.lora_linear_fwd(x, Wd, A, B, y, ALPHA, wsf))
    dx = torch.empty(M, k, dtype=dtype, device="cuda")
    dA = torch.empty(r, k, dtype=torch.float32, device="cuda")
    dB = torch.empty(n, r, dtype=torch.float32, device="cuda")
    wsb = L.workspace(L.OP_BWD | _flag(kind), M, k, n, r, extra=stage)
    bn = _profiled(lambda: L.lora_linear_bwd(x, Wd, A, B, dy, dx, dA, dB, ALPHA, wsb))
    assert L.lora_read_device_status(wsf) == 0 and L.lora_read_device_status(wsb) == 0
    f16 = dtype == F16
    stage_name = "nf4_dequant_kernel" + {(False, False): "", (True, False): "<f16>",
                                         (False, True): "<dq>", (True, True): "<f16,dq>"}[
                                             (f16, kind == "nf4dq")]
    assert fn[0] == stage_name and bn[0] == stage_name, (fn, bn)
    assert not any("nf4" in nm for nm in fn[1:] + bn[1:] if nm.startswith("lora_gemm")), fn + bn
    tol = TOL_F16 if f16 else TOL_BF16
    x64, A64, B64, dy64 = (np64(d[t]) for t in ("x", "A", "B", "dY"))
    assert rel_err(np64(y), ref.lora_fwd(x64, W64, A64, B64, ALPHA)) <= tol
    want = ref.lora_bwd(x64, W64, A64, B64, dy64, ALPHA)
    assert rel_err(np64(dx), want[0]) <= tol
    assert rel_err(np64(dA), want[1]) <= TOL_F32
    assert rel_err(np64(dB), want[2]) <= TOL_F32


@pytest.mark.parametrize("kind", ["dense", "nf4dq"])
def test_fp16_qk_rope_forward_and_backward(kind):
    M, hidden, nqh, nkh, r, theta = 300, 512, 4, 2, 16, 500000.0
    nq, nk = nqh * 128, nkh * 128
    g = torch.Generator().manual_seed(17)
    x = draw_shared_x(g, M, hidden, F16)
    dq_ = draw_projection(g, M, hidden, nq, r, x=x, dtype=F16)
    dk_ = draw_projection(g, M, hidden, nk, r, x=x, dtype=F16)
    Wq, kq, Wq64 = _weight(dq_["W"], kind)
    Wk, kk, Wk64 = _weight(dk_["W"], kind)
    pos = torch.from_numpy(np.random.default_rng(3).integers(0, 4096, M).astype(np.int32))
    posd = cuda(pos)
    xd = cuda(x)
    Aq, Bq, Ak, Bk = (cuda(t) for t in (dq_["A"], dq_["B"], dk_["A"], dk_["B"]))
    q = torch.empty(M, nq, dtype=F16, device="cuda")
    ko = torch.empty(M, nk, dtype=F16, device="cuda")
    ws = L.workspace(L.OP_QK_ROPE_FWD | _flag(kind), M, hidden, nq + nk, r,
                     extra=256 + L.lora_rope_cache_bytes(4096))
    L.lora_qk_rope_fwd(xd, Wq, Aq, Bq, Wk, Ak, Bk, q, ko, ALPHA, theta, posd, None, 4096, ws)
    gq = draw_tensor(g, (M, nq), "normal", 1.0, F16)
    gk = draw_tensor(g, (M, nk), "normal", 1.0, F16)
    dx = torch.empty(M, hidden, dtype=F16, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    dAq, dBq = torch.empty(r, hidden, **f32), torch.empty(nq, r, **f32)
    dAk, dBk = torch.empty(r, hidden, **f32), torch.empty(nk, r, **f32)
    wsb = L.workspace(L.OP_QK_ROPE_BWD | _flag(kind), M, hidden, nq + nk, r,
                      extra=256 + L.lora_rope_cache_bytes(4096))
    L.lora_qk_rope_bwd(xd, Wq, Aq, Bq, Wk, Ak, Bk, cuda(gq), cuda(gk), dx, dAq, dBq, dAk, dBk,
                       ALPHA, theta, posd, None, 4096, wsb)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0 and L.lora_read_device_status(wsb) == 0
    x64 = np64(x)
    P = pos.numpy()
    wq, wk = ref.qk_rope_fwd(x64, Wq64, np64(dq_["A"]), np64(dq_["B"]), Wk64, np64(dk_["A"]),
                             np64(dk_["B"]), ALPHA, P, theta)
    assert rel_err(np64(q), wq) <= TOL_F16 and rel_err(np64(ko), wk) <= TOL_F16
    want = ref.qk_rope_bwd(x64, Wq64, np64(dq_["A"]), np64(dq_["B"]), Wk64, np64(dk_["A"]),
                           np64(dk_["B"]), np64(gq), np64(gk), ALPHA, P, theta)
    assert rel_err(np64(dx), want[0]) <= TOL_F16
    for got, w in zip((dAq, dBq, dAk, dBk), want[1:]):
        assert rel_err(np64(got), w) <= TOL_F32


@pytest.mark.parametrize("kind", ["dense", "nf4", "nf4dq"])
def test_fp16_swiglu_forward_and_backward(kind):
    M, k, n, r = 260, 512, 640, 16
    g = torch.Generator().manual_seed(23)
    x = draw_shared_x(g, M, k, F16)
    gate = draw_projection(g, M, k, n, r, x=x, dtype=F16)
    up = draw_projection(g, M, k, n, r, x=x, dtype=F16)
    Wg, kg, Wg64 = _weight(gate["W"], kind)
    Wu, ku, Wu64 = _weight(up["W"], kind)
    xd = cuda(x)
    Ag, Bg, Au, Bu = (cuda(t) for t in (gate["A"], gate["B"], up["A"], up["B"]))
    h, gg, uu = (torch.empty(M, n, dtype=F16, device="cuda") for _ in range(3))
    ws = L.workspace(L.OP_SWIGLU_FWD | _flag(kind), M, k, n, r)
    L.lora_swiglu_fwd(xd, Wg, Ag, Bg, Wu, Au, Bu, h, ALPHA, ws, g=gg, u=uu)
    dh = draw_tensor(g, (M, n), "normal", 1.0, F16)
    dx = torch.empty(M, k, dtype=F16, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    dAg, dBg = torch.empty(r, k, **f32), torch.empty(n, r, **f32)
    dAu, dBu = torch.empty(r, k, **f32), torch.empty(n, r, **f32)
    wsb = L.workspace(L.OP_SWIGLU_BWD | _flag(kind), M, k, n, r)
    L.lora_swiglu_bwd(xd, Wg, Ag, Bg, Wu, Au, Bu, gg, uu, cuda(dh), dx, dAg, dBg, dAu, dBu,
                      ALPHA, wsb)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0 and L.lora_read_device_status(wsb) == 0
    x64 = np64(x)
    args = (x64, Wg64, np64(gate["A"]), np64(gate["B"]), Wu64, np64(up["A"]), np64(up["B"]))
    hw, gw, uw = ref.swiglu_fwd(*args, ALPHA)
    assert rel_err(np64(h), hw) <= TOL_F16
    assert rel_err(np64(gg), gw) <= TOL_F16 and rel_err(np64(uu), uw) <= TOL_F16
    want = ref.swiglu_bwd(*args, np64(dh), ALPHA)
    assert rel_err(np64(dx), want[0]) <= TOL_F16
    for got, w in zip((dAg, dBg, dAu, dBu), want[1:]):
        assert rel_err(np64(got), w) <= TOL_F32


def test_fp16_dropout_forward_and_backward():
    M, k, n, r, p, seed, off = 300, 512, 768, 16, 0.1, 99, 3
    d = draw_projection(torch.Generator().manual_seed(29), M, k, n, r, dtype=F16)
    x, W, A, B, dy = (cuda(d[t]) for t in ("x", "W", "A", "B", "dY"))
    y = torch.empty(M, n, dtype=F16, device="cuda")
    ws = L.workspace(L.OP_FWD_DROPOUT, M, k, n, r)
    L.lora_linear_fwd_dropout(x, W, A, B, y, ALPHA, p, seed, off, ws)
    dx = torch.empty(M, k, dtype=F16, device="cuda")
    dA = torch.empty(r, k, dtype=torch.float32, device="cuda")
    dB = torch.empty(n, r, dtype=torch.float32, device="cuda")
    wsb = L.workspace(L.OP_BWD_DROPOUT, M, k, n, r)
    L.lora_linear_bwd_dropout(x, W, A, B, dy, dx, dA, dB, ALPHA, p, seed, off, wsb)
    torch.cuda.synchronize()
    x64, W64, A64, B64, dy64 = (np64(d[t]) for t in ("x", "W", "A", "B", "dY"))
    assert rel_err(np64(y), ref.lora_fwd_dropout(x64, W64, A64, B64, ALPHA, p, seed, off)) \
        <= TOL_F16
    want = ref.lora_bwd_dropout(x64, W64, A64, B64, dy64, ALPHA, p, seed, off)
    assert rel_err(np64(dx), want[0]) <= TOL_F16
    assert rel_err(np64(dA), want[1]) <= TOL_F32 and rel_err(np64(dB), want[2]) <= TOL_F32


def test_fp16_merge_and_unmerge_of_a_dense_weight():
    n, k, r = 320, 1024, 16
    d = draw_projection(torch.Generator().manual_seed(31), 1, k, n, r, dtype=F16)
    W, A, B = cuda(d["W"]), cuda(d["A"]), cuda(d["B"])
    L.lora_merge(W, A, B, ALPHA, sign=1)
    torch.cuda.synchronize()
    want = ref.merged_weight(np64(d["W"]), np64(d["A"]), np64(d["B"]), ALPHA)
    # one fp16 rounding of the fp32 sum per element
    assert np.all(np.abs(np64(W) - want) <= np.abs(want) * 2.0 ** -10 + 2.0 ** -24)


@pytest.mark.parametrize("n,k,dtype", [(64, 64, torch.bfloat16), (320, 512, F16),
                                       (1024, 4096, torch.bfloat16), (512, 2048, F16)])
def test_nf4_dequant_of_double_quantised_scales(n, k, dtype):
    g = torch.Generator().manual_seed(n + k)
    W = draw_tensor(g, (n, k), "normal", 1.0 / np.sqrt(k))
    W[0, :64] = 0                                          # an all-zero block
    codes, qc, scale, off = ref.nf4_quantize_dq(np64(W))
    out = torch.empty(n, k, dtype=dtype, device="cuda")
    c_t = cuda(torch.from_numpy(codes))
    q_t = cuda(torch.from_numpy(qc))
    s_t = cuda(torch.from_numpy(scale))
    o_t = cuda(torch.tensor([off], dtype=torch.float32))
    Wd = L.nf4_weight(c_t, q_t, dtype=dtype, absmax_scale=s_t, absmax_offset=o_t)
    L.nf4_dequant(Wd, out)
    torch.cuda.synchronize()
    want = ref.nf4_dequant_dq(codes, qc, scale, off)
    got = np64(out)
    ulp = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11
    assert np.all(np.abs(got - want) <= np.abs(want) * ulp + 1e-30)
    # elements on the ±1 levels are exactly ± the decoded block scale
    idx = ref.nf4_unpack(codes)
    am = np.repeat(ref.dq_decode(qc, scale, off), 64, axis=1)
    ends = (idx == 0) | (idx == 15)
    if dtype == torch.bfloat16:
        np.testing.assert_array_equal(np.abs(got[ends]), am[ends])
    assert np.all(got[0, :64] == 0)


@pytest.mark.parametrize("n,k,dtype", [(64, 256, torch.bfloat16), (320, 1024, F16),
                                       (1024, 4096, torch.bfloat16)])
def test_nf4_quantize_with_double_quantisation(n, k, dtype):
    """Scale codes, group scales and the offset equal the oracle's (both take
    the decisions in fp32); element codes too, except at exact near-ties."""
    g = torch.Generator().manual_seed(7 * n + k)
    W = draw_tensor(g, (n, k), "normal", 1.0 / np.sqrt(k), dtype)
    W[1, 64:128] = 0
    codes_ref, qc_ref, scale_ref, off_ref = ref.nf4_quantize_dq(np64(W), decision="fp32")
    nb = n * k // 64
    codes = torch.empty(n, k // 2, dtype=torch.uint8, device="cuda")
    qc = torch.empty(n, k // 64, dtype=torch.uint8, device="cuda")
    scale = torch.empty((nb + 255) // 256, dtype=torch.float32, device="cuda")
    off = torch.empty(1, dtype=torch.float32, device="cuda")
    L.nf4_quantize(cuda(W), L.nf4_weight(codes, qc, dtype=dtype, absmax_scale=scale,
                                         absmax_offset=off))
    torch.cuda.synchronize()
    assert float(off.item()) == float(off_ref)
    np.testing.assert_array_equal(scale.cpu().numpy(), scale_ref)
    np.testing.assert_array_equal(qc.cpu().numpy(), qc_ref)
    gi, ri = ref.nf4_unpack(codes.cpu().numpy()), ref.nf4_unpack(codes_ref)
    diff = np.argwhere(gi != ri)
    am = ref.dq_decode(qc_ref, scale_ref, off_ref)
    lv = ref.nf4_codebook()
    w = np64(W)
    for i, j in diff:
        t = w[i, j] / am[i, j // 64]
        assert abs(abs(t - lv[gi[i, j]]) - abs(t - lv[ri[i, j]])) < 1e-6
    assert len(diff) <= 1e-4 * n * k


def test_merge_into_a_double_quantised_nf4_weight():
    n, k, r = 512, 1024, 16
    d = draw_projection(torch.Generator().manual_seed(37), 1, k, n, r)
    codes, qc, scale, off = ref.nf4_quantize_dq(np64(d["W"]))
    c, q = cuda(torch.from_numpy(codes)), cuda(torch.from_numpy(qc))
    s, o = cuda(torch.from_numpy(scale)), cuda(torch.tensor([off], dtype=torch.float32))
    L.lora_merge(L.nf4_weight(c, q, absmax_scale=s, absmax_offset=o), cuda(d["A"]),
                 cuda(d["B"]), ALPHA)
    torch.cuda.synchronize()
    got = ref.nf4_dequant_dq(c.cpu().numpy(), q.cpu().numpy(), s.cpu().numpy(), o.item())
    Wm = ref.merged_weight(ref.nf4_dequant_dq(codes, qc, scale, off), np64(d["A"]),
                           np64(d["B"]), ALPHA)
    # within NF4's bound against the new decoded scale, plus the scale's own
    # shortfall and the bf16 rounding of the merged value
    c1 = np.repeat(np.max(np.abs(ref.bf16_round(Wm).reshape(n, k // 64, 64)), axis=2), 64,
                   axis=1)
    am = np.repeat(ref.dq_decode(q.cpu().numpy(), s.cpu().numpy(), o.item()), 64, axis=1)
    gap = np.max(np.diff(ref.nf4_codebook())) / 2
    bound = np.maximum(c1 - am, 0.0) + am * gap * (1 + 2.0 ** -7) + np.abs(Wm) * 2.0 ** -7
    assert np.all(np.abs(got - Wm) <= bound)


def test_full_size_fp16_double_quantised_llama8b_gate_proj():
    """Llama-3-8B gate_proj 4096 -> 14336 at M = 4096, fp16, NF4 with double
    quantisation, fused decode (exact-size workspace): y and dX on 256
    sampled rows, dA and dB in full."""
    M, k, n, r = 4096, 4096, 14336, 16
    d = draw_projection(torch.Generator().manual_seed(43), M, k, n, r, dtype=F16)
    Wd, keep, W64 = _weight(d["W"], "nf4dq")
    x, A, B, dy = (cuda(d[t]) for t in ("x", "A", "B", "dY"))
    y = torch.empty(M, n, dtype=F16, device="cuda")
    dx = torch.empty(M, k, dtype=F16, device="cuda")
    dA = torch.empty(r, k, dtype=torch.float32, device="cuda")
    dB = torch.empty(n, r, dtype=torch.float32, device="cuda")
    wsf = L.workspace(L.OP_FWD | L.OP_FLAG_DQ, M, k, n, r)
    wsb = L.workspace(L.OP_BWD | L.OP_FLAG_DQ, M, k, n, r)
    L.lora_linear_fwd(x, Wd, A, B, y, ALPHA, wsf)
    L.lora_linear_bwd(x, Wd, A, B, dy, dx, dA, dB, ALPHA, wsb)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsf) == 0 and L.lora_read_device_status(wsb) == 0
    rows = np.sort(np.random.default_rng(5).choice(M, 256, replace=False))
    x64, A64, B64, dy64 = (np64(d[t]) for t in ("x", "A", "B", "dY"))
    s = ALPHA / r
    y_want = x64[rows] @ W64.T + s * (x64[rows] @ A64.T) @ B64.T
    assert rel_err(np64(y)[rows], y_want) <= TOL_F16
    dx_want = dy64[rows] @ W64 + s * (dy64[rows] @ B64) @ A64
    assert rel_err(np64(dx)[rows], dx_want) <= TOL_F16
    assert rel_err(np64(dA), s * (dy64 @ B64).T @ x64) <= TOL_F32
    assert rel_err(np64(dB), s * dy64.T @ (x64 @ A64.T)) <= TOL_F32
