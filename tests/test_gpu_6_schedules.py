"""GPU parity of the schedule variants the host picks by shape, each asserted
to have run (kernel names from the library's per-launch timing session):

* the NF4 fused GEMM with two m-blocks per tile (each decoded W K-block
  feeding 512 rows) in the forward and in dX, with a ragged second m-block;
* NF4 weights holding an all-zero 64-block (absmax 0) and a block whose
  absmax is a bf16 subnormal, through the fused forward and dX;
* the rank passes on their cluster schedule and on their stream-K schedule.
"""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, np64, rel_err

pytestmark = pytest.mark.gpu

ALPHA = 16.0


def _nf4(W):
    codes, absmax = ref.nf4_quantize(np64(W))
    c = cuda(torch.from_numpy(codes))
    a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
    return codes, absmax, c, a


def _profiled(fn, cap=16):
    L.lora_profile_begin(cap)
    try:
        fn()
    finally:
        got = L.lora_profile_end(cap)
    return [name for name, _ in got]


def _fwd(d, W, r):
    x, A, B = cuda(d["x"]), cuda(d["A"]), cuda(d["B"])
    M, k = x.shape
    n = d["W"].shape[0]
    y = torch.full((M, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = L.workspace(L.OP_FWD, M, k, n, r)
    names = _profiled(lambda: L.lora_linear_fwd(x, W, A, B, y, ALPHA, ws))
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0
    return y, names


def _bwd(d, W, r):
    x, A, B, dy = cuda(d["x"]), cuda(d["A"]), cuda(d["B"]), cuda(d["dY"])
    M, k = x.shape
    n = dy.shape[1]
    dx = torch.full((M, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    dA = torch.full((r, k), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((n, r), float("nan"), dtype=torch.float32, device="cuda")
    ws = L.workspace(L.OP_BWD, M, k, n, r)
    names = _profiled(lambda: L.lora_linear_bwd(x, W, A, B, dy, dx, dA, dB, ALPHA, ws))
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0
    return (dx, dA, dB), names


def test_nf4_forward_with_two_m_blocks_per_tile():
    # 2 m-blocks (the second holds 44 rows) x 74 n-tiles (the last 64 wide):
    # one wave of 512-row tiles beats two waves of 256-row tiles
    M, k, n, r = 300, 512, 74 * 256 - 192, 16
    d = draw_projection(torch.Generator().manual_seed(61), M, k, n, r)
    codes, absmax, c, a = _nf4(d["W"])
    y, names = _fwd(d, L.nf4_weight(c, a), r)
    assert names[-1] == "lora_gemm_pair_kernel<fwd,nf4,mb2>", names
    want = ref.lora_fwd(np64(d["x"]), ref.nf4_dequant(codes, absmax), np64(d["A"]),
                        np64(d["B"]), ALPHA)
    assert rel_err(np64(y), want) <= TOL_BF16


def test_nf4_backward_dx_with_two_m_blocks_per_tile():
    M, k, n, r = 300, 74 * 256 - 192, 512, 16
    d = draw_projection(torch.Generator().manual_seed(62), M, k, n, r)
    codes, absmax, c, a = _nf4(d["W"])
    got, names = _bwd(d, L.nf4_weight(c, a), r)
    assert "lora_gemm_pair_kernel<dx,nf4,mb2>" in names, names
    want = ref.lora_bwd(np64(d["x"]), ref.nf4_dequant(codes, absmax), np64(d["A"]),
                        np64(d["B"]), np64(d["dY"]), ALPHA)
    assert rel_err(np64(got[0]), want[0]) <= TOL_BF16
    assert rel_err(np64(got[1]), want[1]) <= TOL_F32
    assert rel_err(np64(got[2]), want[2]) <= TOL_F32


@pytest.mark.parametrize("M,k,n", [(16, 512, 320), (200, 512, 320), (300, 512, 74 * 256 - 192)])
def test_nf4_zero_and_subnormal_blocks_in_the_fused_gemms(M, k, n):
    """An all-zero 64-block (absmax 0, every code 7) and a block of bf16
    subnormals decode to zero / tiny values inside the fused forward and dX
    (one- and two-m-block tiles; at 16 tokens the forward's decoding pass)."""
    r = 16
    d = draw_projection(torch.Generator().manual_seed(63), M, k, n, r)
    W = d["W"].clone()
    W[0, :64] = 0
    W[1, 64:128] = (torch.arange(64, dtype=torch.float32) - 32.0) * 1e-40
    W[2:, 128:192] = 0
    d["W"] = W
    codes, absmax, c, a = _nf4(W)
    assert absmax[0, 0] == 0.0 and 0.0 < absmax[1, 1] < 1.17e-38
    Wq = ref.nf4_dequant(codes, absmax)
    y, _ = _fwd(d, L.nf4_weight(c, a), r)
    want = ref.lora_fwd(np64(d["x"]), Wq, np64(d["A"]), np64(d["B"]), ALPHA)
    assert np.isfinite(np64(y)).all()
    assert rel_err(np64(y), want) <= TOL_BF16
    # dX over the same W: as the reduction operand (n rows of W)
    db = draw_projection(torch.Generator().manual_seed(64), M, k, n, r)
    db["W"] = W
    got, _ = _bwd(db, L.nf4_weight(c, a), r)
    want = ref.lora_bwd(np64(db["x"]), Wq, np64(db["A"]), np64(db["B"]), np64(db["dY"]), ALPHA)
    assert np.isfinite(np64(got[0])).all()
    assert rel_err(np64(got[0]), want[0]) <= TOL_BF16


@pytest.mark.parametrize("M,k,n,r,schedule", [
    (2048, 2048, 2048, 64, "lora_skinny_kernel"),     # even tiles: cluster split-K
    (1024, 4096, 4096, 16, "lora_skinny_sk_kernel"),  # few long rank-16 tiles: stream-K
])
def test_rank_pass_schedule_runs_and_matches(M, k, n, r, schedule):
    d = draw_projection(torch.Generator().manual_seed(65), M, k, n, r)
    Wd = cuda(d["W"])
    y, fnames = _fwd(d, L.bf16_weight(Wd), r)
    got, bnames = _bwd(d, L.bf16_weight(Wd), r)
    # the bf16 forward forms s·x·Aᵀ in its GEMM; the backward has two rank passes
    assert not any(nm.startswith("lora_skinny") for nm in fnames), fnames
    rank = [nm for nm in bnames if nm.startswith("lora_skinny")]
    assert len(rank) == 2 and all(nm.startswith(schedule + "<") for nm in rank), rank
    x, W, A, B, dY = (np64(d[t]) for t in ("x", "W", "A", "B", "dY"))
    rows = np.random.default_rng(0).choice(M, 256, replace=False)
    assert rel_err(np64(y)[rows], ref.lora_fwd(x[rows], W, A, B, ALPHA)) <= TOL_BF16
    dx, dA, dB = ref.lora_bwd(x, W, A, B, dY, ALPHA)
    assert rel_err(np64(got[0])[rows], dx[rows]) <= TOL_BF16
    assert rel_err(np64(got[1]), dA) <= TOL_F32
    assert rel_err(np64(got[2]), dB) <= TOL_F32


@pytest.mark.parametrize("M,k,n,r,fused", [
    (700, 1024, 2048, 16, True),     # 3 x 8 tiles: one wave of pairs
    (257, 256, 768, 64, True),
    (2304, 512, 4096, 64, False),    # 9 x 16 tiles: more than one wave
])
def test_bf16_forward_launches(M, k, n, r, fused):
    """A bf16 forward whose tiles fit in one wave of CTA pairs forms s·x·Aᵀ
    inside the fused GEMM ("UnSloth加速微调体验" §算子融合: one pass, no
    intermediate): one launch, s·v only in shared memory.  Larger ones run
    the rank pass first (the measured faster form on B300)."""
    d = draw_projection(torch.Generator().manual_seed(66), M, k, n, r)
    Wd = cuda(d["W"])
    y, names = _fwd(d, L.bf16_weight(Wd), r)
    if fused:
        assert names == ["lora_gemm_pair_kernel<fwd,bf16,xa>"], names
    else:
        assert len(names) == 2 and names[0].startswith("lora_skinny"), names
        assert names[1] == "lora_gemm_pair_kernel<fwd,bf16>", names
    want = ref.lora_fwd(np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]), ALPHA)
    assert rel_err(np64(y), want) <= TOL_BF16


def _nf4_ws(op, M, k, n, r, stage_rows):
    extra = sum(L.lora_nf4_stage_bytes(rows, k) for rows in stage_rows)
    return L.workspace(op, M, k, n, r, extra=extra)


@pytest.mark.parametrize("stage", [True, False])
def test_nf4_linear_staged_in_bf16_when_the_workspace_has_room(stage):
    """M >= 2048 and room past the workspace: W is dequantised once into it
    and the bf16 kernels run; otherwise the codes are decoded in the GEMMs."""
    M, k, n, r = 2048, 512, 768, 16
    d = draw_projection(torch.Generator().manual_seed(67), M, k, n, r)
    codes, absmax, c, a = _nf4(d["W"])
    W = L.nf4_weight(c, a)
    x, A, B, dy = cuda(d["x"]), cuda(d["A"]), cuda(d["B"]), cuda(d["dY"])
    y = torch.empty(M, n, dtype=torch.bfloat16, device="cuda")
    wsf = _nf4_ws(L.OP_FWD, M, k, n, r, [n] if stage else [])
    fn = _profiled(lambda: L.lora_linear_fwd(x, W, A, B, y, ALPHA, wsf))
    dx = torch.empty(M, k, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(r, k, dtype=torch.float32, device="cuda")
    dB = torch.empty(n, r, dtype=torch.float32, device="cuda")
    wsb = _nf4_ws(L.OP_BWD, M, k, n, r, [n] if stage else [])
    bn = _profiled(lambda: L.lora_linear_bwd(x, W, A, B, dy, dx, dA, dB, ALPHA, wsb))
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsf) == 0 and L.lora_read_device_status(wsb) == 0
    if stage:
        assert fn[0] == "nf4_dequant_kernel", fn
        assert any(nm.startswith("lora_gemm_pair_kernel<fwd,bf16") for nm in fn), fn
        assert bn[0] == "nf4_dequant_kernel" and "lora_gemm_pair_kernel<dx,bf16>" in bn, bn
    else:
        assert "nf4_dequant_kernel" not in fn + bn
        assert any(nm.startswith("lora_gemm_pair_kernel<fwd,nf4") for nm in fn), fn
    Wq = ref.nf4_dequant(codes, absmax)
    x64, A64, B64 = np64(d["x"]), np64(d["A"]), np64(d["B"])
    assert rel_err(np64(y), ref.lora_fwd(x64, Wq, A64, B64, ALPHA)) <= TOL_BF16
    want = ref.lora_bwd(x64, Wq, A64, B64, np64(d["dY"]), ALPHA)
    assert rel_err(np64(dx), want[0]) <= TOL_BF16
    assert rel_err(np64(dA), want[1]) <= TOL_F32 and rel_err(np64(dB), want[2]) <= TOL_F32


def test_nf4_qk_pair_staged_in_bf16():
    """Both weights of the q/k pair staged (q then k) for the forward with
    RoPE and the merged backward."""
    from lora_inputs import draw_shared_x
    M, hidden, r, theta = 2048, 256, 16, 500000.0
    g = torch.Generator().manual_seed(68)
    x = draw_shared_x(g, M, hidden)
    q = draw_projection(g, M, hidden, 256, r, x=x)
    k = draw_projection(g, M, hidden, 128, r, x=x)
    (cq, aq, cqd, aqd), (ck, ak, ckd, akd) = _nf4(q["W"]), _nf4(k["W"])
    Wq, Wk = L.nf4_weight(cqd, aqd), L.nf4_weight(ckd, akd)
    pos = np.arange(M)
    posd = cuda(torch.as_tensor(pos, dtype=torch.int32))
    cache = torch.empty(M, 128, dtype=torch.float32, device="cuda")
    L.lora_rope_cache_build(cache, M, 128, theta)
    yq = torch.empty(M, 256, dtype=torch.bfloat16, device="cuda")
    yk = torch.empty(M, 128, dtype=torch.bfloat16, device="cuda")
    wsf = _nf4_ws(L.OP_QK_ROPE_FWD, M, hidden, 384, r, [256, 128])
    dev = {t: cuda(v) for t, v in (("x", x), ("Aq", q["A"]), ("Bq", q["B"]), ("Ak", k["A"]),
                                    ("Bk", k["B"]), ("dq", q["dY"]), ("dk", k["dY"]))}
    fn = _profiled(lambda: L.lora_qk_rope_fwd(dev["x"], Wq, dev["Aq"], dev["Bq"], Wk, dev["Ak"],
                                              dev["Bk"], yq, yk, ALPHA, theta, posd, cache, M,
                                              wsf))
    assert fn[:2] == ["nf4_dequant_kernel", "nf4_dequant_kernel"], fn
    dx = torch.empty(M, hidden, dtype=torch.bfloat16, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    grads = [torch.empty(s, **f32) for s in ((r, hidden), (256, r), (r, hidden), (128, r))]
    wsb = _nf4_ws(L.OP_QK_ROPE_BWD, M, hidden, 384, r, [256, 128])
    L.lora_qk_rope_bwd(dev["x"], Wq, dev["Aq"], dev["Bq"], Wk, dev["Ak"], dev["Bk"], dev["dq"],
                       dev["dk"], dx, *grads, ALPHA, theta, posd, cache, M, wsb)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsf) == 0 and L.lora_read_device_status(wsb) == 0
    Wq64, Wk64 = ref.nf4_dequant(cq, aq), ref.nf4_dequant(ck, ak)
    P = (np64(x), Wq64, np64(q["A"]), np64(q["B"]), Wk64, np64(k["A"]), np64(k["B"]))
    wq, wk = ref.qk_rope_fwd(*P, ALPHA, pos, theta)
    assert rel_err(np64(yq), wq) <= TOL_BF16 and rel_err(np64(yk), wk) <= TOL_BF16
    want = ref.qk_rope_bwd(*P, np64(q["dY"]), np64(k["dY"]), ALPHA, pos, theta)
    assert rel_err(np64(dx), want[0]) <= TOL_BF16
    for got, w in zip(grads, want[1:]):
        assert rel_err(np64(got), w) <= TOL_F32


@pytest.mark.parametrize("M,k,n,r,dtype,kind", [
    (1, 512, 768, 16, torch.bfloat16, "dense"),       # a single token
    (16, 1024, 2048, 64, torch.bfloat16, "dense"),
    (37, 4096, 1024, 8, torch.float16, "dense"),      # ragged token count
    (64, 512, 4096, 32, torch.bfloat16, "dense"),
    (100, 2048, 640, 16, torch.float16, "dense"),     # M in (64, 128]: tokens padded to 128
    (128, 320, 1280, 64, torch.bfloat16, "dense"),
    (1, 1024, 768, 16, torch.bfloat16, "nf4"),
    (16, 4096, 1088, 64, torch.bfloat16, "nf4"),      # W rows not a multiple of 128
    (50, 2048, 2048, 8, torch.float16, "nf4"),
    (100, 576, 640, 32, torch.bfloat16, "nf4"),
    (96, 3072, 1024, 16, torch.bfloat16, "nf4"),      # 96 token columns, 6 CTAs per tile
    (72, 1536, 2560, 32, torch.float16, "nf4"),       # 96 token columns, 3 CTAs per tile
    (24, 1024, 1536, 16, torch.bfloat16, "nf4dq"),
])
def test_small_m_forward_runs_over_the_rows_of_w(M, k, n, r, dtype, kind):
    """With at most 128 tokens the forward is one rank-pass launch over the
    rows of W and of A (yᵀ = W·xᵀ and (s·v)ᵀ = s·A·xᵀ, the reduction split
    across a cluster, so every SM streams a share of W; an NF4 W is decoded
    from its codes inside that launch), then the GEMM adding (s·v)·Bᵀ to y
    in its epilogue."""
    d = draw_projection(torch.Generator().manual_seed(M + k), M, k, n, r, dtype=dtype)
    x, A, B = (cuda(d[t]) for t in ("x", "A", "B"))
    flag = 0
    if kind == "dense":
        Wt = cuda(d["W"])
        Wd, keep, W64 = L.dense_weight(Wt), [Wt], np64(d["W"])
    elif kind == "nf4":
        codes, absmax = ref.nf4_quantize(np64(d["W"]))
        c = cuda(torch.from_numpy(codes))
        a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
        Wd, keep, W64 = L.nf4_weight(c, a, dtype=dtype), [c, a], ref.nf4_dequant(codes, absmax)
    else:
        codes, qc, sc, off = ref.nf4_quantize_dq(np64(d["W"]))
        keep = [cuda(torch.from_numpy(codes)), cuda(torch.from_numpy(qc)),
                cuda(torch.from_numpy(sc)), cuda(torch.tensor([off], dtype=torch.float32))]
        Wd = L.nf4_weight(keep[0], keep[1], dtype=dtype, absmax_scale=keep[2],
                          absmax_offset=keep[3])
        W64 = ref.nf4_dequant_dq(codes, qc, sc, off)
        flag = L.OP_FLAG_DQ
    y = torch.full((M, n), float("nan"), dtype=dtype, device="cuda")
    ws = L.workspace(L.OP_FWD | flag, M, k, n, r)
    names = _profiled(lambda: L.lora_linear_fwd(x, Wd, A, B, y, ALPHA, ws))
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0
    f16 = ",f16" if dtype == torch.float16 else ""
    variant = ",nf4" if kind != "dense" else (",2cta" if M <= 64 else "")
    want_names = (["nf4_dq_expand_kernel"] if kind == "nf4dq" else []) + [
        "lora_skinny_kernel<k_major" + variant + f16 + ">",
        "lora_gemm_pair_kernel<fwd," + ("f16" if f16 else "bf16") + ">"]
    assert names == want_names, names
    want = ref.lora_fwd(np64(d["x"]), W64, np64(d["A"]), np64(d["B"]), ALPHA)
    tol = TOL_BF16 if dtype == torch.bfloat16 else 4e-3
    assert rel_err(np64(y), want) <= tol
