"""GPU parity of the fused backward (dX, dA, dB with x·Aᵀ recomputed)."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, dump, np64, rel_err

pytestmark = pytest.mark.gpu

SHAPES = [  # M, k, n, r
    (256, 512, 512, 8),
    (128, 64, 256, 16),
    (200, 192, 320, 16),
    (130, 512, 1024, 32),
    (257, 256, 768, 64),
    (1, 128, 64, 8),
    (700, 1024, 2048, 16),
]


def run_bwd(d, alpha, nf4=None, accumulate=False, dx0=None):
    x, A, B, dy = cuda(d["x"]), cuda(d["A"]), cuda(d["B"]), cuda(d["dY"])
    M, k = x.shape
    n, r = dy.shape[1], A.shape[0]
    keep = []
    if nf4 is None:
        Wd = cuda(d["W"])
        W = L.bf16_weight(Wd)
        keep.append(Wd)
    else:
        codes, absmax = nf4
        c = cuda(torch.from_numpy(codes))
        a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
        W = L.nf4_weight(c, a)
        keep += [c, a]
    dx = cuda(dx0) if dx0 is not None else torch.full((M, k), float("nan"),
                                                      dtype=torch.bfloat16, device="cuda")
    dA = torch.full((r, k), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((n, r), float("nan"), dtype=torch.float32, device="cuda")
    ws = L.workspace(L.OP_BWD, M, k, n, r)
    L.lora_linear_bwd(x, W, A, B, dy, dx, dA, dB, alpha, ws, accumulate_dx=accumulate)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0
    return dx, dA, dB


def _check(tag, d, got, want):
    errs = [rel_err(np64(g), w) for g, w in zip(got, want)]
    ok = errs[0] <= TOL_BF16 and errs[1] <= TOL_F32 and errs[2] <= TOL_F32
    if not ok:
        dump(tag, x=d["x"], A=d["A"], B=d["B"], dY=d["dY"], dx=got[0], dA=got[1], dB=got[2],
             dx_ref=want[0], dA_ref=want[1], dB_ref=want[2])
    assert ok, errs


@pytest.mark.parametrize("M,k,n,r", SHAPES)
def test_bwd_bf16_parity(M, k, n, r):
    g = torch.Generator().manual_seed(M + 3 * k + n + r)
    d = draw_projection(g, M, k, n, r)
    got = run_bwd(d, 16.0)
    want = ref.lora_bwd(np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]), np64(d["dY"]),
                        16.0)
    _check(f"bwd_{M}_{k}_{n}_{r}", d, got, want)


def test_bwd_accumulates_dx():
    M, k, n, r = 200, 256, 320, 16
    g = torch.Generator().manual_seed(99)
    d = draw_projection(g, M, k, n, r)
    dx0 = torch.randn(M, k, generator=g).to(torch.bfloat16)
    got = run_bwd(d, 16.0, accumulate=True, dx0=dx0)
    dx, dA, dB = ref.lora_bwd(np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]),
                              np64(d["dY"]), 16.0)
    _check("bwd_acc", d, got, (dx + np64(dx0), dA, dB))


def test_bwd_b_zero_gives_plain_gradients():
    """B = 0: dX = dY·W and dA = 0 exactly; dB = s·dYᵀ·(x·Aᵀ) still flows."""
    M, k, n, r = 256, 512, 512, 16
    g = torch.Generator().manual_seed(5)
    d = draw_projection(g, M, k, n, r)
    d["B"] = torch.zeros_like(d["B"])
    dx, dA, dB = run_bwd(d, 16.0)
    assert torch.all(dA == 0)
    want = ref.lora_bwd(np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]), np64(d["dY"]),
                        16.0)
    assert rel_err(np64(dx), np64(d["dY"]) @ np64(d["W"])) <= TOL_BF16
    assert rel_err(np64(dB), want[2]) <= TOL_F32


@pytest.mark.parametrize("M,k,n,r", [(256, 512, 512, 16), (200, 192, 320, 64),
                                     (130, 1024, 768, 16)])
def test_bwd_nf4_parity(M, k, n, r):
    g = torch.Generator().manual_seed(17 + M)
    d = draw_projection(g, M, k, n, r)
    codes, absmax = ref.nf4_quantize(np64(d["W"]))
    got = run_bwd(d, 16.0, nf4=(codes, absmax))
    Wq = ref.nf4_dequant(codes, absmax)
    want = ref.lora_bwd(np64(d["x"]), Wq, np64(d["A"]), np64(d["B"]), np64(d["dY"]), 16.0)
    _check(f"bwd_nf4_{M}_{k}_{n}_{r}", d, got, want)
