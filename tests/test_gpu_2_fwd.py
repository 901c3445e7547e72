"""GPU parity of the fused forward against the fp64 oracle, at sizes the
oracle finishes quickly that still span several tiles and ragged tails."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection
from tests.gpu_util import TOL_BF16, cuda, dump, np64, rel_err

pytestmark = pytest.mark.gpu

SHAPES = [  # M, k, n, r
    (256, 512, 512, 8),      # the single-projection workload
    (128, 64, 256, 16),      # one tile, one K stage
    (200, 192, 320, 16),     # ragged M and n tails
    (130, 512, 1024, 32),
    (257, 256, 768, 64),
    (1, 128, 64, 8),         # a single token
    (700, 1024, 2048, 16),   # several m-blocks and n-tiles per CTA
]


def _run_fwd(d, alpha, nf4=None):
    x, A, B = cuda(d["x"]), cuda(d["A"]), cuda(d["B"])
    M, k = x.shape
    n, r = d["W"].shape[0], A.shape[0]
    if nf4 is None:
        W = L.bf16_weight(Wd := cuda(d["W"]))
        keep = [Wd]
    else:
        codes, absmax = nf4
        c = cuda(torch.from_numpy(codes))
        a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
        W = L.nf4_weight(c, a)
        keep = [c, a]
    y = torch.full((M, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = L.workspace(L.OP_FWD, M, k, n, r)
    L.lora_linear_fwd(x, W, A, B, y, alpha, ws)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0
    del keep
    return y


@pytest.mark.parametrize("M,k,n,r", SHAPES)
def test_fwd_bf16_parity(M, k, n, r):
    g = torch.Generator().manual_seed(M * 7 + k + n + r)
    d = draw_projection(g, M, k, n, r)
    y = _run_fwd(d, 16.0)
    want = ref.lora_fwd(np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]), 16.0)
    err = rel_err(np64(y), want)
    if err > TOL_BF16:
        dump(f"fwd_{M}_{k}_{n}_{r}", x=d["x"], W=d["W"], A=d["A"], B=d["B"], y=y, want=want)
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("M,k,n,r", [(256, 512, 512, 8), (200, 192, 320, 64)])
def test_fwd_base_only_when_b_is_zero(M, k, n, r):
    """B = 0: the adapter vanishes and y is the plain GEMM."""
    g = torch.Generator().manual_seed(11)
    d = draw_projection(g, M, k, n, r)
    d["B"] = torch.zeros_like(d["B"])
    y = _run_fwd(d, 16.0)
    want = np64(d["x"]) @ np64(d["W"]).T
    err = rel_err(np64(y), want)
    if err > TOL_BF16:
        dump(f"fwd_b0_{M}_{k}_{n}_{r}", x=d["x"], W=d["W"], y=y, want=want)
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("r", [8, 16, 32, 64])
def test_fwd_adapter_only_when_w_is_zero(r):
    """W = 0 isolates the adapter branch s·(x·Aᵀ)·Bᵀ."""
    M, k, n = 300, 256, 512
    g = torch.Generator().manual_seed(r)
    d = draw_projection(g, M, k, n, r)
    d["W"] = torch.zeros_like(d["W"])
    y = _run_fwd(d, 32.0)
    want = ref.lora_fwd(np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]), 32.0)
    err = rel_err(np64(y), want)
    if err > TOL_BF16:
        dump(f"fwd_w0_{r}", x=d["x"], A=d["A"], B=d["B"], y=y, want=want)
    assert err <= TOL_BF16, err


@pytest.mark.parametrize("M,k,n,r", [(256, 512, 512, 16), (200, 192, 320, 64),
                                     (130, 1024, 768, 16)])
def test_fwd_nf4_parity(M, k, n, r):
    g = torch.Generator().manual_seed(5 + M)
    d = draw_projection(g, M, k, n, r)
    codes, absmax = ref.nf4_quantize(np64(d["W"]))
    y = _run_fwd(d, 16.0, nf4=(codes, absmax))
    Wq = ref.nf4_dequant(codes, absmax)
    want = ref.lora_fwd(np64(d["x"]), Wq, np64(d["A"]), np64(d["B"]), 16.0)
    err = rel_err(np64(y), want)
    if err > TOL_BF16:
        dump(f"fwd_nf4_{M}_{k}_{n}_{r}", x=d["x"], codes=codes, absmax=absmax, A=d["A"],
             B=d["B"], y=y, want=want)
    assert err <= TOL_BF16, err
