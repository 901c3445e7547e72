"""GPU parity of the fused gate/up + SwiGLU forward and its backward
("Unsloth框架：高效LLM微调与LoRA优化实践" §3.1; SwiGLU per "GLU Variants
Improve Transformer" §2) against the fp64 oracle: small shapes spanning
several tiles with ragged M and n tails, every rank, bf16 and NF4 weights
(one- and two-m-block tiles), accumulated dX, and the Llama-3-8B MLP size."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection, draw_shared_x, draw_tensor
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, np64, rel_err

pytestmark = pytest.mark.gpu

ALPHA = 16.0


def _draw(M, k, n, r, seed):
    g = torch.Generator().manual_seed(seed)
    x = draw_shared_x(g, M, k)
    gate = draw_projection(g, M, k, n, r, x=x)
    up = draw_projection(g, M, k, n, r, x=x)
    return x, gate, up


def _weights(gate, up, nf4):
    if not nf4:
        Wg, Wu = cuda(gate["W"]), cuda(up["W"])
        return L.bf16_weight(Wg), L.bf16_weight(Wu), [Wg, Wu], np64(gate["W"]), np64(up["W"])
    out, keep, refs = [], [], []
    for d in (gate, up):
        codes, absmax = ref.nf4_quantize(np64(d["W"]))
        c = cuda(torch.from_numpy(codes))
        a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
        out.append(L.nf4_weight(c, a))
        keep += [c, a]
        refs.append(ref.nf4_dequant(codes, absmax))
    return out[0], out[1], keep, refs[0], refs[1]


def _run(x, gate, up, nf4=False, accumulate=False, dx0=None, save=True):
    M, k = x.shape
    n, r = gate["W"].shape[0], gate["A"].shape[0]
    Wg, Wu, keep, Wg64, Wu64 = _weights(gate, up, nf4)
    xd = cuda(x)
    Ag, Bg, Au, Bu = (cuda(t) for t in (gate["A"], gate["B"], up["A"], up["B"]))
    bf = dict(dtype=torch.bfloat16, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    h = torch.full((M, n), float("nan"), **bf)
    g = torch.full((M, n), float("nan"), **bf) if save else None
    u = torch.full((M, n), float("nan"), **bf) if save else None
    wsf = L.workspace(L.OP_SWIGLU_FWD, M, k, n, r)
    L.lora_swiglu_fwd(xd, Wg, Ag, Bg, Wu, Au, Bu, h, ALPHA, wsf, g=g, u=u)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsf) == 0
    out = {"h": h, "g": g, "u": u, "Wg64": Wg64, "Wu64": Wu64}
    if not save:
        return out
    dh = cuda(gate["dY"])
    dx = cuda(dx0) if dx0 is not None else torch.full((M, k), float("nan"), **bf)
    grads = [torch.full(s, float("nan"), **f32) for s in ((r, k), (n, r), (r, k), (n, r))]
    wsb = L.workspace(L.OP_SWIGLU_BWD, M, k, n, r)
    L.lora_swiglu_bwd(xd, Wg, Ag, Bg, Wu, Au, Bu, g, u, dh, dx, *grads, ALPHA, wsb,
                      accumulate_dx=accumulate)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsb) == 0
    out.update(dx=dx, grads=grads)
    del keep
    return out


def _check(x, gate, up, out, rows=None, dx0=None):
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    args = (np64(x), out["Wg64"], np64(gate["A"]), np64(gate["B"]), out["Wu64"], np64(up["A"]),
            np64(up["B"]))
    rargs = (sel(args[0]),) + args[1:]
    h, g, u = ref.swiglu_fwd(*rargs, ALPHA)
    assert rel_err(np64(sel(out["h"])), h) <= TOL_BF16
    if out["g"] is not None:
        assert rel_err(np64(sel(out["g"])), g) <= TOL_BF16
        assert rel_err(np64(sel(out["u"])), u) <= TOL_BF16
    if "dx" not in out:
        return
    dx_r = ref.swiglu_bwd(*rargs, sel(np64(gate["dY"])), ALPHA)[0]
    if dx0 is not None:
        dx_r = dx_r + sel(np64(dx0))
    assert rel_err(np64(sel(out["dx"])), dx_r) <= TOL_BF16
    full = ref.swiglu_bwd(*args, np64(gate["dY"]), ALPHA)
    for got, want in zip(out["grads"], full[1:]):
        assert rel_err(np64(got), want) <= TOL_F32


@pytest.mark.parametrize("M,k,n,r", [
    (256, 512, 512, 16),
    (200, 192, 320, 8),       # ragged M and n tails (n not a multiple of 128)
    (300, 512, 1024, 64),
    (130, 256, 384, 32),
    (1, 128, 64, 8),          # a single token, one partial tile
])
def test_swiglu_bf16_parity(M, k, n, r):
    x, gate, up = _draw(M, k, n, r, seed=M + k + n + r)
    _check(x, gate, up, _run(x, gate, up))


@pytest.mark.parametrize("M,k,n,r", [(256, 512, 768, 16), (300, 512, 74 * 128 - 64, 16)])
def test_swiglu_nf4_parity(M, k, n, r):
    # the second shape has 74 tiles of 128 columns per m-block: 512-row tiles
    x, gate, up = _draw(M, k, n, r, seed=7 + M)
    _check(x, gate, up, _run(x, gate, up, nf4=True))


def test_swiglu_without_saved_gate_and_up():
    x, gate, up = _draw(192, 256, 256, 16, seed=3)
    _check(x, gate, up, _run(x, gate, up, save=False))


def test_swiglu_backward_accumulates_dx():
    M, k, n, r = 200, 256, 384, 16
    x, gate, up = _draw(M, k, n, r, seed=9)
    dx0 = draw_tensor(torch.Generator().manual_seed(10), (M, k), "normal", 4.0)
    _check(x, gate, up, _run(x, gate, up, accumulate=True, dx0=dx0), dx0=dx0)


def test_swiglu_llama8b_mlp_full_size():
    """Llama-3-8B gate/up (4096 -> 14336), M = 4096, r = 16: h, g, u and dX on
    512 sampled rows; the adapter gradients in full."""
    M, k, n, r = 4096, 4096, 14336, 16
    x, gate, up = _draw(M, k, n, r, seed=0)
    out = _run(x, gate, up)
    rows = np.unique(np.concatenate([np.random.default_rng(0).choice(M, 510, replace=False),
                                     [0, M - 1]]))
    _check(x, gate, up, out, rows=rows)
