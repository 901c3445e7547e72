"""GPU parity of LoRA dropout on the adapter's input ("微调太慢？试试Unsloth"
§3.3 table, row E: lora_dropout 0.05) against the fp64 oracle, with the mask
drawn from Philox4x64-10 on both sides: the keep pattern bit for bit, the
forward and the backward (mask regenerated), bf16 and NF4 weights."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection, draw_tensor
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, np64, rel_err

pytestmark = pytest.mark.gpu

ALPHA = 16.0


def _weight(d, nf4):
    if not nf4:
        W = cuda(d["W"])
        return L.bf16_weight(W), [W], np64(d["W"])
    codes, absmax = ref.nf4_quantize(np64(d["W"]))
    c = cuda(torch.from_numpy(codes))
    a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
    return L.nf4_weight(c, a), [c, a], ref.nf4_dequant(codes, absmax)


@pytest.mark.parametrize("M,k,n,r,p,nf4", [
    (256, 512, 512, 16, 0.1, False),
    (200, 192, 320, 8, 0.05, False),     # ragged M and n tails
    (300, 512, 1024, 64, 0.5, False),
    (256, 512, 768, 16, 0.3, True),
])
def test_dropout_forward_and_backward_parity(M, k, n, r, p, nf4):
    seed, off = 1234 + M, 7
    d = draw_projection(torch.Generator().manual_seed(M + n), M, k, n, r)
    Wd, keep_alive, W64 = _weight(d, nf4)
    x, A, B, dy = cuda(d["x"]), cuda(d["A"]), cuda(d["B"]), cuda(d["dY"])
    bf = dict(dtype=torch.bfloat16, device="cuda")
    y = torch.full((M, n), float("nan"), **bf)
    wsf = L.workspace(L.OP_FWD_DROPOUT, M, k, n, r)
    L.lora_linear_fwd_dropout(x, Wd, A, B, y, ALPHA, p, seed, off, wsf)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsf) == 0
    # the masked x̃ the forward left after its own workspace: same keep bits
    # as the oracle's Philox mask, kept values bf16(x / q)
    base = L.workspace_size(L.OP_FWD, M, k, n, r)
    xd = np64(wsf[base:base + 2 * M * k].view(torch.bfloat16).view(M, k))
    keep = ref.dropout_keep(M, k, p, seed, off)
    x64 = np64(d["x"])
    nz = x64 != 0
    assert np.array_equal((xd != 0)[nz], keep[nz])
    q = ref.dropout_keep_prob(p)
    np.testing.assert_allclose(xd[keep], (x64 / q)[keep], rtol=2.0 ** -8, atol=0)
    args = (x64, W64, np64(d["A"]), np64(d["B"]))
    assert rel_err(np64(y), ref.lora_fwd_dropout(*args, ALPHA, p, seed, off)) <= TOL_BF16

    dx = torch.full((M, k), float("nan"), **bf)
    dA = torch.full((r, k), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((n, r), float("nan"), dtype=torch.float32, device="cuda")
    wsb = L.workspace(L.OP_BWD_DROPOUT, M, k, n, r)
    L.lora_linear_bwd_dropout(x, Wd, A, B, dy, dx, dA, dB, ALPHA, p, seed, off, wsb)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsb) == 0
    want = ref.lora_bwd_dropout(*args, np64(d["dY"]), ALPHA, p, seed, off)
    errs = [rel_err(np64(g), w) for g, w in zip((dx, dA, dB), want)]
    assert errs[0] <= TOL_BF16 and errs[1] <= TOL_F32 and errs[2] <= TOL_F32, errs
    del keep_alive


def test_dropout_backward_accumulates_dx_and_zero_rate_is_plain_lora():
    M, k, n, r, seed, off = 256, 512, 768, 32, 5, 0
    d = draw_projection(torch.Generator().manual_seed(3), M, k, n, r)
    x, W, A, B, dy = (cuda(d[t]) for t in ("x", "W", "A", "B", "dY"))
    dx0 = draw_tensor(torch.Generator().manual_seed(4), (M, k), "normal", 2.0)
    dx = cuda(dx0)
    f32 = dict(dtype=torch.float32, device="cuda")
    dA, dB = torch.empty(r, k, **f32), torch.empty(n, r, **f32)
    ws = L.workspace(L.OP_BWD_DROPOUT, M, k, n, r)
    L.lora_linear_bwd_dropout(x, W, A, B, dy, dx, dA, dB, ALPHA, 0.2, seed, off, ws,
                              accumulate_dx=True)
    torch.cuda.synchronize()
    args = (np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]), np64(d["dY"]))
    want = ref.lora_bwd_dropout(*args, ALPHA, 0.2, seed, off)
    assert rel_err(np64(dx), want[0] + np64(dx0)) <= TOL_BF16
    # rate 0: the plain LoRA forward
    y = torch.empty(M, n, dtype=torch.bfloat16, device="cuda")
    wsf = L.workspace(L.OP_FWD_DROPOUT, M, k, n, r)
    L.lora_linear_fwd_dropout(x, W, A, B, y, ALPHA, 0.0, seed, off, wsf)
    torch.cuda.synchronize()
    assert rel_err(np64(y), ref.lora_fwd(*args[:4], ALPHA)) <= TOL_BF16
