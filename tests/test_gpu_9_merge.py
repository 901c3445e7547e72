"""GPU parity of merging an adapter into its base weight and taking it back
out ("微调太慢？试试Unsloth" §5.1; "Unsloth自动化优化" §3.2): bf16 in place,
and NF4 (dequantise, merge, re-quantise), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection
from tests.gpu_util import TOL_BF16, cuda, np64, rel_err

pytestmark = pytest.mark.gpu


def _draw(n, k, r, seed):
    return draw_projection(torch.Generator().manual_seed(seed), 64, k, n, r)


@pytest.mark.parametrize("n,k,r,alpha", [
    (512, 768, 16, 16.0),
    (320, 704, 8, 16.0),        # m and n tails of the 256 x 256 tiles
    (1024, 512, 64, 128.0),
    (4096, 14336, 16, 16.0),    # Llama-3-8B down_proj
])
def test_merge_bf16_matches_oracle_elementwise(n, k, r, alpha):
    d = _draw(n, k, r, seed=n + k + r)
    W = cuda(d["W"])
    L.lora_merge(W, cuda(d["A"]), cuda(d["B"]), alpha, sign=1)
    torch.cuda.synchronize()
    want = ref.merged_weight(np64(d["W"]), np64(d["A"]), np64(d["B"]), alpha)
    got = np64(W)
    # one rounding to bf16 (half an ulp: within 2^-8 of the value) of an fp32
    # result whose accumulation error scales with the operands, not with the
    # (possibly cancelling) sum: |W| + s·|B|·|A| at fp32 precision, with room
    mag = np.abs(np64(d["W"])) + (alpha / r) * (np.abs(np64(d["B"])) @ np.abs(np64(d["A"])))
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 2.0 ** -16 * mag)


def test_unmerge_after_merge_returns_the_weight():
    n, k, r, alpha = 768, 1024, 32, 32.0
    d = _draw(n, k, r, seed=5)
    W = cuda(d["W"])
    A, B = cuda(d["A"]), cuda(d["B"])
    L.lora_merge(W, A, B, alpha, sign=1)
    L.lora_merge(W, A, B, alpha, sign=-1)
    torch.cuda.synchronize()
    W0 = np64(d["W"])
    s_ba = np.abs(ref.merged_weight(np.zeros_like(W0), np64(d["A"]), np64(d["B"]), alpha))
    # two bf16 roundings, each at most half an ulp of the merged value
    bound = 2.0 ** -8 * (np.abs(W0) + s_ba) * 2 + 1e-30
    assert np.all(np.abs(np64(W) - W0) <= bound)


def test_merged_forward_equals_lora_forward():
    """Inference on the merged weight (no adapter) reproduces the LoRA
    projection: x·W'ᵀ = x·Wᵀ + s·(x·Aᵀ)·Bᵀ."""
    M, k, n, r, alpha = 256, 512, 768, 16, 16.0
    d = draw_projection(torch.Generator().manual_seed(7), M, k, n, r)
    W = cuda(d["W"])
    L.lora_merge(W, cuda(d["A"]), cuda(d["B"]), alpha)
    y = torch.empty(M, n, dtype=torch.bfloat16, device="cuda")
    ws = L.workspace(L.OP_FWD, M, k, n, r)
    zeroB = torch.zeros(n, r, dtype=torch.bfloat16, device="cuda")
    L.lora_linear_fwd(cuda(d["x"]), W, cuda(d["A"]), zeroB, y, alpha, ws)
    torch.cuda.synchronize()
    want = ref.lora_fwd(np64(d["x"]), np64(d["W"]), np64(d["A"]), np64(d["B"]), alpha)
    assert rel_err(np64(y), want) <= TOL_BF16


@pytest.mark.parametrize("n,k,r,sign", [(256, 512, 16, 1), (320, 1024, 64, -1),
                                        (1024, 4096, 16, 1)])
def test_merge_nf4_requantises_the_merged_weight(n, k, r, sign):
    d = _draw(n, k, r, seed=11 + n)
    alpha = 16.0
    codes, absmax = ref.nf4_quantize(np64(d["W"]))
    c = cuda(torch.from_numpy(codes))
    a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
    L.lora_merge(L.nf4_weight(c, a), cuda(d["A"]), cuda(d["B"]), alpha, sign=sign)
    torch.cuda.synchronize()
    got = ref.nf4_dequant(c.cpu().numpy(), np64(a))
    Wm = ref.nf4_dequant(codes, absmax)
    Wm = (ref.merged_weight if sign > 0 else ref.unmerged_weight)(Wm, np64(d["A"]),
                                                                  np64(d["B"]), alpha)
    # within the NF4 error bound of the merged weight: half the widest level
    # gap times the block scale, plus the bf16 rounding of the merged value
    # and of its block scale
    gaps = np.diff(ref.nf4_codebook()).max()
    scale = np.repeat(np64(a), 64, axis=1)
    bound = scale * (gaps / 2) * (1 + 2.0 ** -7) + np.abs(Wm) * 2.0 ** -7
    assert np.all(np.abs(got - Wm) <= bound)
    # and the codes agree with the oracle's own re-quantisation except where
    # the bf16 merged value sits next to a decision boundary
    c_ref, a_ref = ref.nf4_merge(codes, absmax, np64(d["A"]), np64(d["B"]), alpha, sign)
    same = np.mean(ref.nf4_unpack(c.cpu().numpy()) == ref.nf4_unpack(c_ref))
    assert same >= 0.99, same
