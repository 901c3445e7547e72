"""GPU parity of the non-GEMM kernels: RoPE cache, NF4 dequantise/quantise,
and the RoPE backward rotation (through the q/k backward in a later file)."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection, draw_tensor
from tests.gpu_util import cuda, np64

pytestmark = pytest.mark.gpu


def test_rope_cache_matches_oracle():
    max_pos, D, theta = 8192, 128, 500000.0
    cs = torch.empty(max_pos, D, dtype=torch.float32, device="cuda")
    L.lora_rope_cache_build(cs, max_pos, D, theta)
    torch.cuda.synchronize()
    c, s = ref.rope_cos_sin(np.arange(max_pos), D, theta)
    got = cs.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got[:, :64] - c)) <= 1e-7
    assert np.max(np.abs(got[:, 64:] - s)) <= 1e-7


def _nf4_inputs(n, k, seed=3):
    g = torch.Generator().manual_seed(seed)
    W = draw_tensor(g, (n, k), "normal", 1.0 / np.sqrt(k))
    W[0, :64] = 0                     # an all-zero block
    codes, absmax = ref.nf4_quantize(np64(W))
    return W, codes, absmax


@pytest.mark.parametrize("n,k", [(64, 64), (320, 512), (1024, 4096)])
def test_nf4_dequant_parity(n, k):
    W, codes, absmax = _nf4_inputs(n, k)
    c = cuda(torch.from_numpy(codes))
    a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
    out = torch.empty(n, k, dtype=torch.bfloat16, device="cuda")
    L.nf4_dequant(L.nf4_weight(c, a), out)
    torch.cuda.synchronize()
    want = ref.nf4_dequant(codes, absmax)
    got = np64(out)
    # one bf16 rounding of the fp32 product: within 2^-8 relative per element
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)


@pytest.mark.parametrize("n,k", [(64, 64), (256, 1024), (1024, 4096)])
def test_nf4_quantize_parity(n, k):
    """Codes are the oracle's (decided in fp32, as the kernel does) except
    at exact near-ties, where either neighbour is a correct nearest level."""
    W, _, _ = _nf4_inputs(n, k)
    codes_ref, absmax_ref = ref.nf4_quantize(np64(W), decision="fp32")
    codes = torch.empty(n, k // 2, dtype=torch.uint8, device="cuda")
    absmax = torch.empty(n, k // 64, dtype=torch.bfloat16, device="cuda")
    L.nf4_quantize(cuda(W), L.nf4_weight(codes, absmax))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np64(absmax), absmax_ref)
    gi = ref.nf4_unpack(codes.cpu().numpy())
    ri = ref.nf4_unpack(codes_ref)
    diff = np.argwhere(gi != ri)
    lv = ref.nf4_codebook()
    w = np64(W)
    for i, j in diff:
        a = absmax_ref[i, j // 64]
        ratio = w[i, j] / a
        assert abs(abs(ratio - lv[gi[i, j]]) - abs(ratio - lv[ri[i, j]])) < 1e-6
    assert len(diff) <= 1e-4 * n * k


@pytest.mark.gpu
def test_profile_session_times_each_launch_of_a_call():
    """Per-launch timing: one backward call is four launches (set-up, rank
    pass, dA/dB pass, dX GEMM), each with a positive time, in launch order."""
    M, k, n, r = 512, 512, 768, 16
    d = draw_projection(torch.Generator().manual_seed(5), M, k, n, r)
    x, W, A, B, dy = (cuda(d[t]) for t in ("x", "W", "A", "B", "dY"))
    dx = torch.empty(M, k, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(r, k, dtype=torch.float32, device="cuda")
    dB = torch.empty(n, r, dtype=torch.float32, device="cuda")
    ws = L.workspace(L.OP_BWD, M, k, n, r)
    L.lora_profile_begin(8)
    c0 = L.lora_kernel_launch_count()
    L.lora_linear_bwd(x, W, A, B, dy, dx, dA, dB, 16.0, ws)
    n_launch = L.lora_kernel_launch_count() - c0
    got = L.lora_profile_end(8)
    assert n_launch == 4 and len(got) == 4
    names = [nm for nm, _ in got]
    assert names[0] == "bwd_prep_kernel" and names[3] == "lora_gemm_pair_kernel<dx,bf16>"
    assert names[1].startswith("lora_skinny") and names[2].startswith("lora_skinny")
    assert all(ms > 0.0 for _, ms in got)
    # the session is closed: a second end is an argument error
    with pytest.raises(L.LoraError):
        L.lora_profile_end(8)
