"""lora_linear_bwd_noalloc against lora_linear_bwd, through the C ABI.

Some callers cannot allocate device memory where they run the backward: a
plugin inside another framework's runtime that is handed only its tensors,
or a latency-critical loop that must not enter the driver's allocator.
``lora_linear_bwd_noalloc`` serves them from a fixed scratch array inside
the library instead of a caller workspace.  Its results must be those of
``lora_linear_bwd`` on the same inputs, call after call, even though every
call reuses the same array.

This file is collected last, so a run that stops at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, np64, rel_err

ALPHA = 16.0


def _grads(d, use_noalloc):
    x, A, B, dy, W = (cuda(d[k]) for k in ("x", "A", "B", "dY", "W"))
    M, k = x.shape
    n, r = dy.shape[1], A.shape[0]
    dx = torch.full((M, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    dA = torch.full((r, k), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((n, r), float("nan"), dtype=torch.float32, device="cuda")
    if use_noalloc:
        L.lora_linear_bwd_noalloc(x, W, A, B, dy, dx, dA, dB, ALPHA)
    else:
        ws = L.workspace(L.OP_BWD, M, k, n, r)
        L.lora_linear_bwd(x, W, A, B, dy, dx, dA, dB, ALPHA, ws)
        torch.cuda.synchronize()
        assert L.lora_read_device_status(ws) == 0
    torch.cuda.synchronize()
    return dx, dA, dB


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_on_consecutive_calls():
    # two calls in a row on different shapes and ranks: the second runs on
    # the scratch the first one left behind.  Both entry points run the same
    # deterministic kernels on the same inputs, so the results are equal bit
    # for bit; the first call is also held to the fp64 oracle.
    for i, (M, k, n, r, seed) in enumerate(((700, 1024, 2048, 16, 1), (257, 256, 768, 64, 2))):
        d = draw_projection(torch.Generator().manual_seed(seed), M, k, n, r)
        want = _grads(d, use_noalloc=False)
        got = _grads(d, use_noalloc=True)
        for name, g, w in zip(("dX", "dA", "dB"), got, want):
            assert torch.equal(g, w), (M, name)
        if i == 0:
            f = lambda t: t.float().numpy().astype(np.float64)
            o_dx, o_dA, o_dB = ref.lora_bwd(f(d["x"]), f(d["W"]), f(d["A"]), f(d["B"]),
                                            f(d["dY"]), ALPHA)
            assert rel_err(np64(got[0]), o_dx) <= TOL_BF16
            assert rel_err(np64(got[1]), o_dA) <= TOL_F32
            assert rel_err(np64(got[2]), o_dB) <= TOL_F32


FAKE = 0x10000   # aligned, never dereferenced: these calls return before any CUDA call


def _noalloc(M=256, k=512, n=512, r=8, alpha=16.0, w=None):
    return L.library.lora_linear_bwd_noalloc(FAKE, w or L.Weight(0, FAKE, None, 0), FAKE, FAKE,
                                             FAKE, FAKE, 0, FAKE, FAKE, M, k, n, r, alpha, None)


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_its_scratch():
    assert _noalloc(M=65536, k=4096, n=4096, r=64) == 3    # LORA_ERR_WORKSPACE


def test_noalloc_rejects_what_the_workspace_backward_rejects_before_any_cuda_call():
    # Argument errors come back before the call reaches CUDA (which, on a
    # machine without a GPU, would answer LORA_ERR_CUDA or LORA_ERR_ARCH),
    # so a rejected call has enqueued nothing, not even its status-word reset.
    assert _noalloc(alpha=float("nan")) == 1
    assert _noalloc(alpha=float("inf")) == 1
    assert _noalloc(w=L.Weight(1, FAKE, FAKE, 128)) == 2   # NF4 block size other than 64
    assert _noalloc(w=L.Weight(1, FAKE, None, 64)) == 1    # NF4 without absmax
    assert _noalloc(w=L.Weight(5, FAKE, None, 0)) == 1     # unknown weight type
    assert _noalloc(r=12) == 2
    assert _noalloc(k=100) == 2
    assert _noalloc(M=0) == 1
    assert _noalloc(M=65536, k=4096, n=4096, r=64) == 3
