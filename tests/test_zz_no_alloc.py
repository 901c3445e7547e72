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
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
from lora_inputs import draw_projection
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, np64, rel_err

pytestmark = pytest.mark.gpu


def _grads(d, use_noalloc):
    x, A, B, dy, W = (cuda(d[k]) for k in ("x", "A", "B", "dY", "W"))
    M, k = x.shape
    n, r = dy.shape[1], A.shape[0]
    dx = torch.full((M, k), float("nan"), dtype=torch.bfloat16, device="cuda")
    dA = torch.full((r, k), float("nan"), dtype=torch.float32, device="cuda")
    dB = torch.full((n, r), float("nan"), dtype=torch.float32, device="cuda")
    if use_noalloc:
        L.lora_linear_bwd_noalloc(x, W, A, B, dy, dx, dA, dB, 16.0)
    else:
        ws = L.workspace(L.OP_BWD, M, k, n, r)
        L.lora_linear_bwd(x, W, A, B, dy, dx, dA, dB, 16.0, ws)
        torch.cuda.synchronize()
        assert L.lora_read_device_status(ws) == 0
    torch.cuda.synchronize()
    return dx, dA, dB


def test_noalloc_backward_matches_workspace_backward_on_consecutive_calls():
    # two calls in a row on different shapes and ranks: the second runs on
    # the scratch the first one left behind
    for M, k, n, r, seed in ((700, 1024, 2048, 16, 1), (257, 256, 768, 64, 2)):
        d = draw_projection(torch.Generator().manual_seed(seed), M, k, n, r)
        want = _grads(d, use_noalloc=False)
        got = _grads(d, use_noalloc=True)
        errs = [rel_err(np64(g), np64(w)) for g, w in zip(got, want)]
        assert errs[0] <= TOL_BF16 and errs[1] <= TOL_F32 and errs[2] <= TOL_F32, (M, errs)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    fake = 0x10000   # aligned, never dereferenced: the call returns before any launch
    w = L.Weight(0, fake, None, 0)
    status = L.library.lora_linear_bwd_noalloc(fake, w, fake, fake, fake, fake, 0, fake, fake,
                                               65536, 4096, 4096, 64, 16.0, None)
    assert status == 3    # LORA_ERR_WORKSPACE
