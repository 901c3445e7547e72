"""GPU parity of the q/k projections with the RoPE epilogue, forward and
backward, including the identity case (all positions 0)."""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import draw_projection, draw_shared_x
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, dump, np64, rel_err

pytestmark = pytest.mark.gpu
THETA = 500000.0


def _draw(M, hidden, nqh, nkh, r, seed):
    g = torch.Generator().manual_seed(seed)
    x = draw_shared_x(g, M, hidden)
    q = draw_projection(g, M, hidden, nqh * 128, r, x=x)
    k = draw_projection(g, M, hidden, nkh * 128, r, x=x)
    return x, q, k


def _qk_fwd(x, q, k, pos, max_pos, alpha, use_cache=True):
    M, hidden = x.shape
    r = q["A"].shape[0]
    dev = {n: cuda(t) for n, t in (("x", x), ("Wq", q["W"]), ("Aq", q["A"]), ("Bq", q["B"]),
                                    ("Wk", k["W"]), ("Ak", k["A"]), ("Bk", k["B"]))}
    posd = cuda(torch.as_tensor(pos, dtype=torch.int32))
    nq, nk = q["W"].shape[0], k["W"].shape[0]
    yq = torch.full((M, nq), float("nan"), dtype=torch.bfloat16, device="cuda")
    yk = torch.full((M, nk), float("nan"), dtype=torch.bfloat16, device="cuda")
    cache = None
    extra = 0
    if use_cache:
        cache = torch.empty(max_pos, 128, dtype=torch.float32, device="cuda")
        L.lora_rope_cache_build(cache, max_pos, 128, THETA)
    else:
        extra = L.lora_rope_cache_bytes(max_pos) + 256
    ws = L.workspace(L.OP_QK_ROPE_FWD, M, hidden, nq + nk, r, extra=extra)
    L.lora_qk_rope_fwd(dev["x"], dev["Wq"], dev["Aq"], dev["Bq"], dev["Wk"], dev["Ak"],
                       dev["Bk"], yq, yk, alpha, THETA, posd, cache, max_pos, ws)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0
    return yq, yk


@pytest.mark.parametrize("M,hidden,nqh,nkh,r,use_cache", [
    (300, 256, 2, 1, 16, True),
    (256, 512, 4, 2, 64, False),
    (129, 128, 3, 1, 8, True),
])
def test_qk_rope_fwd_parity(M, hidden, nqh, nkh, r, use_cache):
    x, q, k = _draw(M, hidden, nqh, nkh, r, seed=M + r)
    max_pos = 4096
    pos = np.random.default_rng(M).integers(0, max_pos, size=M)
    yq, yk = _qk_fwd(x, q, k, pos, max_pos, 16.0, use_cache)
    wq, wk = ref.qk_rope_fwd(np64(x), np64(q["W"]), np64(q["A"]), np64(q["B"]), np64(k["W"]),
                             np64(k["A"]), np64(k["B"]), 16.0, pos, THETA)
    eq, ek = rel_err(np64(yq), wq), rel_err(np64(yk), wk)
    if max(eq, ek) > TOL_BF16:
        dump(f"qk_fwd_{M}_{r}", yq=yq, yk=yk, wq=wq, wk=wk)
    assert eq <= TOL_BF16 and ek <= TOL_BF16, (eq, ek)


def test_qk_rope_position_zero_is_plain_projection():
    M, hidden, r = 200, 256, 16
    x, q, k = _draw(M, hidden, 2, 1, r, seed=1)
    yq, yk = _qk_fwd(x, q, k, np.zeros(M, dtype=np.int64), 16, 16.0)
    wq = ref.lora_fwd(np64(x), np64(q["W"]), np64(q["A"]), np64(q["B"]), 16.0)
    wk = ref.lora_fwd(np64(x), np64(k["W"]), np64(k["A"]), np64(k["B"]), 16.0)
    assert rel_err(np64(yq), wq) <= TOL_BF16 and rel_err(np64(yk), wk) <= TOL_BF16


@pytest.mark.parametrize("M,hidden,nqh,nkh,r,accumulate", [
    (300, 256, 2, 1, 16, False), (256, 512, 4, 2, 64, False), (300, 256, 2, 1, 16, True)])
def test_qk_rope_bwd_parity(M, hidden, nqh, nkh, r, accumulate):
    x, q, k = _draw(M, hidden, nqh, nkh, r, seed=7 * M + r)
    max_pos = 8192
    pos = np.random.default_rng(M + 1).integers(0, max_pos, size=M)
    dev = {n: cuda(t) for n, t in (("x", x), ("Wq", q["W"]), ("Aq", q["A"]), ("Bq", q["B"]),
                                    ("Wk", k["W"]), ("Ak", k["A"]), ("Bk", k["B"]),
                                    ("dq", q["dY"]), ("dk", k["dY"]))}
    posd = cuda(torch.as_tensor(pos, dtype=torch.int32))
    nq, nk = q["W"].shape[0], k["W"].shape[0]
    cache = torch.empty(max_pos, 128, dtype=torch.float32, device="cuda")
    L.lora_rope_cache_build(cache, max_pos, 128, THETA)
    dx0 = draw_shared_x(torch.Generator().manual_seed(M + 99), M, hidden)  # prior dX (bf16)
    dx = (cuda(dx0) if accumulate else
          torch.full((M, hidden), float("nan"), dtype=torch.bfloat16, device="cuda"))
    f32 = dict(dtype=torch.float32, device="cuda")
    dAq, dBq = torch.empty(r, hidden, **f32), torch.empty(nq, r, **f32)
    dAk, dBk = torch.empty(r, hidden, **f32), torch.empty(nk, r, **f32)
    ws = L.workspace(L.OP_QK_ROPE_BWD, M, hidden, nq + nk, r)
    L.lora_qk_rope_bwd(dev["x"], dev["Wq"], dev["Aq"], dev["Bq"], dev["Wk"], dev["Ak"],
                       dev["Bk"], dev["dq"], dev["dk"], dx, dAq, dBq, dAk, dBk, 16.0, THETA,
                       posd, cache, max_pos, ws, accumulate_dx=accumulate)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(ws) == 0
    want = list(ref.qk_rope_bwd(np64(x), np64(q["W"]), np64(q["A"]), np64(q["B"]),
                                np64(k["W"]), np64(k["A"]), np64(k["B"]), np64(q["dY"]),
                                np64(k["dY"]), 16.0, pos, THETA))
    if accumulate:       # dX += the q/k gradient
        want[0] = want[0] + np64(dx0)
    got = (dx, dAq, dBq, dAk, dBk)
    errs = [rel_err(np64(g), w) for g, w in zip(got, want)]
    if errs[0] > TOL_BF16 or max(errs[1:]) > TOL_F32:
        dump(f"qk_bwd_{M}_{r}", dx=dx, dx_ref=want[0])
    assert errs[0] <= TOL_BF16 and max(errs[1:]) <= TOL_F32, errs


def test_bad_position_is_reported_not_read():
    """A position outside the cache sets the device status bit (the kernel
    clamps the lookup instead of reading out of bounds)."""
    M, hidden, r = 64, 128, 16
    x, q, k = _draw(M, hidden, 1, 1, r, seed=2)
    max_pos = 32
    pos = np.arange(M)                  # positions 32..63 exceed the cache
    dev = {n: cuda(t) for n, t in (("x", x), ("Wq", q["W"]), ("Aq", q["A"]), ("Bq", q["B"]),
                                    ("Wk", k["W"]), ("Ak", k["A"]), ("Bk", k["B"]))}
    cache = torch.empty(max_pos, 128, dtype=torch.float32, device="cuda")
    L.lora_rope_cache_build(cache, max_pos, 128, THETA)
    yq = torch.empty(M, 128, dtype=torch.bfloat16, device="cuda")
    yk = torch.empty(M, 128, dtype=torch.bfloat16, device="cuda")
    ws = L.workspace(L.OP_QK_ROPE_FWD, M, hidden, 256, r)
    L.lora_qk_rope_fwd(dev["x"], dev["Wq"], dev["Aq"], dev["Bq"], dev["Wk"], dev["Ak"],
                       dev["Bk"], yq, yk, 16.0, THETA, cuda(torch.as_tensor(pos, dtype=torch.int32)),
                       cache, max_pos, ws)
    assert L.lora_read_device_status(ws) == 2   # LORA_DEVSTAT_BAD_POSITION
    L.lora_clear_device_status(ws)
    assert L.lora_read_device_status(ws) == 0
