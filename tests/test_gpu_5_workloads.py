"""Parity at the full workload sizes, through the same calls the bench times.

y and dX are checked on a fixed sample of 512 rows (each row of y and dX
depends only on that row of x and dY, so the oracle computes exactly those
rows); dA and dB are sums over every token and are checked in full.
"""
import numpy as np
import pytest
import torch

import lora_qlora_linear_fwd_b300 as L
import oracle as ref
from lora_inputs import WORKLOADS, draw_workload
from tests.gpu_util import TOL_BF16, TOL_F32, cuda, np64, rel_err

pytestmark = pytest.mark.gpu


def _rows(M, n=512, seed=0):
    if M <= n:
        return np.arange(M)
    rows = np.random.default_rng(seed).choice(M, size=n - 2, replace=False)
    return np.unique(np.concatenate([rows, [0, M - 1]]))


def _weight(p, d, nf4):
    if not nf4:
        W = cuda(d["W"])
        return L.bf16_weight(W), [W], np64(d["W"])
    codes, absmax = ref.nf4_quantize(d["W"].float().numpy())
    c = cuda(torch.from_numpy(codes))
    a = cuda(torch.from_numpy(absmax.astype(np.float32)).to(torch.bfloat16))
    return L.nf4_weight(c, a), [c, a], ref.nf4_dequant(codes, absmax)


@pytest.mark.parametrize("name", [n for n in WORKLOADS if not WORKLOADS[n].rope])
def test_linear_workload_full_size(name):
    wl = WORKLOADS[name]
    data = draw_workload(name, seed=0)
    rows = _rows(wl.M)
    for p in wl.projections:
        d = data[p.name]
        Wdesc, keep, Wref = _weight(p, d, wl.nf4)
        x, A, B, dy = cuda(d["x"]), cuda(d["A"]), cuda(d["B"]), cuda(d["dY"])
        bf = dict(dtype=torch.bfloat16, device="cuda")
        y = torch.full((wl.M, p.n), float("nan"), **bf)
        dx = torch.full((wl.M, p.k), float("nan"), **bf)
        dA = torch.empty(wl.r, p.k, dtype=torch.float32, device="cuda")
        dB = torch.empty(p.n, wl.r, dtype=torch.float32, device="cuda")
        wsf = L.workspace(L.OP_FWD, wl.M, p.k, p.n, wl.r)
        wsb = L.workspace(L.OP_BWD, wl.M, p.k, p.n, wl.r)
        L.lora_linear_fwd(x, Wdesc, A, B, y, wl.alpha, wsf)
        L.lora_linear_bwd(x, Wdesc, A, B, dy, dx, dA, dB, wl.alpha, wsb)
        torch.cuda.synchronize()
        assert L.lora_read_device_status(wsf) == 0 and L.lora_read_device_status(wsb) == 0
        xs, dys = np64(d["x"][rows]), np64(d["dY"][rows])
        A64, B64 = np64(d["A"]), np64(d["B"])
        y_ref = ref.lora_fwd(xs, Wref, A64, B64, wl.alpha)
        dx_ref = ref.lora_bwd(xs, Wref, A64, B64, dys, wl.alpha)[0]
        dA_ref, dB_ref = ref.lora_adapter_grads(np64(d["x"]), A64, B64, np64(d["dY"]), wl.alpha)
        errs = (rel_err(np64(y[rows]), y_ref), rel_err(np64(dx[rows]), dx_ref),
                rel_err(np64(dA), dA_ref), rel_err(np64(dB), dB_ref))
        assert errs[0] <= TOL_BF16 and errs[1] <= TOL_BF16, (p.name, errs)
        assert errs[2] <= TOL_F32 and errs[3] <= TOL_F32, (p.name, errs)
        assert not torch.isnan(y).any() and not torch.isnan(dx).any()
        del keep


def test_qk_rope_workload_full_size():
    name = "llama8b_qk_rope"
    wl = WORKLOADS[name]
    data = draw_workload(name, seed=0)
    q, k = data["q_proj"], data["k_proj"]
    M, hidden, r = wl.M, q["x"].shape[1], wl.r
    nq, nk = q["W"].shape[0], k["W"].shape[0]
    dev = {key: cuda(t) for key, t in (("x", q["x"]), ("Wq", q["W"]), ("Aq", q["A"]),
                                        ("Bq", q["B"]), ("Wk", k["W"]), ("Ak", k["A"]),
                                        ("Bk", k["B"]), ("dq", q["dY"]), ("dk", k["dY"]))}
    pos = np.arange(M)
    posd = cuda(torch.as_tensor(pos, dtype=torch.int32))
    cache = torch.empty(M, 128, dtype=torch.float32, device="cuda")
    L.lora_rope_cache_build(cache, M, 128, wl.rope_theta)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    yq, yk = torch.full((M, nq), float("nan"), **bf), torch.full((M, nk), float("nan"), **bf)
    dx = torch.full((M, hidden), float("nan"), **bf)
    dAq, dBq = torch.empty(r, hidden, **f32), torch.empty(nq, r, **f32)
    dAk, dBk = torch.empty(r, hidden, **f32), torch.empty(nk, r, **f32)
    wsf = L.workspace(L.OP_QK_ROPE_FWD, M, hidden, nq + nk, r)
    wsb = L.workspace(L.OP_QK_ROPE_BWD, M, hidden, nq + nk, r)
    L.lora_qk_rope_fwd(dev["x"], dev["Wq"], dev["Aq"], dev["Bq"], dev["Wk"], dev["Ak"],
                       dev["Bk"], yq, yk, wl.alpha, wl.rope_theta, posd, cache, M, wsf)
    L.lora_qk_rope_bwd(dev["x"], dev["Wq"], dev["Aq"], dev["Bq"], dev["Wk"], dev["Ak"],
                       dev["Bk"], dev["dq"], dev["dk"], dx, dAq, dBq, dAk, dBk, wl.alpha,
                       wl.rope_theta, posd, cache, M, wsb)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(wsf) == 0 and L.lora_read_device_status(wsb) == 0

    rows = _rows(M)
    x64 = np64(q["x"])
    P = {key: np64(t) for key, t in (("Wq", q["W"]), ("Aq", q["A"]), ("Bq", q["B"]),
                                      ("Wk", k["W"]), ("Ak", k["A"]), ("Bk", k["B"]))}
    wq, wk = ref.qk_rope_fwd(x64[rows], P["Wq"], P["Aq"], P["Bq"], P["Wk"], P["Ak"], P["Bk"],
                             wl.alpha, pos[rows], wl.rope_theta)
    assert rel_err(np64(yq[rows]), wq) <= TOL_BF16
    assert rel_err(np64(yk[rows]), wk) <= TOL_BF16
    dq_pre = ref.rope_apply_inverse(np64(q["dY"]), pos, 128, wl.rope_theta)
    dk_pre = ref.rope_apply_inverse(np64(k["dY"]), pos, 128, wl.rope_theta)
    dx_ref = (ref.lora_bwd(x64[rows], P["Wq"], P["Aq"], P["Bq"], dq_pre[rows], wl.alpha)[0]
              + ref.lora_bwd(x64[rows], P["Wk"], P["Ak"], P["Bk"], dk_pre[rows], wl.alpha)[0])
    assert rel_err(np64(dx[rows]), dx_ref) <= TOL_BF16
    gq = ref.lora_adapter_grads(x64, P["Aq"], P["Bq"], dq_pre, wl.alpha)
    gk = ref.lora_adapter_grads(x64, P["Ak"], P["Bk"], dk_pre, wl.alpha)
    for got, want in zip((dAq, dBq, dAk, dBk), (*gq, *gk)):
        assert rel_err(np64(got), want) <= TOL_F32
