"""A device-side wait that runs out is reported, and the device stays usable.

Every wait inside the library's kernels is bounded; past its limit the
kernel records LORA_DEVSTAT_TIMEOUT in the call's status word, lets its
copies in flight land and returns.  The test-only library variant
(liblora_b300_testhooks.so, built with -DLORA_TEST_HOOKS) lets a test make
one such wait run out: in the backward's stream-K rank pass, CTA 1 parks its
partial but never raises its flag, and the flag wait of the CTA that finishes
the tile (CTA 0) gives up after 2 ms.  Nothing faults: the wait is a poll of a global
flag with no copy of the waiting CTA in flight.  The call then reports
LORA_ERR_TIMEOUT through lora_read_device_status, and a clean call afterwards
on the same device (hooks reset, workspace zeroed) matches the fp64 oracle.

The scenario runs in a child process so that the second library instance
and its device state stay out of the other tests' process.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, json, sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import lora_qlora_linear_fwd_b300 as L
from lora_qlora_linear_fwd_b300.build import lib_path
import oracle as ref
from lora_inputs import draw_projection

lib = ctypes.CDLL(lib_path("testhooks"))
for name, (res, args) in L.EXPORTS.items():
    fn = getattr(lib, name)
    fn.restype, fn.argtypes = res, args
lib.lora_test_stream_k_hooks.restype = ctypes.c_int
lib.lora_test_stream_k_hooks.argtypes = [ctypes.c_ulonglong, ctypes.c_int]

# rank 16, 1024 tokens, k = n = 4096: the backward's rank pass runs stream-K
# on 128 CTAs of 8 chunks each, so each 64-chunk row tile is shared by 8 CTAs
# and CTA 0 finishes tile 0 with the partials of CTAs 1-7
M, k, n, r, alpha = 1024, 4096, 4096, 16, 16.0
d = draw_projection(torch.Generator().manual_seed(71), M, k, n, r)
x, W, A, B, dy = (d[t].cuda().contiguous() for t in ("x", "W", "A", "B", "dY"))
dx = torch.zeros(M, k, dtype=torch.bfloat16, device="cuda")
dA = torch.zeros(r, k, dtype=torch.float32, device="cuda")
dB = torch.zeros(n, r, dtype=torch.float32, device="cuda")
ws = torch.zeros(L.workspace_size(L.OP_BWD, M, k, n, r), dtype=torch.uint8, device="cuda")
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
p = lambda t: ctypes.c_void_p(t.data_ptr())

def bwd():
    return lib.lora_linear_bwd(p(x), L.bf16_weight(W), p(A), p(B), p(dy), p(dx), 0, p(dA),
                               p(dB), M, k, n, r, alpha, p(ws), ws.numel(), stream)

def status():
    out = ctypes.c_uint32(0)
    rc = lib.lora_read_device_status(p(ws), ctypes.byref(out), stream)
    return rc, int(out.value)

out = {}
assert lib.lora_test_stream_k_hooks(2_000_000, 1) == 0
lib.lora_profile_begin(8)
out["launch_rc"] = bwd()
torch.cuda.synchronize()
names = (ctypes.c_char_p * 8)(); ms = (ctypes.c_float * 8)(); cnt = ctypes.c_int(0)
lib.lora_profile_end(names, ms, 8, ctypes.byref(cnt))
out["kernels"] = [names[i].decode() for i in range(cnt.value)]
out["timed_out"] = status()
out["cuda_error_after"] = str(torch.cuda.synchronize() or "none")
# a clean call on the same device: hooks off, workspace zeroed
assert lib.lora_test_stream_k_hooks(1_000_000_000, -1) == 0
ws.zero_()
out["clean_rc"] = bwd()
torch.cuda.synchronize()
out["clean"] = status()
f = lambda t: t.float().cpu().numpy().astype(np.float64)
want = ref.lora_bwd(f(d["x"]), f(d["W"]), f(d["A"]), f(d["B"]), f(d["dY"]), alpha)
err = lambda g, w: float(np.max(np.abs(f(g) - w)) / np.max(np.abs(w)))
out["clean_err"] = [err(dx, want[0]), err(dA, want[1]), err(dB, want[2])]
print("RESULT " + json.dumps(out))
'''


@pytest.mark.gpu
def test_stream_k_flag_wait_times_out_reports_status_and_recovers():
    code = "ROOT = " + repr(ROOT) + "\n" + CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")]
    assert r.returncode == 0 and lines, r.stdout[-2000:] + r.stderr[-4000:]
    out = json.loads(lines[-1][len("RESULT "):])
    assert out["launch_rc"] == 0
    assert out["kernels"][1] == "lora_skinny_sk_kernel<k_major>", out["kernels"]
    rc, word = out["timed_out"]
    assert rc == 6 and (word & 0x1), out          # LORA_ERR_TIMEOUT, LORA_DEVSTAT_TIMEOUT
    assert out["clean_rc"] == 0 and out["clean"] == [0, 0], out
    e_dx, e_dA, e_dB = out["clean_err"]
    assert e_dx <= 2e-2 and e_dA <= 5e-3 and e_dB <= 5e-3, out
