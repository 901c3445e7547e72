"""C-ABI boundary tests that need no GPU: the library loads, exports every
function the public header declares, and rejects bad arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

import lora_qlora_linear_fwd_b300 as L

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "lora_b300.h")
lib = L.library
FAKE = 0x10000          # 16-byte aligned, never dereferenced by these calls
MIS = 0x10008           # 8-byte aligned only


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for must in ("lora_linear_fwd", "lora_linear_bwd", "lora_qk_rope_fwd", "lora_qk_rope_bwd",
                 "nf4_dequant", "lora_workspace_size", "lora_rope_cache_build",
                 "lora_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(L.EXPORTS)


def test_status_strings():
    for i, name in enumerate(L.STATUS_NAMES):
        assert L.lora_status_string(i) == name
    assert L.lora_status_string(99) == "LORA_ERR_UNKNOWN"


def _rank_scratch(rp):
    # rank-pass scratch: one 8-byte flag per CTA slot (160), 256-byte aligned,
    # then one parked fp32 partial [rp, 128] per slot
    return (160 * 8 + 255) // 256 * 256 + 160 * rp * 128 * 4


def test_workspace_sizes():
    # forward: status word + the rank block s·x·Aᵀ [M, r] bf16 + rank-pass scratch
    assert L.workspace_size(L.OP_FWD, 256, 512, 512, 8) == 256 + 256 * 8 * 2 + _rank_scratch(16)
    assert L.workspace_size(L.OP_QK_ROPE_FWD, 256, 512, 512, 8) == (
        256 + 256 * 16 * 2 + _rank_scratch(16))
    assert L.workspace_size(L.OP_FWD, 8192, 4096, 4096, 64) == (
        256 + 8192 * 64 * 2 + _rank_scratch(64))
    b = L.workspace_size(L.OP_BWD, 256, 512, 512, 8)
    assert b > 256 and b % 256 == 0
    assert L.workspace_size(L.OP_BWD, 8192, 4096, 4096, 64) > L.workspace_size(
        L.OP_BWD, 4096, 4096, 4096, 64)
    qk = L.workspace_size(L.OP_QK_ROPE_BWD, 8192, 4096, 5120, 64)
    assert qk >= 256 + 8192 * 5120 * 2
    for bad in ((L.OP_FWD, 0, 64, 64, 8), (L.OP_FWD, 64, 64, 64, 12), (99, 64, 64, 64, 8)):
        assert L.workspace_size(*bad) == 0
    assert L.lora_rope_cache_bytes(8192, 128) == 8192 * 128 * 4
    # dropout: the plain op's workspace plus x̃ [M, k] bf16
    assert L.workspace_size(L.OP_FWD_DROPOUT, 256, 512, 512, 8) == (
        L.workspace_size(L.OP_FWD, 256, 512, 512, 8) + 256 * 512 * 2)
    assert L.workspace_size(L.OP_BWD_DROPOUT, 256, 512, 512, 8) == (
        L.workspace_size(L.OP_BWD, 256, 512, 512, 8) + 256 * 512 * 2)
    # merge: the status word; NF4 merge also a bf16 copy of W [n, k]
    assert L.workspace_size(L.OP_MERGE, 1, 512, 256, 16) == 256
    assert L.workspace_size(L.OP_MERGE_NF4, 1, 512, 256, 16) == 256 + 256 * 512 * 2
    # SwiGLU pair: rank 2r layouts
    assert L.workspace_size(L.OP_SWIGLU_FWD, 256, 512, 512, 8) == (
        L.workspace_size(L.OP_QK_ROPE_FWD, 256, 512, 512, 8))


def test_workspace_room_for_double_quantised_scales():
    # OP_FLAG_DQ adds the bf16 expansion of the block scales, n·k/64 · 2
    # bytes per weight (256-aligned); q/k pairs and gate/up hold two weights
    for op in (L.OP_FWD, L.OP_BWD, L.OP_FWD_DROPOUT, L.OP_BWD_DROPOUT):
        assert L.workspace_size(op | L.OP_FLAG_DQ, 512, 4096, 1024, 16) == (
            L.workspace_size(op, 512, 4096, 1024, 16) + 1024 * 64 * 2)
    assert L.workspace_size(L.OP_SWIGLU_BWD | L.OP_FLAG_DQ, 512, 4096, 1024, 16) == (
        L.workspace_size(L.OP_SWIGLU_BWD, 512, 4096, 1024, 16) + 2 * 1024 * 64 * 2)
    assert L.workspace_size(L.OP_QK_ROPE_FWD | L.OP_FLAG_DQ, 512, 4096, 1280, 16) >= (
        L.workspace_size(L.OP_QK_ROPE_FWD, 512, 4096, 1280, 16) + 1280 * 64 * 2)
    # merges decode the scales directly: no extra room
    assert L.workspace_size(L.OP_MERGE_NF4 | L.OP_FLAG_DQ, 1, 512, 256, 16) == (
        L.workspace_size(L.OP_MERGE_NF4, 1, 512, 256, 16))


def _w(ptr=FAKE, typ=0, absmax=None, bs=0, dtype=0, scale=None, offset=None):
    return L.Weight(typ, ptr, absmax, bs, dtype, scale, offset)


def _fwd(M=256, k=512, n=512, r=8, x=FAKE, W=None, A=FAKE, B=FAKE, y=FAKE, ws=FAKE, wsb=8 << 20,
         alpha=16.0):
    return lib.lora_linear_fwd(x, W or _w(), A, B, y, M, k, n, r, alpha, ws, wsb, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(M=0), 1), (dict(k=-64), 1), (dict(k=100), 2), (dict(n=96), 2), (dict(r=12), 2),
    (dict(r=128), 2), (dict(x=0), 1), (dict(x=MIS), 1), (dict(y=MIS), 1), (dict(A=0), 1),
    (dict(ws=0), 1), (dict(wsb=4351), 3), (dict(alpha=float("nan")), 1),
    (dict(W=L.Weight(7, FAKE, None, 0)), 1),
    (dict(W=L.Weight(1, FAKE, None, 64)), 1),            # NF4 without absmax
    (dict(W=L.Weight(1, FAKE, MIS, 64)), 1),             # NF4 absmax not 16-byte aligned
    (dict(W=L.Weight(1, FAKE, FAKE, 128)), 2),           # NF4 block size other than 64
    (dict(W=_w(dtype=2)), 1),                            # 16-bit type neither bf16 nor fp16
    (dict(W=_w(scale=FAKE, offset=FAKE)), 1),            # dense W with DQ scales
    (dict(W=_w(typ=1, absmax=FAKE, bs=64, scale=FAKE)), 1),       # DQ scale without offset
    (dict(W=_w(typ=1, absmax=FAKE, bs=64, scale=MIS, offset=FAKE)), 1),
    # a DQ weight needs the DQ room: the plain workspace is too small
    (dict(W=_w(typ=1, absmax=FAKE, bs=64, scale=FAKE, offset=FAKE),
          wsb=L.workspace_size(L.OP_FWD, 256, 512, 512, 8)), 3),
])
def test_fwd_rejects_bad_arguments(kw, expect):
    assert _fwd(**kw) == expect


def test_bwd_rejects_bad_arguments():
    need = L.workspace_size(L.OP_BWD, 256, 512, 512, 8)
    args = lambda **o: lib.lora_linear_bwd(
        o.get("x", FAKE), _w(), FAKE, FAKE, o.get("dy", FAKE), o.get("dx", FAKE), 0,
        o.get("dA", FAKE), FAKE, 256, 512, 512, 8, 16.0, FAKE, o.get("wsb", need), None)
    assert args(dy=MIS) == 1
    assert args(dA=0) == 1
    assert args(wsb=need - 1) == 3


def test_qk_rope_rejects_bad_arguments():
    def call(head_dim=128, nqh=2, nkh=1, pos=FAKE, cache=FAKE, theta=5e5, wsb=1 << 20, max_pos=64):
        return lib.lora_qk_rope_fwd(FAKE, _w(), FAKE, FAKE, _w(), FAKE, FAKE, FAKE, FAKE, 64, 256,
                                    nqh, nkh, head_dim, 16, 16.0, theta, pos, cache, max_pos,
                                    FAKE, wsb, None)
    assert call(head_dim=64) == 2
    assert call(nqh=0) == 1
    assert call(pos=0) == 1
    assert call(cache=0, theta=-1.0) == 1
    assert call(max_pos=0) == 1
    assert call(cache=0, wsb=256) == 3       # cache built in the workspace needs room


def test_nf4_and_cache_reject_bad_arguments():
    nf4 = lambda **kw: _w(**{**dict(typ=1, absmax=FAKE, bs=64), **kw})
    assert lib.nf4_dequant(nf4(bs=32), FAKE, 64, 64, None) == 2
    assert lib.nf4_dequant(nf4(), FAKE, 64, 100, None) == 2          # k % 64
    assert lib.nf4_dequant(nf4(ptr=MIS), FAKE, 64, 64, None) == 1
    assert lib.nf4_dequant(_w(), FAKE, 64, 64, None) == 1            # dense descriptor
    assert lib.nf4_dequant(nf4(), MIS, 64, 64, None) == 1
    assert lib.nf4_quantize(FAKE, nf4(absmax=0), 64, 64, None) == 1
    assert lib.nf4_quantize(FAKE, nf4(scale=FAKE), 64, 64, None) == 1  # DQ scale, no offset
    assert lib.lora_rope_cache_build(FAKE, 0, 128, 1e4, None) == 1
    assert lib.lora_rope_cache_build(FAKE, 16, 128, 0.0, None) == 1
    assert lib.lora_read_device_status(None, None, None) == 1


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_gpu_fails_loudly():
    """No CPU fallback: a well-formed call on a machine without a GPU
    returns a CUDA error instead of computing anything."""
    assert _fwd() in (4, 5)


def test_profile_session_rejects_bad_use_without_a_gpu_call():
    # capacity outside [1, 65536], or ending a session that is not open,
    # is an argument error decided on the host
    assert lib.lora_profile_begin(0) == 1
    assert lib.lora_profile_begin(1 << 17) == 1
    assert lib.lora_profile_end(None, None, 0, None) == 1



def test_dropout_and_merge_reject_bad_arguments_before_any_cuda_call():
    need = L.workspace_size(L.OP_FWD_DROPOUT, 256, 512, 512, 8)
    fwd = lambda p=0.1, wsb=need: lib.lora_linear_fwd_dropout(
        FAKE, _w(), FAKE, FAKE, FAKE, 256, 512, 512, 8, 16.0, p, 1, 0, FAKE, wsb, None)
    assert fwd(p=1.0) == 1 and fwd(p=-0.1) == 1 and fwd(p=float("nan")) == 1
    assert fwd(wsb=need - 1) == 3
    assert lib.lora_merge(_w(), FAKE, FAKE, 256, 512, 16, 16.0, 0, FAKE, 256, None) == 1  # sign
    assert lib.lora_merge(_w(), FAKE, FAKE, 256, 512, 12, 16.0, 1, FAKE, 256, None) == 2  # rank
    assert lib.lora_merge(_w(), FAKE, FAKE, 256, 512, 16, 16.0, 1, FAKE, 255, None) == 3
    nf4 = _w(typ=1, absmax=FAKE, bs=32)
    assert lib.lora_merge(nf4, FAKE, FAKE, 256, 512, 16, 16.0, 1, FAKE, 1 << 20, None) == 2
    nf4 = _w(typ=1, absmax=FAKE, bs=64)
    need = L.workspace_size(L.OP_MERGE_NF4, 1, 512, 256, 16)
    assert lib.lora_merge(nf4, FAKE, FAKE, 256, 512, 16, 16.0, 1, FAKE, need - 1, None) == 3
