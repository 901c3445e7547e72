"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test ties an oracle function to something independent of its own code:
a special case that reduces to a library routine, an algebraic identity
that takes a different route, finite differences, invariants of rotations,
a published table, brute force on tiny inputs, or a hand-derived example.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def _rand(*shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _golden_kv(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        out[key] = vals
    return out


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------
def test_worked_example_forward_and_backward():
    g = _golden_kv("lora_worked_example.txt")
    f = lambda k: np.array([float(v) for v in g[k]])
    x = f("x").reshape(1, 2)
    W = f("W").reshape(2, 2)
    A = f("A").reshape(2, 2)
    B = f("B").reshape(2, 2)
    alpha = float(g["alpha"][0])
    y = ref.lora_fwd(x, W, A, B, alpha)
    np.testing.assert_array_equal(y, f("y").reshape(1, 2))
    dx, dA, dB = ref.lora_bwd(x, W, A, B, f("dY").reshape(1, 2), alpha)
    np.testing.assert_array_equal(dx, f("dX").reshape(1, 2))
    np.testing.assert_array_equal(dA, f("dA").reshape(2, 2))
    np.testing.assert_array_equal(dB, f("dB").reshape(2, 2))


@pytest.mark.parametrize("M,k,n,r", [(5, 7, 3, 2), (16, 32, 24, 8)])
def test_b_zero_is_plain_linear(M, k, n, r):
    """B = 0 removes the adapter: y is torch's F.linear, dX its autograd
    gradient, and dA = 0."""
    x, W, A = _rand(M, k), _rand(n, k), _rand(r, k)
    B = np.zeros((n, r))
    y = ref.lora_fwd(x, W, A, B, alpha=16.0)
    xt = torch.tensor(x, requires_grad=True)
    yt = torch.nn.functional.linear(xt, torch.tensor(W))
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=0, atol=1e-12)
    G = _rand(M, n)
    yt.backward(torch.tensor(G))
    dx, dA, dB = ref.lora_bwd(x, W, A, B, G, alpha=16.0)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=0, atol=1e-12)
    assert np.all(dA == 0.0)
    # dB = s·dYᵀ·(x·Aᵀ) does not vanish when B = 0
    assert np.abs(dB).max() > 0


def test_merged_weight_identity():
    """y equals the plain linear map with the adapter folded into W
    (different association of the same product)."""
    M, k, n, r, alpha = 9, 12, 10, 3, 6.0
    x, W, A, B = _rand(M, k), _rand(n, k), _rand(r, k), _rand(n, r)
    s = alpha / r
    Wm = np.array(W)
    for i in range(n):                       # W + s·B·A by explicit loops
        for j in range(k):
            Wm[i, j] += s * sum(B[i, l] * A[l, j] for l in range(r))
    y_merged = torch.nn.functional.linear(torch.tensor(x), torch.tensor(Wm)).numpy()
    np.testing.assert_allclose(ref.lora_fwd(x, W, A, B, alpha), y_merged, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ref.merged_weight(W, A, B, alpha), Wm, rtol=1e-13, atol=1e-13)


def test_w_zero_and_alpha_linearity():
    M, k, n, r = 6, 8, 5, 2
    x, W, A, B = _rand(M, k), _rand(n, k), _rand(r, k), _rand(n, r)
    y0 = ref.lora_fwd(x, W, A, B, 0.0)
    y1 = ref.lora_fwd(x, W, A, B, 3.0)
    y2 = ref.lora_fwd(x, W, A, B, 6.0)
    np.testing.assert_allclose(y2 - y0, 2.0 * (y1 - y0), rtol=1e-12, atol=1e-12)
    # W = 0 leaves only the adapter; with r = 1 it is a rank-one outer product
    A1, B1 = _rand(1, k), _rand(n, 1)
    yz = ref.lora_fwd(x, np.zeros((n, k)), A1, B1, 5.0)
    outer = 5.0 * np.outer(x @ A1[0], B1[:, 0])
    np.testing.assert_allclose(yz, outer, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# backward: central finite differences of L = sum(G ⊙ y)
# --------------------------------------------------------------------------
def _fd_grad(fun, P, h=1e-6):
    g = np.zeros_like(P)
    for idx in np.ndindex(P.shape):
        old = P[idx]
        P[idx] = old + h
        fp = fun()
        P[idx] = old - h
        fm = fun()
        P[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


def test_backward_matches_finite_differences():
    M, k, n, r, alpha = 3, 8, 6, 2, 5.0
    x, W, A, B, G = _rand(M, k), _rand(n, k), _rand(r, k), _rand(n, r), _rand(M, n)
    L = lambda: float(np.sum(G * ref.lora_fwd(x, W, A, B, alpha)))
    dx, dA, dB = ref.lora_bwd(x, W, A, B, G, alpha)
    for P, an in ((x, dx), (A, dA), (B, dB)):
        num = _fd_grad(L, P)
        np.testing.assert_allclose(an, num, rtol=1e-7, atol=1e-7)


def test_qk_rope_backward_matches_finite_differences():
    M, k, D, r, alpha, theta = 3, 8, 4, 2, 4.0, 100.0
    nq, nk = 2 * D, D
    x = _rand(M, k)
    Wq, Aq, Bq = _rand(nq, k), _rand(r, k), _rand(nq, r)
    Wk, Ak, Bk = _rand(nk, k), _rand(r, k), _rand(nk, r)
    Gq, Gk = _rand(M, nq), _rand(M, nk)
    pos = np.array([0, 3, 7])

    def L():
        q, kk = ref.qk_rope_fwd(x, Wq, Aq, Bq, Wk, Ak, Bk, alpha, pos, theta, head_dim=D)
        return float(np.sum(Gq * q) + np.sum(Gk * kk))

    dx, dAq, dBq, dAk, dBk = ref.qk_rope_bwd(x, Wq, Aq, Bq, Wk, Ak, Bk, Gq, Gk, alpha, pos,
                                             theta, head_dim=D)
    for P, an in ((x, dx), (Aq, dAq), (Bq, dBq), (Ak, dAk), (Bk, dBk)):
        np.testing.assert_allclose(an, _fd_grad(L, P), rtol=1e-7, atol=1e-7)


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------
D, THETA = 128, 500000.0


def test_rope_position_zero_is_identity():
    y = _rand(4, 2 * D)
    np.testing.assert_array_equal(ref.rope_apply(y, np.zeros(4), D, THETA), y)


def test_rope_preserves_pair_norms():
    y = _rand(5, 3 * D)
    pos = np.array([1, 17, 400, 8191, 3])
    z = ref.rope_apply(y, pos, D, THETA)
    h = D // 2
    yn = y.reshape(5, 3, D)
    zn = z.reshape(5, 3, D)
    np.testing.assert_allclose(yn[..., :h] ** 2 + yn[..., h:] ** 2,
                               zn[..., :h] ** 2 + zn[..., h:] ** 2, rtol=1e-12)


def test_rope_relative_position():
    """<R_m q, R_n k> depends only on m - n."""
    q, k = _rand(1, D), _rand(1, D)
    for m, n, t in ((5, 2, 100), (8191, 10, -7), (0, 0, 4000)):
        a = ref.rope_apply(q, [m], D, THETA) @ ref.rope_apply(k, [n], D, THETA).T
        b = ref.rope_apply(q, [m + t], D, THETA) @ ref.rope_apply(k, [n + t], D, THETA).T
        assert abs(a.item() - b.item()) < 1e-9


def test_rope_single_frequency_closed_form():
    """A unit vector in pair (i, i+D/2) rotates by p·theta^(-2i/D)."""
    for i in (0, 1, 31, 63):
        for p in (1, 5, 1000, 8191):
            y = np.zeros((1, D))
            y[0, i] = 1.0
            z = ref.rope_apply(y, [p], D, THETA)
            phi = p * THETA ** (-2.0 * i / D)
            assert abs(z[0, i] - math.cos(phi)) < 1e-12
            assert abs(z[0, i + D // 2] - math.sin(phi)) < 1e-12
            z[0, i] = z[0, i + D // 2] = 0.0
            assert np.all(z == 0.0)


def test_rope_inverse_is_transpose():
    pos = np.array([0, 1, 2, 999])
    y = _rand(4, 2 * D)
    np.testing.assert_allclose(ref.rope_apply_inverse(ref.rope_apply(y, pos, D, THETA), pos, D,
                                                      THETA), y, rtol=1e-12, atol=1e-12)
    # <R y, z> == <y, R^T z>
    z = _rand(4, 2 * D)
    lhs = np.sum(ref.rope_apply(y, pos, D, THETA) * z)
    rhs = np.sum(y * ref.rope_apply_inverse(z, pos, D, THETA))
    assert abs(lhs - rhs) < 1e-9


# --------------------------------------------------------------------------
# NF4
# --------------------------------------------------------------------------
def test_nf4_codebook_matches_published_table():
    pub = np.array([float(v[0]) for k, v in _golden_kv("nf4_codebook_qlora.txt").items()])
    c = ref.nf4_codebook()
    assert c.shape == (16,)
    np.testing.assert_allclose(c, pub, rtol=0, atol=3e-7)
    assert np.all(np.diff(c) > 0)
    assert c[0] == -1.0 and c[7] == 0.0 and c[15] == 1.0


def test_nf4_hand_example_packing():
    g = _golden_kv("nf4_packing_example.txt")
    w = np.zeros((1, 64))
    w[0, :4] = [-2.0, 2.0, 0.0, 1.0]
    codes, absmax = ref.nf4_quantize(w)
    assert absmax[0, 0] == float(g["absmax"][0])
    assert codes[0, 0] == int(g["byte0"][0], 16)
    assert codes[0, 1] == int(g["byte1"][0], 16)
    assert np.all(codes[0, 2:] == int(g["rest"][0], 16))


def test_nf4_round_trip_on_levels():
    c = ref.nf4_codebook()
    a = 0.8125                             # a bf16 value
    for decision in ("fp64", "fp32"):
        idx = np.tile(np.arange(16), 4)      # 64 elements, every level
        w = (c[idx] * a).reshape(1, 64)
        w[0, 15] = a                         # keep the block's absmax exactly a
        codes, absmax = ref.nf4_quantize(w, decision=decision)
        assert absmax[0, 0] == a
        np.testing.assert_array_equal(ref.nf4_unpack(codes)[0], idx)
        np.testing.assert_array_equal(ref.nf4_dequant(codes, absmax), w)


def test_nf4_absmax_element_maps_to_an_end():
    w = _rand(8, 256)
    w = ref.bf16_round(w)
    codes, absmax = ref.nf4_quantize(w)
    idx = ref.nf4_unpack(codes).reshape(8, 4, 64)
    blocks = w.reshape(8, 4, 64)
    for i in range(8):
        for b in range(4):
            j = int(np.argmax(np.abs(blocks[i, b])))
            assert idx[i, b, j] == (15 if blocks[i, b, j] > 0 else 0)


def test_nf4_zero_block_is_code_7():
    w = np.zeros((2, 128))
    w[1, 64:] = _rand(64)
    codes, absmax = ref.nf4_quantize(w)
    assert absmax[0, 0] == 0 and absmax[0, 1] == 0 and absmax[1, 0] == 0
    idx = ref.nf4_unpack(codes)
    assert np.all(idx[0] == 7) and np.all(idx[1, :64] == 7)


@pytest.mark.parametrize("decision", ["fp64", "fp32"])
def test_nf4_quantiser_is_brute_force_nearest(decision):
    w = ref.bf16_round(_rand(3, 128, scale=0.05))
    codes, absmax = ref.nf4_quantize(w, decision=decision)
    idx = ref.nf4_unpack(codes)
    c = ref.nf4_codebook()
    for i in range(3):
        for j in range(128):
            a = absmax[i, j // 64]
            if decision == "fp32":
                ratio = np.float32(w[i, j]) / np.float32(a)
                best, bestd = 0, None
                for t in range(16):
                    d = abs(ratio - np.float32(c[t]))
                    if bestd is None or d < bestd:
                        best, bestd = t, d
            else:
                ratio = w[i, j] / a
                best = min(range(16), key=lambda t: (abs(ratio - c[t]), t))
            assert idx[i, j] == best


def test_nf4_row_passes_do_not_change_the_result():
    w = ref.bf16_round(_rand(10, 128, scale=0.1))
    for decision in ("fp64", "fp32"):
        c1, a1 = ref.nf4_quantize(w, decision=decision)
        c2, a2 = ref.nf4_quantize(w, decision=decision, rows_per_pass=3)
        np.testing.assert_array_equal(c1, c2)
        np.testing.assert_array_equal(a1, a2)


def test_nf4_dequant_error_bound():
    """Dequantised weights are within half the widest level gap (times
    absmax) of the originals."""
    w = ref.bf16_round(_rand(4, 512, scale=0.02))
    codes, absmax = ref.nf4_quantize(w)
    wd = ref.nf4_dequant(codes, absmax)
    gap = np.max(np.diff(ref.nf4_codebook())) / 2
    bound = np.repeat(absmax, 64, axis=1) * gap
    assert np.all(np.abs(wd - w) <= bound + 1e-15)


def test_bf16_round_matches_torch():
    v = rng.standard_normal(10000).astype(np.float32) * np.float32(10.0) ** rng.integers(
        -30, 30, 10000).astype(np.float32)
    mine = ref.bf16_round(v.astype(np.float64))
    theirs = torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(mine, theirs)


def test_param_count_closed_form():
    """4096x4096 at rank 16: 2 x 4096 x 16 = 131072 trainable parameters
    (the page's "约13万")."""
    assert ref.lora_param_count(4096, 4096, 16) == 131072


# --------------------------------------------------------------------------
# SwiGLU gate/up composition
# --------------------------------------------------------------------------
def test_silu_and_sigmoid_match_torch():
    t = np.concatenate([_rand(200, scale=4.0), [-800.0, -40.0, -1e-300, 0.0, 1e-300, 40.0, 800.0]])
    tt = torch.from_numpy(t)
    np.testing.assert_allclose(ref.silu(t), torch.nn.functional.silu(tt).numpy(),
                               rtol=1e-15, atol=1e-300)
    np.testing.assert_allclose(ref.sigmoid(t), torch.sigmoid(tt).numpy(), rtol=1e-15,
                               atol=1e-300)


def _swiglu_torch(x, Wg, Ag, Bg, Wu, Au, Bu, alpha):
    """The same composition written with torch layers (fp64) for autograd."""
    F = torch.nn.functional
    s = alpha / Ag.shape[0]
    g = F.linear(x, Wg) + s * F.linear(F.linear(x, Ag), Bg)
    u = F.linear(x, Wu) + s * F.linear(F.linear(x, Au), Bu)
    return F.silu(g) * u


def test_swiglu_forward_and_backward_match_torch_autograd():
    M, k, n, r, alpha = 7, 24, 10, 4, 8.0
    arrs = [_rand(M, k), _rand(n, k, scale=0.3), _rand(r, k, scale=0.3), _rand(n, r, scale=0.3),
            _rand(n, k, scale=0.3), _rand(r, k, scale=0.3), _rand(n, r, scale=0.3)]
    dh = _rand(M, n)
    h, g, u = ref.swiglu_fwd(*arrs, alpha)
    ts = [torch.tensor(a, requires_grad=True) for a in arrs]
    ht = _swiglu_torch(*ts, alpha)
    np.testing.assert_allclose(h, ht.detach().numpy(), rtol=1e-12, atol=1e-12)
    ht.backward(torch.from_numpy(dh))
    dx, dAg, dBg, dAu, dBu = ref.swiglu_bwd(*arrs, dh, alpha)
    want = [ts[0].grad, ts[2].grad, ts[3].grad, ts[5].grad, ts[6].grad]
    for got, w in zip((dx, dAg, dBg, dAu, dBu), want):
        np.testing.assert_allclose(got, w.numpy(), rtol=1e-10, atol=1e-12)


def test_swiglu_backward_matches_finite_differences():
    M, k, n, r, alpha = 3, 8, 5, 2, 4.0
    x, Wg, Ag, Bg = _rand(M, k), _rand(n, k), _rand(r, k), _rand(n, r)
    Wu, Au, Bu, G = _rand(n, k), _rand(r, k), _rand(n, r), _rand(M, n)
    L = lambda: float(np.sum(G * ref.swiglu_fwd(x, Wg, Ag, Bg, Wu, Au, Bu, alpha)[0]))
    dx, dAg, dBg, dAu, dBu = ref.swiglu_bwd(x, Wg, Ag, Bg, Wu, Au, Bu, G, alpha)
    for P, an in ((x, dx), (Ag, dAg), (Bg, dBg), (Au, dAu), (Bu, dBu)):
        np.testing.assert_allclose(an, _fd_grad(L, P), rtol=1e-6, atol=1e-7)


def test_swiglu_with_a_zero_gate_has_closed_form_gradients():
    """g ≡ 0 (Wg = 0, Bg = 0): h = 0, silu'(0) = 1/2 so dg = dh·u/2, du = 0,
    and the up projection receives no gradient."""
    M, k, n, r, alpha = 5, 16, 6, 2, 2.0
    x, Ag, Wu, Au, Bu, dh = (_rand(M, k), _rand(r, k), _rand(n, k), _rand(r, k), _rand(n, r),
                             _rand(M, n))
    Wg, Bg = np.zeros((n, k)), np.zeros((n, r))
    h, g, u = ref.swiglu_fwd(x, Wg, Ag, Bg, Wu, Au, Bu, alpha)
    assert np.all(h == 0) and np.all(g == 0)
    dx, dAg, dBg, dAu, dBu = ref.swiglu_bwd(x, Wg, Ag, Bg, Wu, Au, Bu, dh, alpha)
    s = alpha / r
    dg = 0.5 * dh * u
    np.testing.assert_allclose(dx, s * (dg @ Bg) @ Ag + dg @ Wg, atol=1e-12)
    np.testing.assert_allclose(dBg, s * dg.T @ (x @ Ag.T), rtol=1e-12, atol=1e-12)
    assert np.all(dAg == 0) and np.all(dAu == 0) and np.all(dBu == 0)


# --------------------------------------------------------------------------
# merge / unmerge
# --------------------------------------------------------------------------
def test_unmerge_inverts_merge_elementwise_loops():
    n, k, r, alpha = 5, 7, 3, 6.0
    W, A, B = _rand(n, k), _rand(r, k), _rand(n, r)
    Wm = ref.merged_weight(W, A, B, alpha)
    s = alpha / r
    for i in range(n):              # the merged element, summed by hand
        for j in range(k):
            assert abs(Wm[i, j] - (W[i, j] + s * sum(B[i, l] * A[l, j] for l in range(r)))) < 1e-12
    np.testing.assert_allclose(ref.unmerged_weight(Wm, A, B, alpha), W, rtol=0, atol=1e-12)


def test_nf4_merge_with_b_zero_keeps_codes_and_absmax():
    """B = 0 adds nothing: dequantise then quantise gives back the same
    codes and block scales (every level maps to itself, and each block's
    largest level is ±1 times its bf16 absmax)."""
    w = ref.bf16_round(_rand(6, 192))
    codes, absmax = ref.nf4_quantize(w)
    A, B = _rand(4, 192), np.zeros((6, 4))
    for sign in (1.0, -1.0):
        c2, a2 = ref.nf4_merge(codes, absmax, A, B, 16.0, sign)
        np.testing.assert_array_equal(c2, codes)
        np.testing.assert_array_equal(a2, absmax)


def test_nf4_merge_is_within_the_quantisation_bound_of_the_merged_weight():
    w = ref.bf16_round(_rand(8, 256, scale=0.05))
    codes, absmax = ref.nf4_quantize(w)
    A, B, alpha = _rand(4, 256, scale=0.1), _rand(8, 4, scale=0.1), 8.0
    Wm = ref.merged_weight(ref.nf4_dequant(codes, absmax), A, B, alpha)
    c2, a2 = ref.nf4_merge(codes, absmax, A, B, alpha)
    got = ref.nf4_dequant(c2, a2)
    gaps = np.diff(ref.nf4_codebook()).max()
    bound = np.repeat(a2, 64, axis=1) * (gaps / 2) + np.abs(Wm) * 2.0 ** -8
    assert np.all(np.abs(got - Wm) <= bound + 1e-15)


# --------------------------------------------------------------------------
# LoRA dropout: Philox4x64-10 mask
# --------------------------------------------------------------------------
def test_mulhilo64_matches_python_integers():
    r = np.random.default_rng(5)
    a = r.integers(0, 2**63, size=200, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    b = r.integers(0, 2**63, size=200, dtype=np.uint64) | np.uint64(1 << 63)
    from oracle import lora_ref
    hi, lo = lora_ref._mulhilo64(a, b)
    for x, y, h, l in zip(a, b, hi, lo):
        prod = int(x) * int(y)
        assert int(h) == prod >> 64 and int(l) == prod & ((1 << 64) - 1)


@pytest.mark.parametrize("counter,key", [([0, 0, 0, 0], [0, 0]), ([41, 9, 2, 1], [7, 11]),
                                         ([2**64 - 1, 5, 0, 3], [2**64 - 2, 2**63])])
def test_philox4x64_matches_numpy_bit_generator(counter, key):
    """numpy's Philox bit generator is Philox4x64-10; it advances its 256-bit
    counter before each block of four words."""
    c = [int(v) for v in counter]
    prev = (c[0] + (c[1] << 64) + (c[2] << 128) + (c[3] << 192) - 1) % (1 << 256)
    prev_words = [(prev >> (64 * i)) & ((1 << 64) - 1) for i in range(4)]
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.array(prev_words, dtype=np.uint64))
    want = [int(v) for v in bg.random_raw(4)]
    got = [int(v) for v in ref.philox4x64(np.array([c], dtype=np.uint64), key)[0]]
    assert got == want


def test_dropout_mask_element_mapping_and_rate():
    M, k, p, seed, off = 37, 96, 0.25, 2024, 5
    keep = ref.dropout_keep(M, k, p, seed, off)
    t = round(p * 65536)
    # a few elements recomputed one by one from the Philox block they index
    for e in (0, 1, 15, 16, 17, 1000, M * k - 1):
        words = ref.philox4x64(np.array([[e // 16, off, 0, 0]], dtype=np.uint64), (seed, 0))[0]
        u16 = (int(words[(e % 16) // 4]) >> (16 * (e % 4))) & 0xFFFF
        assert keep[e // k, e % k] == (u16 >= t)
    big = ref.dropout_keep(256, 1024, 0.1, 1, 0)
    q = ref.dropout_keep_prob(0.1)
    sd = math.sqrt(q * (1 - q) / big.size)
    assert abs(big.mean() - q) < 5 * sd
    assert np.array_equal(ref.dropout_keep(M, k, p, seed, off), keep)          # regenerated
    assert not np.array_equal(ref.dropout_keep(M, k, p, seed, off + 1), keep)  # per-step offset
    assert ref.dropout_keep(M, k, 0.0, seed, off).all()                         # p = 0 keeps all


def test_dropout_zero_is_plain_lora_and_gradients_match_autograd():
    M, k, n, r, alpha = 9, 32, 12, 4, 8.0
    x, W, A, B, dy = _rand(M, k), _rand(n, k), _rand(r, k), _rand(n, r), _rand(M, n)
    np.testing.assert_allclose(ref.lora_fwd_dropout(x, W, A, B, alpha, 0.0, 3, 0),
                               ref.lora_fwd(x, W, A, B, alpha), rtol=1e-13, atol=1e-13)
    p, seed, off = 0.3, 77, 2
    keep = torch.from_numpy(ref.dropout_keep(M, k, p, seed, off).astype(np.float64))
    q = ref.dropout_keep_prob(p)
    ts = [torch.tensor(a, requires_grad=True) for a in (x, W, A, B)]
    s = alpha / r
    F = torch.nn.functional
    yt = F.linear(ts[0], ts[1]) + s * F.linear(F.linear(ts[0] * keep / q, ts[2]), ts[3])
    np.testing.assert_allclose(ref.lora_fwd_dropout(x, W, A, B, alpha, p, seed, off),
                               yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    yt.backward(torch.from_numpy(dy))
    dx, dA, dB = ref.lora_bwd_dropout(x, W, A, B, dy, alpha, p, seed, off)
    for got, t in zip((dx, dA, dB), (ts[0], ts[2], ts[3])):
        np.testing.assert_allclose(got, t.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_dropout_backward_matches_finite_differences():
    M, k, n, r, alpha, p, seed, off = 3, 16, 5, 2, 4.0, 0.4, 9, 1
    x, W, A, B, G = _rand(M, k), _rand(n, k), _rand(r, k), _rand(n, r), _rand(M, n)
    L = lambda: float(np.sum(G * ref.lora_fwd_dropout(x, W, A, B, alpha, p, seed, off)))
    dx, dA, dB = ref.lora_bwd_dropout(x, W, A, B, G, alpha, p, seed, off)
    for P, an in ((x, dx), (A, dA), (B, dB)):
        np.testing.assert_allclose(an, _fd_grad(L, P), rtol=1e-6, atol=1e-7)


# --------------------------------------------------------------------------
# fp16 rounding and double-quantised NF4 block scales
# --------------------------------------------------------------------------
def test_f16_round_matches_numpy():
    v = rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000)
    # exact ties between neighbours, subnormals and the overflow edge
    ties = np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 2.0 ** -24 * 1.5, 2.0 ** -24 * 2.5,
                     65504.0, 65519.99, 65520.0, -65520.0, 2.0 ** -25, -2.0 ** -26, 0.0])
    v = np.concatenate([v, ties])
    with np.errstate(over="ignore"):                      # 65520 overflows to inf
        theirs = v.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(ref.f16_round(v), theirs)


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    theirs = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = ref.e4m3_values()
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(theirs))
    ok = ~np.isnan(mine)
    np.testing.assert_array_equal(mine[ok], theirs[ok])
    assert np.nanmax(mine) == 448.0 and np.sum(np.isnan(mine)) == 2


def test_e4m3_round_and_encode_match_torch():
    mag = np.exp2(rng.uniform(-12, np.log2(460.0), 20000))
    v = (mag * rng.choice([-1.0, 1.0], 20000)).astype(np.float32)
    # ties (midpoints of the grid), tiny negatives and the saturation edge
    extra = np.array([1.0625, 1.1875, 136.0, 152.0, -2.0 ** -10, 2.0 ** -10, -1e-6, 447.9,
                      448.0, 455.0, -455.0, 0.0], dtype=np.float32)
    v = np.concatenate([v, extra])
    t = torch.tensor(v).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(ref.e4m3_round(v.astype(np.float64)),
                                  t.to(torch.float64).numpy())
    np.testing.assert_array_equal(ref.e4m3_encode(v.astype(np.float64)),
                                  t.view(torch.uint8).numpy())


def test_dq_hand_example():
    g = _golden_kv("dq_worked_example.txt")
    codes, scale, offset = ref.dq_encode(np.array([0.5, 1.0, 1.5, 2.0]))
    assert float(offset) == float(g["offset"][0])
    assert [int(c) for c in codes] == [int(c, 16) for c in g["codes"]]
    assert float(scale[0]) == float(np.float32(0.75) / np.float32(448.0))
    np.testing.assert_array_equal(ref.dq_decode(codes, scale, offset),
                                  [float(x) for x in g["decoded"]])


def test_dq_invariants_over_groups_of_different_spread():
    # three groups of 256 with very different spreads, and a ragged last group
    c1 = np.concatenate([0.02 + 0.001 * rng.random(256), 0.02 + 0.02 * rng.random(256),
                         0.5 * rng.random(256), 0.03 + 0.001 * rng.random(64)])
    c1 = ref.bf16_round(c1).astype(np.float32)
    codes, scale, offset = ref.dq_encode(c1)
    assert scale.shape == (4,)
    # the offset is the fp32 of the exact mean
    assert float(offset) == float(np.float32(math.fsum(map(float, c1)) / c1.size))
    dec = ref.dq_decode(codes, scale, offset)
    d = (c1 - offset).astype(np.float32).astype(np.float64)
    for g in range(4):
        sl = slice(256 * g, 256 * (g + 1))
        assert scale[g] == np.float32(np.max(np.abs(d[sl])) / np.float32(448.0))
        # the element of largest |d| lands on the format's end, ±448
        j = np.argmax(np.abs(d[sl]))
        assert codes[sl][j] in (0x7E, 0xFE)
    r = np.abs(d) / np.repeat(scale.astype(np.float64), 256)[:c1.size]
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(r, 2.0 ** -20))), -6) - 3)
    s_el = np.repeat(scale.astype(np.float64), 256)[:c1.size]
    bound = s_el * step / 2 * (1 + 1e-6) + 2.0 ** -8 * np.abs(c1) + 1e-12
    assert np.all(np.abs(dec - c1) <= bound)
    # the narrow first group is reproduced far better than the wide third one
    err = np.abs(dec - c1)
    assert err[:256].max() < err[512:768].max() / 10


def test_dq_of_constant_scales_is_exact():
    c1 = np.full(300, 0.0390625, dtype=np.float32)      # a bf16 value
    codes, scale, offset = ref.dq_encode(c1)
    assert np.all(scale == 0) and np.all(codes == 0)
    np.testing.assert_array_equal(ref.dq_decode(codes, scale, offset), c1.astype(np.float64))


def test_nf4_quantize_dq_is_brute_force_nearest_against_the_decoded_scale():
    w = ref.bf16_round(_rand(4, 256, scale=0.05))
    w[1, 64:128] = 0.0                                    # an all-zero block
    codes, qc, scale, offset = ref.nf4_quantize_dq(w, decision="fp64", group=4)
    assert scale.shape == (4,) and qc.shape == (4, 4)
    am = ref.dq_decode(qc, scale, offset, group=4)
    lv = ref.nf4_codebook()
    idx = ref.nf4_unpack(codes)
    for i in range(4):
        for j in range(256):
            a = am[i, j // 64]
            if a == 0.0:
                assert idx[i, j] == 7
                continue
            t = min(max(w[i, j] / a, -1.0), 1.0)
            best = min(range(16), key=lambda q: (abs(t - lv[q]), q))
            assert idx[i, j] == best, (i, j)
    assert np.all(idx[1, 64:128] == 7)


def test_nf4_dequant_dq_error_bound():
    w = ref.bf16_round(_rand(8, 1024, scale=0.02))
    codes, qc, scale, offset = ref.nf4_quantize_dq(w)
    wd = ref.nf4_dequant_dq(codes, qc, scale, offset)
    c1 = np.repeat(np.max(np.abs(w.reshape(8, 16, 64)), axis=2), 64, axis=1)
    am = np.repeat(ref.dq_decode(qc, scale, offset), 64, axis=1)
    gap = np.max(np.diff(ref.nf4_codebook())) / 2
    bound = np.maximum(c1 - am, 0.0) + am * gap
    assert np.all(np.abs(wd - w) <= bound * (1 + 1e-6) + 1e-15)
