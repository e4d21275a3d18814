"""Pins of the fp64 oracle against what the pages and the mathematics fix.

No GPU.  Each test checks the oracle against something other than itself: a
hand-derived golden value (tests/golden/), a closed form, an invariant the
pages state, or a library routine (numpy/scipy/torch) computing the same
definition.  tests/test_oracle_mutants.py plants plausible mistakes in a copy
of oracle.cpp and checks that this file catches every one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([p.strip() for p in line.split("|")])
    return rows


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ bf16 ----
def test_bf16_golden_values():
    for inp, exp, why in _golden("bf16_rne.txt"):
        got = orc.bf16_round([float(inp)])[0]
        assert got == float(exp), (inp, exp, got, why)


def test_bf16_matches_torch_for_fp32_inputs():
    # torch's fp32 -> bf16 conversion rounds to nearest even: for inputs that
    # are exact fp32 values both must agree bit for bit.
    g = _rng(1)
    x32 = (g.standard_normal(20000) * np.exp2(g.integers(-30, 30, 20000))).astype(np.float32)
    x32 = np.concatenate([x32, np.float32([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 65504.0, 1e-38])])
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = orc.bf16_round(x32.astype(np.float64))
    np.testing.assert_array_equal(got, want)


# --------------------------------------------------------------- RMSNorm ----
def test_rmsnorm_golden_values():
    gold = {r[0]: np.array([float(v) for v in r[2].split()]) for r in _golden("closed_forms.txt")}
    np.testing.assert_allclose(orc.rmsnorm(np.array([[3.0, 4.0]]), np.ones(2), 0.0)[0],
                               gold["rmsnorm_34_g11_eps0"], rtol=1e-15)
    np.testing.assert_allclose(orc.rmsnorm(np.array([[3.0, 4.0]]), np.array([2.0, 0.5]), 0.0)[0],
                               gold["rmsnorm_34_g2h_eps0"], rtol=1e-15)
    np.testing.assert_allclose(orc.rmsnorm(np.ones((1, 4)), np.ones(4), 1.0)[0], gold["rmsnorm_ones_eps1"],
                               rtol=1e-15)


def test_rmsnorm_matches_torch():
    g = _rng(2)
    x = g.standard_normal((7, 96))
    gain = g.standard_normal(96)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), weight=torch.from_numpy(gain), eps=1e-5)
    np.testing.assert_allclose(orc.rmsnorm(x, gain, 1e-5), want.numpy(), rtol=1e-13, atol=1e-14)


def test_rmsnorm_constant_and_scale_invariance():
    c, eps = 0.37, 1e-5
    out = orc.rmsnorm(np.full((1, 64), c), np.full(64, 1.5), eps)
    np.testing.assert_allclose(out, 1.5 * c / math.sqrt(c * c + eps), rtol=1e-15)
    x = _rng(3).standard_normal((5, 64))
    np.testing.assert_allclose(orc.rmsnorm(12.5 * x, np.ones(64), 0.0), orc.rmsnorm(x, np.ones(64), 0.0),
                               rtol=1e-14)


# ---------------------------------------------------------------- linear ----
def test_linear_matches_numpy():
    # the step's projection is orc_linear's plain sums; numpy's matmul (a library
    # routine) pins it, for output counts below, at and above a group of eight and
    # with a ragged last group
    g = _rng(4)
    for rows, D, nout in ((9, 48, 30), (3, 17, 5), (4, 64, 16), (2, 33, 8), (5, 40, 1)):
        x = g.standard_normal((rows, D))
        W = g.standard_normal((nout, D))
        np.testing.assert_allclose(orc.linear(x, W), x @ W.T, rtol=1e-13, atol=1e-13)
        np.testing.assert_array_equal(orc.project(x, W), orc.linear(x, W))


# ------------------------------------------------------------------ RoPE ----
def test_rope_golden_values():
    for idx, pos, exp in _golden("rope_theta1e4_d8.txt"):
        t = np.zeros((1, 1, 8))
        t[0, 0, int(idx)] = 1.0
        got = orc.rope(t, [int(pos)], 1e4)[0, 0]
        np.testing.assert_allclose(got, [float(v) for v in exp.split()], atol=1e-14)


def test_rope_d2_is_plane_rotation():
    g = _rng(5)
    for theta in (1e4, 5e5, 7.0):
        a, b = g.standard_normal(2)
        for p in (0, 1, 17, 3000):
            got = orc.rope(np.array([[[a, b]]]), [p], theta)[0, 0]
            want = [a * math.cos(p) - b * math.sin(p), b * math.cos(p) + a * math.sin(p)]
            np.testing.assert_allclose(got, want, atol=1e-12)


def test_rope_relative_position_and_norm():
    g = _rng(6)
    d, H = 64, 3
    q = g.standard_normal((1, H, d))
    k = g.standard_normal((1, H, d))
    p, pp, s = 37, 5, 911
    dot0 = np.einsum("hd,hd->h", orc.rope(q, [p], 5e5)[0], orc.rope(k, [pp], 5e5)[0])
    dot1 = np.einsum("hd,hd->h", orc.rope(q, [p + s], 5e5)[0], orc.rope(k, [pp + s], 5e5)[0])
    np.testing.assert_allclose(dot1, dot0, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(np.linalg.norm(orc.rope(q, [p], 5e5), axis=-1), np.linalg.norm(q, axis=-1),
                               rtol=1e-13)
    np.testing.assert_array_equal(orc.rope(q, [0], 5e5), q)


# ------------------------------------------------------------- attention ----
def test_attention_golden_two_keys():
    gold = {(r[0], r[1]): np.array([float(v) for v in r[2].split()]) for r in _golden("closed_forms.txt")}
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    v = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    O, L = orc.attention(q, k, v, 1.0)
    np.testing.assert_allclose(O[0, 0], gold[("attention_two_keys", "O")], rtol=1e-15)
    np.testing.assert_allclose(L[0], gold[("attention_two_keys", "L")], rtol=1e-15)


def test_attention_matches_scipy_softmax():
    g = _rng(7)
    nq, nk, H, d = 6, 23, 3, 16
    q, k, v = g.standard_normal((nq, H, d)), g.standard_normal((nk, H, d)), g.standard_normal((nk, H, d))
    scale = 1 / math.sqrt(d)
    O, L = orc.attention(q, k, v, scale)
    for h in range(H):
        S = scale * q[:, h] @ k[:, h].T
        np.testing.assert_allclose(O[:, h], scipy.special.softmax(S, axis=1) @ v[:, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(L[:, h], scipy.special.logsumexp(S, axis=1), rtol=1e-13)


def test_attention_closed_forms():
    g = _rng(8)
    H, d = 2, 8
    v = g.standard_normal((5, H, d))
    q = g.standard_normal((1, H, d))
    # all keys equal -> O = mean of the values, L = s + ln 5
    k = np.repeat(g.standard_normal((1, H, d)), 5, axis=0)
    O, L = orc.attention(q, k, v, 0.5)
    np.testing.assert_allclose(O[0], v.mean(axis=0), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L[0], 0.5 * np.einsum("hd,hd->h", q[0], k[0]) + math.log(5), rtol=1e-13)
    # one key with a score larger by >= 60 -> O = its value
    k = np.zeros((5, H, d))
    qq = np.zeros((1, H, d))
    qq[0, :, 0] = 1.0
    k[3, :, 0] = 100.0
    O, _ = orc.attention(qq, k, v, 1.0)
    np.testing.assert_allclose(O[0], v[3], rtol=1e-12, atol=1e-12)
    # a single key -> O = v, L = its score
    O, L = orc.attention(q, k[:1] + 1.0, v[:1], 1.0)
    np.testing.assert_allclose(O[0], v[0], rtol=1e-14)


def test_attention_permutation_invariance_and_probabilities():
    g = _rng(9)
    nk, H, d = 16, 2, 16
    q, k = g.standard_normal((4, H, d)), g.standard_normal((nk, H, d))
    v = np.tile(np.eye(nk)[:, None, :], (1, H, 1))  # v_j = e_j -> O rows are the softmax probabilities
    O, _ = orc.attention(q, k, v, 0.25)
    np.testing.assert_allclose(O.sum(axis=-1), 1.0, rtol=1e-14)
    S = 0.25 * np.einsum("qhd,khd->qhk", q, k)
    np.testing.assert_allclose(O[..., 3] / O[..., 7], np.exp(S[..., 3] - S[..., 7]), rtol=1e-12)
    perm = g.permutation(nk)
    O2, _ = orc.attention(q, k[perm], v[perm], 0.25)
    np.testing.assert_allclose(O2, O, rtol=1e-13, atol=1e-15)


# --------------------------------------------- online softmax, Eq. (2)-(6) --
@pytest.mark.parametrize("bc", [1, 3, 7, 64, 45])
def test_online_equals_two_pass(bc):
    g = _rng(10 + bc)
    nq, nk, H, d = 5, 45, 2, 16
    q, k, v = (g.standard_normal((n, H, d)) * 2 for n in (nq, nk, nk))
    O0, L0 = orc.attention(q, k, v, 0.3)
    O1, L1 = orc.attention_online(q, k, v, 0.3, bc)
    np.testing.assert_allclose(O1, O0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L1, L0, rtol=1e-12, atol=1e-13)
    order = g.permutation((nk + bc - 1) // bc)
    O2, L2 = orc.attention_online(q, k, v, 0.3, bc, order)
    np.testing.assert_allclose(O2, O0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2, L0, rtol=1e-12, atol=1e-13)


# ----------------------------------------------- FACache, LaCache §3.3.3 ----
def _qkv(g, N, H, d, s=1.5):
    return (g.standard_normal((N, H, d)) * s for _ in range(3))


@pytest.mark.parametrize("N,c_lo,c_hi,bc", [(50, 16, 24, 8), (50, 0, 8, 7), (50, 42, 50, 64), (33, 5, 30, 3),
                                            (40, 0, 40, 16)])
def test_cached_merge_equals_full_recompute(N, c_lo, c_hi, bc):
    g = _rng(20 + N + c_lo)
    H, d = 2, 16
    q, k, v = _qkv(g, N, H, d)
    U = np.array([r for r in range(N) if not (c_lo <= r < c_hi)], dtype=np.int64)
    scale = 1 / math.sqrt(d)
    m, l, Ot = orc.state_build(q[U], k, v, scale, c_lo, c_hi, bc)
    # the block's keys and values change at the next inner step; U's do not
    k2, v2 = k.copy(), v.copy()
    k2[c_lo:c_hi] = g.standard_normal((c_hi - c_lo, H, d))
    v2[c_lo:c_hi] = g.standard_normal((c_hi - c_lo, H, d))
    O, L = orc.state_merge(q[U], k2, v2, scale, c_lo, c_hi, m, l, Ot, bc)
    Of, Lf = orc.attention(q[U], k2, v2, scale)
    np.testing.assert_allclose(O, Of, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, Lf, rtol=1e-12, atol=1e-13)


def test_cached_state_is_online_state_over_U_keys():
    g = _rng(30)
    N, H, d, c_lo, c_hi = 40, 2, 8, 10, 18
    q, k, v = _qkv(g, N, H, d)
    U = np.r_[0:c_lo, c_hi:N]
    m, l, Ot = orc.state_build(q[U], k, v, 0.5, c_lo, c_hi, 6)
    S = 0.5 * np.einsum("rhd,khd->rhk", q[U], k[U])
    np.testing.assert_allclose(m, S.max(-1), rtol=1e-14)
    P = np.exp(S - S.max(-1, keepdims=True))
    np.testing.assert_allclose(l, P.sum(-1), rtol=1e-12)
    np.testing.assert_allclose(Ot, np.einsum("rhk,khd->rhd", P, v[U]), rtol=1e-11, atol=1e-12)


def test_normalised_state_is_a_convex_combination_of_values():
    """O~ / l of a state is a softmax-weighted average of the value rows of its keys: every
    column lies between that column's smallest and largest value over U, so it is finite in
    any format that holds the values (the cached state is stored as O~ / l); with a single
    key in U it is that key's value row, whatever the query."""
    g = _rng(33)
    N, H, d, c_lo, c_hi = 36, 3, 8, 5, 31
    q, k, v = _qkv(g, N, H, d)
    q *= 4.0  # peaked weights: the average sits close to single values
    U = np.r_[0:c_lo, c_hi:N]
    m, l, Ot = orc.state_build(q[U], k, v, 0.5, c_lo, c_hi, 4)
    o = Ot / l[..., None]
    lo, hi = v[U].min(axis=0), v[U].max(axis=0)  # [H, d] over the keys of U
    assert np.all(o >= lo[None] - 1e-12) and np.all(o <= hi[None] + 1e-12)
    # one key outside C (C = every row but row 0): the state's O~ / l is v[0] for every row
    m1, l1, O1 = orc.state_build(q[:1], k, v, 0.5, 1, N, 4)
    np.testing.assert_allclose(O1 / l1[..., None], np.broadcast_to(v[0], O1.shape), rtol=1e-14)
    np.testing.assert_allclose(l1, 1.0, rtol=1e-14)


def test_merge_invariant_to_reference_max_and_empty_state():
    g = _rng(31)
    N, H, d, c_lo, c_hi = 30, 2, 8, 8, 16
    q, k, v = _qkv(g, N, H, d)
    U = np.r_[0:c_lo, c_hi:N]
    m, l, Ot = orc.state_build(q[U], k, v, 0.5, c_lo, c_hi, 8)
    O0, L0 = orc.state_merge(q[U], k, v, 0.5, c_lo, c_hi, m, l, Ot, 8)
    # re-reference to a larger max (e.g. the full-row max of Algorithm 1): same result
    delta = 3.25
    O1, L1 = orc.state_merge(q[U], k, v, 0.5, c_lo, c_hi, m + delta, l * np.exp(-delta),
                             Ot * np.exp(-delta), 8)
    np.testing.assert_allclose(O1, O0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L1, L0, rtol=1e-12, atol=1e-13)
    # the empty state (-inf, 0, 0) is the identity: result = attention over the block keys only
    O2, L2 = orc.state_merge(q[U], k, v, 0.5, c_lo, c_hi, np.full_like(m, -np.inf), np.zeros_like(l),
                             np.zeros_like(Ot), 8)
    O3, L3 = orc.attention(q[U], k[c_lo:c_hi], v[c_lo:c_hi], 0.5)
    np.testing.assert_allclose(O2, O3, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2, L3, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("br,bc", [(4, 4), (3, 5), (8, 16), (16, 8), (37, 37), (1, 1)])
def test_algorithm1_genstep_then_reuse(br, bc):
    g = _rng(40 + br * 7 + bc)
    N, H, d, c_lo, c_hi = 37, 2, 8, 13, 21
    q, k, v = _qkv(g, N, H, d)
    O, L, cache = orc.alg1(q, k, v, 0.4, c_lo, c_hi, br, bc, True)
    Of, Lf = orc.attention(q, k, v, 0.4)
    np.testing.assert_allclose(O, Of, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L, Lf, rtol=1e-12, atol=1e-13)
    # the next inner step: the block's rows (queries, keys and values) change
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for t in (q2, k2, v2):
        t[c_lo:c_hi] = g.standard_normal((c_hi - c_lo, H, d))
    O2, L2, _ = orc.alg1(q2, k2, v2, 0.4, c_lo, c_hi, br, bc, False, cache)
    Of2, Lf2 = orc.attention(q2, k2, v2, 0.4)
    np.testing.assert_allclose(O2, Of2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2, Lf2, rtol=1e-12, atol=1e-13)


# ---------------------------------------------- the step, LaCache Eq. (1) ----
def test_tokenwise_invariance_of_block_rows():
    # token-wise operators on the block rows alone equal the same rows of the
    # full computation (LaCache §3.3.2)
    g = _rng(50)
    N, D, H, d = 24, 64, 2, 16
    x = g.standard_normal((N, D))
    W = g.standard_normal((3 * H * d, D)) * 0.1
    gain = np.ones(D)
    full = orc.layer_step(x, gain, W, H, d, 1e4, 1e-5)
    q, k, v = orc.qkv(x[8:16], gain, W, H, d, 1e4, 1e-5, np.arange(8, 16))
    np.testing.assert_array_equal(q, full["q"][8:16])
    np.testing.assert_array_equal(k, full["k"][8:16])
    np.testing.assert_array_equal(v, full["v"][8:16])


def test_layer_step_matches_library_composition():
    # The whole step composed from torch fp64 library routines: rms_norm,
    # matmul, RoPE as complex rotation of (x_i + i x_{i+d/2}), and
    # scaled_dot_product_attention; no bf16 mirroring on either side.
    g = _rng(51)
    N, D, H, d, theta = 20, 64, 2, 16, 5e5
    x = g.standard_normal((N, D))
    W = g.standard_normal((3 * H * d, D)) * 0.1
    gain = g.uniform(0.5, 1.5, D)
    ref = orc.layer_step(x, gain, W, H, d, theta, 1e-5, mirror=False)
    xt = torch.from_numpy(x)
    xh = torch.nn.functional.rms_norm(xt, (D,), weight=torch.from_numpy(gain), eps=1e-5)
    y = xh @ torch.from_numpy(W).T
    HD = H * d
    q, k, v = (y[:, i * HD:(i + 1) * HD].reshape(N, H, d) for i in range(3))
    inv = torch.tensor([theta ** (-2.0 * i / d) for i in range(d // 2)], dtype=torch.float64)
    ang = torch.arange(N, dtype=torch.float64)[:, None] * inv[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]

    def rope_c(t):
        z = torch.complex(t[..., :d // 2], t[..., d // 2:]) * rot
        return torch.cat([z.real, z.imag], dim=-1)

    q, k = rope_c(q), rope_c(k)
    O = torch.nn.functional.scaled_dot_product_attention(q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1),
                                                         scale=1 / math.sqrt(d)).transpose(0, 1)
    np.testing.assert_allclose(ref["O"], O.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ref["k"], k.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ref["q"], q.numpy(), rtol=1e-11, atol=1e-12)


# ------------------------------------------------ the block-only epilogue (softmax summary)
def test_softmax_stats_against_library_and_closed_forms():
    """LaCache §3.4 (the sampling stage): per row, lse, the argmax and its
    probability.  Pinned to scipy's logsumexp and numpy's argmax, and to
    closed forms: equal logits give lse = log V, argmax 0 (the lowest index
    among ties) and p_max = 1 / V; a shift by c moves lse by c only."""
    from scipy.special import logsumexp
    rng = np.random.default_rng(11)
    z = rng.normal(scale=3.0, size=(7, 300))
    lse, am, pm = orc.softmax_stats(z)
    assert np.allclose(lse, logsumexp(z, axis=1), rtol=0, atol=1e-12)
    assert np.array_equal(am, z.argmax(axis=1))
    assert np.allclose(pm, np.exp(z.max(axis=1) - lse), rtol=1e-13, atol=0)
    V = 256
    lse, am, pm = orc.softmax_stats(np.full((2, V), 1.5))
    assert np.allclose(lse, 1.5 + np.log(V), atol=1e-13) and np.array_equal(am, [0, 0])
    assert np.allclose(pm, 1.0 / V, rtol=1e-13)
    t = np.zeros((1, 10))
    t[0, [3, 7]] = 5.0  # a tie between 3 and 7: the lowest index
    assert orc.softmax_stats(t)[1][0] == 3
    lse2, am2, pm2 = orc.softmax_stats(z + 4.25)
    lse0, am0, pm0 = orc.softmax_stats(z)
    assert np.allclose(lse2, lse0 + 4.25, atol=1e-12) and np.array_equal(am2, am0) and np.allclose(pm2, pm0)


def test_lm_head_against_torch_composition():
    """RMSNorm (torch's rms_norm), the bf16 operand, the LM head (torch matmul)
    and torch's logsumexp / argmax / softmax reproduce the oracle's block-only
    epilogue."""
    import torch
    rng = np.random.default_rng(12)
    h = rng.normal(size=(5, 64)).astype(np.float64)
    g = rng.uniform(0.5, 1.5, size=64)
    W = rng.normal(scale=0.1, size=(96, 64))
    ref = orc.lm_head(h, g, W, 1e-5)
    th = torch.from_numpy(h)
    xh = torch.nn.functional.rms_norm(th, (64,), torch.from_numpy(g), eps=1e-5)
    xh = xh.to(torch.bfloat16).to(torch.float64)
    z = xh @ torch.from_numpy(W).T
    assert np.allclose(ref["logits"], z.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(ref["lse"], torch.logsumexp(z, 1).numpy(), atol=1e-12)
    assert np.array_equal(ref["argmax"], z.argmax(1).numpy())
    assert np.allclose(ref["p_max"], torch.softmax(z, 1).max(1).values.numpy(), rtol=1e-12)


# ------------------------------------------------ FP8 (e4m3) of the FFN (LaCache §3.4)
def _golden_e4m3():
    codes, rounds = [], []
    for line in open(os.path.join(GOLDEN, "e4m3.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b = line.split()
        (codes if a.startswith("0x") else rounds).append((a, float(b)))
    return codes, rounds


def test_e4m3_golden_values_and_library():
    """Hand-derived codes and roundings (tests/golden/e4m3.txt), torch's
    float8_e4m3fn for every finite code and for in-range rounding."""
    import torch
    codes, rounds = _golden_e4m3()
    for c, v in codes:
        assert orc.e4m3_decode(int(c, 16)) == v, c
    for x, r in rounds:
        assert orc.e4m3_round(float(x)) == r, x
    all_codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = all_codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = orc.e4m3_decode(c)
        if np.isnan(lib[c]):
            assert np.isnan(v), c
        else:
            assert v == lib[c], c
            assert orc.e4m3_round(v) == v  # every finite value rounds to itself
    rng = np.random.default_rng(21)
    xs = rng.uniform(-448, 448, size=4000) * np.exp(rng.uniform(-12, 0, size=4000))
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.array([orc.e4m3_round(x) for x in xs]), ref)


def test_quant_groups_eq7_eq8():
    """Eq. (7)-(8): the group max maps to +-448 exactly, every value within half
    a step (2^-4 relative for the normal range) of its group's grid, a group of
    zeros has scale 0, and a group of equal values comes back unchanged."""
    rng = np.random.default_rng(22)
    x = rng.normal(size=(5, 256)) * np.exp(rng.uniform(-3, 3, size=(5, 1)))
    deq, sc = orc.quant_groups(x)
    x32 = x.astype(np.float32).astype(np.float64)
    for r in range(5):
        for g in range(2):
            blk, d = x32[r, 128 * g:128 * g + 128], deq[r, 128 * g:128 * g + 128]
            s = np.float32(np.abs(blk).max()) / np.float32(448)
            assert sc[r, g] == s
            k = np.abs(blk).argmax()
            assert abs(d[k]) == 448.0 * float(s)
            big = np.abs(blk) > 2.0 ** -6 * s  # normal range of the codes
            assert np.all(np.abs(d - blk)[big] <= np.abs(blk)[big] * 2.0 ** -4 * (1 + 1e-6))
    z = np.zeros((1, 128))
    dz, sz = orc.quant_groups(z)
    assert sz[0, 0] == 0.0 and not dz.any()
    e = np.full((1, 128), 0.37)
    de, _ = orc.quant_groups(e)
    assert np.allclose(de, np.float32(0.37), rtol=1e-6)


def test_ffn_against_torch_composition():
    """The FFN with per-group FP8 reproduced by torch: bf16 residual stream,
    rms_norm, the fp32 quantisation decisions with torch's float8_e4m3fn cast,
    dequantised block-scaled weights, SiLU."""
    import torch
    rng = np.random.default_rng(23)
    M, D, HD, F = 3, 256, 128, 256
    o = rng.normal(size=(M, HD))
    x = rng.normal(size=(M, D))
    Wo = rng.normal(scale=0.05, size=(D, HD))
    g2 = rng.uniform(0.5, 1.5, size=D)
    gu_codes = rng.integers(0, 256, size=(2 * F, D), dtype=np.uint8)
    gu_codes[(gu_codes & 0x7F) == 0x7F] = 0x38  # no NaN codes
    gu_scale = rng.uniform(1e-4, 3e-4, size=(2 * F // 128, D // 128)).astype(np.float32)
    d_codes = rng.integers(0, 256, size=(D, F), dtype=np.uint8)
    d_codes[(d_codes & 0x7F) == 0x7F] = 0x38
    d_scale = rng.uniform(1e-4, 3e-4, size=(D // 128, F // 128)).astype(np.float32)
    ref = orc.ffn(o, x, Wo, g2, gu_codes, gu_scale, d_codes, d_scale, 1e-5)

    def q(t):  # Eq. (7)-(8), decisions in fp32
        t32 = t.to(torch.float32).reshape(t.shape[0], -1, 128)
        s = t32.abs().amax(-1, keepdim=True) / 448.0
        qq = torch.where(s > 0, t32 / s, torch.zeros_like(t32)).to(torch.float8_e4m3fn).to(torch.float64)
        return (qq * s.to(torch.float64)).reshape(t.shape)

    def deq(codes, scale):
        v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
        s = torch.from_numpy(scale).to(torch.float64).repeat_interleave(128, 0).repeat_interleave(128, 1)
        return v * s

    h1 = (torch.from_numpy(x) + torch.from_numpy(o) @ torch.from_numpy(Wo).T).to(torch.bfloat16).to(torch.float64)
    # the quantisation's input in fp32: 1 / rms rounded to fp32, then (h1 * inv) * g2 in fp32
    inv = (1.0 / torch.sqrt(h1.pow(2).mean(1, keepdim=True) + 1e-5)).to(torch.float32)
    x2 = q((h1.to(torch.float32) * inv) * torch.from_numpy(g2).to(torch.float32))
    # and it is RMSNorm: the fp32 values are within fp32 rounding of torch's rms_norm
    assert torch.allclose((h1.to(torch.float32) * inv * torch.from_numpy(g2).to(torch.float32)).double(),
                          torch.nn.functional.rms_norm(h1, (D,), torch.from_numpy(g2), eps=1e-5), rtol=1e-6)
    gu = x2 @ deq(gu_codes, gu_scale).T
    a = q(torch.nn.functional.silu(gu[:, 0::2]) * gu[:, 1::2])
    y = h1 + a @ deq(d_codes, d_scale).T
    assert np.array_equal(ref["h1"], h1.numpy())
    assert np.allclose(ref["y"], y.numpy(), rtol=1e-9, atol=1e-9)


def test_rmsnorm_f32_is_rmsnorm_in_fp32():
    """The quantisation's input (RMSNorm formed in fp32 as the kernels form it) is
    torch's rms_norm up to fp32 rounding (three roundings: 2^-22 relative), for
    rows whose mean square is comparable to eps (so eps counts)."""
    import torch
    rng = np.random.default_rng(24)
    h = rng.normal(size=(6, 256)) * np.array([1.0, 1e-1, 1e-2, 3e-3, 1e-3, 10.0])[:, None]
    g = rng.uniform(0.5, 1.5, size=256)
    got = orc.rmsnorm_f32(h, g, 1e-5)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h), (256,), torch.from_numpy(g), eps=1e-5).numpy()
    assert np.all(np.abs(got - ref) <= 2.0 ** -22 * np.abs(ref) + 1e-30)
    assert np.array_equal(got, got.astype(np.float32).astype(np.float64))  # fp32 values
