"""Pins for the CPU oracle: checks against facts that do not come from the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (``oracle.load()`` or a deliberately broken
build of it) and raises AssertionError when the oracle disagrees with the fact it pins. The kinds
of fact used: closed forms of special cases, values worked by hand (``golden/hand_hc2_d8.json``),
library routines that a special case reduces to (numpy matmul, torch's bfloat16 cast), exact
bit-level identities, and invariants the method guarantees (ranges, column sums).

Definitions pinned (DeepSeek V4.1 model-atlas pages): 'Source layer, pairs pooled' page, Block
excerpts (hc_mixes, hc_pre, hc_post, forward) and Parameters table; 'Reading weights' page,
hc_split_sinkhorn kernel excerpt and the formula for p; 'Final RMSNorm' page, RMSNorm excerpt, the
m_2 formula and the Transformer.forward excerpt (ends of the stack); 'Write the streams' page, the
formula for X'.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf(x):
    """float64 values that are exactly representable in bf16 -> their bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    b = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(orc.bf16_to_double(b), x), "value not exact in bf16"
    return b


def _sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def _hand_case():
    with open(os.path.join(GOLDEN, "hand_hc2_d8.json")) as f:
        g = json.load(f)
    hc, d = g["hc"], g["d"]
    s0 = np.array(g["stream0"], np.float64)
    s1 = np.array(g["stream1"], np.float64)
    sgn = s1
    fn = np.zeros((8, 16), np.float32)
    fn[0, :8] = 0.0625
    fn[1, 8:] = 0.0625 * sgn
    fn[2, :8] = -0.125
    fn[3, 8:] = 0.125 * sgn
    fn[4, :8] = 0.25
    fn[7, 8:] = 0.125 * sgn
    X = np.stack([_bf(s0), _bf(s1)])[None]  # [1, 2, 8]
    return g, hc, d, X, fn


# ---- bf16 rounding ------------------------------------------------------------------------------

def pin_bf16_rounding_matches_torch(lib):
    """double -> bf16 on float32-representable values equals torch's float32 -> bfloat16 cast."""
    import torch
    rng = np.random.default_rng(1)
    vals = [rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000),
            np.array([0.0, -0.0, 1.0, -1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 - 2 ** -9, 3.0e38, -3.4e38,
                      2 ** -133, 2 ** -134, 3 * 2 ** -134, 2 ** -126, 1e-45, np.inf, -np.inf])]
    # exact ties between neighbouring bf16 values, at many exponents
    m = rng.integers(0, 128, 5000)
    e = rng.integers(-120, 120, 5000)
    ties = (1.0 + (2 * m + 1) * 2.0 ** -8) * 2.0 ** e
    vals.append(ties)
    vals.append(-ties)
    x = np.concatenate(vals).astype(np.float32).astype(np.float64)
    ours = orc.double_to_bf16(x, lib=lib)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, "bf16 rounding differs from torch at %r" % (x[bad[:5]],)
    assert lib.oracle_double_to_bf16(float("nan")) & 0x7F80 == 0x7F80


def pin_bf16_ties_to_even(lib):
    """Halfway cases go to the neighbour with an even last bit (1 + 2^-8 -> 1; 1 + 3*2^-8 -> 1 + 2^-6)."""
    assert orc.bf16_to_double([lib.oracle_double_to_bf16(1 + 2 ** -8)])[0] == 1.0
    assert orc.bf16_to_double([lib.oracle_double_to_bf16(1 + 3 * 2 ** -8)])[0] == 1 + 2 ** -6
    assert orc.bf16_to_double([lib.oracle_double_to_bf16(-(1 + 2 ** -8 + 2 ** -40))])[0] == -(1 + 2 ** -7)


# ---- hand-worked case hc=2, d=8 ----------------------------------------------------------------

def pin_hand_case_step_a(lib):
    g, hc, d, X, fn = _hand_case()
    a = g["step_a"]
    out = orc.hc_pre_step(X, np.array([a["pre_mix"]], np.float32), fn, np.array(g["hc_scale"], np.float32),
                          np.array(g["hc_base"], np.float32), np.ones(d, np.float32), g["iters"], g["hc_eps"],
                          g["norm_eps"], lib=lib)
    # closed forms: r = 1/sqrt(1 + eps); the dots are (0.5, 0.5, -1, 1, 2, 0, 0, 1)
    r = 1.0 / math.sqrt(1.0 + 1e-6)
    assert abs(out["r"][0] - r) < 1e-15 and abs(out["r"][0] - a["r"]) < 1e-15
    assert np.allclose(out["mixes"][0], r * np.array([0.5, 0.5, -1, 1, 2, 0, 0, 1]), rtol=1e-14, atol=1e-15)
    pre_cf = [_sig(0.5 * r) + 1e-6, _sig(0.5 * r + 0.25) + 1e-6]
    post_cf = [2 * _sig(-r), 2 * _sig(r)]
    assert np.allclose(out["pre"][0], pre_cf, rtol=1e-14) and np.allclose(out["pre"][0], a["pre"], rtol=1e-14)
    assert np.allclose(out["post"][0], post_cf, rtol=1e-14) and np.allclose(out["post"][0], a["post"], rtol=1e-14)
    assert np.allclose(out["comb"][0], a["comb"], rtol=1e-13)
    lim = math.exp(1.5 * r) / (1 + math.exp(1.5 * r))
    assert abs(out["comb"][0, 0, 0] - lim) < 3e-6  # the eps -> 0 limit, off by the eps effect only
    y = orc.bf16_to_double(out["y"][0])
    assert np.array_equal(y, np.tile([1.0, 0.5], 4))
    yn_cf = np.tile([1.0, 0.5], 4) / math.sqrt(0.625 + 1e-6)
    assert np.allclose(yn_cf[:2], a["y_normed_exact_first_two"], rtol=1e-9)
    assert np.array_equal(orc.bf16_to_double(out["y_normed"][0])[:2], a["y_normed_bf16_first_two"])


def pin_hand_case_step_b(lib):
    g, hc, d, X, fn = _hand_case()
    b = g["step_b"]
    delta = _bf(np.full((1, d), b["delta"]))
    out = orc.hc_post_then_pre(delta, X, np.array([b["post_in"]], np.float32), np.array([b["comb_in"]], np.float32),
                               np.array([b["pre_mix"]], np.float32), fn, np.array(g["hc_scale"], np.float32),
                               np.array(g["hc_base"], np.float32), np.ones(d, np.float32), g["iters"], g["hc_eps"],
                               g["norm_eps"], lib=lib)
    xo = orc.bf16_to_double(out["X_out"][0])
    assert np.array_equal(xo[0], np.tile(b["X_out_stream0_first_two"], 4))
    assert np.array_equal(xo[1], np.tile(b["X_out_stream1_first_two"], 4))
    r = 1.0 / math.sqrt(19.5 / 16 + 1e-6)  # mean of X'^2 over all 16 values is 19.5/16
    assert abs(r - b["r"]) < 1e-15
    pre_cf = [_sig(0.625 * r) + 1e-6, _sig(0.375 * r + 0.25) + 1e-6]
    post_cf = [2 * _sig(-1.25 * r), 2 * _sig(0.75 * r)]
    assert np.allclose(out["pre"][0], pre_cf, rtol=1e-14) and np.allclose(out["pre"][0], b["pre"], rtol=1e-14)
    assert np.allclose(out["post"][0], post_cf, rtol=1e-14) and np.allclose(out["post"][0], b["post"], rtol=1e-14)
    assert np.allclose(out["comb"][0], b["comb"], rtol=1e-13)
    assert np.array_equal(orc.bf16_to_double(out["y_normed"][0])[:2], b["y_normed_bf16_first_two"])


# ---- split + Sinkhorn ---------------------------------------------------------------------------

def _uniform_comb(iters, eps, hc=4):
    v = 1.0 / hc + eps
    v = v / (hc * v + eps)            # the first column normalisation
    for _ in range(iters - 1):
        v = v / (hc * v + eps)        # row
        v = v / (hc * v + eps)        # column
    return v


def pin_uniform_logits_closed_form(lib):
    """mixes == 0 (hc_fn = 0, base = 0): pre = 1/2 + eps, post = 1, comb = the scalar recurrence."""
    for hc, iters, eps in [(4, 20, 1e-6), (4, 50, 1e-6), (4, 1, 1e-3), (2, 7, 1e-2), (3, 5, 0.0),
                           (4, 6, 0.9), (2, 9, 0.5), (4, 3, 2.0), (8, 20, 1e-6), (8, 4, 0.3), (1, 5, 1e-2),
                           (5, 11, 1e-4)]:
        M = (2 + hc) * hc
        pre, post, comb = orc.split_sinkhorn(np.zeros((2, M)), np.array([1.3, 0.7, 2.0], np.float32),
                                             np.zeros(M, np.float32), hc, iters, eps, lib=lib)
        assert np.allclose(pre, 0.5 + eps, rtol=1e-15)
        assert np.allclose(post, 1.0, rtol=1e-15)
        assert np.allclose(comb, _uniform_comb(iters, eps, hc), rtol=1e-14), (hc, iters, eps)


def pin_sinkhorn_2x2_limit(lib):
    """eps = 0, many iterations: a 2x2 positive matrix scales to [[a, 1-a], [1-a, a]],
    a = rho / (1 + rho), rho = sqrt(exp(L00 + L11 - L01 - L10)) (the cross ratio is invariant)."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        m = rng.standard_normal(8) * 1.5
        base = rng.standard_normal(8).astype(np.float32)
        scale = np.array([1.0, 1.0, 0.75], np.float32)
        pre, post, comb = orc.split_sinkhorn(m[None], scale, base, 2, 400, 0.0, lib=lib)
        L = m[4:] * 0.75 + base[4:].astype(np.float64)
        rho = math.sqrt(math.exp(L[0] + L[3] - L[1] - L[2]))
        a = rho / (1 + rho)
        assert np.allclose(comb[0], [[a, 1 - a], [1 - a, a]], atol=1e-9), (comb[0], a)


def pin_sinkhorn_2x2_trajectory(lib):
    """eps = 0, few iterations. After a column normalisation a 2x2 matrix is [[a, b], [1-a, 1-b]];
    a row then a column normalisation map a to
        a' = (a/(a+b)) / (a/(a+b) + (1-a)/(2-a-b)),  b' = (b/(a+b)) / (b/(a+b) + (1-b)/(2-a-b)).
    Far from convergence every iteration moves a, which pins the iteration count."""
    for L in ([[3.0, -1.0], [0.5, 2.5]], [[-2.0, 1.0], [4.0, 0.0]]):
        L = np.array(L)
        m = np.zeros(8)
        m[4:] = L.reshape(4)
        for iters in (1, 2, 3, 5, 8):
            _, _, comb = orc.split_sinkhorn(m[None], np.array([1, 1, 1], np.float32), np.zeros(8, np.float32),
                                            2, iters, 0.0, lib=lib)
            S = np.exp(L - L.max(axis=1, keepdims=True))
            S = S / S.sum(axis=1, keepdims=True)
            S = S / S.sum(axis=0, keepdims=True)
            a, b = S[0, 0], S[0, 1]
            for _ in range(iters - 1):
                r0, r1 = a + b, 2 - a - b
                a, b = (a / r0) / (a / r0 + (1 - a) / r1), (b / r0) / (b / r0 + (1 - b) / r1)
            assert np.allclose(comb[0], [[a, b], [1 - a, 1 - b]], rtol=1e-12), (iters, comb[0], a, b)


def pin_row_softmax_orientation(lib):
    """iters = 1: softmax over each ROW of the logits, + eps, then one column normalisation.
    Logits: row 0 = (c, 0, 0, 0), other rows 0; mixes 8 + 4j + k is row j, column k."""
    hc, eps, c = 4, 1e-3, 2.0
    m = np.zeros(24)
    m[8 + 0 * 4 + 0] = c
    pre, post, comb = orc.split_sinkhorn(m[None], np.array([1, 1, 1], np.float32), np.zeros(24, np.float32),
                                         hc, 1, eps, lib=lib)
    e = math.exp(c)
    S = np.full((4, 4), 0.25 + eps)
    S[0] = np.array([e, 1, 1, 1]) / (e + 3) + eps
    S = S / (S.sum(axis=0, keepdims=True) + eps)
    assert np.allclose(comb[0], S, rtol=1e-14)
    # a logit at (row 1, column 3) lands at comb[1, 3]'s row
    m2 = np.zeros(24)
    m2[8 + 1 * 4 + 3] = 3.0
    _, _, comb2 = orc.split_sinkhorn(m2[None], np.array([1, 1, 1], np.float32), np.zeros(24, np.float32),
                                     hc, 1, 0.0, lib=lib)
    assert comb2[0, 1, 3] == comb2[0].max()
    assert np.allclose(comb2[0, 1, :3], comb2[0, 1, 0]) and comb2[0, 0, 3] < comb2[0, 1, 3]


def pin_split_scales_and_offsets(lib):
    """pre uses hc_scale[0] and base[0:hc]; post uses hc_scale[1] and base[hc:2hc] with factor 2;
    comb uses hc_scale[2] and base[2hc:]. Probed one scale at a time with closed forms."""
    hc = 4
    m = np.arange(24, dtype=np.float64)[None] * 0.01 - 0.1
    base = (np.arange(24) * 0.03 - 0.2).astype(np.float32)
    scale = np.array([0.5, 1.5, 0.0], np.float32)
    pre, post, comb = orc.split_sinkhorn(m, scale, base, hc, 3, 1e-6, lib=lib)
    for j in range(hc):
        assert abs(pre[0, j] - (_sig(m[0, j] * 0.5 + float(base[j])) + 1e-6)) < 1e-15
        assert abs(post[0, j] - 2 * _sig(m[0, 4 + j] * 1.5 + float(base[4 + j]))) < 1e-15
    # with scale 0 the comb logits are the offsets alone
    _, _, comb_b = orc.split_sinkhorn(np.zeros((1, 24)), scale, base, hc, 3, 1e-6, lib=lib)
    assert np.allclose(comb, comb_b, rtol=1e-15)


def pin_split_invariants(lib):
    """pre in [eps, 1+eps], post in [0, 2], every column of comb sums to 1 - O(eps) (the last
    operation is a column normalisation), rows sum to 1 within 1e-3 for mild logits."""
    rng = np.random.default_rng(9)
    n, hc, eps = 4000, 4, 1e-6
    mixes = rng.standard_normal((n, 24)) * 3.0
    base = rng.standard_normal(24).astype(np.float32)
    pre, post, comb = orc.split_sinkhorn(mixes, np.array([1.0, 1.0, 1.0], np.float32), base, hc, 20, eps, lib=lib)
    assert pre.min() >= eps and pre.max() <= 1 + eps
    assert post.min() >= 0 and post.max() <= 2
    cs = comb.sum(axis=1)
    assert np.abs(cs - 1).max() < 5 * hc * eps
    assert comb.min() > 0
    mild = rng.standard_normal((n, 24)) * 0.3
    _, _, comb_m = orc.split_sinkhorn(mild, np.array([1.0, 1.0, 1.0], np.float32), np.zeros(24, np.float32),
                                      hc, 20, eps, lib=lib)
    assert np.abs(comb_m.sum(axis=2) - 1).max() < 1e-3
    assert np.abs(comb_m.sum(axis=1) - 1).max() < 5 * hc * eps


def pin_sinkhorn_permutation_equivariance(lib):
    """Relabelling the streams (rows and columns of the logits together) relabels comb."""
    rng = np.random.default_rng(11)
    hc = 4
    perm = np.array([2, 0, 3, 1])
    m = rng.standard_normal((50, 24))
    L = m[:, 8:].reshape(50, 4, 4)
    m2 = m.copy()
    m2[:, 8:] = L[:, perm][:, :, perm].reshape(50, 16)
    z = np.zeros(24, np.float32)
    s = np.array([1, 1, 1], np.float32)
    _, _, c1 = orc.split_sinkhorn(m, s, z, hc, 20, 1e-6, lib=lib)
    _, _, c2 = orc.split_sinkhorn(m2, s, z, hc, 20, 1e-6, lib=lib)
    assert np.allclose(c2, c1[:, perm][:, :, perm], rtol=1e-12)


# ---- hc_post ------------------------------------------------------------------------------------

def pin_hc_post_identity(lib):
    """comb = I, post = 0 returns X bit for bit."""
    rng = np.random.default_rng(2)
    n, hc, d = 5, 4, 40
    X = (rng.standard_normal((n, hc, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    delta = (rng.standard_normal((n, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    out = orc.hc_post(X, delta, np.zeros((n, hc), np.float32), np.tile(np.eye(hc, dtype=np.float32), (n, 1, 1)),
                      lib=lib)
    assert np.array_equal(out, X)


def pin_hc_post_permutation_orientation(lib):
    """comb[j, k] = 1 iff k = pi(j) sends source stream j to destination k = pi(j):
    X'_{pi(j)} = X_j exactly (the sum in hc_post runs over comb's first stream index)."""
    rng = np.random.default_rng(3)
    n, hc, d = 3, 4, 24
    pi = np.array([1, 3, 0, 2])
    P = np.zeros((hc, hc), np.float32)
    P[np.arange(hc), pi] = 1.0
    X = (rng.standard_normal((n, hc, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    delta = np.zeros((n, d), np.uint16)
    out = orc.hc_post(X, delta, np.zeros((n, hc), np.float32), np.tile(P, (n, 1, 1)), lib=lib)
    for j in range(hc):
        assert np.array_equal(out[:, pi[j]], X[:, j])


def pin_hc_post_dyadic_closed_form(lib):
    """Constant dyadic streams: X'_k = post_k * delta + sum_j comb[j,k] c_j, exact in bf16."""
    hc, d = 4, 16
    c = np.array([1.0, -0.5, 0.25, 2.0])
    delta_v = 0.75
    post = np.array([[0.5, 0.25, -1.0, 0.125]], np.float32)
    comb = np.array([[[0.5, 0.25, 0.0, 0.125],
                      [0.25, 0.5, 0.125, 0.0],
                      [0.125, 0.0, 0.5, 0.25],
                      [0.0, 0.125, 0.25, 0.5]]], np.float32)
    X = _bf(np.repeat(c[:, None], d, axis=1))[None]
    delta = _bf(np.full((1, d), delta_v))
    out = orc.bf16_to_double(orc.hc_post(X, delta, post, comb, lib=lib))[0]
    want = [0.5 * 0.75 + (0.5 * 1 + 0.25 * -0.5 + 0.125 * 0.25 + 0.0 * 2),
            0.25 * 0.75 + (0.25 * 1 + 0.5 * -0.5 + 0.0 * 0.25 + 0.125 * 2),
            -1.0 * 0.75 + (0.0 * 1 + 0.125 * -0.5 + 0.5 * 0.25 + 0.25 * 2),
            0.125 * 0.75 + (0.125 * 1 + 0.0 * -0.5 + 0.25 * 0.25 + 0.5 * 2)]
    for k in range(hc):
        assert np.all(out[k] == want[k]), (k, out[k, 0], want[k])
    # the detailed form returns the same bits, the exact values and the sums of |terms|
    o2, exact, mag = orc.hc_post_detail(X, delta, post, comb, lib=lib)
    assert np.array_equal(o2, orc.hc_post(X, delta, post, comb, lib=lib))
    mag_want = np.abs(post[0, :, None] * 0.75) + np.abs(comb[0].astype(np.float64) * c[:, None]).sum(axis=0)[:, None]
    assert np.allclose(exact[0], np.array(want)[:, None]) and np.allclose(mag[0], mag_want)


# ---- hc_mixes -----------------------------------------------------------------------------------

def pin_mixes_match_numpy_matmul(lib):
    """Special case reducing to a library routine: mixes = (X_flat @ hc_fn^T) * r, with
    r = 1/sqrt(mean over all hc*d flattened values of x^2 + norm_eps), column c = j*d + i."""
    rng = np.random.default_rng(4)
    n, hc, d, eps = 7, 4, 48, 1e-6
    X = (rng.standard_normal((n, hc, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    fn = (rng.standard_normal((24, hc * d)) * 0.02).astype(np.float32)
    mixes, r, S = orc.hc_mixes(X, fn, eps, lib=lib)
    xf = orc.bf16_to_double(X).reshape(n, hc * d)
    r_ref = 1.0 / np.sqrt((xf ** 2).mean(axis=1) + eps)
    assert np.allclose(r, r_ref, rtol=1e-14)
    assert np.allclose(mixes, (xf @ fn.astype(np.float64).T) * r_ref[:, None], rtol=1e-12, atol=1e-14)
    assert np.allclose(S, (np.abs(xf) @ np.abs(fn.astype(np.float64)).T) * r_ref[:, None], rtol=1e-12)


def pin_mixes_stream_constants(lib):
    """Stream j constant c_j: r = 1/sqrt(sum_j c_j^2 / hc + eps) (the mean runs over all hc*d values),
    mixes[m] = r * sum_j c_j * (sum of hc_fn[m] over stream j's block of d columns)."""
    rng = np.random.default_rng(6)
    hc, d, eps = 4, 32, 1e-6
    c = np.array([1.0, -2.0, 0.5, 0.25])
    X = _bf(np.repeat(c[:, None], d, axis=1))[None]
    fn = (rng.standard_normal((24, hc * d)) * 0.1).astype(np.float32)
    mixes, r, _ = orc.hc_mixes(X, fn, eps, lib=lib)
    r_cf = 1.0 / math.sqrt((c ** 2).sum() / hc + eps)
    assert abs(r[0] - r_cf) < 1e-15
    blocks = fn.astype(np.float64).reshape(24, hc, d).sum(axis=2)  # [m, j]
    assert np.allclose(mixes[0], r_cf * blocks @ c, rtol=1e-12, atol=1e-14)


def pin_mixes_scale_invariance(lib):
    """X -> 2^k X (exact in bf16) leaves mixes unchanged except through norm_eps:
    mixes(2^k X) = mixes(X) * sqrt(ms + eps) / sqrt(ms + eps / 4^k), ms = mean(x^2)."""
    rng = np.random.default_rng(7)
    n, hc, d, eps = 4, 4, 40, 1e-2
    X = (rng.standard_normal((n, hc, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    fn = (rng.standard_normal((24, hc * d)) * 0.02).astype(np.float32)
    m0, r0, _ = orc.hc_mixes(X, fn, eps, lib=lib)
    xf = orc.bf16_to_double(X)
    ms = (xf.reshape(n, -1) ** 2).mean(axis=1)
    for k in (-2, -1, 1, 2):
        Xk = _bf(xf * 2.0 ** k)
        mk, _, _ = orc.hc_mixes(Xk, fn, eps, lib=lib)
        f = np.sqrt(ms + eps) / np.sqrt(ms + eps / 4.0 ** k)
        assert np.allclose(mk, m0 * f[:, None], rtol=1e-12, atol=1e-15)


def pin_mixes_stream_permutation(lib):
    """Permuting the streams of X together with hc_fn's column blocks leaves mixes unchanged
    (pins the flattening order c = j*d + i)."""
    rng = np.random.default_rng(8)
    n, hc, d = 3, 4, 16
    X = (rng.standard_normal((n, hc, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    fn = (rng.standard_normal((24, hc * d))).astype(np.float32)
    perm = np.array([3, 1, 0, 2])
    m1, _, _ = orc.hc_mixes(X, fn, 1e-6, lib=lib)
    fn2 = fn.reshape(24, hc, d)[:, perm].reshape(24, hc * d)
    m2, _, _ = orc.hc_mixes(np.ascontiguousarray(X[:, perm]), fn2, 1e-6, lib=lib)
    assert np.allclose(m1, m2, rtol=1e-13, atol=1e-13)
    # a column block of hc_fn over stream j only sees stream j
    fn3 = np.zeros_like(fn)
    fn3[:, 2 * d:3 * d] = 1.0
    m3, r3, _ = orc.hc_mixes(X, fn3, 1e-6, lib=lib)
    assert np.allclose(m3, (orc.bf16_to_double(X[:, 2]).sum(axis=1) * r3)[:, None], rtol=1e-13)


# ---- hc_pre and RMSNorm -------------------------------------------------------------------------

def pin_hc_pre_one_hot(lib):
    """A one-hot pre_mix e_j returns stream j exactly."""
    rng = np.random.default_rng(10)
    n, hc, d = 4, 4, 32
    X = (rng.standard_normal((n, hc, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    for j in range(hc):
        pm = np.zeros((n, hc), np.float32)
        pm[:, j] = 1.0
        y, _ = orc.hc_pre(X, pm, lib=lib)
        assert np.array_equal(y, X[:, j])


def pin_hc_pre_dyadic(lib):
    """Dyadic weights and values: y = sum_j p_j X_j is exact."""
    hc, d = 4, 8
    c = np.array([1.0, -0.5, 0.25, 2.0])
    X = _bf(np.repeat(c[:, None], d, axis=1))[None]
    p = np.array([[0.5, 0.25, 0.125, 0.0625]], np.float32)
    y, ye, ya = orc.hc_pre(X, p, lib=lib, with_abssum=True)
    want = 0.5 * 1 + 0.25 * -0.5 + 0.125 * 0.25 + 0.0625 * 2
    assert np.all(ye == want) and np.all(orc.bf16_to_double(y) == want)
    assert np.all(ya == 0.5 * 1 + 0.25 * 0.5 + 0.125 * 0.25 + 0.0625 * 2)


def pin_rmsnorm_constant(lib):
    """x = c everywhere: out_i = w_i * c / sqrt(c^2 + eps) (eps matters when c^2 ~ eps)."""
    d = 64
    w = np.linspace(0.5, 1.5, d).astype(np.float32)
    for c, eps in [(1.0, 1e-6), (2.0 ** -10, 1e-6), (-3.0, 1e-20), (2.0 ** -12, 1e-6)]:
        x = _bf(np.full((1, d), c))
        out, oe = orc.rmsnorm(x, w, eps, lib=lib)
        want = w.astype(np.float64) * c / math.sqrt(c * c + eps)
        assert np.allclose(oe[0], want, rtol=1e-14)
        assert np.array_equal(out[0], orc.double_to_bf16(want, lib=lib))


def pin_rmsnorm_two_values(lib):
    """x alternating (a, b): mean square (a^2 + b^2)/2."""
    d = 10
    a, b, eps = 1.5, -0.25, 1e-6
    x = _bf(np.tile([a, b], d // 2)[None])
    _, oe = orc.rmsnorm(x, np.ones(d, np.float32), eps, lib=lib)
    s = 1.0 / math.sqrt((a * a + b * b) / 2 + eps)
    assert np.allclose(oe[0], np.tile([a * s, b * s], d // 2), rtol=1e-14)


def pin_pre_step_composition(lib):
    """hc_pre_step rounds y to bf16 before the norm (the collapse is cast back to the stream dtype)
    and takes the norm's statistic from the rounded values."""
    rng = np.random.default_rng(12)
    n, hc, d = 6, 4, 40
    X = (rng.standard_normal((n, hc, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    pm = rng.random((n, hc)).astype(np.float32)
    fn = (rng.standard_normal((24, hc * d)) * 0.02).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    out = orc.hc_pre_step(X, pm, fn, np.array([1, 1, 1], np.float32), np.zeros(24, np.float32), w, 20, 1e-6,
                          1e-6, lib=lib)
    y, _ = orc.hc_pre(X, pm, lib=lib)
    assert np.array_equal(out["y"], y)
    yn, _ = orc.rmsnorm(y, w, 1e-6, lib=lib)
    assert np.array_equal(out["y_normed"], yn)
    # against a float64 numpy evaluation of the same composition on the rounded y
    yf = orc.bf16_to_double(y)
    want = w.astype(np.float64) * yf / np.sqrt((yf ** 2).mean(axis=1, keepdims=True) + 1e-6)
    assert np.array_equal(out["y_normed"], orc.double_to_bf16(want, lib=lib))


def pin_parameter_count(lib):
    """Stream weights per sublayer: 491,547 = mix_hc*hc*dim + mix_hc + 3 at hc=4, dim=5120."""
    hc, dim = 4, 5120
    mix_hc = (2 + hc) * hc
    assert mix_hc * hc * dim + mix_hc + 3 == 491547
    # and the oracle accepts exactly these shapes: a one-token call with hc_fn [24, 20480]
    X = np.zeros((1, hc, dim), np.uint16)
    m, _, _ = orc.hc_mixes(X, np.zeros((mix_hc, hc * dim), np.float32), 1e-6, lib=lib)
    assert m.shape == (1, mix_hc) and np.all(m == 0)


# ---- ends of the stack ('Final RMSNorm' page, Transformer.forward excerpt) ------------------------

def _rand_bf16(rng, shape, scale=1.0):
    return ((rng.standard_normal(shape) * scale).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pin_expand_copies_embedding(lib):
    """The embedding row becomes hc identical streams, stream-major: X[t, j, :] = h[t, :]."""
    h = _rand_bf16(np.random.default_rng(20), (3, 24))
    X = orc.hc_expand(h, hc=4, lib=lib)
    assert X.shape == (3, 4, 24)
    for j in range(4):
        assert np.array_equal(X[:, j], h)


def pin_expand_pre_step_folds(lib):
    """Head of the stack. With weights summing to 1 the collapse of identical streams is the
    embedding itself, so y_normed is the closed-form norm of h; the statistic over the hc*d
    expanded values is the mean over h's d values, and the projection folds over the streams:
    mixes = r * h . (sum over j of hc_fn's j-th column block), computed here with numpy. Any other
    identity-like weights (one-hot e_3) give the same y_normed."""
    rng = np.random.default_rng(21)
    n, d = 5, 16
    h = _rand_bf16(rng, (n, d))
    fn = (rng.standard_normal((24, 4 * d)) * 0.2).astype(np.float32)
    sc = np.array([0.7, 1.3, 0.9], np.float32)
    base = rng.standard_normal(24).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    out = orc.hc_expand_pre_step(h, fn, sc, base, w, 20, 1e-6, 1e-6, lib=lib)
    hf = orc.bf16_to_double(h)
    want = w.astype(np.float64) * hf / np.sqrt((hf ** 2).mean(axis=1, keepdims=True) + 1e-6)
    assert np.array_equal(out["y_normed"], orc.double_to_bf16(want, lib=lib))
    r = 1.0 / np.sqrt((hf ** 2).mean(axis=1) + 1e-6)
    fold = fn.astype(np.float64).reshape(24, 4, d).sum(axis=1)
    m = (hf @ fold.T) * r[:, None]
    pre, post, comb = orc.split_sinkhorn(m, sc, base, 4, 20, 1e-6, lib=lib)
    assert np.allclose(out["pre"], pre, rtol=1e-12, atol=1e-14)
    assert np.allclose(out["post"], post, rtol=1e-12, atol=1e-14)
    assert np.allclose(out["comb"], comb, rtol=1e-10, atol=1e-13)
    pm = np.zeros((n, 4), np.float32)
    pm[:, 3] = 1.0
    o2 = orc.hc_pre_step(out["X_out"], pm, fn, sc, base, w, 20, 1e-6, 1e-6, lib=lib)
    assert np.array_equal(o2["y_normed"], out["y_normed"])
    # small embeddings, where the eps is not negligible: the norm is no longer scale-invariant, so
    # this also pins that the weights sum to 1 (y = h, not a multiple of it)
    hs = _rand_bf16(rng, (n, d), scale=2.0 ** -11)
    hsf = orc.bf16_to_double(hs)
    out = orc.hc_expand_pre_step(hs, fn, sc, base, w, 20, 1e-6, 1e-6, lib=lib)
    want = w.astype(np.float64) * hsf / np.sqrt((hsf ** 2).mean(axis=1, keepdims=True) + 1e-6)
    assert np.array_equal(out["y_normed"], orc.double_to_bf16(want, lib=lib))


def pin_final_norm_epsilon(lib):
    """Tail of the stack on the hand-worked streams: y = 0.75 stream0 + 0.25 stream1 = (1, 0.5, ...),
    z = w * y / sqrt(mean(y^2) + eps). At the final norm's eps = 1e-20 streams scaled by 2^-12 give
    the same z (the eps is negligible against 0.625 * 2^-24); at eps = 1e-6 they do not."""
    g, hc, d, X, _ = _hand_case()
    pm = np.array([[0.75, 0.25]], np.float32)
    w = np.linspace(0.5, 1.5, d).astype(np.float32)
    wd = w.astype(np.float64)
    z, y, ze = orc.hc_final(X, pm, w, 1e-20, lib=lib)
    yv = np.tile([1.0, 0.5], 4)
    assert np.array_equal(orc.bf16_to_double(y[0]), yv)
    assert np.allclose(ze[0], wd * yv / math.sqrt(0.625 + 1e-20), rtol=1e-15)
    assert np.array_equal(z[0], orc.double_to_bf16(ze[0], lib=lib))
    Xs = _bf(orc.bf16_to_double(X) * 2.0 ** -12)
    _, _, zs = orc.hc_final(Xs, pm, w, 1e-20, lib=lib)
    assert np.allclose(zs, ze, rtol=1e-11)
    _, _, zb = orc.hc_final(Xs, pm, w, 1e-6, lib=lib)
    assert np.allclose(zb[0], wd * yv * 2.0 ** -12 / math.sqrt(0.625 * 2.0 ** -24 + 1e-6), rtol=1e-14)
    assert not np.allclose(zb, ze, rtol=1e-3)


def pin_post_then_final_hand_case(lib):
    """Hand-worked step B through the tail of the stack: X' as worked by hand, y = (1.4375, 0.6875,
    ...) and z the final norm of y at eps 1e-20, which is step B's sublayer norm (eps 1e-6) up to the
    eps."""
    g, hc, d, X, _ = _hand_case()
    b = g["step_b"]
    delta = _bf(np.full((1, d), b["delta"]))
    out = orc.hc_post_then_final(delta, X, np.array([b["post_in"]], np.float32), np.array([b["comb_in"]], np.float32),
                                 np.array([b["pre_mix"]], np.float32), np.ones(d, np.float32), 1e-20, lib=lib)
    xo = orc.bf16_to_double(out["X_out"][0])
    assert np.array_equal(xo[0], np.tile(b["X_out_stream0_first_two"], 4))
    assert np.array_equal(xo[1], np.tile(b["X_out_stream1_first_two"], 4))
    y = np.tile(b["y_first_two"], 4)
    want = y / math.sqrt((y ** 2).mean() + 1e-20)
    assert np.array_equal(out["z"][0], orc.double_to_bf16(want, lib=lib))
    assert np.allclose(want[:2], b["y_normed_exact_first_two"], rtol=1e-6)


def pin_stream_mean(lib):
    """The tap of the multi-token-prediction head: mean over the streams. Identical streams give the
    value itself; (a, -a, b, -b) gives 0; dyadic streams give their exact mean; random streams match
    numpy's float64 mean rounded once; the mean is over the stream axis, not the columns."""
    d = 16
    a = _bf(np.arange(-8, 8) * 0.375)
    X = np.stack([a, a, a, a])[None]
    out, ex = orc.stream_mean(X, lib=lib)
    assert np.array_equal(out[0], a)
    b = _bf(np.arange(1, d + 1) * 0.125)
    neg = lambda v: (v ^ 0x8000).astype(np.uint16)  # noqa: E731
    out, ex = orc.stream_mean(np.stack([a, neg(a), b, neg(b)])[None], lib=lib)
    assert np.all(ex == 0)
    c = np.array([1.0, 0.5, 0.25, 2.0])
    X = _bf(np.repeat(c[:, None], d, axis=1))[None]
    _, ex = orc.stream_mean(X, lib=lib)
    assert np.all(ex == c.mean())
    rng = np.random.default_rng(30)
    X = _rand_bf16(rng, (3, 4, d))
    out, ex = orc.stream_mean(X, lib=lib)
    want = orc.bf16_to_double(X).mean(axis=1)
    assert np.allclose(ex, want, rtol=1e-15, atol=0)
    assert np.array_equal(out, orc.double_to_bf16(want, lib=lib))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
