"""How close an fp32 evaluation of the split can come to the exact one: the evidence behind the
coefficient tolerances of the GPU parity tests (gpu_util).

The "Reading weights" page's hc_split_sinkhorn kernel excerpt runs the split in fp32: sigmoid + eps,
2 sigmoid, a row softmax (max subtracted) + eps, one column normalisation, then iters - 1 rounds of
row and column normalisation, each dividing by its sum + eps. `split_fp32` below evaluates exactly
those steps in IEEE binary32 with numpy (every operation rounded once, plain division), as the
model's own fp32 kernel would, and compares the comb it returns with the double-precision oracle.
It is test-side only and never used to check the GPU.

What it shows, on mixes of the workloads' scale (the oracle's own mixes of workload tokens and
Gaussian mixes of the same spread):
  * at 20 rounds (the model's setting and that of every workload but the stress one) the fp32
    evaluation stays far inside the flat tolerance rel 1e-5 / abs 1e-6;
  * at 50 rounds on the stress workload's extreme logits it still meets the flat tolerance, with a
    thinner margin (up to 0.9 of it on 10 million such tokens), and it stays inside the first-order
    fp32 bound 2 iters (hc + 2) u |comb| (gpu_util.sinkhorn_fp32_bound).
So an fp32 implementation of the page's split can meet the flat tolerance at every round count of
the workloads, and the GPU's split is held to it without any widening.
"""

import numpy as np
import pytest

import oracle as orc
from hyper_connection_residual_hc_gb300 import synth
from hyper_connection_residual_hc_gb300.synth import T_X

import gpu_util as gu

F = np.float32


def split_fp32(m, hc_scale, hc_base, hc, iters, eps):
    """comb [n, hc, hc] of the page's split evaluated in IEEE fp32, steps in the page's order."""
    m = np.asarray(m, dtype=F)
    s2, eps = F(hc_scale[2]), F(eps)
    b = np.asarray(hc_base, dtype=F)[2 * hc:]
    n = m.shape[0]
    L = (m[:, 2 * hc:] * s2 + b).astype(F).reshape(n, hc, hc)      # logits, row j = source stream
    e = np.exp((L - L.max(axis=2, keepdims=True)).astype(F)).astype(F)
    C = (e / e.sum(axis=2, keepdims=True, dtype=F) + eps).astype(F)   # row softmax, + eps
    C = (C / (C.sum(axis=1, keepdims=True, dtype=F) + eps)).astype(F)  # first column normalisation
    for _ in range(iters - 1):
        C = (C / (C.sum(axis=2, keepdims=True, dtype=F) + eps)).astype(F)  # rows
        C = (C / (C.sum(axis=1, keepdims=True, dtype=F) + eps)).astype(F)  # columns
    return C


def _ratios(m, prm, iters, eps):
    _, _, exact = orc.split_sinkhorn(m, prm["hc_scale"], prm["hc_base"], 4, iters, eps)
    c32 = split_fp32(m, prm["hc_scale"], prm["hc_base"], 4, iters, eps).astype(np.float64)
    err = np.abs(c32 - exact)
    flat = np.maximum(1e-5 * np.abs(exact), 1e-6)
    bound = gu.sinkhorn_fp32_bound(exact, 4, iters)
    return float((err / flat).max()), float((err / bound).max())


def _mixes_samples(w, steps, gauss_tokens, gauss_sd, seed):
    """(mixes, params) pairs: the oracle's mixes of 256 workload tokens per parameter set, and
    Gaussian mixes with the spread those have (hc_fn ~ N(0, 0.02^2) over 20,480 inputs: sd 2.9)."""
    rng = np.random.default_rng(seed)
    for l in steps:
        prm = synth.params(w, l)
        x = synth.tokens(w, T_X, 0, 256 * l, 256 * l + 256)
        m, _, _ = orc.hc_mixes(x, prm["hc_fn"], w.norm_eps)
        yield m, prm
        g = (rng.standard_normal((gauss_tokens, w.M)) * gauss_sd).astype(F).astype(np.float64)
        yield g, prm


def test_fp32_sinkhorn_at_20_rounds_meets_the_flat_tolerance():
    """Workload distributions at the model's 20 rounds: an fp32 evaluation stays well inside rel 1e-5 /
    abs 1e-6, and inside the first-order bound."""
    w = synth.WORKLOADS["prefill_b4_t4096"]
    worst_flat = worst_bound = 0.0
    for m, prm in _mixes_samples(w, range(4), 1 << 14, 2.9, 11):
        a, b = _ratios(m, prm, w.iters, w.hc_eps)
        worst_flat, worst_bound = max(worst_flat, a), max(worst_bound, b)
    print("20 rounds: worst err/flat %.3f, err/bound %.3f" % (worst_flat, worst_bound))
    assert worst_flat < 0.5
    assert worst_bound < 1.0


def test_fp32_sinkhorn_at_50_rounds_on_stress_logits():
    """The stress workload (hc_scale ~ U(5, 10), hc_base ~ N(0, 3^2), 50 rounds): the fp32 evaluation
    meets the flat tolerance on this sample with a thinner margin, and stays inside the first-order
    bound."""
    w = synth.WORKLOADS["stress_b2_t8192_80steps"]
    worst_flat = worst_bound = 0.0
    for m, prm in _mixes_samples(w, range(6), 1 << 14, 4.0, 12):
        a, b = _ratios(m, prm, w.iters, w.hc_eps)
        worst_flat, worst_bound = max(worst_flat, a), max(worst_bound, b)
    print("50 rounds: worst err/flat %.3f, err/bound %.3f" % (worst_flat, worst_bound))
    assert worst_flat < 1.0
    assert worst_flat > 0.2   # not a loose margin: 50 rounds of fp32 use a good part of the flat tolerance
    assert worst_bound < 1.0


@pytest.mark.parametrize("iters", [1, 2, 20])
def test_split_fp32_agrees_with_the_oracle_on_mild_logits(iters):
    """The fp32 evaluation is the same computation as the oracle's: on mild logits (sd 0.3) where
    nothing is ill-conditioned it agrees to a few fp32 rounding errors, for every round count."""
    w = synth.WORKLOADS["step_b1_t64"]
    prm = synth.params(w, 0)
    m = np.random.default_rng(5).standard_normal((512, w.M)) * 0.3
    _, _, exact = orc.split_sinkhorn(m, prm["hc_scale"], prm["hc_base"], 4, iters, w.hc_eps)
    c32 = split_fp32(m, prm["hc_scale"], prm["hc_base"], 4, iters, w.hc_eps).astype(np.float64)
    assert np.abs(c32 - exact).max() <= 64 * iters * gu.U
