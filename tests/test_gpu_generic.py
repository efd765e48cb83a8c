"""The generic path (the projection on the tensor cores, the other steps on CUDA cores) against the
oracle: any number of streams hc in 1..8 and any stream width d that is a multiple of 8, through
every entry point. hc = 4 at widths the fused kernel does not take (not a multiple of 256, or above
5120) runs here too. The formulas are the model's for any hc ("Source layer, pairs pooled" page,
Block excerpts; "Reading weights" page, hc_split_sinkhorn; "Write the streams" and "Final RMSNorm"
pages); tolerances as in gpu_util.
"""

import numpy as np
import pytest
import torch

import hyper_connection_residual_hc_gb300 as hc
import oracle as orc
from hyper_connection_residual_hc_gb300 import synth
from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_EMBED, T_POST, T_PREMIX, T_X

import gpu_util as gu

pytestmark = pytest.mark.gpu

CASES = [(1, 17, 256), (2, 37, 64), (2, 300, 1000), (3, 50, 200), (5, 20, 128), (8, 1, 64), (8, 33, 520),
         (8, 129, 5120), (4, 130, 1000), (4, 40, 6144)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()
    gu.device_error_clear()
    yield
    gu.device_error_clear()


def _setup(hcn, n, d, seed):
    w = synth.small("step_b1_t64", 1, n, d, seed=seed, hc=hcn)
    inp = {k: synth.tokens(w, t, 0) for k, t in (("X", T_X), ("delta", T_DELTA), ("post", T_POST),
                                                  ("comb", T_COMB), ("pre_mix", T_PREMIX), ("h", T_EMBED))}
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d, hcn)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    return w, inp, prm, P, dev


@pytest.mark.parametrize("hcn,n,d", CASES)
def test_generic_reading_and_writing(hcn, n, d):
    w, inp, prm, P, dev = _setup(hcn, n, d, 1200 + 10 * hcn + n + d)
    s = gu.shape_of(w)
    label = "hc=%d n=%d d=%d" % (hcn, n, d)
    # reading half alone
    out = gu.run_pre_step(dev["X"], dev["pre_mix"], P, s, n)
    ref = orc.hc_pre_step(inp["X"], inp["pre_mix"], prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"],
                          w.iters, w.hc_eps, w.norm_eps)
    gu.check_y_normed(gu.host_u16(out["y_normed"]), inp["X"], inp["pre_mix"], prm["norm_w"], w.norm_eps,
                      label + " y_normed")
    m_gpu = gu.host_f32(gu.debug_mixes(dev["X"], P, s, n))
    gu.check_step(out, ref, m_gpu, ref["mixes"], ref["S"], prm, w.iters, w.hc_eps, label + " pre_step")
    # writing half + next reading half, and the tap
    o = gu.alloc_outputs(n, d, True, hcn)
    mean = gu.guarded((n, d), torch.bfloat16)
    hc.hc_post_then_pre_tap(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P.c, n, s, o["X_out"],
                            o["y_normed"], o["pre"], o["post"], o["comb"], mean, gu.workspace())
    xo = gu.host_u16(o["X_out"])
    gu.check_xprime(xo, inp["X"], inp["delta"], inp["post"], inp["comb"], label + " X'")
    ref2 = orc.hc_pre_step(xo, inp["pre_mix"], prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"],
                           w.iters, w.hc_eps, w.norm_eps)
    gu.check_y_normed(gu.host_u16(o["y_normed"]), xo, inp["pre_mix"], prm["norm_w"], w.norm_eps,
                      label + " post y_normed")
    gu.check_step(o, ref2, gu.host_f32(gu.debug_mixes(o["X_out"], P, s, n)), ref2["mixes"], ref2["S"], prm, w.iters,
                  w.hc_eps, label + " post_then_pre")
    mref, mex = orc.stream_mean(xo)
    g = orc.bf16_to_double(gu.host_u16(mean))
    mag = np.abs(orc.bf16_to_double(xo)).sum(axis=1) / hcn
    assert np.all(np.abs(g - mex) <= gu.bf16_spacing(mex) + (hcn + 1) * gu.U * mag), label + " stream mean"
    # the plain call gives the same bits as the tap
    o2 = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, s, n)
    for k in ("X_out", "y_normed", "pre", "post", "comb"):
        assert torch.equal(o[k], o2[k]), k
    # hc_post alone, also in place
    Xp = gu.guarded(dev["X"].shape, dev["X"].dtype)
    hc.hc_post(dev["delta"], dev["X"], dev["post"], dev["comb"], n, s, Xp)
    assert torch.equal(Xp, o["X_out"])
    gu.device_error_clear()


@pytest.mark.parametrize("hcn,n,d", CASES)
def test_generic_stack_ends(hcn, n, d):
    w, inp, prm, P, dev = _setup(hcn, n, d, 1300 + 10 * hcn + n + d)
    s = gu.shape_of(w)
    label = "hc=%d n=%d d=%d" % (hcn, n, d)
    # head of the stack
    o = gu.alloc_outputs(n, d, True, hcn)
    hc.hc_expand_pre_step(dev["h"], P.c, n, s, o["X_out"], o["y_normed"], o["pre"], o["post"], o["comb"],
                          gu.workspace())
    want = np.repeat(inp["h"][:, None, :], hcn, axis=1)
    assert np.array_equal(gu.host_u16(o["X_out"]), want), label + " expanded streams"
    ref = orc.hc_expand_pre_step(inp["h"], prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"], w.iters,
                                 w.hc_eps, w.norm_eps, hc=hcn)
    m_ref, _, S = orc.hc_mixes(want, prm["hc_fn"], w.norm_eps)
    gu.check_y_normed(gu.host_u16(o["y_normed"]), want, np.full((n, hcn), 1.0 / hcn, np.float32), prm["norm_w"],
                      w.norm_eps, label + " expand y_normed")
    gu.check_step(o, ref, gu.host_f32(gu.debug_mixes(o["X_out"], P, s, n)), m_ref, S, prm, w.iters, w.hc_eps,
                  label + " expand")
    # tail of the stack
    fw = synth.final_norm_w(w)
    sf = hc.shape(d=d, norm_eps=1e-20, hc=hcn)
    z = gu.guarded((n, d), torch.bfloat16)
    hc.hc_final(dev["X"], dev["pre_mix"], gu.dev_f32(fw), n, sf, z)
    gu.check_y_normed(gu.host_u16(z), inp["X"], inp["pre_mix"], fw, 1e-20, label + " final z")
    Xo = gu.guarded(dev["X"].shape, dev["X"].dtype)
    z2 = gu.guarded(z.shape, z.dtype)
    hc.hc_post_then_final(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], gu.dev_f32(fw), n, sf, Xo,
                          z2)
    xo = gu.host_u16(Xo)
    gu.check_xprime(xo, inp["X"], inp["delta"], inp["post"], inp["comb"], label + " tail X'")
    gu.check_y_normed(gu.host_u16(z2), xo, inp["pre_mix"], fw, 1e-20, label + " tail z")
    z3 = gu.guarded(z.shape, z.dtype)
    hc.hc_post_then_final(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], gu.dev_f32(fw), n, sf,
                          None, z3)
    assert torch.equal(z2, z3)
    gu.device_error_clear()


def test_generic_uniform_logits_closed_form_hc8():
    """hc = 8, hc_fn = 0 and base = 0: pre = 1/2 + eps, post = 1, and every comb entry follows the
    scalar recurrence v <- v / (8 v + eps) from 1/8 + eps (one column step, then a row and a column
    step per round)."""
    hcn, n, d = 8, 9, 64
    w = synth.small("step_b1_t64", 1, n, d, seed=1400, hc=hcn)
    prm = synth.params(w, 0)
    prm["hc_fn"][:] = 0
    prm["hc_base"][:] = 0
    P = gu.DevParams(prm, d, hcn)
    X = gu.dev_bf16(synth.tokens(w, T_X, 0))
    pm = gu.dev_f32(synth.tokens(w, T_PREMIX, 0))
    for iters, eps in [(20, 1e-6), (3, 0.25)]:
        s = hc.shape(d=d, sinkhorn_iters=iters, hc_eps=eps, hc=hcn)
        out = gu.run_pre_step(X, pm, P, s, n)
        v = 1.0 / hcn + eps
        v = v / (hcn * v + eps)
        for _ in range(iters - 1):
            v = v / (hcn * v + eps)
            v = v / (hcn * v + eps)
        assert np.allclose(gu.host_f32(out["pre"]), 0.5 + np.float32(eps), rtol=1e-6)
        assert np.array_equal(gu.host_f32(out["post"]), np.ones((n, hcn)))
        assert np.allclose(gu.host_f32(out["comb"]), v, rtol=1e-5)


@pytest.mark.parametrize("name", ["prefill_b4_t4096_hc8", "prefill_b4_t4096_hc2", "prefill_b4_t4096_d7168",
                                  "prefill_b4_t4096_d2048"])
def test_prefill_batch_at_other_shapes(name):
    """The 16,384-token prefill batch at 8 or 2 streams, or at d = 7168 (the generic kernels) or
    d = 2048 (the fused kernel), in the call bench.py times: one hc_post_then_pre on all tokens,
    checked against the oracle on the first and last tokens, tile edges and 128 random tokens."""
    gu.COEF_STATS.clear()
    w = synth.WORKLOADS[name]
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, w.d, w.hc)
    inp = dict(X=synth.tokens(w, T_X, 0), delta=synth.tokens(w, T_DELTA, 0), post=synth.tokens(w, T_POST, 0),
               comb=synth.tokens(w, T_COMB, 0), pre_mix=synth.tokens(w, T_PREMIX, 0))
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    del inp
    out = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, gu.shape_of(w),
                               w.n)
    idx = gu.sample_tokens(w.n, 128, np.random.default_rng(3))
    gu.check_sampled(w, 0, dev, out, prm, idx, True, name)
    assert torch.isfinite(out["y_normed"].float()).all()
    assert float((out["comb"].sum(dim=1) - 1).abs().max()) < 1e-4
    gu.check_guards()
    gu.device_error_clear()
    print("%s: coefficients beyond the flat rel 1e-5 / abs 1e-6\n%s" % (name, gu.coef_stats_report()))
