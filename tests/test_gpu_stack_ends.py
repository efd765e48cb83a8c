"""Ends of the stack on the GPU against the oracle, through the C ABI ("Final RMSNorm" page,
Transformer.forward excerpt):
  hc_expand_pre_step   the embedding copied into the four streams (checked bit-exact), then the
                       first reading half with the identity pre_mix;
  hc_final             the last collapse and the final RMSNorm (the page's eps 1e-20);
  hc_post_then_final   the last writing half fused with hc_final, with and without writing X';
and a whole stack of 80 sublayers from the embedding to the final norm, every step checked
teacher-forced. Tolerances are those of gpu_util: the final norm is the same collapse + RMSNorm
arithmetic as a reading half's y_normed.
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

FINAL_EPS = 1e-20  # the final RMSNorm's eps on the "Final RMSNorm" page


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()
    gu.device_error_clear()
    yield
    gu.device_error_clear()


def _identity(n):
    return np.full((n, 4), 0.25, np.float32)


def run_expand(h, P, s, n):
    o = gu.alloc_outputs(n, s.d, True)
    hc.hc_expand_pre_step(h, P.c, n, s, o["X_out"], o["y_normed"], o["pre"], o["post"], o["comb"], gu.workspace())
    return o


def check_expand(w, h_host, out, prm, idx, label):
    """Streams bit-exact copies of h; y_normed and the coefficients as a reading half of them."""
    h = h_host[idx]
    want = np.repeat(h[:, None, :], 4, axis=1)
    got = gu.host_u16(out["X_out"][idx])
    assert np.array_equal(got, want), "%s: streams are not copies of the embedding" % label
    ref = orc.hc_expand_pre_step(h, prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"], w.iters, w.hc_eps,
                                 w.norm_eps)
    m_ref, _, S = orc.hc_mixes(want, prm["hc_fn"], w.norm_eps)
    gu.check_y_normed(gu.host_u16(out["y_normed"][idx]), want, _identity(len(idx)), prm["norm_w"], w.norm_eps,
                      label + " y_normed")
    # the identity collapse gives y = h exactly, so y_normed is the sublayer norm of h itself
    yn_h, _ = orc.rmsnorm(h, prm["norm_w"], w.norm_eps)
    gu.assert_bf16_close(gu.host_u16(out["y_normed"][idx]), yn_h, label + " y_normed vs norm(h)")
    sub = {k: out[k][idx] for k in ("pre", "post", "comb")}
    P = gu.DevParams(prm, w.d)
    # the GPU's own mixes of these tokens, with the group size of the call on all w.n tokens
    m_gpu = gu.host_f32(gu.debug_mixes(gu.dev_bf16(want), P, gu.shape_of(w), len(idx),
                                       gu.plan_group(w.n, gu.shape_of(w))))
    gu.check_step(sub, ref, m_gpu, m_ref, S, prm, w.iters, w.hc_eps, label)


# ---- head of the stack ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,d", [(1, 5120), (3, 5120), (127, 5120), (300, 5120), (129, 1024), (33, 256),
                                 (5000, 256)])
def test_expand_pre_step_matches_oracle(n, d):
    w = synth.small("step_b1_t64", 1, n, d, seed=600 + n)
    h = synth.tokens(w, T_EMBED, 0)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    out = run_expand(gu.dev_bf16(h), P, gu.shape_of(w), n)
    idx = np.arange(n) if n <= 300 else gu.sample_tokens(n, 300, np.random.default_rng(n))
    check_expand(w, h, out, prm, idx, "expand n=%d d=%d" % (n, d))
    gu.device_error_clear()


def test_expand_pre_step_prefill_b4_t4096():
    w = synth.WORKLOADS["prefill_b4_t4096"]
    h = synth.tokens(w, T_EMBED, 0)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, w.d)
    out = run_expand(gu.dev_bf16(h), P, gu.shape_of(w), w.n)
    idx = gu.sample_tokens(w.n, 256, np.random.default_rng(1))
    check_expand(w, h, out, prm, idx, "expand prefill")
    # every token: the four streams are the embedding
    Xo = out["X_out"]
    hd = gu.dev_bf16(h)
    for j in range(4):
        assert torch.equal(Xo[:, j], hd)
    gu.device_error_clear()


def test_expand_matches_pre_step_on_expanded_streams():
    """The expand path (one operand tile for all four streams, identity pre_mix) and the plain
    reading half of the same four copies give identical bits."""
    n, d = 257, 5120
    w = synth.small("step_b1_t64", 1, n, d, seed=610)
    h = synth.tokens(w, T_EMBED, 0)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = gu.shape_of(w)
    a = run_expand(gu.dev_bf16(h), P, s, n)
    b = gu.run_pre_step(a["X_out"].clone(), gu.dev_f32(_identity(n)), P, s, n)
    for k in ("y_normed", "pre", "post", "comb"):
        assert torch.equal(a[k], b[k]), k


# ---- tail of the stack ---------------------------------------------------------------------------

def _final_inputs(w, scale=None):
    X = synth.tokens(w, T_X, 0)
    if scale is not None:
        X = orc.double_to_bf16(orc.bf16_to_double(X) * scale)
    return X, synth.tokens(w, T_PREMIX, 0), synth.final_norm_w(w)


@pytest.mark.parametrize("n,d,eps", [(1, 5120, FINAL_EPS), (3, 5120, FINAL_EPS), (300, 5120, FINAL_EPS),
                                     (129, 1024, 1e-6), (5, 8, FINAL_EPS), (77, 5112, FINAL_EPS),
                                     (40, 136, FINAL_EPS)])
def test_final_matches_oracle(n, d, eps):
    w = synth.small("step_b1_t64", 1, n, d, seed=700 + n + d)
    X, pm, fw = _final_inputs(w)
    z = gu.guarded((n, d), torch.bfloat16)
    hc.hc_final(gu.dev_bf16(X), gu.dev_f32(pm), gu.dev_f32(fw), n, hc.shape(d=d, norm_eps=eps), z)
    exact, worst = gu.check_y_normed(gu.host_u16(z), X, pm, fw, eps, "z")
    ref, _, _ = orc.hc_final(X, pm, fw, eps)
    dd = gu.ulp_diff(gu.host_u16(z), ref)
    print("n=%d d=%d eps=%g z bit-exact %.5f, max ulp %d" % (n, d, eps, exact, int(dd.max())))


def test_final_small_values_see_the_eps():
    """Streams of size ~2^-14: mean(y^2) ~ 1e-9, so eps 1e-6 and 1e-20 give different z; both match
    the oracle."""
    n, d = 64, 5120
    w = synth.small("step_b1_t64", 1, n, d, seed=720)
    X, pm, fw = _final_inputs(w, scale=2.0 ** -14)
    zs = {}
    for eps in (FINAL_EPS, 1e-6):
        z = gu.guarded((n, d), torch.bfloat16)
        hc.hc_final(gu.dev_bf16(X), gu.dev_f32(pm), gu.dev_f32(fw), n, hc.shape(d=d, norm_eps=eps), z)
        gu.check_y_normed(gu.host_u16(z), X, pm, fw, eps, "z eps=%g" % eps)
        zs[eps] = gu.host_u16(z)
    assert (gu.ulp_diff(zs[FINAL_EPS], zs[1e-6]) > 8).mean() > 0.5


@pytest.mark.parametrize("n,d", [(1, 5120), (300, 5120), (129, 1024), (6, 8), (50, 5112)])
def test_post_then_final_matches_oracle(n, d):
    w = synth.small("step_b1_t64", 1, n, d, seed=800 + n + d)
    X = synth.tokens(w, T_X, 0)
    delta, post, comb = synth.tokens(w, T_DELTA, 0), synth.tokens(w, T_POST, 0), synth.tokens(w, T_COMB, 0)
    pm, fw = synth.tokens(w, T_PREMIX, 0), synth.final_norm_w(w)
    s = hc.shape(d=d, norm_eps=FINAL_EPS)
    dev = [gu.dev_bf16(delta), gu.dev_bf16(X), gu.dev_f32(post), gu.dev_f32(comb), gu.dev_f32(pm), gu.dev_f32(fw)]
    Xo = gu.guarded((n, 4, d), torch.bfloat16)
    z = gu.guarded((n, d), torch.bfloat16)
    hc.hc_post_then_final(*dev, n, s, Xo, z)
    xo = gu.host_u16(Xo)
    ex_x, _ = gu.check_xprime(xo, X, delta, post, comb)
    ex_z, _ = gu.check_y_normed(gu.host_u16(z), xo, pm, fw, FINAL_EPS, "z")  # teacher-forced on the GPU's X'
    free = orc.hc_post_then_final(delta, X, post, comb, pm, fw, FINAL_EPS)
    dd = gu.ulp_diff(gu.host_u16(z), free["z"])
    # without writing the streams: the same z, bit for bit
    z2 = gu.guarded(z.shape, z.dtype)
    hc.hc_post_then_final(*dev, n, s, None, z2)
    assert torch.equal(z, z2)
    print("n=%d d=%d X' bit-exact %.5f, z bit-exact %.5f, free-running z max ulp %d" % (n, d, ex_x, ex_z, int(dd.max())))


def test_post_then_final_prefill_b4_t4096():
    w = synth.WORKLOADS["prefill_b4_t4096"]
    inp = {k: synth.tokens(w, t, 0) for k, t in (("X", T_X), ("delta", T_DELTA), ("post", T_POST),
                                                  ("comb", T_COMB), ("pre_mix", T_PREMIX))}
    fw = synth.final_norm_w(w)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    Xo = gu.guarded(dev["X"].shape, dev["X"].dtype)
    z = gu.guarded((w.n, w.d), torch.bfloat16)
    hc.hc_post_then_final(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], gu.dev_f32(fw), w.n,
                          hc.shape(d=w.d, norm_eps=FINAL_EPS), Xo, z)
    idx = gu.sample_tokens(w.n, 384, np.random.default_rng(2))
    xo = gu.host_u16(Xo[idx])
    gu.check_xprime(xo, inp["X"][idx], inp["delta"][idx], inp["post"][idx], inp["comb"][idx], "prefill X'")
    gu.check_y_normed(gu.host_u16(z[idx]), xo, inp["pre_mix"][idx], fw, FINAL_EPS, "prefill z")
    assert torch.isfinite(z.float()).all()


# ---- a whole stack -------------------------------------------------------------------------------

def test_stack_from_embedding_to_final_norm():
    """80 sublayers on 256 tokens, as the decode chain (stand-in sublayer delta = bf16(y_normed *
    w_diag)), entered through hc_expand_pre_step and left through hc_post_then_final; each step
    checked on every token against the oracle fed that step's device inputs."""
    w = synth.WORKLOADS["decode_chain_b256_80steps"]
    n, s = w.n, gu.shape_of(w)
    h = synth.tokens(w, T_EMBED, 0)
    prm = synth.params(w, 0)
    out = run_expand(gu.dev_bf16(h), gu.DevParams(prm, w.d), s, n)
    idx = np.arange(n)
    check_expand(w, h, out, prm, idx, "stack step 0")
    state = dict(X=out["X_out"], post=out["post"], comb=out["comb"], pre_mix=out["pre"], y=out["y_normed"])
    wd = prm["w_diag"]
    for l in range(1, w.steps):
        delta = (state["y"].float() * gu.dev_f32(wd)).to(torch.bfloat16)
        prm = synth.params(w, l)
        out = gu.run_post_then_pre(delta, state["X"], state["post"], state["comb"], state["pre_mix"],
                                   gu.DevParams(prm, w.d), s, n)
        dev_in = dict(X=state["X"], delta=delta, post=state["post"], comb=state["comb"], pre_mix=state["pre_mix"])
        gu.check_sampled(w, l, dev_in, out, prm, idx, True, "stack step %d" % l)
        state = dict(X=out["X_out"], post=out["post"], comb=out["comb"], pre_mix=out["pre"], y=out["y_normed"])
        wd = prm["w_diag"]
    delta = (state["y"].float() * gu.dev_f32(wd)).to(torch.bfloat16)
    fw = synth.final_norm_w(w)
    Xo = gu.guarded(state["X"].shape, state["X"].dtype)
    z = gu.guarded((n, w.d), torch.bfloat16)
    hc.hc_post_then_final(delta, state["X"], state["post"], state["comb"], state["pre_mix"], gu.dev_f32(fw), n,
                          hc.shape(d=w.d, norm_eps=FINAL_EPS), Xo, z)
    xo = gu.host_u16(Xo)
    gu.check_xprime(xo, gu.host_u16(state["X"]), gu.host_u16(delta), gu.host_f32(state["post"]).astype(np.float32),
                    gu.host_f32(state["comb"]).astype(np.float32), "stack tail X'")
    gu.check_y_normed(gu.host_u16(z), xo, gu.host_f32(state["pre_mix"]).astype(np.float32), fw, FINAL_EPS,
                      "stack tail z")
    gu.device_error_clear()
