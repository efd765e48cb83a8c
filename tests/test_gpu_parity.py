"""CUDA path against the CPU oracle, element by element, through the C ABI.

Small cases run every output of every token through the oracle; they span several tiles and a
ragged last tile (n = 1, 3, 127, 129, 300) and several stream widths (d = 256 ... 5120). The
full-size workloads are checked on sampled tokens (tokens are independent, so a sample is exact)
and the chained workloads step by step, teacher-forced: each step's oracle takes the GPU's own
inputs for that step. Tolerances are defined in gpu_util.
"""

import numpy as np
import pytest
import torch

import hyper_connection_residual_hc_gb300 as hc
import oracle as orc
from hyper_connection_residual_hc_gb300 import synth
from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_POST, T_PREMIX, T_X

import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()
    gu.device_error_clear()
    yield
    gu.device_error_clear()


def _inputs(w, step=0, lo=0, hi=None):
    hi = w.n if hi is None else hi
    return dict(X=synth.tokens(w, T_X, step, lo, hi), delta=synth.tokens(w, T_DELTA, step, lo, hi),
                post=synth.tokens(w, T_POST, step, lo, hi), comb=synth.tokens(w, T_COMB, step, lo, hi),
                pre_mix=synth.tokens(w, T_PREMIX, step, lo, hi))


def _shape(w):
    return hc.shape(d=w.d, sinkhorn_iters=w.iters, hc_eps=w.hc_eps, norm_eps=w.norm_eps)


# ---- pieces ----------------------------------------------------------------------------------------

def test_prepare_params_split_is_exact():
    w = synth.WORKLOADS["prefill_b4_t4096"]
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, w.d)
    planes = gu.host_u16(P.planes).reshape(72, 4 * w.d)
    vals = orc.bf16_to_double(planes)
    rec = np.zeros((24, 4 * w.d))
    for h in range(2):
        for p in range(3):
            rec[12 * h:12 * h + 12] += vals[36 * h + 12 * p:36 * h + 12 * p + 12]
    assert np.array_equal(rec, prm["hc_fn"].astype(np.float64))
    # the hi plane is the nearest bf16 of each weight
    hi = np.concatenate([planes[0:12], planes[36:48]])
    assert np.array_equal(hi, orc.double_to_bf16(prm["hc_fn"].astype(np.float64)))


@pytest.mark.parametrize("n,d,group", [(600, 5120, 32), (1200, 5120, 16), (700, 1024, 32), (300, 5120, 8)])
def test_debug_mixes_forced_group(n, d, group):
    """The projection with a forced group size over several tiles per CTA (groups of 16 and 32 fold
    their tiles; 600 tokens over 4 groups of 32 is 3 tiles per CTA), against the oracle."""
    w = synth.small("step_b1_t64", 1, n, d, seed=150 + n + group)
    x = synth.tokens(w, T_X, 0)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    m_gpu = gu.host_f32(gu.debug_mixes(gu.dev_bf16(x), P, _shape(w), n, group))
    m_ref, _, S = orc.hc_mixes(x, prm["hc_fn"], w.norm_eps)
    gu.assert_mixes_close(m_gpu, m_ref, S)
    gu.device_error_clear()


@pytest.mark.parametrize("n,d", [(1, 5120), (3, 5120), (127, 5120), (300, 5120), (129, 1024), (40, 256)])
def test_debug_mixes_match_oracle(n, d):
    w = synth.small("step_b1_t64", 1, n, d, seed=100 + n)
    x = synth.tokens(w, T_X, 0)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = _shape(w)
    m_gpu = gu.host_f32(gu.debug_mixes(gu.dev_bf16(x), P, s, n))
    m_ref, r_ref, S = orc.hc_mixes(x, prm["hc_fn"], w.norm_eps)
    worst = gu.assert_mixes_close(m_gpu, m_ref, S)
    print("n=%d d=%d worst |err|/(uS) = %.3f" % (n, d, worst))
    gu.device_error_clear()


@pytest.mark.parametrize("n,d", [(1, 5120), (3, 5120), (127, 5120), (300, 5120), (129, 512), (33, 256)])
def test_pre_step_matches_oracle(n, d):
    w = synth.small("step_b1_t64", 1, n, d, seed=200 + n)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = _shape(w)
    X = gu.dev_bf16(inp["X"])
    out = gu.run_pre_step(X, gu.dev_f32(inp["pre_mix"]), P, s, n)
    m_gpu = gu.host_f32(gu.debug_mixes(X, P, s, n))
    ref = orc.hc_pre_step(inp["X"], inp["pre_mix"], prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"],
                          w.iters, w.hc_eps, w.norm_eps)
    exact, worst = gu.check_y_normed(gu.host_u16(out["y_normed"]), inp["X"], inp["pre_mix"], prm["norm_w"], w.norm_eps)
    gu.check_step(out, ref, m_gpu, ref["mixes"], ref["S"], prm, w.iters, w.hc_eps, "pre_step")
    print("n=%d d=%d y_normed bit-exact %.5f, max ulp %d" % (n, d, exact, worst))
    gu.device_error_clear()


@pytest.mark.parametrize("n,d", [(1, 5120), (3, 5120), (127, 5120), (300, 5120), (129, 1024), (65, 256)])
def test_post_then_pre_matches_oracle(n, d):
    w = synth.small("step_b1_t64", 1, n, d, seed=300 + n)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = _shape(w)
    out = gu.run_post_then_pre(gu.dev_bf16(inp["delta"]), gu.dev_bf16(inp["X"]), gu.dev_f32(inp["post"]),
                               gu.dev_f32(inp["comb"]), gu.dev_f32(inp["pre_mix"]), P, s, n)
    xo = gu.host_u16(out["X_out"])
    ex_x, _ = gu.check_xprime(xo, inp["X"], inp["delta"], inp["post"], inp["comb"])
    # reading half teacher-forced on the GPU's X'
    ref = orc.hc_pre_step(xo, inp["pre_mix"], prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"],
                          w.iters, w.hc_eps, w.norm_eps)
    ex_y, _ = gu.check_y_normed(gu.host_u16(out["y_normed"]), xo, inp["pre_mix"], prm["norm_w"], w.norm_eps)
    m_gpu = gu.host_f32(gu.debug_mixes(out["X_out"], P, s, n))
    gu.check_step(out, ref, m_gpu, ref["mixes"], ref["S"], prm, w.iters, w.hc_eps, "post_then_pre")
    # and free running: the oracle's own X' all the way (reported; bf16 ties may differ by 1 ulp)
    free = orc.hc_post_then_pre(inp["delta"], inp["X"], inp["post"], inp["comb"], inp["pre_mix"], prm["hc_fn"],
                                prm["hc_scale"], prm["hc_base"], prm["norm_w"], w.iters, w.hc_eps, w.norm_eps)
    dd = gu.ulp_diff(gu.host_u16(out["y_normed"]), free["y_normed"])
    print("n=%d d=%d X' bit-exact %.5f, y_normed bit-exact %.5f, free-running y_normed max ulp %d"
          % (n, d, ex_x, ex_y, int(dd.max())))
    gu.device_error_clear()


@pytest.mark.parametrize("n,d", [(1, 5120), (5, 24), (300, 5120), (77, 1024)])
def test_hc_post_matches_oracle(n, d):
    w = synth.small("step_b1_t64", 1, n, d, seed=400 + n)
    inp = _inputs(w)
    s = hc.shape(d=d)
    X = gu.dev_bf16(inp["X"])
    out = gu.guarded(X.shape, X.dtype)
    hc.hc_post(gu.dev_bf16(inp["delta"]), X, gu.dev_f32(inp["post"]), gu.dev_f32(inp["comb"]), n, s, out)
    ex, worst = gu.check_xprime(gu.host_u16(out), inp["X"], inp["delta"], inp["post"], inp["comb"], "hc_post")
    print("n=%d d=%d hc_post bit-exact %.6f, max ulp %d" % (n, d, ex, worst))
    # in place gives the same bits
    hc.hc_post(gu.dev_bf16(inp["delta"]), X, gu.dev_f32(inp["post"]), gu.dev_f32(inp["comb"]), n, s, X)
    assert np.array_equal(gu.host_u16(X), gu.host_u16(out))


@pytest.mark.parametrize("d", [256, 512])
def test_many_tiles_per_group_short_rows(d):
    """d = 256 gives one 32-column stage per CTA and tile: tiles end every stage, so the group
    exchange, the r_y hand-over and the y ring turn over at their fastest (about 17 tiles per group)."""
    n = 40000
    w = synth.small("step_b1_t64", 1, n, d, seed=500 + d)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = _shape(w)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    out = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, s, n)
    idx = gu.sample_tokens(n, 600, np.random.default_rng(d))
    gu.check_sampled(w, 0, dev, out, prm, idx, True, "short rows d=%d" % d)
    gu.device_error_clear()


@pytest.mark.parametrize("n,d,group,waves", [(100, 1024, 16, 1), (257, 5120, 16, 1), (544, 1024, 16, 1),
                                             (1000, 5120, 16, 2), (256, 5120, 32, 1), (129, 5120, 32, 1),
                                             (64, 5120, 32, 1), (2468, 2048, 8, 2), (2468, 1024, 8, 2)])
def test_group_sizes(n, d, group, waves):
    """Every group size the launch plan uses (8, 16 or 32 CTAs per token tile), single and multi-wave,
    with ragged last tiles. Groups of 16 and 32 fold their tiles (two column stages per pass): an even
    stage count (d = 1024 over 16 CTAs: 2 stages, one pass), an odd one whose last pass holds one
    stage (d = 5120 over 32 CTAs: 5 stages, 3 passes), and several tiles per CTA (1000 tokens)."""
    g, tm, nt = hc.hc_plan_tiles(n, d, hc.hc_fused_ctas())
    assert g == group and -(-nt // (hc.hc_fused_ctas() // g)) == waves, (g, tm, nt)
    w = synth.small("step_b1_t64", 1, n, d, seed=900 + n + d)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    out = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, _shape(w), n)
    idx = np.arange(n) if n <= 600 else gu.sample_tokens(n, 400, np.random.default_rng(n), tile=tm)
    gu.check_sampled(w, 0, dev, out, prm, idx, True, "group %d n=%d d=%d" % (g, n, d))
    # the reading half alone on the same streams
    o2 = gu.run_pre_step(dev["X"], dev["pre_mix"], P, _shape(w), n)
    gu.check_sampled(w, 0, dict(X=dev["X"], pre_mix=dev["pre_mix"]), o2, prm, idx, False,
                     "pre_step group %d n=%d d=%d" % (g, n, d))
    gu.device_error_clear()


# ---- special cases with closed forms ------------------------------------------------------------

def test_identity_comb_returns_streams_bit_exact():
    n, d = 130, 5120
    w = synth.small("step_b1_t64", 1, n, d, seed=7)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    post = np.zeros((n, 4), np.float32)
    comb = np.tile(np.eye(4, dtype=np.float32), (n, 1, 1))
    out = gu.run_post_then_pre(gu.dev_bf16(inp["delta"]), gu.dev_bf16(inp["X"]), gu.dev_f32(post), gu.dev_f32(comb),
                               gu.dev_f32(inp["pre_mix"]), P, _shape(w), n)
    assert np.array_equal(gu.host_u16(out["X_out"]), inp["X"])


def test_uniform_logits_closed_form_on_gpu():
    """hc_fn = 0 and base = 0 give mixes = 0: pre = 1/2 + eps, post = 1, comb = the scalar recurrence
    v <- v / (4 v + eps) from 1/4 + eps (one column step, then a row and a column step per round)."""
    n, d = 70, 5120
    w = synth.small("step_b1_t64", 1, n, d, seed=8)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    prm["hc_fn"][:] = 0
    prm["hc_base"][:] = 0
    P = gu.DevParams(prm, d)
    for iters, eps in [(20, 1e-6), (50, 1e-6), (3, 0.25)]:
        s = hc.shape(d=d, sinkhorn_iters=iters, hc_eps=eps)
        out = gu.run_pre_step(gu.dev_bf16(inp["X"]), gu.dev_f32(inp["pre_mix"]), P, s, n)
        v = 0.25 + eps
        v = v / (4 * v + eps)
        for _ in range(iters - 1):
            v = v / (4 * v + eps)
            v = v / (4 * v + eps)
        assert np.allclose(gu.host_f32(out["pre"]), 0.5 + np.float32(eps), rtol=1e-6)
        assert np.array_equal(gu.host_f32(out["post"]), np.ones((n, 4)))
        assert np.allclose(gu.host_f32(out["comb"]), v, rtol=1e-5), (gu.host_f32(out["comb"])[0, 0, 0], v)


def test_one_hot_pre_mix_reads_one_stream():
    n, d = 64, 5120
    w = synth.small("step_b1_t64", 1, n, d, seed=9)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    for j in range(4):
        pm = np.zeros((n, 4), np.float32)
        pm[:, j] = 1.0
        out = gu.run_pre_step(gu.dev_bf16(inp["X"]), gu.dev_f32(pm), P, _shape(w), n)
        want, _ = orc.rmsnorm(inp["X"][:, j], prm["norm_w"], w.norm_eps)
        gu.assert_bf16_close(gu.host_u16(out["y_normed"]), want, "one-hot y_normed stream %d" % j)


def test_model_norm_eps_1e20():
    """The model's own norm_eps (1e-20) instead of the workloads' 1e-6."""
    n, d = 129, 5120
    w = synth.small("step_b1_t64", 1, n, d, seed=10, norm_eps=1e-20)
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = _shape(w)
    X = gu.dev_bf16(inp["X"])
    out = gu.run_pre_step(X, gu.dev_f32(inp["pre_mix"]), P, s, n)
    ref = orc.hc_pre_step(inp["X"], inp["pre_mix"], prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"],
                          w.iters, w.hc_eps, w.norm_eps)
    gu.check_y_normed(gu.host_u16(out["y_normed"]), inp["X"], inp["pre_mix"], prm["norm_w"], w.norm_eps)
    gu.check_step(out, ref, gu.host_f32(gu.debug_mixes(X, P, s, n)), ref["mixes"], ref["S"], prm, w.iters, w.hc_eps,
                  "eps1e-20")


def test_zero_tokens_is_a_noop():
    d = 5120
    w = synth.small("step_b1_t64", 1, 4, d, seed=11)
    P = gu.DevParams(synth.params(w, 0), d)
    o = gu.alloc_outputs(4, d, True)
    o["y_normed"].fill_(3.0)
    X = torch.zeros((4, 4, d), dtype=torch.bfloat16, device="cuda")
    pm = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    hc.hc_pre_step(X, pm, P.c, 0, hc.shape(), o["y_normed"], o["pre"], o["post"], o["comb"], gu.workspace())
    torch.cuda.synchronize()
    assert bool((o["y_normed"] == 3.0).all())


# ---- the five workloads ------------------------------------------------------------------------------

def _report(name):
    print("%s: coefficients beyond the flat rel 1e-5 / abs 1e-6\n%s" % (name, gu.coef_stats_report()))


def test_workload_step_b1_t64():
    gu.COEF_STATS.clear()
    w = synth.WORKLOADS["step_b1_t64"]
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, w.d)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    out = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, _shape(w), w.n)
    gu.check_sampled(w, 0, dev, out, prm, np.arange(w.n), True, "step_b1_t64")
    gu.device_error_clear()
    _report(w.name)


def test_workload_prefill_b4_t4096():
    gu.COEF_STATS.clear()
    w = synth.WORKLOADS["prefill_b4_t4096"]
    inp = _inputs(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, w.d)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    out = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, _shape(w), w.n)
    idx = gu.sample_tokens(w.n, 384, np.random.default_rng(0))
    gu.check_sampled(w, 0, dev, out, prm, idx, True, "prefill_b4_t4096")
    # properties on every token: X_out differs from X, y_normed finite, comb columns sum to 1
    comb = out["comb"]
    assert torch.isfinite(out["y_normed"].float()).all()
    assert float((comb.sum(dim=1) - 1).abs().max()) < 1e-4
    pre = out["pre"]
    assert float(pre.min()) >= 1e-6 * 0.999 and float(pre.max()) <= 1 + 2e-6
    gu.device_error_clear()
    _report(w.name)


def _extreme_tokens(X_in, out, P, s, n, k=8):
    """Tokens at the extremes of one step, picked on the device: the largest |X| among the streams read
    and among those written, the largest |comb logit| (s2 * mix + base, from the GPU's own mixes of
    every token), the most nearly one-hot comb (largest sum of row maxima), and tokens whose pre or
    post saturated in fp32 (pre = 1 + eps, post = 2 or 0)."""
    picks = []

    def top(v):
        picks.append(torch.topk(v, min(k, n)).indices)

    top(X_in.float().abs().amax(dim=(1, 2)))
    if "X_out" in out:
        top(out["X_out"].float().abs().amax(dim=(1, 2)))
    m = gu.debug_mixes(out["X_out"] if "X_out" in out else X_in, P, s, n, gu.plan_group(n, s))
    logits = m[:, 2 * s.hc:] * P.hc_scale[2] + P.hc_base[2 * s.hc:]
    top(logits.abs().amax(dim=1))
    top(out["comb"].amax(dim=2).sum(dim=1))
    sat = ((out["pre"] == float(np.float32(1.0 + s.hc_eps))).any(dim=1) | (out["post"] == 2.0).any(dim=1) |
           (out["post"] == 0.0).any(dim=1)).nonzero().flatten()
    picks.append(sat[:k])
    return set(torch.cat(picks).cpu().numpy().tolist())


def _with_extremes(idx, X_in, out, P, s, n):
    return np.array(sorted(set(idx.tolist()) | _extreme_tokens(X_in, out, P, s, n)), dtype=np.int64)


def _run_chain(w, sample_k, first_pre_step, fresh_delta):
    """Steps: [hc_pre_step], then hc_post_then_pre ... ; every step checked teacher-forced on a sample:
    random tokens, the first and last, tile edges, and the step's extreme tokens (_extreme_tokens)."""
    rng = np.random.default_rng(w.seed)
    s = _shape(w)
    n = w.n
    X = gu.dev_bf16(synth.tokens(w, T_X, 0))
    pre_mix = gu.dev_f32(synth.tokens(w, T_PREMIX, 0))
    steps = w.steps
    worst = 0
    if first_pre_step:
        prm = synth.params(w, 0)
        P = gu.DevParams(prm, w.d)
        out = gu.run_pre_step(X, pre_mix, P, s, n)
        idx = _with_extremes(gu.sample_tokens(n, sample_k, rng), X, out, P, s, n)
        gu.check_sampled(w, 0, dict(X=X, pre_mix=pre_mix), out, prm, idx, False, "%s step 0" % w.name)
        state = dict(X=X, post=out["post"], comb=out["comb"], pre_mix=out["pre"], y=out["y_normed"])
        start = 1
        wd = prm["w_diag"]
    else:
        state = dict(X=X, post=gu.dev_f32(synth.tokens(w, T_POST, 0)), comb=gu.dev_f32(synth.tokens(w, T_COMB, 0)),
                     pre_mix=pre_mix, y=None)
        start = 0
        wd = None
    for l in range(start, steps):
        if fresh_delta:
            delta = gu.dev_bf16(synth.tokens(w, T_DELTA, l))
        else:
            delta = (state["y"].float() * gu.dev_f32(wd)).to(torch.bfloat16)  # stand-in sublayer
        prm = synth.params(w, l)
        P = gu.DevParams(prm, w.d)
        out = gu.run_post_then_pre(delta, state["X"], state["post"], state["comb"], state["pre_mix"], P, s, n)
        idx = _with_extremes(gu.sample_tokens(n, sample_k, rng), state["X"], out, P, s, n)
        dev_in = dict(X=state["X"], delta=delta, post=state["post"], comb=state["comb"], pre_mix=state["pre_mix"])
        gu.check_sampled(w, l, dev_in, out, prm, idx, True, "%s step %d" % (w.name, l))
        state = dict(X=out["X_out"], post=out["post"], comb=out["comb"], pre_mix=out["pre"], y=out["y_normed"])
        wd = prm["w_diag"]
        worst = max(worst, float(state["X"].float().abs().max()))
    gu.device_error_clear()
    return state, worst


def test_workload_decode_chain_b256_80steps():
    gu.COEF_STATS.clear()
    w = synth.WORKLOADS["decode_chain_b256_80steps"]
    state, worst = _run_chain(w, 256, first_pre_step=True, fresh_delta=False)
    # the chain's tail: the last writing half alone
    delta = gu.dev_bf16(synth.tokens(w, T_DELTA, w.steps))
    Xf = gu.guarded(state["X"].shape, state["X"].dtype)
    hc.hc_post(delta, state["X"], state["post"], state["comb"], w.n, _shape(w), Xf)
    gu.check_xprime(gu.host_u16(Xf), gu.host_u16(state["X"]), gu.host_u16(delta),
                    gu.host_f32(state["post"]).astype(np.float32), gu.host_f32(state["comb"]).astype(np.float32),
                    "decode chain tail")
    print("decode chain: max |X| after 80 steps %.3g" % worst)
    _report(w.name)


@pytest.mark.slow
def test_workload_long_prefill_b1_t65536_4steps():
    gu.COEF_STATS.clear()
    w = synth.WORKLOADS["long_prefill_b1_t65536_4steps"]
    _run_chain(w, 256, first_pre_step=False, fresh_delta=True)
    _report(w.name)


@pytest.mark.slow
def test_workload_stress_b2_t8192_80steps():
    gu.COEF_STATS.clear()
    w = synth.WORKLOADS["stress_b2_t8192_80steps"]
    _run_chain(w, 48, first_pre_step=True, fresh_delta=True)
    _report(w.name)
