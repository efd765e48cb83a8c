"""The multi-token-prediction tap on the GPU ("Final RMSNorm" page, Transformer.forward excerpt: at the
head's target layers the model keeps the mean over the hc streams entering the layer): the mean
hc_post_then_pre_tap writes against the oracle's mean of the call's own X' (within 1 bf16 ulp of an
fp32 evaluation), and every other output identical, bit for bit, to hc_post_then_pre's.
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


def check_mean(gpu_u16, Xp, what="stream_mean"):
    ref, exact = orc.stream_mean(Xp)
    mag = orc.bf16_to_double(Xp).__abs__().sum(axis=1) / 4
    g = orc.bf16_to_double(gpu_u16)
    tol = gu.bf16_spacing(exact) + 4 * gu.U * mag
    bad = np.abs(g - exact) > tol
    assert not bad.any(), "%s: %d values beyond 1 ulp + fp32 bound" % (what, int(bad.sum()))
    dd = gu.ulp_diff(np.asarray(gpu_u16), ref)
    return float((dd == 0).mean()), int(dd.max())


@pytest.mark.parametrize("n,d", [(1, 5120), (300, 5120), (129, 1024), (2468, 1024), (16384, 5120)])
def test_tap_matches_oracle_and_plain_call(n, d):
    w = synth.small("step_b1_t64", 1, n, d, seed=1100 + n + d) if n != 16384 else synth.WORKLOADS["prefill_b4_t4096"]
    inp = {k: synth.tokens(w, t, 0) for k, t in (("X", T_X), ("delta", T_DELTA), ("post", T_POST),
                                                  ("comb", T_COMB), ("pre_mix", T_PREMIX))}
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    s = gu.shape_of(w)
    ref = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, s, n)
    o = gu.alloc_outputs(n, d, True)
    mean = gu.guarded((n, d), torch.bfloat16)
    hc.hc_post_then_pre_tap(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P.c, n, s, o["X_out"],
                            o["y_normed"], o["pre"], o["post"], o["comb"], mean, gu.workspace())
    for k in ("X_out", "y_normed", "pre", "post", "comb"):
        assert torch.equal(o[k], ref[k]), k
    idx = np.arange(n) if n <= 3000 else gu.sample_tokens(n, 300, np.random.default_rng(3))
    exact, worst = check_mean(gu.host_u16(mean[idx]), gu.host_u16(o["X_out"][idx]))
    print("n=%d d=%d stream mean bit-exact %.5f, max ulp %d" % (n, d, exact, worst))
    gu.device_error_clear()
