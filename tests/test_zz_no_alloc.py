"""hc_post_then_pre_noalloc: the step for callers that may not allocate device memory.

Some callers cannot call cudaMalloc where they run the step (an engine plugin that is handed no
workspace, a runtime whose memory plan is fixed after start-up). This entry point keeps its scratch
in a fixed array inside the library instead of a caller workspace. The test calls it twice in a
row through the C ABI, on two different batches, and checks each result against hc_post_then_pre
with a caller workspace on the same inputs, with the tolerances of the other parity tests (the
two calls run the same kernel, so in practice they agree bit for bit).

This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test.
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


def _batch(n, d, seed, hcn=4):
    w = synth.small("step_b1_t64", 1, n, d, seed=seed, hc=hcn)
    dev = dict(X=gu.dev_bf16(synth.tokens(w, T_X, 0)), delta=gu.dev_bf16(synth.tokens(w, T_DELTA, 0)),
               post=gu.dev_f32(synth.tokens(w, T_POST, 0)), comb=gu.dev_f32(synth.tokens(w, T_COMB, 0)),
               pre_mix=gu.dev_f32(synth.tokens(w, T_PREMIX, 0)))
    return w, dev


def _two_calls(d, hcn, cases):
    """Two calls in a row of the no-allocation step, each against the workspace call on the same inputs."""
    for n, seed in cases:
        w, dev = _batch(n, d, seed, hcn)
        prm = synth.params(w, 0)
        P = gu.DevParams(prm, d, hcn)
        s = hc.shape(d=d, sinkhorn_iters=w.iters, hc_eps=w.hc_eps, norm_eps=w.norm_eps, hc=hcn)
        ref = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, s, n)
        got = gu.alloc_outputs(n, d, True, hcn)
        hc.hc_post_then_pre_noalloc(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P.c, n, s,
                                    got["X_out"], got["y_normed"], got["pre"], got["post"], got["comb"])
        torch.cuda.synchronize()
        assert hc.hc_device_error(clear=True) == 0
        for k in ("X_out", "y_normed"):
            gu.assert_bf16_close(gu.host_u16(got[k]), gu.host_u16(ref[k]), "noalloc " + k)
        for k in ("pre", "post", "comb"):
            gu.assert_coef_close(gu.host_f32(got[k]), gu.host_f32(ref[k]), "noalloc " + k)
        same = all(torch.equal(got[k].view(torch.int16) if got[k].dtype == torch.bfloat16 else got[k],
                               ref[k].view(torch.int16) if ref[k].dtype == torch.bfloat16 else ref[k])
                   for k in got)
        print("hc=%d d=%d n=%d: noalloc call %s the workspace call bit for bit"
              % (hcn, d, n, "matches" if same else "differs from"))
        yield w, dev, prm, got


def _skip_without_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()


def test_noalloc_matches_the_workspace_call_twice_in_a_row():
    """The model's shape (hc = 4, d = 5120): the fused kernel with the fixed array as its exchange
    workspace."""
    _skip_without_gpu()
    for _ in _two_calls(5120, 4, ((300, 901), (1000, 902))):
        pass


def test_noalloc_generic_shape_twice_in_a_row():
    """A shape outside the fused kernel (hc = 3, d = 1000): the generic kernels, which take their chunked
    mixes and sums of squares from the fixed array. Also checked against the oracle."""
    _skip_without_gpu()
    for w, dev, prm, got in _two_calls(1000, 3, ((300, 903), (77, 904))):
        X, dl = gu.host_u16(dev["X"]), gu.host_u16(dev["delta"])
        po, co, pm = (gu.host_f32(dev[k]).astype(np.float32) for k in ("post", "comb", "pre_mix"))
        xo = gu.host_u16(got["X_out"])
        gu.check_xprime(xo, X, dl, po, co, "noalloc generic X_out")
        gu.check_y_normed(gu.host_u16(got["y_normed"]), xo, pm, prm["norm_w"], w.norm_eps, "noalloc generic y_normed")
        ref = orc.hc_pre_step(xo, pm, prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"], w.iters,
                              w.hc_eps, w.norm_eps)
        s = hc.shape(d=w.d, sinkhorn_iters=w.iters, hc_eps=w.hc_eps, norm_eps=w.norm_eps, hc=w.hc)
        m_gpu = gu.host_f32(gu.debug_mixes(got["X_out"], gu.DevParams(prm, w.d, w.hc), s, w.n))
        gu.check_step(got, ref, m_gpu, ref["mixes"], ref["S"], prm, w.iters, w.hc_eps, "noalloc generic")


def test_noalloc_after_clearing_the_error_word():
    """hc_device_error with `clear` zeroes the fixed array when a wait had given up: a bounded flag wait
    that runs out (on flags nothing sets) sets the word, and the no-allocation step is still right after
    the clear, its launch counters starting afresh."""
    _skip_without_gpu()
    flags = torch.zeros(4, dtype=torch.int64, device="cuda")
    hc.hc_debug_wait_flag(flags, 4, 1, 2_000_000)
    torch.cuda.synchronize()
    assert hc.hc_device_error(clear=True) != 0
    assert hc.hc_device_error(clear=True) == 0
    for _ in _two_calls(5120, 4, ((129, 905), (64, 906))):
        pass
