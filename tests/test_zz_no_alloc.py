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
from hyper_connection_residual_hc_gb300 import synth
from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_POST, T_PREMIX, T_X

import gpu_util as gu

pytestmark = pytest.mark.gpu


def _batch(n, d, seed):
    w = synth.small("step_b1_t64", 1, n, d, seed=seed)
    dev = dict(X=gu.dev_bf16(synth.tokens(w, T_X, 0)), delta=gu.dev_bf16(synth.tokens(w, T_DELTA, 0)),
               post=gu.dev_f32(synth.tokens(w, T_POST, 0)), comb=gu.dev_f32(synth.tokens(w, T_COMB, 0)),
               pre_mix=gu.dev_f32(synth.tokens(w, T_PREMIX, 0)))
    return w, dev


def test_noalloc_matches_the_workspace_call_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()
    d = 5120
    for n, seed in ((300, 901), (1000, 902)):
        w, dev = _batch(n, d, seed)
        P = gu.DevParams(synth.params(w, 0), d)
        s = hc.shape(d=d, sinkhorn_iters=w.iters, hc_eps=w.hc_eps, norm_eps=w.norm_eps)
        ref = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, s, n)
        got = gu.alloc_outputs(n, d, True)
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
        print("n=%d: noalloc call %s the workspace call bit for bit" % (n, "matches" if same else "differs from"))
