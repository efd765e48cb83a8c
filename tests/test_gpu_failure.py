"""Failure detection without a GPU fault: every wait in the library's kernels is bounded, and a wait
that runs out records a bit in the device error word and returns, leaving the context usable. Here
a wait is made to run out on exchange counters nothing advances (hc_debug_wait_flag runs the fused
kernel's own bounded counter wait with a short limit); the host reads the bit, and the same context
then runs a normal step correctly.
"""

import time

import numpy as np
import pytest
import torch

import hyper_connection_residual_hc_gb300 as hc
from hyper_connection_residual_hc_gb300 import synth
from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_POST, T_PREMIX, T_X

import gpu_util as gu

pytestmark = pytest.mark.gpu

EXCHANGE_BIT = 64  # the device error word's bit for a wait on the group's arrival counter


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()
    hc.hc_device_error(clear=True)
    yield
    hc.hc_device_error(clear=True)


def test_flag_wait_runs_out_and_reports():
    flags = torch.zeros(8, dtype=torch.int64, device="cuda")  # nothing will set these
    t0 = time.perf_counter()
    hc.hc_debug_wait_flag(flags, 8, 1, 20_000_000)  # give up after 20 ms
    word = hc.hc_device_error(clear=True)  # synchronises
    elapsed = time.perf_counter() - t0
    assert word & EXCHANGE_BIT, "the wait that ran out was not reported (word 0x%x)" % word
    assert elapsed < 0.9, "the wait did not stop at its limit (%.3f s)" % elapsed
    assert hc.hc_device_error(clear=True) == 0  # cleared


def test_flag_wait_that_is_met_reports_nothing():
    flags = torch.full((8,), 5, dtype=torch.int64, device="cuda")
    hc.hc_debug_wait_flag(flags, 8, 5, 20_000_000)
    hc.hc_debug_wait_flag(flags, 8, 3, 20_000_000)  # a counter past its target also meets it
    assert hc.hc_device_error(clear=True) == 0


def test_context_usable_after_a_wait_ran_out():
    flags = torch.zeros(4, dtype=torch.int64, device="cuda")
    hc.hc_debug_wait_flag(flags, 4, 7, 5_000_000)
    assert hc.hc_device_error(clear=True) & EXCHANGE_BIT
    n, d = 70, 5120
    w = synth.small("step_b1_t64", 1, n, d, seed=1500)
    inp = {k: synth.tokens(w, t, 0) for k, t in (("X", T_X), ("delta", T_DELTA), ("post", T_POST),
                                                  ("comb", T_COMB), ("pre_mix", T_PREMIX))}
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    dev = {k: (gu.dev_bf16(v) if v.dtype == np.uint16 else gu.dev_f32(v)) for k, v in inp.items()}
    out = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, gu.shape_of(w), n)
    gu.check_sampled(w, 0, dev, out, prm, np.arange(n), True, "after a wait ran out")
    assert hc.hc_device_error(clear=True) == 0
