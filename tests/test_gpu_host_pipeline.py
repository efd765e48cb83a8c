"""The host-buffer executor (hc_host_post_then_pre): every per-token array in host memory, streamed
through the GPU in chunks whose copies, in both directions, overlap the fused step.

Each chunk is hc_post_then_pre on that chunk's tokens, so the executor's results must equal, bit
for bit, the device call run on the same chunk slices. That checks the plumbing exactly (offsets,
ragged last chunks, the reuse of the three staging buffers within a call and across calls, the
ordering on other streams); the oracle then checks the results themselves (every token of the small
cases, sampled tokens of the full prefill batch).
"""

import numpy as np
import pytest
import torch

import hyper_connection_residual_hc_gb300 as hc
from hyper_connection_residual_hc_gb300 import synth
from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_POST, T_PREMIX, T_X

import gpu_util as gu

pytestmark = pytest.mark.gpu

IN = ("delta", "X", "post", "comb", "pre_mix")
OUT = ("X_out", "y_normed", "pre", "post", "comb")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()
    gu.device_error_clear()
    yield
    gu.device_error_clear()


def _draw(w, step=0):
    return dict(X=synth.tokens(w, T_X, step), delta=synth.tokens(w, T_DELTA, step),
                post=synth.tokens(w, T_POST, step), comb=synth.tokens(w, T_COMB, step),
                pre_mix=synth.tokens(w, T_PREMIX, step))


def _host(a, pinned):
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.pin_memory() if pinned else t.clone()


def _host_outputs(n, hcn, d, pinned):
    def e(shape, dt):
        return torch.empty(shape, dtype=dt, pin_memory=pinned)
    return dict(X_out=e((n, hcn, d), torch.bfloat16), y_normed=e((n, d), torch.bfloat16),
                pre=e((n, hcn), torch.float32), post=e((n, hcn), torch.float32), comb=e((n, hcn, hcn), torch.float32))


def _run_host(pipe, hin, P, n, s, hout, stream=None):
    hc.hc_host_post_then_pre(pipe, hin["delta"], hin["X"], hin["post"], hin["comb"], hin["pre_mix"], P.c, n, s,
                             hout["X_out"], hout["y_normed"], hout["pre"], hout["post"], hout["comb"], stream)


def _per_chunk_reference(dev, P, s, n, chunk):
    """hc_post_then_pre on the device over the executor's chunks, gathered on the host."""
    parts = {k: [] for k in OUT}
    for t0, m in hc.hc_host_chunk_plan(n, chunk):
        sl = {k: dev[k][t0:t0 + m].clone() for k in IN}  # own allocations: 16-byte aligned at any t0
        o = gu.run_post_then_pre(sl["delta"], sl["X"], sl["post"], sl["comb"], sl["pre_mix"], P, s, m)
        for k in OUT:
            parts[k].append(o[k].cpu())
    return {k: torch.cat(v) for k, v in parts.items()}


def _chunk_groups(n, chunk, s, idx):
    """The group size of the fused call that computed each sampled token (that of its chunk)."""
    plan = hc.hc_host_chunk_plan(n, chunk)
    starts = np.array([t0 for t0, _ in plan])
    sizes = np.array([m for _, m in plan])
    which = np.searchsorted(starts, idx, side="right") - 1
    return np.array([gu.plan_group(int(sizes[c]), s) for c in which])


def _assert_same(hout, ref, label):
    for k in OUT:
        a, b = hout[k], ref[k]
        assert a.shape == b.shape, (label, k)
        same = torch.equal(a.view(torch.int16), b.view(torch.int16)) if a.dtype == torch.bfloat16 else \
            torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert same, "%s: %s differs from the per-chunk device calls" % (label, k)


@pytest.mark.parametrize("n,chunk,d,hcn", [(1000, 384, 5120, 4), (2500, 256, 1024, 4), (3000, 512, 2048, 4),
                                           (5, 1024, 5120, 4), (1, 1, 256, 4), (40, 1, 256, 4),
                                           (140000, 4096, 256, 4), (300, 128, 1000, 2), (500, 128, 64, 8)])
def test_host_pipeline_matches_device_chunks_and_oracle(n, chunk, d, hcn):
    """Ramped plans with a ragged middle chunk, even splits, a single chunk smaller than the chunk
    size, one-token chunks, more chunks than staging buffers, three segments of coefficient copies
    (140,000 tokens: 65,536 + 65,536 + the rest, the first segment buffer used twice), and shapes of
    the generic path with per-chunk coefficient copies (hc = 2, d = 1000) and with segments (hc = 8)."""
    w = synth.small("step_b1_t64", 1, n, d, seed=1300 + n + d, hc=hcn)
    inp = _draw(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d, hcn)
    s = gu.shape_of(w)
    hin = {k: _host(inp[k], True) for k in IN}
    hout = _host_outputs(n, hcn, d, True)
    with hc.HostPipeline(hcn, d, chunk) as pipe:
        assert pipe.chunk_tokens == chunk
        _run_host(pipe, hin, P, n, s, hout)
        torch.cuda.current_stream().synchronize()
    dev = {k: hin[k].cuda() for k in IN}
    _assert_same(hout, _per_chunk_reference(dev, P, s, n, chunk), "n=%d chunk=%d" % (n, chunk))
    idx = np.arange(n) if n <= 400 else gu.sample_tokens(n, 300, np.random.default_rng(n))
    gu.check_sampled(w, 0, dev, hout, prm, idx, True, "host pipeline n=%d d=%d hc=%d" % (n, d, hcn),
                     _chunk_groups(n, chunk, s, idx))
    gu.device_error_clear()


def test_back_to_back_calls_other_stream_and_pageable_memory():
    """Three calls enqueued without a host wait in between (different inputs and outputs, so a
    staging buffer reused too early would show), the second on a side stream, the third with
    pageable host arrays; each equals its own per-chunk reference."""
    n, d, chunk = 2100, 2048, 256
    ws = [synth.small("step_b1_t64", 1, n, d, seed=1400 + k) for k in range(3)]
    prm = synth.params(ws[0], 0)
    P = gu.DevParams(prm, d)
    s = gu.shape_of(ws[0])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    hins, houts = [], []
    with hc.HostPipeline(4, d, chunk) as pipe:
        for k, w in enumerate(ws):
            pinned = k < 2
            inp = _draw(w)
            hins.append({key: _host(inp[key], pinned) for key in IN})
            houts.append(_host_outputs(n, 4, d, pinned))
            _run_host(pipe, hins[-1], P, n, s, houts[-1], side if k == 1 else None)
        torch.cuda.synchronize()
    for k in range(3):
        dev = {key: hins[k][key].cuda() for key in IN}
        _assert_same(houts[k], _per_chunk_reference(dev, P, s, n, chunk), "call %d" % k)
    gu.device_error_clear()


def test_host_pipeline_validation():
    n, d = 64, 1024
    w = synth.small("step_b1_t64", 1, n, d, seed=1500)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = gu.shape_of(w)
    hin = {k: _host(v, True) for k, v in _draw(w).items()}
    hout = _host_outputs(n, 4, d, True)

    base = dict(delta=hin["delta"], X=hin["X"], post=hin["post"], comb=hin["comb"], pre_mix=hin["pre_mix"],
                P=P.c, n=n, s=s, X_out=hout["X_out"], y_normed=hout["y_normed"], pre_out=hout["pre"],
                post_out=hout["post"], comb_out=hout["comb"])

    def expect(status, **over):
        a = dict(base, **over)
        with pytest.raises(hc.HCError) as e:
            hc.hc_host_post_then_pre(pipe, a["delta"], a["X"], a["post"], a["comb"], a["pre_mix"], a["P"], a["n"],
                                     a["s"], a["X_out"], a["y_normed"], a["pre_out"], a["post_out"], a["comb_out"])
        assert e.value.status == status

    with hc.HostPipeline(4, d, 32) as pipe:
        expect(hc.HC_ERR_SHAPE, s=hc.shape(d=2048))
        expect(hc.HC_ERR_SHAPE, s=hc.shape(d=d, hc=2))
        expect(hc.HC_ERR_SHAPE, n=-1)
        expect(hc.HC_ERR_ARG, s=hc.shape(d=d, sinkhorn_iters=0))
        expect(hc.HC_ERR_NULL, P=hc.params(None, P.hc_scale, P.hc_base, P.norm_w))
        expect(hc.HC_ERR_ALIAS, X_out=hin["X"])
        expect(hc.HC_ERR_ALIAS, y_normed=hin["delta"][8:])
        # n == 0 is a no-op that leaves the outputs untouched
        before = hout["y_normed"].clone()
        hc.hc_host_post_then_pre(pipe, hin["delta"], hin["X"], hin["post"], hin["comb"], hin["pre_mix"], P.c, 0, s,
                                 hout["X_out"], hout["y_normed"], hout["pre"], hout["post"], hout["comb"])
        torch.cuda.synchronize()
        assert torch.equal(before.view(torch.int16), hout["y_normed"].view(torch.int16))
    with pytest.raises(hc.HCError) as e:
        hc.HostPipeline(4, 1004, 0)
    assert e.value.status == hc.HC_ERR_SHAPE


@pytest.mark.slow
def test_host_pipeline_prefill_b4_t4096():
    """The full prefill batch (16,384 tokens, d = 5120) in the default chunks, as bench.py's
    end-to-end run streams it: X_out bit-exact against one device call on the whole batch (the
    writing half is per element), the rest against the oracle on sampled tokens."""
    w = synth.WORKLOADS["prefill_b4_t4096"]
    n, d = w.n, w.d
    inp = _draw(w)
    prm = synth.params(w, 0)
    P = gu.DevParams(prm, d)
    s = gu.shape_of(w)
    hin = {k: _host(inp[k], True) for k in IN}
    hout = _host_outputs(n, 4, d, True)
    with hc.HostPipeline(4, d, 0) as pipe:
        _run_host(pipe, hin, P, n, s, hout)
        torch.cuda.current_stream().synchronize()
    dev = {k: hin[k].cuda() for k in IN}
    full = gu.run_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, s, n)
    assert torch.equal(hout["X_out"].view(torch.int16), full["X_out"].cpu().view(torch.int16))
    del full
    idx = gu.sample_tokens(n, 400, np.random.default_rng(4096))
    gu.check_sampled(w, 0, dev, hout, prm, idx, True, "host pipeline prefill", _chunk_groups(n, 0, s, idx))
    gu.device_error_clear()
