"""A whole decode stack captured in one CUDA graph: 80 sublayers on 256 tokens (the decode chain's
stand-in sublayer delta = bf16(y_normed * w_diag) between the HC calls), entered through
hc_expand_pre_step and left through hc_post_then_final. The graph is replayed on two different
embeddings; each replay must reproduce an eager run of the same calls bit for bit. (The fused
kernel tags its exchange flags with launch numbers kept in the workspace, so replays, whose kernel
parameters are frozen at capture, still never accept a flag from an earlier launch; different
inputs per replay make a stale flag visible as wrong results.) The eager result itself is checked
against the oracle at the first and last step.
"""

import numpy as np
import pytest
import torch

import hyper_connection_residual_hc_gb300 as hc
import oracle as orc
from hyper_connection_residual_hc_gb300 import synth
from hyper_connection_residual_hc_gb300.synth import T_EMBED

import gpu_util as gu

pytestmark = pytest.mark.gpu

FINAL_EPS = 1e-20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hc.load()
    gu.device_error_clear()
    yield
    gu.device_error_clear()


class Stack:
    """Static buffers and parameters of an L-sublayer HC stack on n tokens (decode chain shape)."""

    def __init__(self, w, steps):
        n, d = w.n, w.d
        self.n, self.d, self.steps = n, d, steps
        self.s = gu.shape_of(w)
        self.sf = hc.shape(d=d, norm_eps=FINAL_EPS)
        self.P = [gu.DevParams(synth.params(w, l), d) for l in range(steps)]
        self.wd = [gu.dev_f32(synth.params(w, l)["w_diag"]) for l in range(steps)]
        self.fw = gu.dev_f32(synth.final_norm_w(w))
        bf = dict(dtype=torch.bfloat16, device="cuda")
        f32 = dict(dtype=torch.float32, device="cuda")
        self.h = torch.empty((n, d), **bf)
        self.X = [torch.empty((n, 4, d), **bf) for _ in range(2)]
        self.y = torch.empty((n, d), **bf)
        self.delta = torch.empty((n, d), **bf)
        self.coef = [dict(pre=torch.empty((n, 4), **f32), post=torch.empty((n, 4), **f32),
                          comb=torch.empty((n, 4, 4), **f32)) for _ in range(2)]
        self.z = torch.empty((n, d), **bf)
        self.Xf = torch.empty((n, 4, d), **bf)
        self.ws = hc.new_workspace()

    def run(self):
        """The whole stack on the current stream (what the graph captures)."""
        n, s = self.n, self.s
        c = self.coef[0]
        hc.hc_expand_pre_step(self.h, self.P[0].c, n, s, self.X[0], self.y, c["pre"], c["post"], c["comb"], self.ws)
        for l in range(1, self.steps):
            self.delta.copy_((self.y.float() * self.wd[l - 1]).to(torch.bfloat16))  # stand-in sublayer
            a, b = self.coef[(l - 1) % 2], self.coef[l % 2]
            hc.hc_post_then_pre(self.delta, self.X[(l - 1) % 2], a["post"], a["comb"], a["pre"], self.P[l].c, n, s,
                                self.X[l % 2], self.y, b["pre"], b["post"], b["comb"], self.ws)
        self.delta.copy_((self.y.float() * self.wd[self.steps - 1]).to(torch.bfloat16))
        last = self.coef[(self.steps - 1) % 2]
        hc.hc_post_then_final(self.delta, self.X[(self.steps - 1) % 2], last["post"], last["comb"], last["pre"],
                              self.fw, n, self.sf, self.Xf, self.z)


def test_decode_stack_graph_replays_match_eager():
    w = synth.WORKLOADS["decode_chain_b256_80steps"]
    st = Stack(w, w.steps)
    embeds = [synth.tokens(w, T_EMBED, 0), synth.tokens(w, T_EMBED, 1)]
    eager = []
    for e in embeds:
        st.h.copy_(gu.dev_bf16(e))
        st.run()
        torch.cuda.synchronize()
        eager.append((st.z.clone(), st.Xf.clone(), st.coef[(w.steps - 1) % 2]["pre"].clone()))
    assert not torch.equal(eager[0][0], eager[1][0])
    gu.device_error_clear()

    # the eager stack is right: first step and tail against the oracle
    st.h.copy_(gu.dev_bf16(embeds[1]))
    prm0 = synth.params(w, 0)
    ref0 = orc.hc_expand_pre_step(embeds[1], prm0["hc_fn"], prm0["hc_scale"], prm0["hc_base"], prm0["norm_w"],
                                  w.iters, w.hc_eps, w.norm_eps)
    hc.hc_expand_pre_step(st.h, st.P[0].c, st.n, st.s, st.X[0], st.y, st.coef[0]["pre"], st.coef[0]["post"],
                          st.coef[0]["comb"], st.ws)
    gu.check_y_normed(gu.host_u16(st.y), ref0["X_out"], np.full((st.n, 4), 0.25, np.float32), prm0["norm_w"],
                      w.norm_eps, "stack head")

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.run()  # warm the side stream once outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        st.run()
    for rep in range(2):
        for k, e in enumerate(embeds):
            st.h.copy_(gu.dev_bf16(e))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(st.z, eager[k][0]), "replay %d, embedding %d: z differs from eager" % (rep, k)
            assert torch.equal(st.Xf, eager[k][1]), "replay %d, embedding %d: X differs from eager" % (rep, k)
            assert torch.equal(st.coef[(w.steps - 1) % 2]["pre"], eager[k][2])
    gu.device_error_clear()

    # the tail of the replayed stack against the oracle, fed the replay's last streams
    # (teacher-forced: the final step recomputed on the CPU from the GPU's inputs of that step)
    last = st.coef[(w.steps - 1) % 2]
    Xl = gu.host_u16(st.X[(w.steps - 1) % 2])
    delta = gu.host_u16(st.delta)
    ref = orc.hc_post_then_final(delta, Xl, gu.host_f32(last["post"]).astype(np.float32),
                                 gu.host_f32(last["comb"]).astype(np.float32),
                                 gu.host_f32(last["pre"]).astype(np.float32), synth.final_norm_w(w), FINAL_EPS)
    gu.check_xprime(gu.host_u16(st.Xf), Xl, delta, gu.host_f32(last["post"]).astype(np.float32),
                    gu.host_f32(last["comb"]).astype(np.float32), "stack tail X'")
    gu.check_y_normed(gu.host_u16(st.z), gu.host_u16(st.Xf), gu.host_f32(last["pre"]).astype(np.float32),
                      synth.final_norm_w(w), FINAL_EPS, "stack tail z")
    dd = gu.ulp_diff(gu.host_u16(st.z), ref["z"])
    print("graph stack: tail z max ulp vs oracle %d" % int(dd.max()))
