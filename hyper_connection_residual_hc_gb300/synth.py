"""Seeded synthetic inputs for the Hyper-Connection stream step.

This module only draws random numbers and rounds them to the storage formats. It holds none of
the step's arithmetic, so both the CUDA path and the CPU oracle can take their inputs from it.

Every per-token tensor is drawn in independent blocks of ``BLOCK`` tokens, each block from its own
PCG64 stream seeded by (workload seed, step, tensor id, block index). Any token range can therefore
be regenerated on its own, which lets the parity tests check sampled tokens of a 65,536-token
workload without drawing all of it twice.

Distributions (per workload, see ``WORKLOADS``):
  X        bf16 [n, hc, d]   N(0,1), or 4 * Student-t(3) for the stress workload
  delta    bf16 [n, d]       N(0, delta_sd^2)
  post     fp32 [n, hc]      2 * sigmoid(N(0,1))
  comb     fp32 [n, hc, hc]  softmax over each row of a N(0,1) matrix
  pre_mix  fp32 [n, hc]      sigmoid(N(0,1)) + 1e-6
  hc_fn    fp32 [(2+hc)*hc, hc*d]  N(0, 0.02^2)
  hc_base  fp32 [(2+hc)*hc]  N(0, base_sd^2)
  hc_scale fp32 [3]          U(scale_lo, scale_hi)
  norm_w   fp32 [d]          1 + N(0, 0.1^2), rounded to a bf16 value (stored as fp32)
  w_diag   fp32 [d]          N(0, 0.5^2), the stand-in sublayer of the decode chain
  embed    bf16 [n, d]       N(0,1): the embedding rows the head of the stack expands into streams
  final_w  fp32 [d]          1 + N(0, 0.1^2) rounded to bf16: the final norm's gain
bf16 values are drawn in float32 (float64 for Student-t), then rounded to nearest-even bf16.
"""

from __future__ import annotations

import dataclasses

import numpy as np

BLOCK = 1024

# tensor ids, part of the seed
T_X, T_DELTA, T_POST, T_COMB, T_PREMIX, T_FN, T_BASE, T_SCALE, T_NORMW, T_WDIAG, T_EMBED, T_FINALW = range(12)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    T: int
    hc: int = 4
    d: int = 5120
    steps: int = 1             # number of HC sublayer steps (parameter sets)
    chain: str = "single"      # "single": one hc_post_then_pre; "decode": pre_step, post_then_pre..., post
                               # with delta = bf16(y_normed * w_diag); "fresh": chained post_then_pre
                               # with a fresh delta per step; "stress": like decode but fresh deltas
    iters: int = 20
    hc_eps: float = 1e-6
    norm_eps: float = 1e-6
    x_dist: str = "normal"
    delta_sd: float = 1.0
    scale_lo: float = 0.5
    scale_hi: float = 2.0
    base_sd: float = 1.0
    fn_sd: float = 0.02

    @property
    def n(self) -> int:
        return self.B * self.T

    @property
    def M(self) -> int:
        return (2 + self.hc) * self.hc


WORKLOADS = {
    w.name: w
    for w in [
        Workload("step_b1_t64", seed=0, B=1, T=64),
        Workload("decode_chain_b256_80steps", seed=1000, B=256, T=1, steps=80, chain="decode"),
        Workload("prefill_b4_t4096", seed=2000, B=4, T=4096),
        Workload("long_prefill_b1_t65536_4steps", seed=3000, B=1, T=65536, steps=4, chain="fresh"),
        Workload("stress_b2_t8192_80steps", seed=4000, B=2, T=8192, steps=80, chain="stress", iters=50,
                 x_dist="t3x4", delta_sd=4.0, scale_lo=5.0, scale_hi=10.0, base_sd=3.0),
        # the prefill batch at other stream counts and widths (the formulas hold for any hc and d)
        Workload("prefill_b4_t4096_hc8", seed=2100, B=4, T=4096, hc=8),
        Workload("prefill_b4_t4096_hc2", seed=2200, B=4, T=4096, hc=2),
        Workload("prefill_b4_t4096_d7168", seed=2300, B=4, T=4096, d=7168),
        Workload("prefill_b4_t4096_d2048", seed=2400, B=4, T=4096, d=2048),
    ]
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, step: int, tensor: int, block: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, step, tensor, block])))


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _draw_block(w: Workload, tensor: int, step: int, block: int, rows: int) -> np.ndarray:
    g = _rng(w.seed, step, tensor, block)
    hc, d = w.hc, w.d
    if tensor == T_X:
        if w.x_dist == "normal":
            v = g.standard_normal((rows, hc, d), dtype=np.float32)
        else:
            v = (4.0 * g.standard_t(3.0, size=(rows, hc, d))).astype(np.float32)
        return f32_to_bf16_bits(v)
    if tensor == T_DELTA:
        v = g.standard_normal((rows, d), dtype=np.float32)
        if w.delta_sd != 1.0:
            v *= np.float32(w.delta_sd)
        return f32_to_bf16_bits(v)
    if tensor == T_EMBED:
        return f32_to_bf16_bits(g.standard_normal((rows, d), dtype=np.float32))
    if tensor == T_POST:
        return (2.0 * _sigmoid(g.standard_normal((rows, hc)))).astype(np.float32)
    if tensor == T_COMB:
        z = g.standard_normal((rows, hc, hc))
        z = np.exp(z - z.max(axis=2, keepdims=True))
        return (z / z.sum(axis=2, keepdims=True)).astype(np.float32)
    if tensor == T_PREMIX:
        return (_sigmoid(g.standard_normal((rows, hc))) + 1e-6).astype(np.float32)
    raise ValueError("not a per-token tensor: %d" % tensor)


def tokens(w: Workload, tensor: int, step: int, lo: int = 0, hi: int | None = None) -> np.ndarray:
    """Rows [lo, hi) of a per-token input tensor of workload ``w`` at chain step ``step``."""
    hi = w.n if hi is None else hi
    if not (0 <= lo <= hi <= w.n):
        raise ValueError("token range out of bounds")
    parts = []
    b0, b1 = lo // BLOCK, (hi + BLOCK - 1) // BLOCK
    for b in range(b0, b1):
        rows = min(BLOCK, w.n - b * BLOCK)
        blk = _draw_block(w, tensor, step, b, rows)
        s = max(lo - b * BLOCK, 0)
        e = min(hi - b * BLOCK, rows)
        parts.append(blk[s:e])
    if not parts:
        return _draw_block(w, tensor, step, 0, 0)
    return np.ascontiguousarray(np.concatenate(parts, axis=0)) if len(parts) > 1 else np.ascontiguousarray(parts[0])


def token_rows(w: Workload, tensor: int, step: int, idx) -> np.ndarray:
    """The rows listed in ``idx`` (any order) of a per-token tensor."""
    idx = np.asarray(idx, dtype=np.int64)
    out = None
    for b in np.unique(idx // BLOCK):
        rows = min(BLOCK, w.n - int(b) * BLOCK)
        blk = _draw_block(w, tensor, step, int(b), rows)
        if out is None:
            out = np.empty((idx.size,) + blk.shape[1:], blk.dtype)
        sel = np.nonzero(idx // BLOCK == b)[0]
        out[sel] = blk[idx[sel] - int(b) * BLOCK]
    return out


def params(w: Workload, step: int) -> dict:
    """The HC parameter set of sublayer ``step`` (and the stand-in sublayer's diagonal)."""
    hc, d, M = w.hc, w.d, w.M
    hc_fn = (_rng(w.seed, step, T_FN).standard_normal((M, hc * d)) * w.fn_sd).astype(np.float32)
    hc_base = (_rng(w.seed, step, T_BASE).standard_normal(M) * w.base_sd).astype(np.float32)
    hc_scale = _rng(w.seed, step, T_SCALE).uniform(w.scale_lo, w.scale_hi, 3).astype(np.float32)
    nw = (1.0 + 0.1 * _rng(w.seed, step, T_NORMW).standard_normal(d)).astype(np.float32)
    norm_w = bf16_bits_to_f32(f32_to_bf16_bits(nw))
    w_diag = (_rng(w.seed, step, T_WDIAG).standard_normal(d) * 0.5).astype(np.float32)
    return dict(hc_fn=hc_fn, hc_base=hc_base, hc_scale=hc_scale, norm_w=norm_w, w_diag=w_diag)


def small(name: str, B: int, T: int, d: int, seed: int = 77, **kw) -> Workload:
    """A reduced-size workload with the distributions of ``name`` (for fast parity tests)."""
    base = WORKLOADS[name]
    return dataclasses.replace(base, name="%s_small_b%d_t%d_d%d" % (name, B, T, d), seed=seed, B=B, T=T, d=d, **kw)


def final_norm_w(w: Workload) -> np.ndarray:
    """The final RMSNorm's gain [d] (one per stack)."""
    nw = (1.0 + 0.1 * _rng(w.seed, 0, T_FINALW).standard_normal(w.d)).astype(np.float32)
    return bf16_bits_to_f32(f32_to_bf16_bits(nw))
