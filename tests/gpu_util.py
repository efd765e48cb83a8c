"""Helpers for the GPU parity tests: device buffers, calls through the C ABI, comparisons with
the oracle and the tolerances they use.

Tolerances (stated once, used everywhere):
  bf16 outputs (X', y_normed): 1 bf16 ulp after fp32 accumulation. The model evaluates hc_post and
    hc_pre on float32 tensors and then casts; an fp32 evaluation of a k-term sum is off from the exact
    value by at most k u A (A = sum of |terms|, u = 2^-24). So X' must lie within 1 bf16 ulp of an
    fp32 evaluation: |gpu - exact| <= ulp_bf16(exact) + 6 u A. Away from cancellation this is the
    plain "at most 1 ulp from the oracle's rounded value"; only where the terms nearly cancel does the
    fp32 bound (several ulps of the tiny result) take over. y_normed likewise, with y's admissible
    bf16 values pushed through the norm. Both checks also report the plain ulp histogram and require
    99.9% of the values within 1 ulp of the oracle's rounding.
  mixes: |gpu - oracle| <= max(1e-5 |m|, 1e-6) + 2 u S, with u = 2^-24 and S = r sum_c |x_c w_mc|:
    a 20,480-term dot product accumulated in fp32 is off by a few u S whatever the order.
  pre/post/comb given the GPU's own mixes (stage isolated): rel 1e-5 or abs 1e-6, flat, for every
    Sinkhorn round count. The model runs hc_split_sinkhorn in fp32; an IEEE fp32 evaluation of the
    page's steps meets this even at the stress workload's 50 rounds on extreme logits, with less
    margin than at 20 (tests/test_split_fp32.py).
  pre/post/comb end to end: the flat tolerance plus the mixes bound pushed through the split: pre and
    post through the sigmoid's slope, comb through the oracle split's sensitivities (central
    differences). The elements beyond the flat tolerance are counted and reported (COEF_STATS).
"""

from __future__ import annotations

import collections

import numpy as np
import torch

import hyper_connection_residual_hc_gb300 as hc
import oracle as orc

U = 2.0 ** -24


def dev_bf16(a_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().astype(np.float64)


class DevParams:
    """One sublayer's parameters on the device, with hc_fn split by hc_prepare_params."""

    def __init__(self, prm: dict, d: int, hcn: int = 4):
        self.hc_fn = dev_f32(prm["hc_fn"])
        self.hc_scale = dev_f32(prm["hc_scale"])
        self.hc_base = dev_f32(prm["hc_base"])
        self.norm_w = dev_f32(prm["norm_w"])
        nbytes = hc.hc_prepare_params_size(hcn, d)
        self.planes = torch.empty(nbytes // 2, dtype=torch.bfloat16, device="cuda")
        hc.hc_prepare_params(self.hc_fn, hcn, d, self.planes)
        self.c = hc.params(self.planes, self.hc_scale, self.hc_base, self.norm_w)


_WS = None


def workspace():
    """One zero-filled workspace shared by the (sequential) test calls."""
    global _WS
    if _WS is None:
        _WS = hc.new_workspace()
    return _WS


# ---- guard bands around outputs ------------------------------------------------------------------
# An output allocated through `guarded` sits between two 4 KB bands of 0xA5 bytes. A kernel that writes
# past either end of the output (a ragged last tile, a wrong row count in a tensor map, an index one
# row too far) lands in a band, which no parity check of the output itself would see. `check_guards`
# verifies the bands of every output allocated since the last check; conftest runs it after every
# test, and `guarded` runs it once the held outputs reach 8 GB, so that long chains stay bounded.
GUARD_BYTES = 4096
GUARD_VALUE = 0xA5
_GUARD_CHECK_BYTES = 8 << 30
_guarded = []        # (buffer, output bytes) of the outputs allocated since the last check
_guarded_bytes = 0


def guarded(shape, dtype=torch.bfloat16, device="cuda") -> torch.Tensor:
    """An uninitialised tensor of `shape` and `dtype` with a guard band on each side (its address stays
    16-byte aligned: the band is 4 KB and the allocator's blocks are aligned further)."""
    global _guarded_bytes
    count = 1
    for e in shape:
        count *= int(e)
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    if _guarded_bytes + nbytes > _GUARD_CHECK_BYTES:
        check_guards()
    buf = torch.empty(2 * GUARD_BYTES + nbytes, dtype=torch.uint8, device=device)
    buf[:GUARD_BYTES].fill_(GUARD_VALUE)
    buf[GUARD_BYTES + nbytes:].fill_(GUARD_VALUE)
    _guarded.append((buf, nbytes))
    _guarded_bytes += nbytes
    return buf[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(tuple(shape))


def check_guards():
    """Raise if any guard band of an output allocated since the last check was written; forget them."""
    global _guarded, _guarded_bytes
    held, _guarded, _guarded_bytes = _guarded, [], 0
    if not held:
        return
    if any(b.is_cuda for b, _ in held):
        torch.cuda.synchronize()
    for buf, nbytes in held:
        for side, band in (("before", buf[:GUARD_BYTES]), ("after", buf[GUARD_BYTES + nbytes:])):
            bad = (band != GUARD_VALUE).nonzero()
            if bad.numel():
                raise AssertionError("%d bytes of the guard band %s an output of %d bytes were written (first at "
                                     "band byte %d)" % (bad.numel(), side, nbytes, int(bad[0])))


def alloc_outputs(n: int, d: int, post_mode: bool, hcn: int = 4):
    o = dict(y_normed=guarded((n, d), torch.bfloat16),
             pre=guarded((n, hcn), torch.float32),
             post=guarded((n, hcn), torch.float32),
             comb=guarded((n, hcn, hcn), torch.float32))
    if post_mode:
        o["X_out"] = guarded((n, hcn, d), torch.bfloat16)
    return o


def run_pre_step(X, pre_mix, P: DevParams, s, n):
    o = alloc_outputs(n, s.d, False, s.hc)
    hc.hc_pre_step(X, pre_mix, P.c, n, s, o["y_normed"], o["pre"], o["post"], o["comb"], workspace())
    return o


def run_post_then_pre(delta, X, post, comb, pre_mix, P: DevParams, s, n):
    o = alloc_outputs(n, s.d, True, s.hc)
    hc.hc_post_then_pre(delta, X, post, comb, pre_mix, P.c, n, s, o["X_out"], o["y_normed"], o["pre"], o["post"],
                        o["comb"], workspace())
    return o


def debug_mixes(X, P: DevParams, s, n, group=0):
    """The GPU's own mixes of n tokens; `group` as the call being checked used (plan_group)."""
    m = guarded((n, (2 + s.hc) * s.hc), torch.float32)
    hc.hc_debug_mixes(X, P.c, n, s, group, m, workspace())
    return m


def plan_group(n, s):
    """The group size (CTAs per token tile) of a fused call on n tokens of shape s; 0 for the
    generic path. A token's mixes depend on it, not on its tile's other tokens."""
    if s.hc != 4 or s.d % 256 or s.d > 5120 or n == 0:
        return 0
    return hc.hc_plan_tiles(n, s.d, hc.hc_fused_ctas())[0]


def device_error_clear():
    w = hc.hc_device_error(clear=True)
    assert w == 0, "a kernel gave up a bounded wait (word 0x%x)" % w


# ---- comparisons --------------------------------------------------------------------------------

def bf16_key(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_diff(a_u16: np.ndarray, b_u16: np.ndarray) -> np.ndarray:
    return np.abs(bf16_key(a_u16) - bf16_key(b_u16))


def assert_bf16_close(gpu_u16, ref_u16, what, max_ulp=1):
    gpu_u16 = np.asarray(gpu_u16)
    ref_u16 = np.asarray(ref_u16)
    nan_g = (gpu_u16 & 0x7F80) == 0x7F80
    nan_r = (ref_u16 & 0x7F80) == 0x7F80
    assert np.array_equal(nan_g, nan_r), "%s: non-finite values differ" % what
    dd = ulp_diff(gpu_u16[~nan_g], ref_u16[~nan_r])
    worst = int(dd.max()) if dd.size else 0
    assert worst <= max_ulp, "%s: %d values beyond %d ulp (worst %d ulp)" % (what, int((dd > max_ulp).sum()), max_ulp, worst)
    return float((dd == 0).mean()) if dd.size else 1.0


def bf16_spacing(v):
    """Distance between consecutive bf16 values around |v| (float64 array)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return np.where(a < 2.0 ** -126, 2.0 ** -133, 2.0 ** (e - 7))


def check_xprime(gpu_u16, X, delta, post, comb, what="X_out"):
    """hc_post output against the oracle: within 1 bf16 ulp of an fp32 evaluation."""
    ref, exact, mag = orc.hc_post_detail(X, delta, post, comb)
    g = orc.bf16_to_double(gpu_u16)
    tol = bf16_spacing(exact) + (np.asarray(X).shape[1] + 2) * U * mag
    bad = np.abs(g - exact) > tol
    assert not bad.any(), "%s: %d values beyond 1 ulp + fp32 bound" % (what, int(bad.sum()))
    dd = ulp_diff(np.asarray(gpu_u16), ref)
    assert (dd <= 1).mean() >= 0.999, "%s: only %.5f within 1 ulp" % (what, float((dd <= 1).mean()))
    return float((dd == 0).mean()), int(dd.max())


def check_y_normed(gpu_u16, Xp, pre_mix, norm_w, norm_eps, what="y_normed"):
    """y_normed against the oracle fed the same X': y may be any bf16 value an fp32 evaluation of
    sum_j pre_mix_j X'_j can round to; the norm of each must be within 1 bf16 ulp."""
    y_ref, y_exact, y_abs = orc.hc_pre(Xp, pre_mix, with_abssum=True)
    yn_ref, _ = orc.rmsnorm(y_ref, norm_w, norm_eps)
    yr = orc.bf16_to_double(y_ref)
    r = 1.0 / np.sqrt((yr ** 2).mean(axis=1, keepdims=True) + norm_eps)
    Ey = (np.asarray(Xp).shape[1] + 1) * U * y_abs
    y_lo = orc.bf16_to_double(orc.double_to_bf16(y_exact - Ey))
    y_hi = orc.bf16_to_double(orc.double_to_bf16(y_exact + Ey))
    w = np.asarray(norm_w, dtype=np.float64)[None, :]
    a, b = w * y_lo * r, w * y_hi * r
    lo, hi = np.minimum(a, b), np.maximum(a, b)
    lo = lo - bf16_spacing(lo) - 4 * U * np.abs(lo)
    hi = hi + bf16_spacing(hi) + 4 * U * np.abs(hi)
    g = orc.bf16_to_double(gpu_u16)
    bad = (g < lo) | (g > hi)
    assert not bad.any(), "%s: %d values outside the admissible range" % (what, int(bad.sum()))
    dd = ulp_diff(np.asarray(gpu_u16), yn_ref)
    assert (dd <= 1).mean() >= 0.999, "%s: only %.5f within 1 ulp" % (what, float((dd <= 1).mean()))
    return float((dd == 0).mean()), int(dd.max())


def mixes_tol(m_ref, S):
    return np.maximum(1e-5 * np.abs(m_ref), 1e-6) + 2 * U * S


def assert_mixes_close(m_gpu, m_ref, S, what="mixes"):
    err = np.abs(m_gpu - m_ref)
    tol = mixes_tol(m_ref, S)
    bad = err > tol
    assert not bad.any(), "%s: %d beyond tolerance, worst err/tol %.3g" % (what, int(bad.sum()), float((err / tol).max()))
    return float((err / (U * S)).max())


def sinkhorn_fp32_bound(comb_ref, hcn, iters):
    """First-order error of an fp32 evaluation of the split's Sinkhorn iteration: 2 iters normalisations
    of (hc + 2) u each ((hc - 1) additions, + eps, the division). Not a tolerance of the GPU checks; the
    fp32 evidence test (test_split_fp32) shows an IEEE evaluation stays inside it."""
    return 2 * iters * (hcn + 2) * U * np.abs(comb_ref)


# per check kind (e.g. "comb (isolated)"): [elements, beyond the flat tolerance, worst err / flat]
COEF_STATS = collections.defaultdict(lambda: [0, 0, 0.0])


def coef_stats_report(reset=True):
    """One line per check kind: how many coefficients needed more than the flat rel 1e-5 / abs 1e-6."""
    lines = ["%-26s %9d elements, %6d beyond flat (%.2e), worst err/flat %.3f"
             % (k, v[0], v[1], v[1] / max(v[0], 1), v[2]) for k, v in sorted(COEF_STATS.items())]
    if reset:
        COEF_STATS.clear()
    return "\n".join(lines)


def assert_coef_close(gpu, ref, what, extra=None, kind=None):
    """|gpu - ref| <= max(1e-5 |ref|, 1e-6) + extra; the elements beyond the flat part are counted
    under `kind` in COEF_STATS."""
    flat = np.maximum(1e-5 * np.abs(ref), 1e-6)
    err = np.abs(gpu - ref)
    tol = flat if extra is None else flat + extra
    bad = err > tol
    assert not bad.any(), "%s: %d beyond tolerance, worst err %.3g (tol %.3g)" % (
        what, int(bad.sum()), float(err[bad].max()), float(tol[bad][np.argmax(err[bad])]))
    if kind is not None:
        st = COEF_STATS[kind]
        st[0] += err.size
        st[1] += int((err > flat).sum())
        st[2] = max(st[2], float((err / flat).max()) if err.size else 0.0)


def hc_of(M):
    """The number of streams whose mix count (2 + hc) hc is M."""
    return next(h for h in range(1, 9) if (2 + h) * h == M)


def split_sensitivity_bound(m_ref, S, hc_scale, hc_base, iters, eps):
    """Bound on |d(pre, post, comb)| from mixes errors up to E = 2 u S + 1e-5|m| + 1e-6, pushed through
    the oracle split: analytic for pre/post, central differences for comb."""
    n, M = m_ref.shape
    h_ = hc_of(M)
    E = 2 * U * S + 1e-5 * np.abs(m_ref) + 1e-6
    pre0, post0, comb0 = orc.split_sinkhorn(m_ref, hc_scale, hc_base, h_, iters, eps)
    s0, s1 = float(hc_scale[0]), float(hc_scale[1])
    sg = pre0 - eps
    b_pre = abs(s0) * sg * (1 - sg) * E[:, 0:h_]
    sp = post0 / 2
    b_post = 2 * abs(s1) * sp * (1 - sp) * E[:, h_:2 * h_]
    b_comb = np.zeros((n, h_, h_))
    for k in range(2 * h_, M):
        h = np.maximum(E[:, k], 1e-9)
        mp = m_ref.copy()
        mm = m_ref.copy()
        mp[:, k] += h
        mm[:, k] -= h
        _, _, cp = orc.split_sinkhorn(mp, hc_scale, hc_base, h_, iters, eps)
        _, _, cm = orc.split_sinkhorn(mm, hc_scale, hc_base, h_, iters, eps)
        b_comb += np.abs(cp - cm) / 2
    return b_pre, b_post, b_comb


def check_step(out, ref, m_gpu, m_ref, S, prm, iters, eps, label):
    """Compare one reading half (pre_step outputs) with the oracle's, both ways:
    stage-isolated (oracle split on the GPU's mixes) and end to end."""
    pre_g, post_g, comb_g = host_f32(out["pre"]), host_f32(out["post"]), host_f32(out["comb"])
    assert_mixes_close(m_gpu, m_ref, S, label + " mixes")
    h_ = hc_of(m_gpu.shape[1])
    pre_i, post_i, comb_i = orc.split_sinkhorn(m_gpu, prm["hc_scale"], prm["hc_base"], h_, iters, eps)
    assert_coef_close(pre_g, pre_i, label + " pre (isolated)", kind="pre (isolated)")
    assert_coef_close(post_g, post_i, label + " post (isolated)", kind="post (isolated)")
    assert_coef_close(comb_g, comb_i, label + " comb (isolated)", kind="comb (isolated)")
    bp, bq, bc = split_sensitivity_bound(m_ref, S, prm["hc_scale"], prm["hc_base"], iters, eps)
    assert_coef_close(pre_g, ref["pre"], label + " pre", bp, kind="pre (end to end)")
    assert_coef_close(post_g, ref["post"], label + " post", bq, kind="post (end to end)")
    assert_coef_close(comb_g, ref["comb"], label + " comb", bc, kind="comb (end to end)")


# ---- sampled checks of a full-size step -----------------------------------------------------------

def shape_of(w):
    return hc.shape(d=w.d, sinkhorn_iters=w.iters, hc_eps=w.hc_eps, norm_eps=w.norm_eps, hc=w.hc)


def sample_tokens(n, k, rng, tile=128):
    """First and last tokens, tile edges, and k random tokens of n (sorted, unique)."""
    idx = set(range(min(n, 8))) | set(range(max(0, n - 8), n))
    for b in range(0, n, tile * 16):
        idx.update([b, min(n - 1, b + tile - 1), min(n - 1, b + tile)])
    idx.update(rng.choice(n, size=min(k, n), replace=False).tolist())
    return np.array(sorted(idx), dtype=np.int64)


def check_sampled(w, step, dev_in, out, prm, idx, post_mode, label, groups=None):
    """Oracle on the sampled tokens of one step, fed that step's device inputs (teacher-forced).
    The stage-isolated check feeds the oracle split the GPU's own mixes of those tokens, taken with
    the group size of the call that produced `out` (that of a call on w.n tokens, or `groups[i]`
    per sampled token), so that they are the very mixes that call used."""
    X = host_u16(dev_in["X"][idx])
    pm = host_f32(dev_in["pre_mix"][idx]).astype(np.float32)
    if post_mode:
        delta = host_u16(dev_in["delta"][idx])
        post = host_f32(dev_in["post"][idx]).astype(np.float32)
        comb = host_f32(dev_in["comb"][idx]).astype(np.float32)
        xo = host_u16(out["X_out"][idx])
        check_xprime(xo, X, delta, post, comb, label + " X_out")
        X = xo
    ref = orc.hc_pre_step(X, pm, prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"], w.iters, w.hc_eps,
                          w.norm_eps)
    check_y_normed(host_u16(out["y_normed"][idx]), X, pm, prm["norm_w"], w.norm_eps, label + " y_normed")
    sub = {k: out[k][idx] for k in ("pre", "post", "comb")}
    P = DevParams(prm, w.d, w.hc)
    shp = shape_of(w)
    gs = np.full(len(idx), plan_group(w.n, shp)) if groups is None else np.asarray(groups)
    m_gpu = np.empty((len(idx), w.M))
    for g in np.unique(gs):
        sel = np.nonzero(gs == g)[0]
        m_gpu[sel] = host_f32(debug_mixes(dev_bf16(X[sel]), P, shp, len(sel), int(g)))
    check_step(sub, ref, m_gpu, ref["mixes"], ref["S"], prm, w.iters, w.hc_eps, label)
