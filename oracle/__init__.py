"""Plain CPU oracle for the Hyper-Connection stream step (double precision, C++).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference arms are the only callers. The product path (the CUDA library and its Python
binding) never imports this package, and this package imports nothing from it.

The arithmetic lives in ``hc_oracle.cpp``; this module only compiles it with the host C++
compiler and marshals numpy arrays through ctypes. bf16 tensors travel as their raw 16-bit
patterns (``numpy.uint16``).

Sources, cited per function in ``hc_oracle.cpp`` (DeepSeek V4.1 model-atlas pages):
"Source layer, pairs pooled" (Block excerpts), "Reading weights" (hc_split_sinkhorn excerpt and the
formula for p), "Final RMSNorm" (RMSNorm excerpt and formula, Transformer.forward excerpt for the
ends of the stack), "Write the streams" (formula for X').
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hc_oracle.cpp")
_LIB = os.path.join(_HERE, "libhc_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle into a shared library with g++ (portable flags, x86 and Arm alike)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_D = ctypes.c_double


def _declare(lib):
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.oracle_double_to_bf16.argtypes = [_D]
    lib.oracle_bf16_to_double.restype = _D
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_round_bf16.argtypes = [_I64, _P, _P]
    lib.oracle_hc_post.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _I]
    lib.oracle_hc_mixes.argtypes = [_I64, _I, _I, _P, _P, _D, _P, _P, _P, _I]
    lib.oracle_split_sinkhorn.argtypes = [_I64, _I, _P, _P, _P, _I, _D, _P, _P, _P, _I]
    lib.oracle_hc_pre.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _I]
    lib.oracle_hc_post_detail.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _P, _P, _I]
    lib.oracle_rmsnorm.argtypes = [_I64, _I, _P, _P, _D, _P, _P, _I]
    lib.oracle_hc_pre_step.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _P, _I, _D, _D,
                                       _P, _P, _P, _P, _P, _P, _P, _P, _I]
    lib.oracle_hc_post_then_pre.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                            _I, _D, _D, _P, _P, _P, _P, _P, _I]
    lib.oracle_hc_expand.argtypes = [_I64, _I, _I, _P, _P, _I]
    lib.oracle_hc_expand_pre_step.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _I, _D, _D, _P, _P, _P, _P, _P, _I]
    lib.oracle_hc_final.argtypes = [_I64, _I, _I, _P, _P, _P, _D, _P, _P, _P, _I]
    lib.oracle_hc_post_then_final.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P, _P, _D, _P, _P, _I]
    lib.oracle_stream_mean.argtypes = [_I64, _I, _I, _P, _P, _P, _I]
    lib.oracle_hardware_threads.restype = _I
    lib.oracle_hardware_threads.argtypes = []


def load(path: str | None = None):
    """Load (building first if needed) the oracle library. A ``path`` loads another build of it."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            _declare(lib)
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads(lib=None) -> int:
    return int((lib or load()).oracle_hardware_threads())


def double_to_bf16(x, lib=None) -> np.ndarray:
    lib = lib or load()
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib.oracle_round_bf16(x.size, _p(x), _p(out))
    return out


def bf16_to_double(b) -> np.ndarray:
    """bf16 bit patterns to float64 (exact: a bf16 is the top half of a binary32)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def hc_post(X, delta, post, comb, threads=0, lib=None):
    """X' = bf16(post_k * delta + sum_j comb[j,k] X_j). X [n,hc,d] u16, delta [n,d] u16."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    delta, post, comb = _c(delta, np.uint16), _c(post, np.float32), _c(comb, np.float32)
    out = np.empty_like(X)
    lib.oracle_hc_post(n, hc, d, _p(X), _p(delta), _p(post), _p(comb), _p(out), threads)
    return out


def hc_mixes(X, hc_fn, norm_eps, threads=0, lib=None):
    """Returns (mixes [n,M], r [n], S [n,M]) in float64."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    M = (2 + hc) * hc
    hc_fn = _c(hc_fn, np.float32)
    mixes = np.empty((n, M), np.float64)
    r = np.empty((n,), np.float64)
    S = np.empty((n, M), np.float64)
    lib.oracle_hc_mixes(n, hc, d, _p(X), _p(hc_fn), float(norm_eps), _p(mixes), _p(r), _p(S), threads)
    return mixes, r, S


def split_sinkhorn(mixes, hc_scale, hc_base, hc, iters, eps, threads=0, lib=None):
    """Returns (pre [n,hc], post [n,hc], comb [n,hc,hc]) in float64."""
    lib = lib or load()
    mixes = _c(mixes, np.float64)
    n = mixes.shape[0]
    hc_scale, hc_base = _c(hc_scale, np.float32), _c(hc_base, np.float32)
    pre = np.empty((n, hc), np.float64)
    post = np.empty((n, hc), np.float64)
    comb = np.empty((n, hc, hc), np.float64)
    lib.oracle_split_sinkhorn(n, hc, _p(mixes), _p(hc_scale), _p(hc_base), int(iters), float(eps),
                              _p(pre), _p(post), _p(comb), threads)
    return pre, post, comb


def hc_post_detail(X, delta, post, comb, threads=0, lib=None):
    """hc_post plus, per element, the value before rounding and the sum of |terms| (float64)."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    delta, post, comb = _c(delta, np.uint16), _c(post, np.float32), _c(comb, np.float32)
    out = np.empty_like(X)
    exact = np.empty(X.shape, np.float64)
    mag = np.empty(X.shape, np.float64)
    lib.oracle_hc_post_detail(n, hc, d, _p(X), _p(delta), _p(post), _p(comb), _p(out), _p(exact), _p(mag), threads)
    return out, exact, mag


def hc_pre(X, pre_mix, threads=0, lib=None, with_abssum=False):
    """Returns (y bf16 bits [n,d], y before rounding float64 [n,d][, sum of |terms| [n,d]])."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    pre_mix = _c(pre_mix, np.float32)
    y = np.empty((n, d), np.uint16)
    ye = np.empty((n, d), np.float64)
    ya = np.empty((n, d), np.float64)
    lib.oracle_hc_pre(n, hc, d, _p(X), _p(pre_mix), _p(y), _p(ye), _p(ya), threads)
    return (y, ye, ya) if with_abssum else (y, ye)


def rmsnorm(x, w, eps, threads=0, lib=None):
    """Returns (out bf16 bits [n,d], out before rounding float64 [n,d])."""
    lib = lib or load()
    x = _c(x, np.uint16)
    n, d = x.shape
    w = _c(w, np.float32)
    out = np.empty((n, d), np.uint16)
    oe = np.empty((n, d), np.float64)
    lib.oracle_rmsnorm(n, d, _p(x), _p(w), float(eps), _p(out), _p(oe), threads)
    return out, oe


def hc_pre_step(X, pre_mix, hc_fn, hc_scale, hc_base, norm_w, iters, hc_eps, norm_eps, threads=0, lib=None):
    """One reading half. Returns a dict: y_normed, pre, post, comb, mixes, r, S, y."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    M = (2 + hc) * hc
    pre_mix, hc_fn = _c(pre_mix, np.float32), _c(hc_fn, np.float32)
    hc_scale, hc_base, norm_w = _c(hc_scale, np.float32), _c(hc_base, np.float32), _c(norm_w, np.float32)
    out = dict(
        y_normed=np.empty((n, d), np.uint16), pre=np.empty((n, hc)), post=np.empty((n, hc)),
        comb=np.empty((n, hc, hc)), mixes=np.empty((n, M)), r=np.empty((n,)), S=np.empty((n, M)),
        y=np.empty((n, d), np.uint16))
    lib.oracle_hc_pre_step(n, hc, d, _p(X), _p(pre_mix), _p(hc_fn), _p(hc_scale), _p(hc_base), _p(norm_w),
                           int(iters), float(hc_eps), float(norm_eps), _p(out["y_normed"]), _p(out["pre"]),
                           _p(out["post"]), _p(out["comb"]), _p(out["mixes"]), _p(out["r"]), _p(out["S"]),
                           _p(out["y"]), threads)
    return out


def hc_post_then_pre(delta, X, post, comb, pre_mix, hc_fn, hc_scale, hc_base, norm_w, iters, hc_eps, norm_eps,
                     threads=0, lib=None):
    """Writing half then the next reading half. Returns a dict: X_out, y_normed, pre, post, comb."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    delta, post, comb, pre_mix = (_c(delta, np.uint16), _c(post, np.float32), _c(comb, np.float32),
                                  _c(pre_mix, np.float32))
    hc_fn, hc_scale, hc_base, norm_w = (_c(hc_fn, np.float32), _c(hc_scale, np.float32),
                                        _c(hc_base, np.float32), _c(norm_w, np.float32))
    out = dict(X_out=np.empty_like(X), y_normed=np.empty((n, d), np.uint16), pre=np.empty((n, hc)),
               post=np.empty((n, hc)), comb=np.empty((n, hc, hc)))
    lib.oracle_hc_post_then_pre(n, hc, d, _p(delta), _p(X), _p(post), _p(comb), _p(pre_mix), _p(hc_fn),
                                _p(hc_scale), _p(hc_base), _p(norm_w), int(iters), float(hc_eps), float(norm_eps),
                                _p(out["X_out"]), _p(out["y_normed"]), _p(out["pre"]), _p(out["post"]),
                                _p(out["comb"]), threads)
    return out


def hc_expand(h, hc=4, threads=0, lib=None):
    """The embedding rows h [n,d] (u16) copied into hc streams: [n,hc,d]."""
    lib = lib or load()
    h = _c(h, np.uint16)
    n, d = h.shape
    out = np.empty((n, hc, d), np.uint16)
    lib.oracle_hc_expand(n, hc, d, _p(h), _p(out), threads)
    return out


def hc_expand_pre_step(h, hc_fn, hc_scale, hc_base, norm_w, iters, hc_eps, norm_eps, hc=4, threads=0, lib=None):
    """Head of the stack: expand, then the first reading half with the identity pre_mix. Returns a
    dict: X_out, y_normed, pre, post, comb."""
    lib = lib or load()
    h = _c(h, np.uint16)
    n, d = h.shape
    hc_fn, hc_scale, hc_base, norm_w = (_c(hc_fn, np.float32), _c(hc_scale, np.float32),
                                        _c(hc_base, np.float32), _c(norm_w, np.float32))
    out = dict(X_out=np.empty((n, hc, d), np.uint16), y_normed=np.empty((n, d), np.uint16), pre=np.empty((n, hc)),
               post=np.empty((n, hc)), comb=np.empty((n, hc, hc)))
    lib.oracle_hc_expand_pre_step(n, hc, d, _p(h), _p(hc_fn), _p(hc_scale), _p(hc_base), _p(norm_w), int(iters),
                                  float(hc_eps), float(norm_eps), _p(out["X_out"]), _p(out["y_normed"]),
                                  _p(out["pre"]), _p(out["post"]), _p(out["comb"]), threads)
    return out


def hc_final(X, pre_mix, norm_w, norm_eps, threads=0, lib=None):
    """Tail of the stack: collapse with pre_mix, then the final RMSNorm. Returns (z, y, z before
    rounding)."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    pre_mix, norm_w = _c(pre_mix, np.float32), _c(norm_w, np.float32)
    z = np.empty((n, d), np.uint16)
    y = np.empty((n, d), np.uint16)
    ze = np.empty((n, d), np.float64)
    lib.oracle_hc_final(n, hc, d, _p(X), _p(pre_mix), _p(norm_w), float(norm_eps), _p(z), _p(y), _p(ze), threads)
    return z, y, ze


def hc_post_then_final(delta, X, post, comb, pre_mix, norm_w, norm_eps, threads=0, lib=None):
    """The last writing half, then the tail of the stack. Returns a dict: X_out, z."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    delta, post, comb, pre_mix = (_c(delta, np.uint16), _c(post, np.float32), _c(comb, np.float32),
                                  _c(pre_mix, np.float32))
    norm_w = _c(norm_w, np.float32)
    out = dict(X_out=np.empty_like(X), z=np.empty((n, d), np.uint16))
    lib.oracle_hc_post_then_final(n, hc, d, _p(delta), _p(X), _p(post), _p(comb), _p(pre_mix), _p(norm_w),
                                  float(norm_eps), _p(out["X_out"]), _p(out["z"]), threads)
    return out


def stream_mean(X, threads=0, lib=None):
    """The mean over the hc streams of X [n,hc,d] (u16), rounded to bf16: (out [n,d] u16, exact)."""
    lib = lib or load()
    X = _c(X, np.uint16)
    n, hc, d = X.shape
    out = np.empty((n, d), np.uint16)
    ex = np.empty((n, d), np.float64)
    lib.oracle_stream_mean(n, hc, d, _p(X), _p(out), _p(ex), threads)
    return out, ex
