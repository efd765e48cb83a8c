"""GB300 (sm_103a) Hyper-Connection stream step: Python binding of the C-ABI library libhc.so.

Every function here has the name and the argument order of the C entry point it wraps
(``include/hc.h``); the binding only turns tensors into raw device pointers, picks the current
CUDA stream when none is given and raises :class:`HCError` on a nonzero status. All arithmetic
runs in the library's CUDA kernels. There is no fallback: if libhc.so is missing or cannot be
loaded, :func:`load` raises.

Device buffers are torch tensors (or integer device addresses); the caller allocates and owns
them, and must keep them alive until the stream has finished with them.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhc.so")

HC_OK = 0
HC_ERR_NULL = -1
HC_ERR_SHAPE = -2
HC_ERR_UNSUPPORTED = -3
HC_ERR_ALIGN = -4
HC_ERR_ALIAS = -5
HC_ERR_ARG = -6
HC_ERR_CUDA = -7
HC_ERR_DEVICE = -8

# every symbol include/hc.h declares
SYMBOLS = (
    "hc_prepare_params_size", "hc_prepare_params", "hc_workspace_size", "hc_pre_step", "hc_post_then_pre",
    "hc_post_then_pre_tap", "hc_post_then_pre_noalloc", "hc_post", "hc_expand_pre_step", "hc_final", "hc_post_then_final", "hc_debug_mixes",
    "hc_plan_tiles", "hc_fused_ctas", "hc_debug_wait_flag", "hc_device_error", "hc_status_string",
    "hc_host_pipeline_create", "hc_host_pipeline_chunk_tokens", "hc_host_pipeline_destroy", "hc_host_chunk_plan",
    "hc_host_post_then_pre",
)


class HCError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__("%s failed: %s (status %d)" % (fn, message, status))
        self.status = status


class hc_shape_t(ctypes.Structure):
    _fields_ = [("hc", ctypes.c_int), ("d", ctypes.c_int), ("sinkhorn_iters", ctypes.c_int),
                ("hc_eps", ctypes.c_float), ("norm_eps", ctypes.c_float)]


class hc_params_t(ctypes.Structure):
    _fields_ = [("hc_fn_planes", ctypes.c_void_p), ("hc_scale", ctypes.c_void_p), ("hc_base", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libhc.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libhc.so not found at %s: build it with hyper_connection_residual_hc_gb300.build.build()"
                           % path)
    lib = ctypes.CDLL(path)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.hc_prepare_params_size.argtypes = [I, I, ctypes.POINTER(ctypes.c_size_t)]
    lib.hc_prepare_params.argtypes = [P, I, I, P, P]
    lib.hc_workspace_size.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
    lib.hc_pre_step.argtypes = [P, P, hc_params_t, I64, hc_shape_t, P, P, P, P, P, P]
    lib.hc_post_then_pre.argtypes = [P, P, P, P, P, hc_params_t, I64, hc_shape_t, P, P, P, P, P, P, P]
    lib.hc_post_then_pre_tap.argtypes = [P, P, P, P, P, hc_params_t, I64, hc_shape_t, P, P, P, P, P, P, P, P]
    lib.hc_post_then_pre_noalloc.argtypes = [P, P, P, P, P, hc_params_t, I64, hc_shape_t, P, P, P, P, P, P]
    lib.hc_post.argtypes = [P, P, P, P, I64, hc_shape_t, P, P]
    lib.hc_expand_pre_step.argtypes = [P, hc_params_t, I64, hc_shape_t, P, P, P, P, P, P, P]
    lib.hc_final.argtypes = [P, P, P, I64, hc_shape_t, P, P]
    lib.hc_post_then_final.argtypes = [P, P, P, P, P, P, I64, hc_shape_t, P, P, P]
    lib.hc_debug_mixes.argtypes = [P, hc_params_t, I64, hc_shape_t, I, P, P, P]
    lib.hc_plan_tiles.argtypes = [I64, I, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I64)]
    lib.hc_fused_ctas.argtypes = [ctypes.POINTER(I)]
    lib.hc_debug_wait_flag.argtypes = [P, I, ctypes.c_uint64, I64, P]
    lib.hc_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), I, P]
    lib.hc_status_string.argtypes = [I]
    lib.hc_host_pipeline_create.argtypes = [I, I, I64, ctypes.POINTER(P)]
    lib.hc_host_pipeline_chunk_tokens.argtypes = [P, ctypes.POINTER(I64)]
    lib.hc_host_pipeline_destroy.argtypes = [P]
    PI64 = ctypes.POINTER(I64)
    lib.hc_host_chunk_plan.argtypes = [I64, I64, I64, PI64, PI64, PI64]
    lib.hc_host_post_then_pre.argtypes = [P, P, P, P, P, P, hc_params_t, I64, hc_shape_t, P, P, P, P, P, P]
    lib.hc_status_string.restype = ctypes.c_char_p
    for name in SYMBOLS:
        if name != "hc_status_string":
            getattr(lib, name).restype = I
    if path == LIB_PATH:
        _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn: str, status: int):
    if status != HC_OK:
        raise HCError(fn, status, load().hc_status_string(status).decode())


def shape(d: int = 5120, sinkhorn_iters: int = 20, hc_eps: float = 1e-6, norm_eps: float = 1e-6, hc: int = 4):
    return hc_shape_t(hc, d, sinkhorn_iters, hc_eps, norm_eps)


def params(hc_fn_planes, hc_scale, hc_base, norm_w) -> hc_params_t:
    """An hc_params_t of device pointers (the tensors must outlive its use)."""
    return hc_params_t(_ptr(hc_fn_planes), _ptr(hc_scale), _ptr(hc_base), _ptr(norm_w))


def hc_status_string(status: int) -> str:
    return load().hc_status_string(status).decode()


def hc_prepare_params_size(hc: int, d: int) -> int:
    out = ctypes.c_size_t(0)
    _check("hc_prepare_params_size", load().hc_prepare_params_size(hc, d, ctypes.byref(out)))
    return out.value


def hc_prepare_params(hc_fn, hc: int, d: int, planes, stream=None) -> None:
    _check("hc_prepare_params", load().hc_prepare_params(_ptr(hc_fn), hc, d, _ptr(planes), _stream(stream)))


def hc_workspace_size() -> int:
    out = ctypes.c_size_t(0)
    _check("hc_workspace_size", load().hc_workspace_size(ctypes.byref(out)))
    return out.value


def new_workspace(device=None):
    """A zero-filled device workspace for the fused calls (torch uint8 tensor)."""
    import torch
    return torch.zeros(hc_workspace_size(), dtype=torch.uint8, device=device or "cuda")


def hc_pre_step(X, pre_mix, p: hc_params_t, n: int, s: hc_shape_t, y_normed, pre, post, comb, workspace,
                stream=None) -> None:
    _check("hc_pre_step", load().hc_pre_step(_ptr(X), _ptr(pre_mix), p, n, s, _ptr(y_normed), _ptr(pre), _ptr(post),
                                             _ptr(comb), _ptr(workspace), _stream(stream)))


def hc_post_then_pre(delta, X, post, comb, pre_mix, nxt: hc_params_t, n: int, s: hc_shape_t, X_out, y_normed,
                     pre_out, post_out, comb_out, workspace, stream=None) -> None:
    _check("hc_post_then_pre", load().hc_post_then_pre(
        _ptr(delta), _ptr(X), _ptr(post), _ptr(comb), _ptr(pre_mix), nxt, n, s, _ptr(X_out), _ptr(y_normed),
        _ptr(pre_out), _ptr(post_out), _ptr(comb_out), _ptr(workspace), _stream(stream)))


def hc_post_then_pre_tap(delta, X, post, comb, pre_mix, nxt: hc_params_t, n: int, s: hc_shape_t, X_out, y_normed,
                         pre_out, post_out, comb_out, stream_mean, workspace, stream=None) -> None:
    """hc_post_then_pre that also writes bf16(mean over the 4 new streams) to stream_mean [n, d]."""
    _check("hc_post_then_pre_tap", load().hc_post_then_pre_tap(
        _ptr(delta), _ptr(X), _ptr(post), _ptr(comb), _ptr(pre_mix), nxt, n, s, _ptr(X_out), _ptr(y_normed),
        _ptr(pre_out), _ptr(post_out), _ptr(comb_out), _ptr(stream_mean), _ptr(workspace), _stream(stream)))


def hc_post_then_pre_noalloc(delta, X, post, comb, pre_mix, nxt: hc_params_t, n: int, s: hc_shape_t, X_out,
                             y_normed, pre_out, post_out, comb_out, stream=None) -> None:
    """hc_post_then_pre with the library's own fixed scratch instead of a caller workspace, for
    callers that may not allocate device memory (see include/hc.h)."""
    _check("hc_post_then_pre_noalloc", load().hc_post_then_pre_noalloc(
        _ptr(delta), _ptr(X), _ptr(post), _ptr(comb), _ptr(pre_mix), nxt, n, s, _ptr(X_out), _ptr(y_normed),
        _ptr(pre_out), _ptr(post_out), _ptr(comb_out), _stream(stream)))


def hc_post(delta, X, post, comb, n: int, s: hc_shape_t, X_out, stream=None) -> None:
    _check("hc_post", load().hc_post(_ptr(delta), _ptr(X), _ptr(post), _ptr(comb), n, s, _ptr(X_out),
                                     _stream(stream)))


def hc_expand_pre_step(h, p: hc_params_t, n: int, s: hc_shape_t, X_out, y_normed, pre, post, comb, workspace,
                       stream=None) -> None:
    _check("hc_expand_pre_step", load().hc_expand_pre_step(
        _ptr(h), p, n, s, _ptr(X_out), _ptr(y_normed), _ptr(pre), _ptr(post), _ptr(comb), _ptr(workspace),
        _stream(stream)))


def hc_final(X, pre_mix, norm_w, n: int, s: hc_shape_t, z, stream=None) -> None:
    _check("hc_final", load().hc_final(_ptr(X), _ptr(pre_mix), _ptr(norm_w), n, s, _ptr(z), _stream(stream)))


def hc_post_then_final(delta, X, post, comb, pre_mix, norm_w, n: int, s: hc_shape_t, X_out, z, stream=None) -> None:
    """X_out may be None: the streams after the last block are then not written."""
    _check("hc_post_then_final", load().hc_post_then_final(
        _ptr(delta), _ptr(X), _ptr(post), _ptr(comb), _ptr(pre_mix), _ptr(norm_w), n, s, _ptr(X_out), _ptr(z),
        _stream(stream)))


def hc_debug_mixes(X, p: hc_params_t, n: int, s: hc_shape_t, group: int, mixes, workspace, stream=None) -> None:
    _check("hc_debug_mixes", load().hc_debug_mixes(_ptr(X), p, n, s, group, _ptr(mixes), _ptr(workspace),
                                                   _stream(stream)))


def hc_plan_tiles(n: int, d: int, ctas: int):
    """(CTAs per tile, tokens per tile, tiles) of the fused calls."""
    g = ctypes.c_int(0)
    tm = ctypes.c_int(0)
    nt = ctypes.c_int64(0)
    _check("hc_plan_tiles", load().hc_plan_tiles(n, d, ctas, ctypes.byref(g), ctypes.byref(tm), ctypes.byref(nt)))
    return g.value, tm.value, nt.value


def hc_fused_ctas() -> int:
    c = ctypes.c_int(0)
    _check("hc_fused_ctas", load().hc_fused_ctas(ctypes.byref(c)))
    return c.value


def hc_debug_wait_flag(flags, count: int, value: int, limit_ns: int, stream=None) -> None:
    _check("hc_debug_wait_flag", load().hc_debug_wait_flag(_ptr(flags), count, value, limit_ns, _stream(stream)))


def hc_device_error(clear: bool = True, stream=None) -> int:
    w = ctypes.c_uint(0)
    _check("hc_device_error", load().hc_device_error(ctypes.byref(w), 1 if clear else 0, _stream(stream)))
    return w.value


class HostPipeline:
    """The host-buffer executor (hc_host_pipeline_t): device staging for three chunks of tokens, two
    copy streams and a workspace, owned until :meth:`close`. Its calls take host tensors (pinned ones
    let the copies overlap)."""

    def __init__(self, hc: int = 4, d: int = 5120, chunk_tokens: int = 0):
        h = ctypes.c_void_p()
        _check("hc_host_pipeline_create", load().hc_host_pipeline_create(hc, d, chunk_tokens, ctypes.byref(h)))
        self.handle = h.value

    @property
    def chunk_tokens(self) -> int:
        c = ctypes.c_int64(0)
        _check("hc_host_pipeline_chunk_tokens", load().hc_host_pipeline_chunk_tokens(self.handle, ctypes.byref(c)))
        return c.value

    def close(self) -> None:
        if self.handle:
            h, self.handle = self.handle, None
            _check("hc_host_pipeline_destroy", load().hc_host_pipeline_destroy(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def hc_host_pipeline_create(hc: int, d: int, chunk_tokens: int = 0) -> HostPipeline:
    return HostPipeline(hc, d, chunk_tokens)


def hc_host_pipeline_chunk_tokens(p: HostPipeline) -> int:
    return p.chunk_tokens


def hc_host_pipeline_destroy(p: HostPipeline) -> None:
    p.close()


def hc_host_chunk_plan(n: int, chunk_tokens: int = 0):
    """The chunks [(first token, tokens), ...] the executor cuts a call on n tokens into."""
    L = load()
    count, t0, m = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    _check("hc_host_chunk_plan", L.hc_host_chunk_plan(n, chunk_tokens, -1, ctypes.byref(count), None, None))
    out = []
    for i in range(count.value):
        _check("hc_host_chunk_plan", L.hc_host_chunk_plan(n, chunk_tokens, i, ctypes.byref(count), ctypes.byref(t0),
                                                          ctypes.byref(m)))
        out.append((t0.value, m.value))
    return out


def hc_host_post_then_pre(p, delta, X, post, comb, pre_mix, nxt: hc_params_t, n: int, s: hc_shape_t, X_out, y_normed,
                          pre_out, post_out, comb_out, stream=None) -> None:
    """hc_post_then_pre on HOST tensors through the executor `p` (a HostPipeline, a raw handle or None);
    the results are in the host tensors once `stream` has passed the call."""
    handle = p.handle if isinstance(p, HostPipeline) else p
    _check("hc_host_post_then_pre", load().hc_host_post_then_pre(
        handle, _ptr(delta), _ptr(X), _ptr(post), _ptr(comb), _ptr(pre_mix), nxt, n, s, _ptr(X_out), _ptr(y_normed),
        _ptr(pre_out), _ptr(post_out), _ptr(comb_out), _stream(stream)))
