"""Host-side checks of the C-ABI library that need no GPU: it builds for sm_103a, loads, exports
every entry point include/hc.h declares, validates arguments before touching the device, and
plans tiles sensibly. Pointers here are fake device addresses that are never dereferenced:
every call below returns from host-side validation (or is a no-op) before any CUDA call."""

import os
import re
import subprocess

import pytest

import hyper_connection_residual_hc_gb300 as hc
from hyper_connection_residual_hc_gb300 import build as hcbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    hcbuild.build()
    return hc.load()


def _declared_functions():
    with open(os.path.join(ROOT, "include", "hc.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(hc_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_symbols():
    assert _declared_functions() == sorted(hc.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", hc.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (hc_\w+)", out))
    missing = [s for s in _declared_functions() if s not in exported]
    assert not missing, missing
    for s in _declared_functions():
        assert hasattr(lib, s)


def test_status_strings(lib):
    for code in range(0, -9, -1):
        assert hc.hc_status_string(code)
    assert hc.hc_status_string(-100) == "unknown status"


def test_prepare_params_size(lib):
    assert hc.hc_prepare_params_size(4, 5120) == 3 * 24 * 20480 * 2
    with pytest.raises(hc.HCError) as e:
        hc.hc_prepare_params_size(4, 0)
    assert e.value.status == hc.HC_ERR_SHAPE


# fake, 256-byte aligned device addresses far apart (never dereferenced)
A = [0x7F0000000000 + i * (1 << 36) for i in range(16)]


def _p():
    return hc.params(A[10], A[11], A[12], A[13])


def _expect(status, fn, *args):
    with pytest.raises(hc.HCError) as e:
        fn(*args)
    assert e.value.status == status, (e.value.status, status)


def test_workspace_size(lib):
    # partial sums [256 CTAs][2 parities][28][128] fp32, an arrival counter per group slot on its own
    # 128-byte line [32][16] u64, a base per group slot [32] u64
    assert hc.hc_workspace_size() == 256 * 2 * 28 * 128 * 4 + 32 * 16 * 8 + 32 * 8 == 7344384


def test_pre_step_validation(lib):
    s = hc.shape()
    st = 0
    W = A[14]
    _expect(hc.HC_ERR_NULL, hc.hc_pre_step, None, A[1], _p(), 8, s, A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_NULL, hc.hc_pre_step, A[0], A[1], _p(), 8, s, A[2], A[3], A[4], A[5], None, st)
    _expect(hc.HC_ERR_NULL, hc.hc_pre_step, A[0], A[1], hc.params(None, A[11], A[12], A[13]), 8, s, A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_SHAPE, hc.hc_pre_step, A[0], A[1], _p(), -1, s, A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_SHAPE, hc.hc_pre_step, A[0], A[1], _p(), 8, hc.shape(d=5004), A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_SHAPE, hc.hc_pre_step, A[0], A[1], _p(), 8, hc.shape(hc=0), A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_UNSUPPORTED, hc.hc_pre_step, A[0], A[1], _p(), 8, hc.shape(hc=9), A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_UNSUPPORTED, hc.hc_pre_step, A[0], A[1], _p(), 8, hc.shape(d=65544), A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_ARG, hc.hc_pre_step, A[0], A[1], _p(), 8, hc.shape(sinkhorn_iters=0), A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_ARG, hc.hc_pre_step, A[0], A[1], _p(), 8, hc.shape(hc_eps=float("nan")), A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_ARG, hc.hc_pre_step, A[0], A[1], _p(), 8, hc.shape(norm_eps=-1.0), A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_ALIGN, hc.hc_pre_step, A[0] + 8, A[1], _p(), 8, s, A[2], A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_ALIGN, hc.hc_pre_step, A[0], A[1], _p(), 8, s, A[2], A[3], A[4], A[5], W + 8, st)
    _expect(hc.HC_ERR_ALIGN, hc.hc_pre_step, A[0], A[1], hc.params(A[10] + 4, A[11], A[12], A[13]), 8, s, A[2], A[3], A[4], A[5], W, st)
    # y_normed overlapping X, pre overlapping post, the workspace overlapping X
    _expect(hc.HC_ERR_ALIAS, hc.hc_pre_step, A[0], A[1], _p(), 8, s, A[0] + 1024, A[3], A[4], A[5], W, st)
    _expect(hc.HC_ERR_ALIAS, hc.hc_pre_step, A[0], A[1], _p(), 8, s, A[2], A[3], A[3] + 64, A[5], W, st)
    _expect(hc.HC_ERR_ALIAS, hc.hc_pre_step, A[0], A[1], _p(), 8, s, A[2], A[3], A[4], A[5], A[0] + 256, st)
    # n == 0 is a no-op
    hc.hc_pre_step(A[0], A[1], _p(), 0, s, A[2], A[3], A[4], A[5], W, st)


def test_post_then_pre_validation(lib):
    s = hc.shape()
    st = 0
    args = [A[0], A[1], A[2], A[3], A[4], _p(), 8, s, A[5], A[6], A[7], A[8], A[9], A[14], st]
    for i in (0, 1, 2, 3, 4, 8, 9, 10, 11, 12, 13):
        bad = list(args)
        bad[i] = None
        _expect(hc.HC_ERR_NULL, hc.hc_post_then_pre, *bad)
    bad = list(args)
    bad[8] = A[1] + 4096  # X_out inside X
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_pre, *bad)
    bad = list(args)
    bad[8] = A[1]  # exactly in place is not allowed for the fused call
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_pre, *bad)
    bad = list(args)
    bad[9] = A[0]  # y_normed on delta
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_pre, *bad)
    bad = list(args)
    bad[13] = A[5] + 64  # workspace inside X_out
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_pre, *bad)
    bad = list(args)
    bad[2] = A[2] + 12
    _expect(hc.HC_ERR_ALIGN, hc.hc_post_then_pre, *bad)
    bad = list(args)
    bad[6] = 1 << 31
    _expect(hc.HC_ERR_SHAPE, hc.hc_post_then_pre, *bad)
    bad = list(args)
    bad[6] = 0
    hc.hc_post_then_pre(*bad)


def test_post_then_pre_tap_validation(lib):
    s = hc.shape()
    st = 0
    args = [A[0], A[1], A[2], A[3], A[4], _p(), 8, s, A[5], A[6], A[7], A[8], A[9], A[15], A[14], st]
    bad = list(args)
    bad[13] = None  # the tap is this call's point
    _expect(hc.HC_ERR_NULL, hc.hc_post_then_pre_tap, *bad)
    bad = list(args)
    bad[13] = A[6] + 512  # stream_mean inside y_normed
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_pre_tap, *bad)
    bad = list(args)
    bad[13] = A[1]  # on X
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_pre_tap, *bad)
    bad = list(args)
    bad[13] = A[15] + 2
    _expect(hc.HC_ERR_ALIGN, hc.hc_post_then_pre_tap, *bad)
    bad = list(args)
    bad[6] = 0
    hc.hc_post_then_pre_tap(*bad)


def test_post_validation(lib):
    s = hc.shape(d=24)  # hc_post only needs d % 8 == 0
    _expect(hc.HC_ERR_SHAPE, hc.hc_post, A[0], A[1], A[2], A[3], 4, hc.shape(d=20), A[4], 0)
    _expect(hc.HC_ERR_ALIAS, hc.hc_post, A[0], A[1], A[2], A[3], 4, s, A[1] + 16, 0)
    _expect(hc.HC_ERR_ALIAS, hc.hc_post, A[0], A[1], A[2], A[3], 4, s, A[0], 0)
    hc.hc_post(A[0], A[1], A[2], A[3], 0, s, A[1], 0)  # exactly in place is allowed; n == 0 no-op


def test_expand_pre_step_validation(lib):
    s = hc.shape()
    st = 0
    args = [A[0], _p(), 8, s, A[1], A[2], A[3], A[4], A[5], A[14], st]
    for i in (0, 4, 5, 6, 7, 8, 9):
        bad = list(args)
        bad[i] = None
        _expect(hc.HC_ERR_NULL, hc.hc_expand_pre_step, *bad)
    bad = list(args)
    bad[1] = hc.params(A[10], None, A[12], A[13])
    _expect(hc.HC_ERR_NULL, hc.hc_expand_pre_step, *bad)
    bad = list(args)
    bad[4] = A[0] + 2048  # the streams written over the embedding
    _expect(hc.HC_ERR_ALIAS, hc.hc_expand_pre_step, *bad)
    bad = list(args)
    bad[5] = A[1] + 512  # y_normed inside the streams
    _expect(hc.HC_ERR_ALIAS, hc.hc_expand_pre_step, *bad)
    bad = list(args)
    bad[0] = A[0] + 2
    _expect(hc.HC_ERR_ALIGN, hc.hc_expand_pre_step, *bad)
    bad = list(args)
    bad[3] = hc.shape(d=260)
    _expect(hc.HC_ERR_SHAPE, hc.hc_expand_pre_step, *bad)
    bad = list(args)
    bad[3] = hc.shape(sinkhorn_iters=0)
    _expect(hc.HC_ERR_ARG, hc.hc_expand_pre_step, *bad)
    bad = list(args)
    bad[2] = 0
    hc.hc_expand_pre_step(*bad)


def test_final_validation(lib):
    s = hc.shape(norm_eps=1e-20)
    st = 0
    args = [A[0], A[1], A[2], 8, s, A[3], st]
    for i in (0, 1, 2, 5):
        bad = list(args)
        bad[i] = None
        _expect(hc.HC_ERR_NULL, hc.hc_final, *bad)
    _expect(hc.HC_ERR_SHAPE, hc.hc_final, A[0], A[1], A[2], 8, hc.shape(d=12), A[3], st)
    _expect(hc.HC_ERR_SHAPE, hc.hc_final, A[0], A[1], A[2], -1, s, A[3], st)
    _expect(hc.HC_ERR_UNSUPPORTED, hc.hc_final, A[0], A[1], A[2], 8, hc.shape(d=65544), A[3], st)
    _expect(hc.HC_ERR_UNSUPPORTED, hc.hc_final, A[0], A[1], A[2], 8, hc.shape(hc=9), A[3], st)
    _expect(hc.HC_ERR_ARG, hc.hc_final, A[0], A[1], A[2], 8, hc.shape(norm_eps=float("inf")), A[3], st)
    _expect(hc.HC_ERR_ALIGN, hc.hc_final, A[0], A[1], A[2] + 4, 8, s, A[3], st)
    _expect(hc.HC_ERR_ALIAS, hc.hc_final, A[0], A[1], A[2], 8, s, A[0] + 16, st)
    _expect(hc.HC_ERR_ALIAS, hc.hc_final, A[0], A[1], A[2], 8, s, A[2], st)
    # the Sinkhorn fields are not used here: an invalid iteration count is accepted
    hc.hc_final(A[0], A[1], A[2], 0, hc.shape(d=8, sinkhorn_iters=0, norm_eps=1e-20), A[3], st)


def test_post_then_final_validation(lib):
    s = hc.shape(norm_eps=1e-20)
    st = 0
    args = [A[0], A[1], A[2], A[3], A[4], A[5], 8, s, A[6], A[7], st]
    for i in (0, 1, 2, 3, 4, 5, 9):
        bad = list(args)
        bad[i] = None
        _expect(hc.HC_ERR_NULL, hc.hc_post_then_final, *bad)
    bad = list(args)
    bad[8] = A[1]  # X_out on X
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_final, *bad)
    bad = list(args)
    bad[9] = A[6] + 1024  # z inside X_out
    _expect(hc.HC_ERR_ALIAS, hc.hc_post_then_final, *bad)
    bad = list(args)
    bad[8] = A[6] + 8
    _expect(hc.HC_ERR_ALIGN, hc.hc_post_then_final, *bad)
    bad = list(args)
    bad[6] = 0
    bad[8] = None  # X_out is optional
    hc.hc_post_then_final(*bad)


def test_debug_wait_flag_validation(lib):
    _expect(hc.HC_ERR_NULL, hc.hc_debug_wait_flag, None, 8, 1, 1000, 0)
    _expect(hc.HC_ERR_SHAPE, hc.hc_debug_wait_flag, A[0], 0, 1, 1000, 0)
    _expect(hc.HC_ERR_SHAPE, hc.hc_debug_wait_flag, A[0], 33, 1, 1000, 0)
    _expect(hc.HC_ERR_ARG, hc.hc_debug_wait_flag, A[0], 8, 1, -1, 0)
    _expect(hc.HC_ERR_ARG, hc.hc_debug_wait_flag, A[0], 8, 1, 2_000_000_000, 0)
    _expect(hc.HC_ERR_ALIGN, hc.hc_debug_wait_flag, A[0] + 4, 8, 1, 1000, 0)


def test_plan_tiles(lib):
    for ctas in (8, 56, 128, 152, 256):
        for d in (256, 512, 1024, 5120):
            for n in [1, 2, 31, 32, 33, 64, 100, 127, 128, 129, 255, 256, 1000, 4096, 16384, 16385, 65536, 100003]:
                g, tm, nt = hc.hc_plan_tiles(n, d, ctas)
                assert g in (8, 16, 32) and d % (32 * g) == 0 and g <= ctas
                assert 1 <= tm <= 128
                assert nt * tm >= n and (nt - 1) * tm < n
                if nt > 1:
                    assert tm % 32 == 0 or 96 <= tm <= 128
    # the prefill batch over 19 groups of 8 (all 152 SMs of a GB300): 133 tiles of 124 tokens fill
    # exactly 7 waves, where 128 tiles of 128 would leave 5 groups idle in the last
    assert hc.hc_plan_tiles(16384, 5120, 152) == (8, 124, 133)
    # balanced heights only for several waves and only from 96 rows up
    assert hc.hc_plan_tiles(4096, 5120, 152) == (8, 108, 38)
    assert hc.hc_plan_tiles(2468, 1024, 152) == (8, 96, 26)
    assert hc.hc_plan_tiles(65536, 5120, 152) == (8, 128, 512)
    # a decode batch spreads each tile over more CTAs: fewer column stages per CTA
    g, tm, nt = hc.hc_plan_tiles(256, 5120, 152)
    assert g == 32 and g * nt <= 152
    g, tm, nt = hc.hc_plan_tiles(64, 5120, 152)
    assert g == 32 and g * nt <= 152
    # d = 256 only divides into groups of 8
    assert hc.hc_plan_tiles(64, 256, 152)[0] == 8
    assert hc.hc_plan_tiles(0, 5120, 152)[2] == 0
    _expect(hc.HC_ERR_SHAPE, hc.hc_plan_tiles, 16, 5000, 152)
    _expect(hc.HC_ERR_SHAPE, hc.hc_plan_tiles, 16, 5120, 4)


def test_host_pipeline_validation(lib):
    """The host-buffer executor's checks that come before any CUDA call (creating a real executor
    needs a GPU: tests/test_gpu_host_pipeline.py)."""
    import ctypes
    h = ctypes.c_void_p()
    assert lib.hc_host_pipeline_create(4, 5120, 0, None) == hc.HC_ERR_NULL
    for hcn, d, chunk, status in [(0, 5120, 0, hc.HC_ERR_SHAPE), (4, 0, 0, hc.HC_ERR_SHAPE),
                                  (4, 5004, 0, hc.HC_ERR_SHAPE), (4, 5120, -1, hc.HC_ERR_SHAPE),
                                  (4, 5120, (1 << 20) + 1, hc.HC_ERR_SHAPE), (9, 5120, 0, hc.HC_ERR_UNSUPPORTED),
                                  (4, 65544, 0, hc.HC_ERR_UNSUPPORTED)]:
        assert lib.hc_host_pipeline_create(hcn, d, chunk, ctypes.byref(h)) == status, (hcn, d, chunk)
        assert h.value is None
    assert lib.hc_host_pipeline_destroy(None) == hc.HC_OK
    c = ctypes.c_int64(0)
    assert lib.hc_host_pipeline_chunk_tokens(None, ctypes.byref(c)) == hc.HC_ERR_NULL
    # a NULL executor or host array is refused before anything is dereferenced
    s = hc.shape()
    args = [A[0], A[1], A[2], A[3], A[4], _p(), 8, s, A[5], A[6], A[7], A[8], A[9], 0]
    _expect(hc.HC_ERR_NULL, hc.hc_host_post_then_pre, None, *args)
    for i in (0, 1, 2, 3, 4, 8, 9, 10, 11, 12):
        bad = list(args)
        bad[i] = None
        _expect(hc.HC_ERR_NULL, hc.hc_host_post_then_pre, None, *bad)


@pytest.mark.parametrize("n,chunk", [(0, 0), (1, 0), (5, 1024), (31, 0), (300, 128), (1000, 384), (2500, 256),
                                     (5631, 2048), (5632, 2048), (16384, 0), (16384, 4096), (16384, 8192), (65536, 1024),
                                     (1000, 256), (1152, 256), (4480, 4096), (4479, 4096),
                                     (100, 1), (1 << 20, 1 << 20), (12345, 7)])
def test_host_chunk_plan(lib, n, chunk):
    """The executor's chunks tile [0, n) in order, none above the chunk size; large calls ramp
    up and down by halving sizes (C/2 down to the last one of at least max(128, C/32) tokens)
    around full chunks, small ones are cut evenly."""
    plan = hc.hc_host_chunk_plan(n, chunk)
    C = chunk or 1024
    pos = 0
    for t0, m in plan:
        assert t0 == pos and 1 <= m <= C
        pos += m
    assert pos == n
    ramp = [C >> j for j in range(1, 6) if (C >> j) >= max(128, C // 32)]
    sizes = [m for _, m in plan]
    if ramp and n >= 2 * sum(ramp) + C:
        r = len(ramp)
        assert sizes[:r] == ramp[::-1] and sizes[-r:] == ramp
        assert all(m == C for m in sizes[r:-r - 1]) and 1 <= sizes[-r - 1] <= C
    elif n:
        assert max(sizes) - min(sizes) <= 1
        assert len(plan) == max(-(-n // C), min(8, n // 32), 1)


def test_host_chunk_plan_validation(lib):
    import ctypes
    c = ctypes.c_int64(0)
    assert lib.hc_host_chunk_plan(10, 0, -1, None, None, None) == hc.HC_ERR_NULL
    assert lib.hc_host_chunk_plan(-1, 0, -1, ctypes.byref(c), None, None) == hc.HC_ERR_SHAPE
    assert lib.hc_host_chunk_plan(10, -1, -1, ctypes.byref(c), None, None) == hc.HC_ERR_SHAPE
    assert lib.hc_host_chunk_plan(10, (1 << 20) + 1, -1, ctypes.byref(c), None, None) == hc.HC_ERR_SHAPE
    assert lib.hc_host_chunk_plan(10, 0, 0, ctypes.byref(c), None, None) == hc.HC_ERR_NULL
    t, m = ctypes.c_int64(0), ctypes.c_int64(0)
    assert lib.hc_host_chunk_plan(10, 0, 1, ctypes.byref(c), ctypes.byref(t), ctypes.byref(m)) == hc.HC_ERR_ARG
    assert lib.hc_host_chunk_plan(0, 0, -1, ctypes.byref(c), None, None) == hc.HC_OK and c.value == 0


def test_debug_mixes_group_validation(lib):
    s = hc.shape()
    W = A[15]
    _expect(hc.HC_ERR_NULL, hc.hc_debug_mixes, None, _p(), 8, s, 0, A[1], W, 0)
    _expect(hc.HC_ERR_ARG, hc.hc_debug_mixes, A[0], _p(), 8, s, 4, A[1], W, 0)
    _expect(hc.HC_ERR_ARG, hc.hc_debug_mixes, A[0], _p(), 8, s, 64, A[1], W, 0)
    # d = 256 splits over 8 CTAs only (32 columns each)
    _expect(hc.HC_ERR_ARG, hc.hc_debug_mixes, A[0], _p(), 8, hc.shape(d=256), 16, A[1], W, 0)
    _expect(hc.HC_ERR_ALIGN, hc.hc_debug_mixes, A[0] + 4, _p(), 8, s, 32, A[1], W, 0)
    hc.hc_debug_mixes(A[0], _p(), 0, s, 32, A[1], W, 0)  # n == 0: no-op
