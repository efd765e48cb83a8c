"""bench.py's host arithmetic, on CPU: the algorithmic bytes behind every roofline figure and the
launch counts it reports. Each count is the sum of the tensors an entry point reads and writes once
("Source layer, pairs pooled" page, Block.forward excerpt: the streams, Delta and the coefficients in,
the new streams, y and the next coefficients out)."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from hyper_connection_residual_hc_gb300 import synth  # noqa: E402


def test_step_bytes_at_the_model_shape():
    # X 4*5120 bf16 + Delta 5120 bf16 + post 4, comb 16, pre_mix 4 fp32 in; X', y and pre, post, comb out
    assert bench.step_bytes_per_token(4, 5120) == bench.BYTES_PER_TOKEN == 2 * (40960 + 10240 + 96)
    # hc_fn [24, 20480] fp32 + norm_w [5120] + hc_base [24] + hc_scale [3]
    assert bench.step_param_bytes(4, 5120) == bench.PARAM_BYTES == 24 * 20480 * 4 + 5120 * 4 + 24 * 4 + 12


def test_step_bytes_small_case_by_hand():
    # hc = 2, d = 8: X 2*8*2 = 32 B, Delta 16 B, post 8 + comb 16 + pre_mix 8 = 32 B, each way
    assert bench.step_bytes_per_token(2, 8) == 2 * (32 + 16 + 32)
    # M = 8 mixes: hc_fn [8, 16] fp32 = 512 B, norm_w 32 B, hc_base 32 B, hc_scale 12 B
    assert bench.step_param_bytes(2, 8) == 512 + 32 + 32 + 12


def test_every_step_op_counts_its_own_workload():
    for op, spec in bench.OPS.items():
        if spec.get("call", op) != "post_then_pre":
            continue
        w = synth.WORKLOADS[bench._workload_name(op)]
        assert spec["bytes_per_token"] == bench.step_bytes_per_token(w.hc, w.d), op
        assert spec["param_bytes"] == bench.step_param_bytes(w.hc, w.d), op


def test_other_entry_points_at_the_model_shape():
    x, row, coef = 4 * 5120 * 2, 5120 * 2, 4 * (4 + 4 + 16)
    expect = {
        "post_then_pre_tap": bench.BYTES_PER_TOKEN + row,        # + the stream mean
        "pre_step": x + 16 + row + coef,                         # X, pre_mix in; y, coefficients out
        "expand_pre_step": row + x + row + coef,                 # h in; X', y, coefficients out
        "post_then_final": x + row + 16 + 64 + 16 + row,         # X, Delta, post, comb, pre_mix in; z out
        "final": x + 16 + row,                                   # X, pre_mix in; z out
        "post": x + row + 16 + 64 + x,                           # X, Delta, post, comb in; X' out
    }
    for op, b in expect.items():
        assert bench.OPS[op]["bytes_per_token"] == b, op


def test_metric_names_the_shape_of_other_workloads():
    assert bench._metric("post_then_pre") == bench.METRIC
    assert bench._metric("post_then_pre_hc8").endswith("hc=8 d=5120")
    assert bench._metric("post_then_pre_d7168").endswith("hc=4 d=7168")
