#!/usr/bin/env python3
"""Benchmark of the fused Hyper-Connection step (hc_post -> hc_mixes -> split/Sinkhorn -> hc_pre ->
RMSNorm) on GB300: one step = one hc_post_then_pre over the prefill batch B=4, T=4096 (16,384
tokens, hc=4, d=5120) of seeded synthetic inputs already resident in HBM.

Prints one JSON line. `value` is tokens/s over all ranks; `roofline` rates the fused kernel
against the measured HBM copy bandwidth; `e2e` repeats the step through the same C-ABI call with
the inputs copied from pinned host memory and the results copied back inside the timed region;
`cpu_baseline` times the CPU oracle (double precision) on this host's cores on a sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--op OP]
Under torchrun every rank runs its own batch (weak scaling, no data-path collective).
`--impl reference` times the CPU oracle itself as the reference arm.
`--op` times another entry point on the same batch, against its own algorithmic bytes:
post_then_pre (the default step), pre_step, expand_pre_step (head of the stack), post_then_final
and final (tail of the stack, eps 1e-20), post (writing half alone), decode_chain (80 sublayers on 256
tokens captured in one CUDA graph); or the step on the other single-step workloads: step_b1_t64 (one
hc_post_then_pre on 64 tokens, each launch timed alone with L2 flushed before it: latency) and
long_prefill_b1_t65536 (one hc_post_then_pre on 65,536 tokens).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HC step tokens/s and achieved HBM GB/s vs peak, prefill B=4 T=4096"
WORKLOAD = "prefill_b4_t4096"
SPEC_HBM_GBS = 8000.0         # GB300 HBM3e, nominal
BYTES_PER_TOKEN = 102592      # read X 40960 + delta 10240 + post 16 + comb 64 + pre_mix 16;
                              # write X' 40960 + y_normed 10240 + pre/post/comb 96
PARAM_BYTES = 1986668         # hc_fn fp32 1966080 + norm_w 20480 + hc_base 96 + hc_scale 12
FINAL_EPS = 1e-20             # the final RMSNorm's eps ("Final RMSNorm" page)


def step_bytes_per_token(hc: int, d: int) -> int:
    """hc_post_then_pre's bytes per token for hc streams of width d: read X, Delta, post, comb and
    pre_mix; write X', y_normed and pre, post, comb (BYTES_PER_TOKEN at hc = 4, d = 5120)."""
    coefs = 4 * (2 * hc + hc * hc)  # post, comb, pre_mix in; pre, post, comb out: the same count
    return 2 * (hc * d * 2 + d * 2 + coefs)


def step_param_bytes(hc: int, d: int) -> int:
    """Bytes of one parameter set: hc_fn fp32 [(2 + hc) hc, hc d], norm_w, hc_base, hc_scale
    (PARAM_BYTES at hc = 4, d = 5120)."""
    M = (2 + hc) * hc
    return M * hc * d * 4 + d * 4 + M * 4 + 3 * 4
CSRC = "hyper_connection_residual_hc_gb300/csrc/"
FUSED_SOURCES = [CSRC + "hc_fused.cu", CSRC + "hc_ptx.cuh"]
FINAL_SOURCES = [CSRC + "hc_final.cu"]
GENERIC_SOURCES = [CSRC + "hc_generic.cu", CSRC + "hc_proj.cu"]
GENERIC_KERNELS = "gen_post_kernel, gen_proj_tc_kernel, gen_tail_kernel"

# Per op: algorithmic bytes per token and per call (parameters), the kernel it launches, the sources
# that kernel is built from, and the ncu summary of that kernel on this workload; `call` is the entry
# point (default: the op's own name), `workload` the synthetic workload (default: the prefill batch),
# `flush_l2` times each launch alone after writing a buffer larger than L2.
OPS = {
    "post_then_pre": dict(bytes_per_token=BYTES_PER_TOKEN, param_bytes=PARAM_BYTES, kernel="hc_fused_kernel<1>",
                          sources=FUSED_SOURCES, traffic="hc_fused_prefill_b4_t4096_traffic.json"),
    # the step plus the mean of the 4 new streams: + 10240 written
    "post_then_pre_tap": dict(bytes_per_token=BYTES_PER_TOKEN + 10240, param_bytes=PARAM_BYTES,
                              kernel="hc_fused_kernel<1>", sources=FUSED_SOURCES,
                              traffic="hc_fused_tap_prefill_b4_t4096_traffic.json"),
    # read X 40960 + pre_mix 16; write y_normed 10240 + pre/post/comb 96
    "pre_step": dict(bytes_per_token=51312, param_bytes=PARAM_BYTES, kernel="hc_fused_kernel<0>",
                     sources=FUSED_SOURCES, traffic="hc_fused_pre_step_prefill_b4_t4096_traffic.json"),
    # read h 10240; write X' 40960 + y_normed 10240 + pre/post/comb 96
    "expand_pre_step": dict(bytes_per_token=61536, param_bytes=PARAM_BYTES, kernel="hc_fused_kernel<2>",
                            sources=FUSED_SOURCES, traffic="hc_fused_expand_prefill_b4_t4096_traffic.json"),
    # read X 40960 + delta 10240 + post 16 + comb 64 + pre_mix 16; write z 10240 (X' not written)
    "post_then_final": dict(bytes_per_token=61536, param_bytes=20480, kernel="hc_final_kernel<true,false>",
                            sources=FINAL_SOURCES, traffic="hc_final_post_then_final_prefill_b4_t4096_traffic.json"),
    # read X 40960 + pre_mix 16; write z 10240
    "final": dict(bytes_per_token=51216, param_bytes=20480, kernel="hc_final_kernel<false,false>",
                  sources=FINAL_SOURCES, traffic="hc_final_final_prefill_b4_t4096_traffic.json"),
    # read X 40960 + delta 10240 + post 16 + comb 64; write X' 40960
    "post": dict(bytes_per_token=92240, param_bytes=0, kernel="hc_post_kernel", sources=[CSRC + "hc_api.cu"],
                 traffic="hc_post_prefill_b4_t4096_traffic.json"),
    # the step on the single-step workload of 64 tokens: a latency (each launch alone, L2 flushed)
    "step_b1_t64": dict(bytes_per_token=BYTES_PER_TOKEN, param_bytes=PARAM_BYTES, kernel="hc_fused_kernel<1>",
                        sources=FUSED_SOURCES, traffic=None, call="post_then_pre", workload="step_b1_t64",
                        flush_l2=True),
    # the step on the long-prefill workload's 65,536 tokens (its first step)
    "long_prefill_b1_t65536": dict(bytes_per_token=BYTES_PER_TOKEN, param_bytes=PARAM_BYTES,
                                   kernel="hc_fused_kernel<1>", sources=FUSED_SOURCES, traffic=None,
                                   call="post_then_pre", workload="long_prefill_b1_t65536_4steps"),
    # the step on the prefill batch at other shapes: 8 or 2 streams, or d = 7168, on the generic kernels
    # (the writing half, then per chunk of tokens the tensor-core projection and the split + norm);
    # d = 2048 on the fused kernel
    "post_then_pre_hc8": dict(bytes_per_token=step_bytes_per_token(8, 5120), param_bytes=step_param_bytes(8, 5120),
                              kernel=GENERIC_KERNELS, sources=GENERIC_SOURCES, traffic=None, call="post_then_pre",
                              workload="prefill_b4_t4096_hc8"),
    "post_then_pre_hc2": dict(bytes_per_token=step_bytes_per_token(2, 5120), param_bytes=step_param_bytes(2, 5120),
                              kernel=GENERIC_KERNELS, sources=GENERIC_SOURCES, traffic=None, call="post_then_pre",
                              workload="prefill_b4_t4096_hc2"),
    "post_then_pre_d7168": dict(bytes_per_token=step_bytes_per_token(4, 7168),
                                param_bytes=step_param_bytes(4, 7168), kernel=GENERIC_KERNELS,
                                sources=GENERIC_SOURCES, traffic=None, call="post_then_pre",
                                workload="prefill_b4_t4096_d7168"),
    "post_then_pre_d2048": dict(bytes_per_token=step_bytes_per_token(4, 2048),
                                param_bytes=step_param_bytes(4, 2048), kernel="hc_fused_kernel<1>",
                                sources=FUSED_SOURCES, traffic=None, call="post_then_pre",
                                workload="prefill_b4_t4096_d2048"),
}


def _call(op):
    return OPS[op].get("call", op)


def _workload_name(op):
    return OPS[op].get("workload", WORKLOAD)


def workload_config(w, op):
    """The `config` of a bench line: the workload and the call, nothing measured, so that both arms
    print the same dict."""
    spec = OPS[op]
    alg = w.n * spec["bytes_per_token"] + spec["param_bytes"]
    l2 = ("flushed before every launch (a 256 MB write); each launch timed alone" if spec.get("flush_l2") else
          "no flush: every step moves %d MB, far above the 129 MB L2" % (alg // 10 ** 6))
    return {"workload": w.name, "entry_point": "hc_" + _call(op), "tokens_per_gpu": w.n, "B": w.B, "T": w.T,
            "hc": w.hc, "d": w.d, "sinkhorn_iters": w.iters, "hc_eps": w.hc_eps, "norm_eps": w.norm_eps,
            "stream_dtype": "bf16", "coefficient_dtype": "f32", "l2": l2}


def _metric(op):
    if op == "post_then_pre":
        return METRIC
    if op == "step_b1_t64":
        return "HC step latency and tokens/s, single step B=1 T=64"
    if op == "long_prefill_b1_t65536":
        return "HC step tokens/s and achieved HBM GB/s vs peak, long prefill B=1 T=65536"
    if _workload_name(op) != WORKLOAD:  # the prefill batch at another shape
        from hyper_connection_residual_hc_gb300 import synth
        w = synth.WORKLOADS[_workload_name(op)]
        return "HC step tokens/s and achieved HBM GB/s vs peak, prefill B=4 T=4096, hc=%d d=%d" % (w.hc, w.d)
    return "HC %s tokens/s and achieved HBM GB/s vs peak, prefill B=4 T=4096" % op


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_workload(w0, rank: int):
    """This rank's batch: the workload's shapes and distributions with a seed of its own. Tokens are
    independent, so each rank steps its own batch and no data crosses ranks (weak scaling)."""
    import dataclasses
    return dataclasses.replace(w0, seed=w0.seed + 17 * rank) if rank else w0


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's value of a timing (x itself when there is one process). The only
    collective of a run: the step has no data-path exchange."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units all ranks processed per second of the slowest rank."""
    return units_per_rank * world / seconds


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _source_hash(sources=FUSED_SOURCES):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profile(op="post_then_pre"):
    """The committed ncu summary of the op's kernel on its workload (DRAM bytes of one launch, and pipe
    utilisations where captured); None when absent or taken on another version of the kernel."""
    spec = OPS[op]
    if not spec.get("traffic"):
        return None
    try:
        with open(os.path.join(ROOT, "profiles", spec["traffic"])) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("source_sha256_16") != _source_hash(spec["sources"]):
        return None
    return t


def _traffic_per_launch(n_tokens, op="post_then_pre"):
    """DRAM bytes per launch of the op's kernel from the committed ncu summary, scaled to this
    launch's token count; None when absent or taken on another version of the kernel."""
    t = _profile(op)
    if t is None:
        return None
    return float(t["dram_bytes_per_launch"]) * n_tokens / float(t["tokens"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _oracle_call(w, tokens, threads, op="post_then_pre"):
    """A no-argument call of the oracle's version of the op on the first `tokens` tokens of the
    workload, its inputs drawn beforehand."""
    import oracle as orc
    from hyper_connection_residual_hc_gb300 import synth
    from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_EMBED, T_POST, T_PREMIX, T_X
    prm = synth.params(w, 0)

    def tk(t):
        return synth.tokens(w, t, 0, 0, tokens)

    coef = (prm["hc_fn"], prm["hc_scale"], prm["hc_base"], prm["norm_w"], w.iters, w.hc_eps, w.norm_eps)
    op = _call(op) if op in OPS else op
    if op in ("post_then_pre", "post_then_pre_tap"):
        args = (tk(T_DELTA), tk(T_X), tk(T_POST), tk(T_COMB), tk(T_PREMIX))
        if op == "post_then_pre":
            fn = lambda: orc.hc_post_then_pre(*args, *coef, threads=threads)  # noqa: E731
        else:
            def fn():
                out = orc.hc_post_then_pre(*args, *coef, threads=threads)
                orc.stream_mean(out["X_out"], threads=threads)
    elif op == "pre_step":
        args = (tk(T_X), tk(T_PREMIX))
        fn = lambda: orc.hc_pre_step(*args, *coef, threads=threads)  # noqa: E731
    elif op == "expand_pre_step":
        h = tk(T_EMBED)
        fn = lambda: orc.hc_expand_pre_step(h, *coef, threads=threads)  # noqa: E731
    elif op == "post_then_final":
        args = (tk(T_DELTA), tk(T_X), tk(T_POST), tk(T_COMB), tk(T_PREMIX), synth.final_norm_w(w))
        fn = lambda: orc.hc_post_then_final(*args, FINAL_EPS, threads=threads)  # noqa: E731
    elif op == "final":
        args = (tk(T_X), tk(T_PREMIX), synth.final_norm_w(w))
        fn = lambda: orc.hc_final(*args, FINAL_EPS, threads=threads)  # noqa: E731
    else:
        args = (tk(T_X), tk(T_DELTA), tk(T_POST), tk(T_COMB))
        fn = lambda: orc.hc_post(*args, threads=threads)  # noqa: E731
    return fn


def _oracle_sample_rate(w, tokens, threads, op="post_then_pre"):
    """The oracle's version of the op on the first `tokens` tokens: tokens/s (input drawing untimed)."""
    fn = _oracle_call(w, tokens, threads, op)
    t0 = time.perf_counter()
    fn()
    return tokens / (time.perf_counter() - t0)


def run_reference(args):
    """Reference arm: the CPU oracle as it stands, on this host's cores, a bounded sample per step."""
    rank, world, _ = _dist()
    if rank != 0:
        return
    import oracle as orc
    from hyper_connection_residual_hc_gb300 import synth
    op, unit, metric = args.op, "tokens/s", _metric(args.op)
    if args.op == "decode_chain":  # the chain's sublayer steps, one hc_post_then_pre per sublayer
        wname, op, unit = DECODE, "post_then_pre", "sublayer-tokens/s"
        metric = DECODE_METRIC
        config = decode_config(synth.WORKLOADS[DECODE])
    else:
        wname = _workload_name(op)
        config = workload_config(synth.WORKLOADS[wname], op)
    w = synth.WORKLOADS[wname]
    threads = orc.hardware_threads()
    # size each step so that warmup + steps take about two minutes at most
    rate = _oracle_sample_rate(w, min(w.n, 4 * threads), threads, op)
    per_step = min(w.n, max(threads, int(rate * 120.0 / max(1, args.steps + args.warmup))))
    fn = _oracle_call(w, per_step, threads, op)  # the same sample every step, drawn once
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    sample = "first %d of the %d tokens of %s per step (hc_%s, float64 oracle)" % (per_step, w.n, wname,
                                                                                    _call(op) if op in OPS else op)
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch

    import hyper_connection_residual_hc_gb300 as hc
    from hyper_connection_residual_hc_gb300 import synth
    from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_EMBED, T_POST, T_PREMIX, T_X

    op = args.op
    spec = OPS[op]
    call = _call(op)
    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hc.load()

    w = rank_workload(synth.WORKLOADS[_workload_name(op)], rank)
    n, d, hcn = w.n, w.d, w.hc
    prm = synth.params(w, 0)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))

    # per-token inputs of the op (copied host -> device every step of the e2e run)
    names = {"post_then_pre": ("delta", "X", "post", "comb", "pre_mix"), "pre_step": ("X", "pre_mix"),
             "post_then_pre_tap": ("delta", "X", "post", "comb", "pre_mix"),
             "expand_pre_step": ("h",), "post_then_final": ("delta", "X", "post", "comb", "pre_mix"),
             "final": ("X", "pre_mix"), "post": ("delta", "X", "post", "comb")}[call]
    draw = dict(delta=lambda: bf(synth.tokens(w, T_DELTA, 0)), X=lambda: bf(synth.tokens(w, T_X, 0)),
                post=lambda: f32(synth.tokens(w, T_POST, 0)), comb=lambda: f32(synth.tokens(w, T_COMB, 0)),
                pre_mix=lambda: f32(synth.tokens(w, T_PREMIX, 0)), h=lambda: bf(synth.tokens(w, T_EMBED, 0)))
    host = {k: draw[k]() for k in names}
    dev = {k: v.cuda() for k, v in host.items()}
    hc_fn = f32(prm["hc_fn"]).cuda()
    planes = torch.empty(hc.hc_prepare_params_size(hcn, d) // 2, dtype=torch.bfloat16, device="cuda")
    hc.hc_prepare_params(hc_fn, hcn, d, planes)
    scale, base, nw = f32(prm["hc_scale"]).cuda(), f32(prm["hc_base"]).cuda(), f32(prm["norm_w"]).cuda()
    P = hc.params(planes, scale, base, nw)
    s = hc.shape(d=d, sinkhorn_iters=w.iters, hc_eps=w.hc_eps, norm_eps=w.norm_eps, hc=hcn)
    sf = hc.shape(d=d, norm_eps=FINAL_EPS, hc=hcn)
    fw = f32(synth.final_norm_w(w)).cuda()

    def empty(*shape, dt=torch.bfloat16):
        return torch.empty(shape, dtype=dt, device="cuda")

    coef = lambda: dict(pre=empty(n, hcn, dt=torch.float32), post=empty(n, hcn, dt=torch.float32),  # noqa: E731
                        comb=empty(n, hcn, hcn, dt=torch.float32))
    if call in ("post_then_pre", "expand_pre_step"):
        out = dict(X_out=empty(n, hcn, d), y_normed=empty(n, d), **coef())
    elif call == "post_then_pre_tap":
        out = dict(X_out=empty(n, hcn, d), y_normed=empty(n, d), stream_mean=empty(n, d), **coef())
    elif call == "pre_step":
        out = dict(y_normed=empty(n, d), **coef())
    elif call in ("post_then_final", "final"):
        out = dict(z=empty(n, d))
    else:
        out = dict(X_out=empty(n, hcn, d))
    stream = torch.cuda.current_stream()
    ws = hc.new_workspace()

    def step():
        if call == "post_then_pre":
            hc.hc_post_then_pre(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, n, s,
                                out["X_out"], out["y_normed"], out["pre"], out["post"], out["comb"], ws, stream)
        elif call == "post_then_pre_tap":
            hc.hc_post_then_pre_tap(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], P, n, s,
                                    out["X_out"], out["y_normed"], out["pre"], out["post"], out["comb"],
                                    out["stream_mean"], ws, stream)
        elif call == "pre_step":
            hc.hc_pre_step(dev["X"], dev["pre_mix"], P, n, s, out["y_normed"], out["pre"], out["post"], out["comb"],
                           ws, stream)
        elif call == "expand_pre_step":
            hc.hc_expand_pre_step(dev["h"], P, n, s, out["X_out"], out["y_normed"], out["pre"], out["post"],
                                  out["comb"], ws, stream)
        elif call == "post_then_final":
            hc.hc_post_then_final(dev["delta"], dev["X"], dev["post"], dev["comb"], dev["pre_mix"], fw, n, sf, None,
                                  out["z"], stream)
        elif call == "final":
            hc.hc_final(dev["X"], dev["pre_mix"], fw, n, sf, out["z"], stream)
        else:
            hc.hc_post(dev["delta"], dev["X"], dev["post"], dev["comb"], n, s, out["X_out"], stream)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
    barrier()
    werr = hc.hc_device_error(clear=True)

    # timed region: one call per step (one fused launch; the CUDA-core path's launches for other
    # shapes), CUDA events on the launching stream around each call; with flush_l2, a 256 MB write
    # before every call (outside its events), and the steps' time is the sum of the calls' own times
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if spec.get("flush_l2") else None
    clocks = ClockSampler(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    per_launch = sorted(a.elapsed_time(b) for a, b in ev)
    kern_ms = sum(per_launch) / args.steps
    el_ms = sum(per_launch) if flush is not None else t_start.elapsed_time(t_end)
    el_ms = max_over_ranks(el_ms, dist, "cuda")
    derr = hc.hc_device_error(clear=True)

    # end to end through the C ABI: pinned host inputs in, results out, every step
    pin_in = {k: v.pin_memory() for k, v in host.items()}
    pin_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in out.items()}
    e2e_steps = max(3, min(50, args.steps))
    h2d = sum(v.numel() * v.element_size() for v in pin_in.values())
    d2h = sum(v.numel() * v.element_size() for v in pin_out.values())

    pipe = None
    if call == "post_then_pre":
        # the library's host-buffer executor: chunks of tokens copied in, stepped and copied out on
        # overlapping streams, all behind one C-ABI call on host arrays
        pipe = hc.HostPipeline(hcn, d, args.e2e_chunk)
        e2e_path = "hc_host_post_then_pre, chunks of %d tokens" % pipe.chunk_tokens
    else:
        e2e_path = "copies in, hc_%s, copies out, one after another" % op

    def e2e_step():
        if pipe is not None:
            hc.hc_host_post_then_pre(pipe, pin_in["delta"], pin_in["X"], pin_in["post"], pin_in["comb"],
                                     pin_in["pre_mix"], P, n, s, pin_out["X_out"], pin_out["y_normed"], pin_out["pre"],
                                     pin_out["post"], pin_out["comb"], stream)
        else:
            for k in dev:
                dev[k].copy_(pin_in[k], non_blocking=True)
            step()
            for k in out:
                pin_out[k].copy_(out[k], non_blocking=True)
        stream.synchronize()

    for _ in range(10):  # the host link's first transfers of a run are slower
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    barrier()
    e2e_s = time.perf_counter() - t0
    if pipe is not None:
        pipe.close()
    e2e_s = max_over_ranks(e2e_s, dist, "cuda")

    value = whole_job_rate(n * args.steps, world, el_ms / 1e3)
    peak, peak_kind = _peaks()
    alg_bytes = n * spec["bytes_per_token"] + spec["param_bytes"]
    achieved = alg_bytes / (kern_ms / 1e3) / 1e9
    med_ms = statistics.median(per_launch)
    ctas = hc.hc_fused_ctas()
    if spec["kernel"] == GENERIC_KERNELS:
        # the writing half in one launch, then per chunk of tokens (as many as the workspace holds raw
        # mixes and sums of squares for) a projection launch and a split + norm launch
        chunk = hc.hc_workspace_size() // (((2 + hcn) * hcn + 1) * 4)
        launches = 1 + 2 * -(-n // chunk)
        plan = {"path": "generic kernels (projection on tcgen05)", "chunk_tokens": chunk,
                "launches_per_step": launches}
    else:
        group, tile_m, tiles = hc.hc_plan_tiles(n, d, ctas)
        launches = 1
        plan = {"tile_tokens": tile_m, "tiles": tiles, "ctas_per_tile": group, "resident_ctas": ctas}
    prof = _profile(op)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as orc
        threads = orc.hardware_threads()
        r0 = _oracle_sample_rate(w, min(n, 2 * threads), threads, op)
        sample_tokens = int(max(threads, min(n, r0 * 15.0)))  # about 15 s of wall time at most
        rate = _oracle_sample_rate(w, sample_tokens, threads, op)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": "hc_%s on the first %d of the %d tokens of %s, float64 oracle, %d threads"
                         % (call, sample_tokens, n, w.name, threads)}

    if rank == 0:
        line = {
            "metric": _metric(op), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": el_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, op),
            "plan": plan,
            "latency_us": {"median": 1e3 * med_ms, "best": 1e3 * per_launch[0], "mean": 1e3 * kern_ms,
                           "launches": args.steps},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "frac_spec": achieved / SPEC_HBM_GBS, "spec_peak": SPEC_HBM_GBS,
                         "achieved_median": alg_bytes / (med_ms / 1e3) / 1e9,
                         "achieved_best": alg_bytes / (per_launch[0] / 1e3) / 1e9,
                         "region_gb_per_s": alg_bytes * args.steps / (el_ms / 1e3) / 1e9,
                         "traffic": _traffic_per_launch(n, op), "algorithmic_bytes": alg_bytes,
                         "pipes": prof.get("pipes") if prof else None,
                         "kernel": spec["kernel"], "kernel_ms": kern_ms},
            "cpu_baseline": cpu,
            "e2e": {"value": whole_job_rate(n * e2e_steps, world, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "path": e2e_path},
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "gpu_launches": launches * args.steps,
            "device_error": werr | derr,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


DECODE = "decode_chain_b256_80steps"
DECODE_METRIC = "HC decode chain sublayer-tokens/s (80 sublayers x 256 tokens, one CUDA graph)"


def decode_config(w):
    """The decode chain's `config`, the same in both arms."""
    return {"workload": w.name, "entry_point": "graph of hc_expand_pre_step, 79 x hc_post_then_pre, "
            "hc_post_then_final", "tokens_per_gpu": w.n, "sublayers": w.steps, "hc": w.hc, "d": w.d,
            "sinkhorn_iters": w.iters, "hc_eps": w.hc_eps, "norm_eps": w.norm_eps, "final_norm_eps": FINAL_EPS,
            "l2": "no flush: the 80 parameter sets (236 MB of weight planes) exceed the 129 MB L2, the 10 MB of "
                  "streams stay resident between sublayers as in a real decode step"}


def run_decode_chain(args):
    """The decode chain: 80 sublayers on 256 tokens, the whole stack as one CUDA graph of the
    library's calls (hc_expand_pre_step, 79 x hc_post_then_pre, hc_post_then_final). The sublayers'
    outputs Delta are drawn beforehand (the sublayer itself is not part of the path), so the graph
    holds only the library's 81 launches. Timed by CUDA events around graph replays."""
    import numpy as np
    import torch

    import hyper_connection_residual_hc_gb300 as hc
    from hyper_connection_residual_hc_gb300 import synth
    from hyper_connection_residual_hc_gb300.synth import T_DELTA, T_EMBED

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hc.load()
    w = rank_workload(synth.WORKLOADS[DECODE], rank)
    n, d, L = w.n, w.d, w.steps

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))

    params = []
    for l in range(L):
        prm = synth.params(w, l)
        planes = torch.empty(hc.hc_prepare_params_size(4, d) // 2, dtype=torch.bfloat16, device="cuda")
        fn = f32(prm["hc_fn"]).cuda()
        hc.hc_prepare_params(fn, 4, d, planes)
        keep = (planes, f32(prm["hc_scale"]).cuda(), f32(prm["hc_base"]).cuda(), f32(prm["norm_w"]).cuda())
        params.append((hc.params(*keep), keep))
    fw = f32(synth.final_norm_w(w)).cuda()
    h_host = bf(synth.tokens(w, T_EMBED, 0)).pin_memory()
    h = h_host.cuda()
    delta = torch.stack([bf(synth.tokens(w, T_DELTA, l)) for l in range(L)]).cuda()
    s = hc.shape(d=d, sinkhorn_iters=w.iters, hc_eps=w.hc_eps, norm_eps=w.norm_eps)
    sf = hc.shape(d=d, norm_eps=FINAL_EPS)
    X = [torch.empty((n, 4, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    y = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    coef = [dict(pre=torch.empty((n, 4), device="cuda"), post=torch.empty((n, 4), device="cuda"),
                 comb=torch.empty((n, 4, 4), device="cuda")) for _ in range(2)]
    z = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    ws = hc.new_workspace()

    def chain():
        c = coef[0]
        hc.hc_expand_pre_step(h, params[0][0], n, s, X[0], y, c["pre"], c["post"], c["comb"], ws)
        for l in range(1, L):
            a, b = coef[(l - 1) % 2], coef[l % 2]
            hc.hc_post_then_pre(delta[l - 1], X[(l - 1) % 2], a["post"], a["comb"], a["pre"], params[l][0], n, s,
                                X[l % 2], y, b["pre"], b["post"], b["comb"], ws)
        last = coef[(L - 1) % 2]
        hc.hc_post_then_final(delta[L - 1], X[(L - 1) % 2], last["post"], last["comb"], last["pre"], fw, n, sf, None,
                              z)

    for _ in range(max(3, args.warmup)):
        chain()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        chain()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    werr = hc.hc_device_error(clear=True)
    stream = torch.cuda.current_stream()
    steps = max(1, args.steps)
    clocks = ClockSampler(local)
    clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    t0.record(stream)
    marks[0].record(stream)
    for i in range(steps):
        graph.replay()
        marks[i + 1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    chain_samples = [marks[i].elapsed_time(marks[i + 1]) for i in range(steps)]
    el_ms = max_over_ranks(t0.elapsed_time(t1), dist, "cuda")
    derr = hc.hc_device_error(clear=True)

    # end to end: the embedding in from pinned host memory and z out, every chain
    z_host = torch.empty(z.shape, dtype=z.dtype, pin_memory=True)
    e2e_steps = max(3, min(50, steps))
    torch.cuda.synchronize()
    w0t = time.perf_counter()
    for _ in range(e2e_steps):
        h.copy_(h_host, non_blocking=True)
        graph.replay()
        z_host.copy_(z, non_blocking=True)
        stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - w0t, dist, "cuda")

    chain_ms = el_ms / steps
    sub_tokens = n * L * world
    # algorithmic bytes of one chain: head (h in; streams, y_normed, coefficients out), 79 middle
    # steps, tail (streams, Delta, coefficients in; z out); each sublayer's parameters once
    alg = (n * 61536 + PARAM_BYTES) + (L - 1) * (n * BYTES_PER_TOKEN + PARAM_BYTES) + (n * 61536 + 20480)
    peak, peak_kind = _peaks()
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as orc
        threads = orc.hardware_threads()
        k = 32  # tokens of the sample, every sublayer
        prm0 = synth.params(w, 0)
        sub = lambda t: synth.tokens(w, t, 0, 0, k)  # noqa: E731
        from hyper_connection_residual_hc_gb300.synth import T_COMB, T_POST, T_PREMIX, T_X
        args_ = (sub(T_DELTA), sub(T_X), sub(T_POST), sub(T_COMB), sub(T_PREMIX))
        ts = time.perf_counter()
        for _ in range(8):
            orc.hc_post_then_pre(*args_, prm0["hc_fn"], prm0["hc_scale"], prm0["hc_base"], prm0["norm_w"], w.iters,
                                 w.hc_eps, w.norm_eps, threads=threads)
        rate = 8 * k / (time.perf_counter() - ts)
        cpu = {"value": rate, "unit": "sublayer-tokens/s", "cores": threads, "kind": "oracle",
               "sample": "8 sublayer steps (hc_post_then_pre) on %d of the %d tokens, float64 oracle" % (k, n)}
    if rank == 0:
        line = {
            "metric": DECODE_METRIC,
            "value": sub_tokens / (chain_ms / 1e3), "unit": "sublayer-tokens/s", "n_gpus": world, "steps": steps,
            "warmup": max(3, args.warmup), "ms_per_step": chain_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": decode_config(w),
            "plan": dict(zip(("ctas_per_tile", "tile_tokens", "tiles"), hc.hc_plan_tiles(n, d, hc.hc_fused_ctas()))),
            "latency_us": {"per_sublayer": chain_ms * 1e3 / L, "per_chain": chain_ms * 1e3,
                           "per_sublayer_median": 1e3 * statistics.median(chain_samples) / L,
                           "per_sublayer_best": 1e3 * min(chain_samples) / L, "chains": len(chain_samples)},
            "roofline": {"bound": "latency (launch chain)", "achieved": alg / (chain_ms / 1e3) / 1e9, "peak": peak,
                         "unit": "GB/s", "frac": alg / (chain_ms / 1e3) / 1e9 / peak, "peak_kind": peak_kind,
                         "frac_spec": alg / (chain_ms / 1e3) / 1e9 / SPEC_HBM_GBS, "spec_peak": SPEC_HBM_GBS,
                         "traffic": None, "algorithmic_bytes": alg},
            "cpu_baseline": cpu,
            "e2e": {"value": sub_tokens * e2e_steps / e2e_s, "unit": "sublayer-tokens/s",
                    "h2d_bytes_per_step": h.numel() * 2, "d2h_bytes_per_step": z.numel() * 2},
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "gpu_launches": (L + 1) * steps,
            "device_error": werr | derr,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunk", type=int, default=0,
                    help="tokens per chunk of the host-buffer executor in the end-to-end run (0: the library's default)")
    ap.add_argument("--op", default="post_then_pre", choices=sorted(OPS) + ["decode_chain"])
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "decode_chain":
        run_decode_chain(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
