"""bench.py's multi-process path, on CPU: two processes joined by a gloo process group over
127.0.0.1, as torchrun joins one process per GPU.

The step shards by tokens with no exchange (weak scaling): each rank draws its own batch of the
workload and steps it alone; the only collective is the MAX over ranks of a timing. Checked here:
the ranks' batches differ but have the workload's shapes; a rank's results (the oracle on its own
batch) equal the rows of one call on the two batches together, so nothing had to cross ranks;
max_over_ranks returns the slowest rank's value on every rank; the whole-job rate counts the
units of all ranks over that time; and the reference arm does its work on rank 0 only.
"""

import multiprocessing
import os
import socket
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(WORLD))
        sys.path.insert(0, ROOT)
        import torch.distributed as dist

        import bench
        import oracle as orc
        from hyper_connection_residual_hc_gb300 import synth
        from hyper_connection_residual_hc_gb300.synth import T_COMB, T_DELTA, T_POST, T_PREMIX, T_X

        dist.init_process_group("gloo", rank=rank, world_size=WORLD)
        w0 = synth.small("step_b1_t64", 1, 6, 256, seed=31)
        w = bench.rank_workload(w0, rank)
        inp = dict(X=synth.tokens(w, T_X, 0), delta=synth.tokens(w, T_DELTA, 0), post=synth.tokens(w, T_POST, 0),
                   comb=synth.tokens(w, T_COMB, 0), pre_mix=synth.tokens(w, T_PREMIX, 0))
        prm = synth.params(w0, 0)  # every rank holds the same parameters
        out = orc.hc_post_then_pre(inp["delta"], inp["X"], inp["post"], inp["comb"], inp["pre_mix"], prm["hc_fn"],
                                   prm["hc_scale"], prm["hc_base"], prm["norm_w"], w.iters, w.hc_eps, w.norm_eps,
                                   threads=1)
        slowest = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, w.seed, inp, out, slowest))
    except Exception as e:  # surface the failure in the parent
        q.put((rank, "error", repr(e), None, None))


def test_two_ranks_shard_tokens_without_exchange():
    ctx = multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(WORLD):
        rank, seed, inp, out, slowest = q.get(timeout=240)
        assert seed != "error", inp
        res[rank] = (seed, inp, out, slowest)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (s0, in0, out0, m0), (s1, in1, out1, m1) = res[0], res[1]
    assert s0 != s1
    for k in in0:
        assert in0[k].shape == in1[k].shape and in0[k].dtype == in1[k].dtype
    assert not np.array_equal(in0["X"], in1["X"])
    assert m0 == m1 == 2.5  # both ranks hold the slowest rank's value

    # one call on both batches together gives each rank's rows: no data had to cross ranks
    sys.path.insert(0, ROOT)
    import oracle as orc
    from hyper_connection_residual_hc_gb300 import synth
    w0 = synth.small("step_b1_t64", 1, 6, 256, seed=31)
    prm = synth.params(w0, 0)
    cat = {k: np.concatenate([in0[k], in1[k]]) for k in in0}
    both = orc.hc_post_then_pre(cat["delta"], cat["X"], cat["post"], cat["comb"], cat["pre_mix"], prm["hc_fn"],
                                prm["hc_scale"], prm["hc_base"], prm["norm_w"], w0.iters, w0.hc_eps, w0.norm_eps)
    n = in0["X"].shape[0]
    for k in both:
        assert np.array_equal(both[k][:n], out0[k]), k
        assert np.array_equal(both[k][n:], out1[k]), k


def test_whole_job_rate_and_single_process_reduce():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(16384, 4, 0.5) == 16384 * 4 / 0.5
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    from hyper_connection_residual_hc_gb300 import synth
    w = synth.WORKLOADS["prefill_b4_t4096"]
    assert bench.rank_workload(w, 0) is w
    assert bench.rank_workload(w, 3).seed == w.seed + 51 and bench.rank_workload(w, 3).n == w.n


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
