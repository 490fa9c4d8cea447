"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The hot path does not shard across GPUs in this library (replicas only): each
rank runs the whole workload on its own GPU, ranks meet at a barrier around
the timed steps, the step time is the maximum over ranks, and the reported
rate is all ranks' units over that time.  These host-side pieces are what a
multi-GPU run adds, and they run here without a GPU.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    d = bench.init_dist(w)
    try:
        bench.barrier(d)
        # each rank reports its own step time; the job takes the slowest
        t_ms = 1.0 + rank            # rank 0: 1 ms, rank 1: 2 ms
        t_max = bench.max_over_ranks(d, t_ms)
        rate = bench.whole_job_rate(w, 1000.0, t_max)
        bench.barrier(d)
        results[rank] = (r, w, local, t_max, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), results), nprocs=world,
                           join=True, start_method="spawn")
        got = dict(results)
    assert sorted(got) == [0, 1]
    for rank, (r, w, local, t_max, rate) in got.items():
        assert (r, w, local) == (rank, world, rank)
        assert t_max == pytest.approx(2.0)                    # the slowest rank
        assert rate == pytest.approx(2 * 1000.0 / 2.0e-3)     # all ranks' units / max time


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1) is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.whole_job_rate(1, 10.0, 5.0) == pytest.approx(2000.0)


def test_cpu_baseline_reports_all_cores_and_one_thread():
    """bench.py's CPU-oracle leg on the small fp32 workload: a positive rate
    on all cores and on one thread, each with its sample described."""
    import bench
    from sparse_voxel_convolution_coord_b300 import synth
    cb = bench.cpu_baseline(synth.make_problem(1), target_s=0.5, single_s=0.2)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert "whole workload" in cb["sample"] or "sampled" in cb["sample"]
    assert cb["cpu_model"] and cb["nproc"] >= 1


@pytest.mark.parametrize("key,bound", [(3, "tensor"), (5, "hbm"), (1, "hbm")])
def test_roofline_takes_the_binding_limit(key, bound):
    """64^3 C=256 is bound by the tensor pipe, 256^3 C=32 by HBM (its
    algorithmic bytes take longer than its flops at the measured peaks), the
    fp32 path is reported against HBM."""
    import bench
    from sparse_voxel_convolution_coord_b300 import synth
    cfg = synth.CONFIGS[key]
    p = synth.make_problem(key)
    cin, cout = cfg.cin, cfg.cout
    es = 4 if cfg.dtype == "f32" else 2
    pairs = 20 * p.n
    flops = 2.0 * pairs * cin * cout
    fwd_bytes = p.n * cin * es + 108 * p.n + 4 * p.n * cout + 27 * cin * cout * es
    peaks = {"hbm_gbs": 6491.5, "bf16_tflops": 1804.9, "bf16_tflops_sustained": 1396.2,
             "source": "test"}
    r = bench.roofline_object(cfg.dtype, flops, fwd_bytes, 0.1, peaks, None)
    assert r["bound"] == bound
    want = flops / 1e-4 / 1e12 if bound == "tensor" else fwd_bytes / 1e-4 / 1e9
    assert abs(r["achieved"] - want) <= 1e-9 * want
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12


def test_clock_sampler_summary_and_cleanup(tmp_path):
    """The clock record's parsing: median SM clock, max clock, throttle
    reasons that were active, and the scratch file removed afterwards."""
    import os
    import bench

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

        def kill(self):
            pass

    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "clocks.csv")
    rows = ["0, 2032, 2032, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2000, 2032, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2032, 2032, 980.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    with open(cs.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    cs.f = open(os.devnull, "w")
    cs.proc = FakeProc()
    out = cs.stop()
    assert out["sm_mhz"] == 2032 and out["sm_max_mhz"] == 2032 and out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(cs.path)
