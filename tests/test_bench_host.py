"""bench.py's host-side logic, on CPU.

The path runs on one GPU: our arm refuses more than one (it prints one
"unavailable" line from rank 0 and exits 0, since the tensor-core kernel's
weight multicast within a CTA pair is kept to single-GPU runs), and the
reference arm (the CPU oracle) runs on rank 0 alone.  Both are checked under a
real two-process launch (torch.distributed.run on 127.0.0.1), which needs no
GPU.  The rest covers the CPU-baseline leg, the roofline choice and the clock
record.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(text):
    return [json.loads(ln) for ln in text.splitlines() if ln.startswith("{")]


def test_more_than_one_gpu_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2
    assert "multicast" in lines[0]["unavailable"]


@pytest.mark.parametrize("impl", ["ours", "reference"])
def test_two_process_launch(impl):
    """Under a two-rank launcher: rank 0 prints exactly one line (the refusal
    for our arm, the CPU oracle's line for the reference arm), rank 1 nothing,
    and both exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--impl", impl, "--config", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout
    if impl == "ours":
        assert "unavailable" in lines[0]
    else:
        assert lines[0]["impl"] == "reference" and lines[0]["value"] > 0
        assert lines[0]["cpu_baseline"]["kind"] == "oracle"


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


def test_mma_rows_per_pair():
    """Rows the tensor core runs per present pair: 1 when every row of every
    unit has the unit's offsets; units of two tiles take their union."""
    import numpy as np
    import bench
    nbr = np.zeros((256, 27), np.int32)            # two full tiles: every offset present
    assert bench.mma_rows_per_pair(nbr, 256 * 27, 1) == 1.0
    nbr = -np.ones((300, 27), np.int32)            # three tiles (the last ragged)
    nbr[:, 13] = np.arange(300)                    # centre everywhere
    nbr[0, 0] = 5                                  # one extra offset in tile 0
    pairs = 301
    # cl = 1: tile 0 runs 2 offsets x 128 rows, tiles 1, 2 one offset x 128
    # (the kernel runs every tile's 128 rows, pad rows included)
    assert bench.mma_rows_per_pair(nbr, pairs, 1) == (2 * 128 + 128 + 128) / pairs
    # cl = 2: unit 0 (tiles 0, 1) runs 2 offsets x 256 rows, unit 1 (tile 2) 1 x 128
    assert bench.mma_rows_per_pair(nbr, pairs, 2) == (2 * 256 + 128) / pairs
