"""Benchmark of the 3x3x3 submanifold sparse convolution hot path on B300.

One step = the whole hot path over one synthetic voxel set: coordinate hash
build + neighbour map (sc_build_map), gather-implicit-GEMM with the fused
bias (sc_forward).  Inputs are resident in HBM when the timed region starts;
L2 is flushed (256 MB write) before every timed step.  The printed JSON line
reports effective TFLOP/s = 2 * pairs * cin * cout / step time (pairs = the
present (output, neighbour) pairs only) and active voxels/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3]
    python bench.py --impl reference ...   # the CPU oracle, on host cores

One GPU only: the path does not shard (replicas at most), and the tensor-core
convolution shares its weight slices between the two CTAs of a cluster by TMA
multicast, which is kept to single-GPU runs.  With --gpus N > 1, or under a
launcher with WORLD_SIZE > 1, our arm prints one "unavailable" line (rank 0)
and exits 0.  The reference arm (the CPU oracle) runs on rank 0 alone.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse conv3d effective TFLOP/s + active voxels/s (1 B300, % of roofline)"
FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = same as --steps (max 500)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-map-gate", action="store_true",
                    help="skip timing the 256^3 ~400k-voxel map build beside the workload")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


MULTI_GPU_UNAVAILABLE = (
    "multi-GPU runs are not made: the path runs on one GPU (replicas only, no data-path "
    "exchange), and k_conv_tc multicasts W slices between the two CTAs of a cluster "
    "(cp.async.bulk.tensor .multicast::cluster), which is kept to single-GPU runs")


def multi_gpu_line(n_gpus):
    """The line our arm prints instead of running on more than one GPU."""
    return {"metric": METRIC, "n_gpus": n_gpus, "unavailable": MULTI_GPU_UNAVAILABLE}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        # raw samples in a scratch file; the line carries their summary
        self.path = os.path.join(tempfile.gettempdir(),
                                 "sc_bench_clocks_%d_rank%d.csv" % (os.getpid(), gpu_index))

    def one_shot(self):
        """One synchronous query, appended to the record (a timed region
        shorter than the sampling period still gets a sample on each side)."""
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                                "--format=csv,noheader,nounits"], capture_output=True,
                               text=True, timeout=10)
            if r.returncode == 0 and r.stdout.strip():
                with open(self.path, "a") as f:
                    f.write(r.stdout.strip() + "\n")
        except Exception:
            pass

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            open(self.path, "w").close()
            self.one_shot()
            self.f = open(self.path, "a")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        self.one_shot()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle legs (the only places bench.py runs oracle/)

def cpu_model():
    """The host CPU's model name (from /proc/cpuinfo), or the platform's."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def oracle_sample_run(p, rows, threads=0):
    """Oracle map build over all voxels + fp64 convolution of `rows`."""
    import oracle
    t0 = time.perf_counter()
    nbr = oracle.build_neighbor_table(p.coords, p.res)
    oracle.conv(nbr[rows], p.feats, p.weight, p.bias, threads)
    dt = time.perf_counter() - t0
    pairs = int((nbr[rows] >= 0).sum())
    return dt, pairs


def cpu_baseline(p, target_s=20.0, single_s=4.0):
    """The oracle as it stands on the host cores, for ~target_s seconds: the
    whole workload (map build + fp64 convolution of every row) repeated while
    it fits, else the map build and a row sample sized to the target.  Also
    the same oracle on one thread (its map build is single-threaded anyway),
    on a row sample of ~single_s seconds."""
    import oracle
    cin, cout = p.feats.shape[1], p.weight.shape[2]
    rng = np.random.default_rng(0)
    t0 = time.perf_counter()
    nbr = oracle.build_neighbor_table(p.coords, p.res)
    t_map = time.perf_counter() - t0
    # pilot large enough to occupy every thread (the oracle hands out rows
    # 64 at a time)
    pilot = rng.choice(p.n, size=min(p.n, max(2048, 256 * oracle.max_threads())),
                       replace=False)
    t0 = time.perf_counter()
    oracle.conv(nbr[pilot], p.feats, p.weight, p.bias)
    per_row = max((time.perf_counter() - t0) / len(pilot), 1e-9)
    t_full = t_map + per_row * p.n
    if t_full <= target_s:
        reps = max(1, int(target_s / t_full))
        rows = np.arange(p.n)
        dt, pairs = 0.0, 0
        for _ in range(reps):
            d, pr = oracle_sample_run(p, rows)
            dt += d
            pairs += pr
        what = "the whole workload (oracle map build + fp64 conv of all %d rows) %d times" % (
            p.n, reps)
        rows_done = reps * p.n
    else:
        m = int(min(p.n, max(256, (target_s - t_map) / per_row)))
        rows = np.sort(rng.choice(p.n, size=m, replace=False))
        dt, pairs = oracle_sample_run(p, rows)
        what = "oracle map build over all %d voxels + fp64 conv of %d sampled output rows" % (
            p.n, m)
        rows_done = m
    tflops = 2.0 * pairs * cin * cout / dt / 1e12
    # the same oracle on one thread, on a sample of ~single_s seconds
    per_row1 = per_row * oracle.max_threads()
    m1 = int(min(p.n, max(64, (single_s - t_map) / per_row1)))
    rows1 = np.sort(rng.choice(p.n, size=m1, replace=False))
    dt1, pairs1 = oracle_sample_run(p, rows1, threads=1)
    return {"value": tflops, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "sample": "%s: %d pairs in %.1f s; voxels/s %.3g" % (what, pairs, dt, rows_done / dt),
            "single_thread": {
                "value": 2.0 * pairs1 * cin * cout / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                "sample": "oracle map build over all %d voxels + fp64 conv of %d sampled rows "
                          "on one thread: %d pairs in %.1f s" % (p.n, m1, pairs1, dt1)}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from sparse_voxel_convolution_coord_b300 import synth
    import oracle
    p = synth.make_problem(args.config)
    cin, cout = p.feats.shape[1], p.weight.shape[2]
    rng = np.random.default_rng(1)
    # bounded sample per step: the full map build + the conv of 16 output rows
    samples = [np.sort(rng.choice(p.n, size=16, replace=False)) for _ in range(4)]
    for i in range(args.warmup):
        oracle_sample_run(p, samples[i % 4])
    tot_t, tot_pairs = 0.0, 0
    for i in range(args.steps):
        dt, pairs = oracle_sample_run(p, samples[i % 4])
        tot_t += dt
        tot_pairs += pairs
    value = 2.0 * tot_pairs * cin * cout / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": p.config.name, "n_voxels": p.n, "cin": cin, "cout": cout,
                   "res": p.res},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": "per step: oracle map build over all %d voxels + fp64 conv "
                                   "of 16 sampled output rows" % p.n},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# of the convolution kernel, from the ncu capture summarised in profiles/,
# valid only for the kernel source it was measured on (sha1 of the file).
MEASURED_TRAFFIC = {
    # workload name: (sha1 of sc_conv_tc.cu, bytes per launch)
    "sq3x64_30k_c256_bf16": ("c673aed9615fe250034075d9bc52bd3538000c69", 33265664 + 27392),
    "sq4x256_400k_c32_bf16": ("c673aed9615fe250034075d9bc52bd3538000c69", 68185088 + 13070592),
}


def _file_sha1(path):
    import hashlib
    return hashlib.sha1(open(path, "rb").read()).hexdigest()


def time_forward_alone(sc, torch, m, feats, weight, bias, out, flush, stream, reps=200):
    """Median device time of one forward launch: the stream is first held by a
    GPU sleep so that every (flush, event, forward, event) group is queued
    before the GPU reaches it (no host gaps inside the events); L2 is flushed
    before each launch."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(int(5e7))
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        sc.sc_forward(m, feats, weight, bias, out)
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs[10:])


def mma_rows_per_pair(nbr, pairs, cl):
    """Tensor-core rows issued per present (output, neighbour) pair for the
    map in input order: a unit of `cl` consecutive 128-row tiles runs one
    stage group per offset present in any of its rows, for all its rows."""
    n = nbr.shape[0]
    if n == 0 or pairs == 0:
        return None
    tiles = (n + 127) // 128
    pres = np.zeros((tiles * 128, 27), bool)
    pres[:n] = nbr >= 0
    tile_any = pres.reshape(tiles, 128, 27).any(axis=1)
    units = (tiles + cl - 1) // cl
    pad = np.zeros((units * cl, 27), bool)
    pad[:tiles] = tile_any
    unit_any = pad.reshape(units, cl, 27).any(axis=1)
    rows_per_unit = np.minimum(cl, tiles - np.arange(units) * cl) * 128
    return float((unit_any.sum(axis=1) * rows_per_unit).sum() / pairs)


def roofline_object(dtype, flops, fwd_bytes, t_kernel_ms, peaks, traffic):
    """The bench line's roofline for one forward launch of t_kernel_ms: the
    tensor pipe or HBM, whichever the algorithmic flops or bytes would take
    longer on (fp16 takes the bf16 measured peak x the nominal fp16/bf16
    ratio, 1); the fp32 FFMA path against HBM."""
    t_s = t_kernel_ms * 1e-3
    if dtype == "f32":
        gbs = fwd_bytes / t_s / 1e9
        return {"kernel": "k_conv_simt_f32 (fp32 FFMA gather-GEMM)", "bound": "hbm",
                "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"] + " hbm",
                "traffic": None, "kernel_us": t_kernel_ms * 1e3,
                "algorithmic_bytes_per_launch": fwd_bytes}
    kernel = "k_conv_tc (gather-implicit-GEMM, tcgen05, %s -> fp32 TMEM)" % dtype
    tensor_bound = (flops / (peaks["bf16_tflops"] * 1e12)
                    >= fwd_bytes / (peaks["hbm_gbs"] * 1e9))
    if tensor_bound:
        achieved = flops / t_s / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "frac_of_sustained": (achieved / peaks["bf16_tflops_sustained"]
                                      if peaks.get("bf16_tflops_sustained") else None),
                "peak_source": peaks["source"] + " bf16 burst (MEASURED_PEAKS.json)"
                               + (" x nominal fp16/bf16 ratio 1" if dtype == "f16" else ""),
                "traffic": traffic, "kernel_us": t_kernel_ms * 1e3,
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": fwd_bytes}
    gbs = fwd_bytes / t_s / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
            "peak_source": peaks["source"] + " hbm", "traffic": traffic,
            "kernel_us": t_kernel_ms * 1e3, "algorithmic_flops_per_launch": flops,
            "tensor_tflops": flops / t_s / 1e12, "algorithmic_bytes_per_launch": fwd_bytes}


def time_build(sc, torch, coords, res, nbatch, flush, stream, reps=60):
    """Map build timed two ways on the same coordinates, L2 flushed before each:
    device-only (CUDA events around sc_build_map_async: init, insert and query
    kernels, with the stream held by a GPU sleep so host gaps do not count)
    and host-inclusive (host time of sc_build_map, which synchronises once to
    read the status and pair count).  Returns medians in ms."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    maps = []
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e7))
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        maps.append(sc.sc_build_map_async(coords, res, nbatch))
        e1.record(stream)
    torch.cuda.synchronize()
    sc.sc_map_status(maps[-1])
    for m in maps:
        m.free()
    dev_ms = statistics.median(a.elapsed_time(b) for a, b in evs[5:])
    host = []
    for _ in range(reps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        m = sc.sc_build_map(coords, res)
        host.append((time.perf_counter() - t0) * 1e3)
        m.free()
    torch.cuda.synchronize()
    return dev_ms, statistics.median(host[5:])


def map_build_object(n, dev_ms, host_ms, peaks, what):
    """The map build against its algorithmic bytes (coords 16N + one slot write
    8N + neighbour table 108N)."""
    b = 132 * n
    return {"workload": what, "bound": "hbm", "n_voxels": n, "algorithmic_bytes": b,
            "device_us": dev_ms * 1e3, "achieved_gbs": b / (dev_ms * 1e-3) / 1e9,
            "frac_of_hbm": b / (dev_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "host_inclusive_us": host_ms * 1e3,
            "achieved_gbs_host_inclusive": b / (host_ms * 1e-3) / 1e9,
            "frac_of_hbm_host_inclusive": b / (host_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "peak_source": peaks["source"] + " hbm"}


def run_ours(args):
    rank, world, local = dist_env()
    if args.gpus > 1 or world > 1:
        if rank == 0:
            print(json.dumps(multi_gpu_line(max(args.gpus, world))), flush=True)
        return
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import sparse_voxel_convolution_coord_b300 as sc
    from sparse_voxel_convolution_coord_b300 import build_lib, synth
    build_lib.build()
    sc.load_library()

    p = synth.make_problem(args.config)
    cin, cout = p.feats.shape[1], p.weight.shape[2]
    nbatch = int(p.coords[:, 0].max()) + 1 if p.n else 1
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[p.config.dtype]
    esize = 4 if p.config.dtype == "f32" else 2
    coords = torch.from_numpy(p.coords).to(dev)
    feats = torch.from_numpy(p.feats).to(dev).to(tdt)
    weight = torch.from_numpy(p.weight).to(dev).to(tdt)
    bias = torch.from_numpy(p.bias).to(dev)
    out = torch.empty((p.n, cout), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    m = sc.sc_build_map(coords, p.res)
    pairs = m.pairs
    m.free()
    flops = 2.0 * pairs * cin * cout
    # algorithmic bytes (every byte the path must move once)
    fwd_bytes = p.n * cin * esize + 108 * p.n + 4 * p.n * cout + 27 * cin * cout * esize

    # -- the timed step: map build (asynchronous: no host synchronisation) +
    # forward, L2 flushed before each step outside the events
    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        mp = sc.sc_build_map_async(coords, p.res, nbatch)
        if evs is not None:
            evs[1].record(stream)
        sc.sc_forward(mp, feats, weight, bias, out)
        if evs is not None:
            evs[2].record(stream)
        return mp

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step().free()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    launches0 = sc.sc_kernel_launches()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        step(evs[i]).free()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    gpu_launches = sc.sc_kernel_launches() - launches0
    clk = clocks.stop()
    # the timed builds ran on the same coordinates: one more must report no error
    mp = step()
    sc.sc_map_status(mp)
    sc.sc_device_status(mp)
    mp.free()
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    build_ms = [e[0].elapsed_time(e[1]) for e in evs]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    t_step = sum(step_ms) / K
    t_build = sum(build_ms) / K
    t_fwd = sum(fwd_ms) / K

    # -- the convolution kernel alone (roofline), on one map
    mp = sc.sc_build_map(coords, p.res)
    for _ in range(5):
        sc.sc_forward(mp, feats, weight, bias, out)
    t_kernel = time_forward_alone(sc, torch, mp, feats, weight, bias, out, flush, stream)
    sc.sc_device_status(mp)
    mma_rows = mma_rows_per_pair(sc.sc_get_neighbor_table(mp).cpu().numpy(), pairs,
                                 2 if cout > 64 and p.config.dtype != "f32" else 1)
    # the same forward over rows ordered by neighbour mask (sc_map_order_rows,
    # a one-off cost per map), and that cost
    o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e7))
    o0.record(stream)
    sc.sc_map_order_rows(mp)
    o1.record(stream)
    for _ in range(5):
        sc.sc_forward(mp, feats, weight, bias, out)
    t_kernel_ordered = time_forward_alone(sc, torch, mp, feats, weight, bias, out, flush, stream)
    t_order = o0.elapsed_time(o1)
    sc.sc_device_status(mp)
    mp.free()

    # -- the map build alone: this workload, and the 256^3 ~400k-voxel shells
    # (the largest single build, where the HBM target is set)
    peaks = load_peaks()
    dev_b, host_b = time_build(sc, torch, coords, p.res, nbatch, flush, stream)
    map_build = map_build_object(p.n, dev_b, host_b, peaks, p.config.name)
    gate = None
    if args.config != 5 and not args.no_map_gate:
        p5 = synth.make_problem(5)
        c5 = torch.from_numpy(p5.coords).to(dev)
        dev5, host5 = time_build(sc, torch, c5, p5.res, 1, flush, stream)
        gate = map_build_object(p5.n, dev5, host5, peaks, p5.config.name)
        del c5

    # -- end to end through the public API from pinned host buffers
    h_coords = torch.from_numpy(p.coords).pin_memory()
    h_feats = torch.from_numpy(p.feats).to(tdt).pin_memory()
    h_weight = torch.from_numpy(p.weight).to(tdt).pin_memory()
    h_bias = torch.from_numpy(p.bias).pin_memory()
    h_out = torch.empty((p.n, cout), dtype=torch.float32).pin_memory()
    d_coords = torch.empty_like(coords)
    d_feats = torch.empty_like(feats)
    d_weight = torch.empty_like(weight)
    d_bias = torch.empty_like(bias)
    h2d = sum(t.numel() * t.element_size() for t in (h_coords, h_feats, h_weight, h_bias))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_coords.copy_(h_coords, non_blocking=True)
        d_feats.copy_(h_feats, non_blocking=True)
        d_weight.copy_(h_weight, non_blocking=True)
        d_bias.copy_(h_bias, non_blocking=True)
        mp = sc.sc_build_map_async(d_coords, p.res, nbatch)
        sc.sc_forward(mp, d_feats, d_weight, d_bias, out)
        h_out.copy_(out, non_blocking=True)
        mp.free()

    KE = args.e2e_steps or min(K, 500)
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(KE):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = e0.elapsed_time(e1) / KE

    # The same steps pipelined, as a serving loop would run them: two sets of
    # device buffers; step i's inputs go up on one copy stream while the
    # main stream computes step i - 1 and another copy stream brings step
    # i - 2's result down (PCIe carries both directions at once).  Every
    # step still copies all its inputs up and its whole result down.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    dbufs = [(d_coords, d_feats, d_weight, d_bias, out)] + [
        (torch.empty_like(coords), torch.empty_like(feats), torch.empty_like(weight),
         torch.empty_like(bias), torch.empty_like(out))]
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # step's inputs landed
    ev_used = [torch.cuda.Event() for _ in range(2)]  # step's compute done with its buffers
    ev_down = [torch.cuda.Event() for _ in range(2)]  # step's result left the device
    for ev in ev_in + ev_used + ev_down:
        ev.record(stream)

    def pipe_step(i):
        b = i % 2
        dc, df, dw, db, do = dbufs[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_used[b])
            dc.copy_(h_coords, non_blocking=True)
            df.copy_(h_feats, non_blocking=True)
            dw.copy_(h_weight, non_blocking=True)
            db.copy_(h_bias, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_down[b])
        mp = sc.sc_build_map_async(dc, p.res, nbatch)
        sc.sc_forward(mp, df, dw, db, do)
        ev_used[b].record(stream)
        mp.free()
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_used[b])
            h_outs[b].copy_(do, non_blocking=True)
            ev_down[b].record(s_out)

    for i in range(3):
        pipe_step(i)
    torch.cuda.synchronize()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(KE):
        pipe_step(i)
    stream.wait_event(ev_down[(KE - 1) % 2])
    stream.wait_event(ev_in[(KE - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e_pipe = e0.elapsed_time(e1) / KE

    conv_src = os.path.join(ROOT, "sparse_voxel_convolution_coord_b300", "csrc", "sc_conv_tc.cu")
    traffic = None
    rec = MEASURED_TRAFFIC.get(p.config.name)
    if rec is not None and p.config.dtype != "f32" and rec[0] == _file_sha1(conv_src):
        traffic = rec[1]
    roofline = roofline_object(p.config.dtype, flops, fwd_bytes, t_kernel, peaks, traffic)
    line = {
        "metric": METRIC,
        "value": flops / (t_step * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": p.config.dtype,
        "data": "synthetic (seeded superquadric voxel shells; random N(0,1) features, "
                "N(0, 1/sqrt(27 cin)) weights)",
        "config": {"workload": p.config.name, "description": p.config.description,
                   "n_voxels": p.n, "pairs": pairs, "cin": cin, "cout": cout, "res": p.res,
                   "parallelism": "single",
                   "step": "sc_build_map_async (hash + neighbour map, no host sync) + "
                           "sc_forward (gather-GEMM + bias); build errors checked after",
                   "l2": "flushed before every timed step (256 MB write, outside the events)"},
        "voxels_per_s": p.n / (t_step * 1e-3),
        "breakdown_ms": {"build_map_in_step": t_build, "forward_in_step": t_fwd,
                         "forward_kernel_alone": t_kernel,
                         "forward_kernel_alone_rows_ordered": t_kernel_ordered,
                         "order_rows_once_per_map": t_order,
                         "wall_per_step_incl_flush": wall / K * 1e3},
        "mma_rows_issued_per_pair": mma_rows,
        "roofline": roofline,
        "map_build": map_build,
        "map_build_256cubed_400k": gate,
        "e2e": {"value": flops / (t_e2e_pipe * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": t_e2e_pipe, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": KE,
                "how": "public API (sc_build_map_async + sc_forward) from pinned host buffers; "
                       "inputs up on one copy stream, result down on another, compute on "
                       "the main stream, two device buffer sets (steps overlap)",
                "serial": {"value": flops / (t_e2e * 1e-3) / 1e12, "ms_per_step": t_e2e,
                           "how": "copy up, build, forward, copy down on one stream"}},
        # counted by the library at each of its launches over the timed steps
        # (map build: init, insert, query; forward: conv, plus the zeroing
        # kernel when a partial last round of tiles is split)
        "gpu_launches": gpu_launches,
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
