"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Maps (neighbour table, pair lists) must match bit for bit.  Convolution
outputs must meet the bars of the method's acceptance criteria: fp32 inputs
relative L2 <= 1e-5; bf16 inputs relative L2 <= 2e-3 and max |err| <=
1e-2 * rms(ref), against the oracle fed the same bf16-rounded values.
relative L2 = ||gpu - ref||_2 / ||ref||_2 over the compared outputs,
rms(ref) = ||ref||_2 / sqrt(count).
"""
import numpy as np
import pytest

import oracle
from sparse_voxel_convolution_coord_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32_REL_L2 = 1e-5
BF16_REL_L2 = 2e-3
BF16_MAX_ABS_OVER_RMS = 1e-2


@pytest.fixture(scope="module")
def sc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_voxel_convolution_coord_b300 as m
    from sparse_voxel_convolution_coord_b300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(dtype) if dtype is not None else t


def gpu_map(sc, coords, res):
    m = sc.sc_build_map(to_dev(coords.astype(np.int32)), res)
    nbr = sc.sc_get_neighbor_table(m).cpu().numpy()
    return m, nbr


TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def gpu_conv(sc, m, feats, weight, bias, dtype):
    tdt = TORCH_DT[dtype]
    out = sc.sc_forward(m, to_dev(feats, tdt), to_dev(weight, tdt),
                        None if bias is None else to_dev(bias))
    sc.sc_device_status(m)
    return out.cpu().numpy().astype(np.float64)


def assert_close(got, ref, dtype, what=""):
    err = got - ref
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / max(nref, 1e-300)
    if dtype == "f32":
        assert rel <= F32_REL_L2, "%s rel L2 %.3e > %.0e" % (what, rel, F32_REL_L2)
    else:  # bf16 and fp16 inputs: the half-precision bars
        rms = nref / np.sqrt(ref.size)
        mx = np.abs(err).max() if err.size else 0.0
        assert rel <= BF16_REL_L2, "%s rel L2 %.3e" % (what, rel)
        assert mx <= BF16_MAX_ABS_OVER_RMS * rms, "%s max abs %.3e > 1e-2 rms %.3e" % (what, mx, rms)
    return rel


def random_coords(rng, nbatch, res, density, batch_ids=None):
    rows = []
    ids = batch_ids if batch_ids is not None else range(nbatch)
    for b in ids:
        occ = rng.random((res, res, res)) < density
        xyz = np.argwhere(occ)
        rows.append(np.concatenate([np.full((len(xyz), 1), b), xyz], axis=1))
    return np.concatenate(rows).astype(np.int32)


# ---------------------------------------------------------------------------
# maps

@pytest.mark.parametrize("key", [1, 2, 3, 4, 5])
def test_map_bit_exact_configs(sc, key):
    p = synth.make_problem(key)
    m, nbr = gpu_map(sc, p.coords, p.res)
    want = oracle.build_neighbor_table(p.coords, p.res)
    np.testing.assert_array_equal(nbr, want)
    assert sc.sc_map_pairs(m) == int((want >= 0).sum())
    off, pin, pout = sc.sc_get_pairs(m)
    woff, wpin, wpout = oracle.pairs(want)
    np.testing.assert_array_equal(off.numpy(), woff)
    np.testing.assert_array_equal(pin.cpu().numpy(), wpin)
    np.testing.assert_array_equal(pout.cpu().numpy(), wpout)
    m.free()


def test_map_shuffled_and_repeatable(sc):
    p = synth.make_problem(3)
    rng = np.random.default_rng(1)
    perm = rng.permutation(p.n)
    c = p.coords[perm]
    m1, nbr1 = gpu_map(sc, c, p.res)
    m2, nbr2 = gpu_map(sc, c, p.res)
    np.testing.assert_array_equal(nbr1, nbr2)
    np.testing.assert_array_equal(nbr1, oracle.build_neighbor_table(c, p.res))
    m1.free()
    m2.free()


@pytest.mark.parametrize("case", ["full_cube", "res1_batches", "batch_gaps", "single",
                                  "line_z", "sparse_big_res", "k32_last_batch",
                                  "k32_overflow_retry"])
def test_map_edge_cases(sc, case):
    rng = np.random.default_rng(2)
    if case == "full_cube":
        L = 9
        xyz = np.argwhere(np.ones((L, L, L), bool))
        coords, res = np.concatenate([np.zeros((len(xyz), 1)), xyz], 1).astype(np.int32), L
    elif case == "res1_batches":
        coords, res = np.array([[b, 0, 0, 0] for b in range(5)], np.int32), 1
    elif case == "batch_gaps":
        coords, res = random_coords(rng, 0, 12, 0.2, batch_ids=[0, 3, 7]), 12
    elif case == "single":
        coords, res = np.array([[2, 5, 0, 7]], np.int32), 8
    elif case == "line_z":
        coords, res = np.array([[0, 3, 3, z] for z in range(300)], np.int32), 300
    elif case == "k32_last_batch":
        # res 64: 32-bit keys hold batch indices < (2^32 - 1) // 64^3 = 16383
        coords, res = random_coords(rng, 0, 64, 0.01, batch_ids=[0, 16382]), 64
    elif case == "k32_overflow_retry":
        # batch 16383 reaches key 2^32 - 1 and 20000 lies beyond: 64-bit keys
        coords, res = random_coords(rng, 0, 64, 0.01, batch_ids=[0, 16383, 20000]), 64
    else:
        coords, res = random_coords(rng, 1, 64, 0.002), 1 << 14
        coords[:, 1:] *= 200
    m, nbr = gpu_map(sc, coords, res)
    want = oracle.build_neighbor_table(coords, res)
    np.testing.assert_array_equal(nbr, want)
    if case == "full_cube":
        assert sc.sc_map_pairs(m) == (3 * 9 - 2) ** 3
    m.free()


def test_map_empty(sc):
    m = sc.sc_build_map(torch.zeros((0, 4), dtype=torch.int32, device="cuda"), 16)
    assert sc.sc_map_size(m) == 0 and sc.sc_map_pairs(m) == 0
    off, pin, pout = sc.sc_get_pairs(m)
    assert off.abs().sum() == 0 and pin.numel() == 0
    out = sc.sc_forward(m, torch.zeros((0, 32), dtype=torch.bfloat16, device="cuda"),
                        torch.zeros((27, 32, 32), dtype=torch.bfloat16, device="cuda"))
    assert out.shape == (0, 32)
    m.free()


@pytest.mark.parametrize("coords,res,code", [
    ([[0, 0, 0, 8]], 8, 2),                       # x/y/z == res
    ([[0, 0, -1, 0]], 8, 2),                      # negative coordinate
    ([[-1, 0, 0, 0]], 8, 2),                      # negative batch
    ([[0, 1, 2, 3], [0, 1, 2, 3]], 8, 3),         # duplicate
    ([[0, 1, 2, 3], [0, 1, 2, 3], [0, 9, 0, 0]], 8, 2),  # range wins over duplicate
])
def test_map_errors(sc, coords, res, code):
    with pytest.raises(sc.ScError) as e:
        sc.sc_build_map(to_dev(np.array(coords, np.int32)), res)
    assert e.value.code == code
    # the oracle agrees on the class of error
    with pytest.raises(oracle.OracleError) as eo:
        oracle.build_neighbor_table(np.array(coords, np.int32), res)
    assert eo.value.code == {2: oracle.COORD_RANGE, 3: oracle.DUPLICATE}[code]


def test_key_space_overflow_is_unsupported(sc):
    # n = 1 leaves 63 key bits; res = 2^14 uses 42 of them, so batch < 2^21.
    with pytest.raises(sc.ScError) as e:
        sc.sc_build_map(to_dev(np.array([[1 << 22, 0, 0, 0]], np.int32)), 1 << 14)
    assert e.value.code == sc.SC_ERR_UNSUPPORTED
    m = sc.sc_build_map(to_dev(np.array([[(1 << 21) - 1, 5, 5, 5]], np.int32)), 1 << 14)
    m.free()


def test_double_free_is_caught(sc):
    m = sc.sc_build_map(to_dev(np.array([[0, 1, 1, 1]], np.int32)), 4)
    ptr = m.ptr
    m.free()
    import ctypes
    assert sc.load_library().sc_free_map(ctypes.c_void_p(ptr), None) == sc.SC_ERR_BAD_HANDLE


# ---------------------------------------------------------------------------
# convolution

def check_problem(sc, coords, res, feats, weight, bias, dtype, rows=None, what=""):
    """The GPU map equals the oracle's bit for bit, and the GPU convolution
    matches the oracle's convolution over the ORACLE's map (nothing the
    reference computes comes from the CUDA path)."""
    m, nbr = gpu_map(sc, coords, res)
    want = oracle.build_neighbor_table(coords, res)
    np.testing.assert_array_equal(nbr, want)
    got = gpu_conv(sc, m, feats, weight, bias, dtype)
    if rows is None:
        ref = oracle.conv(want, feats, weight, bias)
        rel = assert_close(got, ref, dtype, what)
    else:
        ref = oracle.conv(want[rows], feats, weight, bias)
        rel = assert_close(got[rows], ref, dtype, what)
    m.free()
    return rel


@pytest.mark.parametrize("key", [1, 2, 5])
def test_conv_configs_full(sc, key):
    p = synth.make_problem(key)
    check_problem(sc, p.coords, p.res, p.feats, p.weight, p.bias, p.config.dtype,
                  what="config %d" % key)


@pytest.mark.parametrize("key", [3, 4])
def test_conv_configs_sampled(sc, key):
    p = synth.make_problem(key)
    rng = np.random.default_rng(10 + key)
    n = p.n
    rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(n - 300, n),
                                     rng.choice(n, size=3000, replace=False)]))
    check_problem(sc, p.coords, p.res, p.feats, p.weight, p.bias, p.config.dtype, rows=rows,
                  what="config %d" % key)


SHAPES = [(16, 16), (32, 48), (64, 64), (64, 192), (128, 32), (192, 256), (256, 256),
          (1024, 16), (32, 256), (128, 128), (256, 96), (512, 64)]


@pytest.mark.parametrize("cin,cout", SHAPES)
def test_conv_bf16_shapes(sc, cin, cout):
    rng = np.random.default_rng(cin * 1000 + cout)
    coords = random_coords(rng, 2, 14, 0.25)          # ~1370 rows: 11 tiles, ragged tail
    feats, weight, bias = synth.make_tensors(len(coords), cin, cout, "bf16", cin + cout)
    check_problem(sc, coords, 14, feats, weight, bias, "bf16", what="%dx%d" % (cin, cout))


@pytest.mark.parametrize("cin,cout", [(16, 16), (64, 192), (256, 256), (32, 256)])
def test_conv_f16_shapes(sc, cin, cout):
    """fp16 operands on the tensor cores (tcgen05 kind::f16 with fp16 A and B)."""
    rng = np.random.default_rng(cin * 1000 + cout + 1)
    coords = random_coords(rng, 2, 14, 0.25)
    feats, weight, bias = synth.make_tensors(len(coords), cin, cout, "f16", cin + cout)
    check_problem(sc, coords, 14, feats, weight, bias, "f16", what="f16 %dx%d" % (cin, cout))


@pytest.mark.parametrize("key", [2, 3])
def test_conv_f16_configs(sc, key):
    """Configs 2 and 3 with their inputs rounded to fp16 instead of bf16."""
    p = synth.make_problem(key)
    feats, weight, bias = synth.make_tensors(p.n, p.feats.shape[1], p.weight.shape[2], "f16", key)
    rows = None
    if key == 3:
        rng = np.random.default_rng(44)
        rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(p.n - 300, p.n),
                                         rng.choice(p.n, size=3000, replace=False)]))
    check_problem(sc, p.coords, p.res, feats, weight, bias, "f16", rows=rows,
                  what="f16 config %d" % key)


@pytest.mark.parametrize("cin,cout", [(32, 32), (3, 5), (100, 256), (64, 128)])
def test_conv_f32_shapes(sc, cin, cout):
    rng = np.random.default_rng(cin + 7 * cout)
    coords = random_coords(rng, 2, 12, 0.3)
    feats, weight, bias = synth.make_tensors(len(coords), cin, cout, "f32", cin)
    check_problem(sc, coords, 12, feats, weight, bias, "f32", what="f32 %dx%d" % (cin, cout))


@pytest.mark.parametrize("dtype,c", [("bf16", 64), ("f32", 32), ("bf16", 32)])
def test_identity_centre_tap_is_exact(sc, dtype, c):
    p = synth.make_problem(2)
    feats = p.feats[:, :c] if dtype == "bf16" else p.feats[:, :c].copy()
    w = np.zeros((27, c, c), np.float32)
    w[13] = np.eye(c)
    m, _ = gpu_map(sc, p.coords, p.res)
    got = gpu_conv(sc, m, feats, w, None, dtype)
    np.testing.assert_array_equal(got, feats.astype(np.float64))
    m.free()


def test_isolated_voxels(sc):
    coords = np.array([[0, 1, 1, 1], [0, 5, 5, 5], [1, 1, 1, 1], [3, 0, 0, 0]], np.int32)
    feats, weight, bias = synth.make_tensors(4, 64, 64, "bf16", 77)
    m, nbr = gpu_map(sc, coords, 8)
    assert (nbr >= 0).sum() == 4
    got = gpu_conv(sc, m, feats, weight, bias, "bf16")
    want = feats.astype(np.float64) @ weight[13].astype(np.float64) + bias
    assert_close(got, want, "bf16")
    m.free()


def test_permutation_equivariance(sc):
    p = synth.make_problem(2)
    m, _ = gpu_map(sc, p.coords, p.res)
    base = gpu_conv(sc, m, p.feats, p.weight, p.bias, "bf16")
    m.free()
    perm = np.random.default_rng(3).permutation(p.n)
    m, _ = gpu_map(sc, p.coords[perm], p.res)
    got = gpu_conv(sc, m, p.feats[perm], p.weight, p.bias, "bf16")
    assert_close(got, base[perm], "bf16")
    m.free()


@pytest.mark.parametrize("key,fwd", [(3, 2), (5, 1)])
def test_launch_counter(sc, key, fwd):
    """Map build = 3 kernels; a forward = the conv kernel, plus the zeroing
    kernel where the last partial round of tiles is split (64^3, C=256)."""
    p = synth.make_problem(key)
    c0 = sc.sc_kernel_launches()
    m, _ = gpu_map(sc, p.coords, p.res)
    c1 = sc.sc_kernel_launches()
    gpu_conv(sc, m, p.feats, p.weight, p.bias, "bf16")
    c2 = sc.sc_kernel_launches()
    m.free()
    assert c2 - c1 == fwd
    assert c1 - c0 == 4  # the build's 3, plus the row-major copy of the table gpu_map reads


@pytest.mark.parametrize("key", [2, 3, 4])
def test_forward_deterministic_mode(sc, key):
    """Deterministic mode: repeated forwards are bit-identical."""
    p = synth.make_problem(key)
    m, _ = gpu_map(sc, p.coords, p.res)
    sc.sc_set_deterministic(True)
    try:
        a = gpu_conv(sc, m, p.feats, p.weight, p.bias, "bf16")
        b = gpu_conv(sc, m, p.feats, p.weight, p.bias, "bf16")
    finally:
        sc.sc_set_deterministic(False)
    np.testing.assert_array_equal(a, b)
    m.free()


@pytest.mark.parametrize("key", [2, 3, 4])
def test_forward_repeat_default_mode(sc, key):
    """Default mode: rows of split tiles may differ between runs, by fp32
    rounding of a reordered sum of at most 8 partial accumulators."""
    p = synth.make_problem(key)
    m, _ = gpu_map(sc, p.coords, p.res)
    a = gpu_conv(sc, m, p.feats, p.weight, p.bias, "bf16")
    b = gpu_conv(sc, m, p.feats, p.weight, p.bias, "bf16")
    scale = np.abs(a).max()
    assert np.abs(a - b).max() <= 8 * 2.0 ** -23 * 2 * scale
    m.free()


def test_forward_rejects_bad_arguments(sc):
    import ctypes
    p = synth.make_problem(2)
    m, _ = gpu_map(sc, p.coords, p.res)
    lib = sc.load_library()
    f = to_dev(p.feats, torch.bfloat16)
    w = to_dev(p.weight, torch.bfloat16)
    out = torch.empty((p.n, 64), device="cuda")
    P = ctypes.c_void_p
    # unaligned feats
    assert lib.sc_forward(P(m.ptr), P(f.data_ptr() + 2), P(w.data_ptr()), None,
                          P(out.data_ptr()), 64, 64, 1, None) == sc.SC_ERR_INVALID_ARG
    # unsupported shapes
    assert lib.sc_forward(P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None,
                          P(out.data_ptr()), 48, 64, 1, None) == sc.SC_ERR_UNSUPPORTED
    assert lib.sc_forward(P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None,
                          P(out.data_ptr()), 64, 72, 1, None) == sc.SC_ERR_UNSUPPORTED
    assert lib.sc_forward(P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None,
                          P(out.data_ptr()), 64, 64, 7, None) == sc.SC_ERR_UNSUPPORTED
    assert lib.sc_forward(P(m.ptr), None, P(w.data_ptr()), None,
                          P(out.data_ptr()), 64, 64, 1, None) == sc.SC_ERR_INVALID_ARG
    m.free()


# ---------------------------------------------------------------------------
# fused epilogue: out = act(conv + bias) + residual, rounded once to the
# output dtype ("Porting TRELLIS.2 From Python to Rust and Metal", section V)

_ORACLE_CONV = {}


def _oracle_conv_full(key):
    if key not in _ORACLE_CONV:
        p = synth.make_problem(key)
        _ORACLE_CONV[key] = oracle.sparse_conv(p.coords, p.res, p.feats, p.weight, p.bias)
    return _ORACLE_CONV[key]


def half_ulp(x, odt):
    """Spacing of bf16 (8 significant bits, 2^-133 below 2^-126) or fp16 (11
    significant bits, 2^-24 below 2^-14) values at |x|."""
    sig, emin = (8, -125) if odt == "bf16" else (11, -13)
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, np.maximum(e, emin) - sig)


def check_epilogue_out(got, ref, odt, in_dtype, what):
    """fp32 output: the convolution's bars.  bf16 / fp16 output: within one
    spacing of the oracle's value rounded to that format (the GPU rounds its
    fp32 result, which can sit on the other side of a rounding boundary),
    plus the fp32 accumulation error, and equal to it for nearly every element
    (fp16's finer spacing leaves more elements near a boundary)."""
    if odt == "f32":
        assert_close(got, ref, in_dtype, what)
        return
    rref = oracle.round_bf16(ref) if odt == "bf16" else oracle.round_f16(ref)
    rms = np.linalg.norm(ref) / np.sqrt(ref.size)
    err = np.abs(got - rref)
    bound = half_ulp(ref, odt) + 1e-4 * rms
    assert np.all(err <= bound), "%s: %d elements beyond one %s spacing" % (
        what, int((err > bound).sum()), odt)
    frac = np.mean(got == rref)
    floor = 0.95 if odt == "bf16" else 0.9
    assert frac >= floor, "%s: only %.3f of elements equal the rounded oracle" % (what, frac)


def _residual(n, cout, odt, seed):
    r = np.random.default_rng(seed).standard_normal((n, cout)).astype(np.float32)
    if odt != "f32":
        r = torch.from_numpy(r).to(TORCH_DT[odt]).to(torch.float32).numpy()
    return r


@pytest.mark.parametrize("key", [1, 2])
@pytest.mark.parametrize("act", ["none", "relu", "silu"])
@pytest.mark.parametrize("resid", [False, True])
@pytest.mark.parametrize("odt", ["f32", "bf16", "f16"])
def test_fused_epilogue(sc, key, act, resid, odt):
    p = synth.make_problem(key)
    cout = p.weight.shape[2]
    tin = TORCH_DT[p.config.dtype]
    tout = TORCH_DT[odt]
    r = _residual(p.n, cout, odt, 100 + key) if resid else None
    m, _ = gpu_map(sc, p.coords, p.res)
    out = sc.sc_forward_ex(m, to_dev(p.feats, tin), to_dev(p.weight, tin), to_dev(p.bias),
                           residual=None if r is None else to_dev(r, tout), act=act,
                           out_dtype=tout)
    sc.sc_device_status(m)
    got = out.float().cpu().numpy().astype(np.float64)
    m.free()
    acts = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "silu": oracle.ACT_SILU}
    ref = oracle.epilogue(_oracle_conv_full(key), acts[act], r)
    check_epilogue_out(got, ref, odt, p.config.dtype, "config %d %s resid=%s %s" % (
        key, act, resid, odt))


@pytest.mark.parametrize("act,odt", [("none", "f32"), ("silu", "bf16"), ("relu", "f32"),
                                     ("none", "f16")])
def test_fused_epilogue_split_shapes(sc, act, odt):
    """64^3, C=256: with act none and fp32 output the last partial round of
    tiles is split and its parts add the residual in the last part; an
    activation or bf16 output runs unsplit."""
    p = synth.make_problem(3)
    cout = p.weight.shape[2]
    tout = TORCH_DT[odt]
    r = _residual(p.n, cout, odt, 7)
    m, nbr = gpu_map(sc, p.coords, p.res)
    want = oracle.build_neighbor_table(p.coords, p.res)
    np.testing.assert_array_equal(nbr, want)
    out = sc.sc_forward_ex(m, to_dev(p.feats, torch.bfloat16), to_dev(p.weight, torch.bfloat16),
                           to_dev(p.bias), residual=to_dev(r, tout), act=act, out_dtype=tout)
    sc.sc_device_status(m)
    got = out.float().cpu().numpy().astype(np.float64)
    m.free()
    rng = np.random.default_rng(33)
    rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(p.n - 2000, p.n),
                                     rng.choice(p.n, size=2000, replace=False)]))
    acts = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "silu": oracle.ACT_SILU}
    ref = oracle.epilogue(oracle.conv(want[rows], p.feats, p.weight, p.bias), acts[act], r[rows])
    check_epilogue_out(got[rows], ref, odt, "bf16", "split %s %s" % (act, odt))


@pytest.mark.parametrize("cin,cout", [(32, 32), (16, 16), (128, 32), (128, 128), (256, 64)])
@pytest.mark.parametrize("act,odt,resid", [("silu", "bf16", True), ("relu", "f32", True),
                                           ("none", "f16", False)])
def test_fused_epilogue_stage_shapes(sc, cin, cout, act, odt, resid):
    """The fused epilogue on every stage layout: N = 32 outputs (cout <= 32),
    several offsets per stage (cin <= 64), two 64-channel blocks of one
    offset per stage (cin a multiple of 128, cout <= 128, with and without the
    CTA-pair W multicast), against the oracle's map and convolution."""
    rng = np.random.default_rng(cin * 7 + cout)
    coords = random_coords(rng, 2, 14, 0.25)          # ~1370 rows: 11 tiles, ragged tail
    feats, weight, bias = synth.make_tensors(len(coords), cin, cout, "bf16", cin + cout + 5)
    tout = TORCH_DT[odt]
    r = _residual(len(coords), cout, odt, cin + cout) if resid else None
    m, nbr = gpu_map(sc, coords, 14)
    want = oracle.build_neighbor_table(coords, 14)
    np.testing.assert_array_equal(nbr, want)
    out = sc.sc_forward_ex(m, to_dev(feats, torch.bfloat16), to_dev(weight, torch.bfloat16),
                           to_dev(bias), residual=None if r is None else to_dev(r, tout),
                           act=act, out_dtype=tout)
    sc.sc_device_status(m)
    got = out.float().cpu().numpy().astype(np.float64)
    m.free()
    acts = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "silu": oracle.ACT_SILU}
    ref = oracle.epilogue(oracle.conv(want, feats, weight, bias), acts[act], r)
    check_epilogue_out(got, ref, odt, "bf16", "%dx%d %s %s" % (cin, cout, act, odt))


@pytest.mark.parametrize("odt", ["f32", "bf16"])
def test_in_place_residual(sc, odt):
    """residual == out (an in-place skip connection) at 64^3, C=256, whose
    last partial round of tiles is split when the output is fp32 and there is
    no activation: the library runs it unsplit, so every row reads its
    residual before writing it.  Compared on the first tile, the last 2,000
    rows (the split tail) and 2,000 random rows."""
    p = synth.make_problem(3)
    cout = p.weight.shape[2]
    tout = TORCH_DT[odt]
    r = _residual(p.n, cout, odt, 8)
    m, _ = gpu_map(sc, p.coords, p.res)
    buf = to_dev(r, tout)
    got_t = sc.sc_forward_ex(m, to_dev(p.feats, torch.bfloat16), to_dev(p.weight, torch.bfloat16),
                             to_dev(p.bias), residual=buf, act="none", out_dtype=tout, out=buf)
    assert got_t.data_ptr() == buf.data_ptr()
    sc.sc_device_status(m)
    got = buf.float().cpu().numpy().astype(np.float64)
    m.free()
    rng = np.random.default_rng(34)
    rows = np.unique(np.concatenate([np.arange(0, 128), np.arange(p.n - 2000, p.n),
                                     rng.choice(p.n, size=2000, replace=False)]))
    want = oracle.build_neighbor_table(p.coords, p.res)
    ref = oracle.epilogue(oracle.conv(want[rows], p.feats, p.weight, p.bias), oracle.ACT_NONE,
                          r[rows])
    check_epilogue_out(got[rows], ref, odt, "bf16", "in place %s" % odt)


def test_forward_ex_rejects_bad_epilogue_arguments(sc):
    import ctypes
    p = synth.make_problem(1)
    m, _ = gpu_map(sc, p.coords, p.res)
    f = to_dev(p.feats)
    w = to_dev(p.weight)
    out = torch.empty((p.n, p.weight.shape[2]), device="cuda")
    lib = sc.load_library()
    P = ctypes.c_void_p
    args = (P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None, None, P(out.data_ptr()),
            f.shape[1], out.shape[1], sc.SC_F32)
    assert lib.sc_forward_ex(*args, 7, sc.SC_F32, None) == sc.SC_ERR_INVALID_ARG
    assert lib.sc_forward_ex(*args, sc.SC_ACT_RELU, 5, None) == sc.SC_ERR_INVALID_ARG
    misaligned = P(out.data_ptr() + 4)
    assert lib.sc_forward_ex(P(m.ptr), P(f.data_ptr()), P(w.data_ptr()), None, misaligned,
                             P(out.data_ptr()), f.shape[1], out.shape[1], sc.SC_F32,
                             sc.SC_ACT_NONE, sc.SC_F32, None) == sc.SC_ERR_INVALID_ARG
    m.free()


def test_decoder_scale_config(sc):
    """1024^3, 3.26M voxels, C=64 fp16 (the decoder-scale workload): the whole
    neighbour map bit-exact, outputs on sampled rows (first tile, ragged last
    tile, 3,000 random rows) within the half-precision bars."""
    scm = sc
    p = synth.make_problem(6)
    m, nbr = gpu_map(scm, p.coords, p.res)
    want = oracle.build_neighbor_table(p.coords, p.res)
    np.testing.assert_array_equal(nbr, want)
    assert scm.sc_map_pairs(m) == int((want >= 0).sum())
    out = scm.sc_forward(m, to_dev(p.feats, torch.float16), to_dev(p.weight, torch.float16),
                         to_dev(p.bias))
    scm.sc_device_status(m)
    rng = np.random.default_rng(66)
    rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(p.n - 300, p.n),
                                     rng.choice(p.n, size=3000, replace=False)]))
    got = out[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    m.free()
    ref = oracle.conv(want[rows], p.feats, p.weight, p.bias)
    assert_close(got, ref, "f16", "config 6")


def test_release_cached_memory_then_rebuild(sc):
    """Trimming the library's pool after a map is freed (and its stream has
    run the free) leaves later builds working."""
    p = synth.make_problem(2)
    m, nbr = gpu_map(sc, p.coords, p.res)
    m.free()
    torch.cuda.synchronize()
    sc.sc_release_cached_memory()
    m2, nbr2 = gpu_map(sc, p.coords, p.res)
    np.testing.assert_array_equal(nbr, nbr2)
    m2.free()


# ---------------------------------------------------------------------------
# rows ordered by neighbour mask (sc_map_order_rows): the same results, every
# output in its own row

@pytest.mark.parametrize("key", [1, 2, 3, 4, 5])
def test_ordered_rows_match_oracle(sc, key):
    p = synth.make_problem(key)
    m, nbr = gpu_map(sc, p.coords, p.res)
    want = oracle.build_neighbor_table(p.coords, p.res)
    np.testing.assert_array_equal(nbr, want)
    sc.sc_map_order_rows(m)
    # the neighbour table the caller sees is unchanged
    np.testing.assert_array_equal(sc.sc_get_neighbor_table(m).cpu().numpy(), want)
    got = gpu_conv(sc, m, p.feats, p.weight, p.bias, p.config.dtype)
    m.free()
    rows = None
    if key in (3, 4):
        rng = np.random.default_rng(70 + key)
        rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(p.n - 300, p.n),
                                         rng.choice(p.n, size=3000, replace=False)]))
    if rows is None:
        assert_close(got, oracle.conv(want, p.feats, p.weight, p.bias), p.config.dtype,
                     "ordered config %d" % key)
    else:
        assert_close(got[rows], oracle.conv(want[rows], p.feats, p.weight, p.bias),
                     p.config.dtype, "ordered config %d" % key)


@pytest.mark.parametrize("act,odt,inplace", [("none", "f32", False), ("silu", "bf16", False),
                                             ("none", "f32", True)])
def test_ordered_rows_fused_epilogue(sc, act, odt, inplace):
    """64^3, C=256 over ordered rows: the split tail (zeroed through the row
    indirection), a fused SiLU with bf16 output, and an in-place residual."""
    p = synth.make_problem(3)
    cout = p.weight.shape[2]
    tout = TORCH_DT[odt]
    r = _residual(p.n, cout, odt, 9)
    m, _ = gpu_map(sc, p.coords, p.res)
    sc.sc_map_order_rows(m)
    rbuf = to_dev(r, tout)
    out = sc.sc_forward_ex(m, to_dev(p.feats, torch.bfloat16), to_dev(p.weight, torch.bfloat16),
                           to_dev(p.bias), residual=rbuf, act=act, out_dtype=tout,
                           out=rbuf if inplace else None)
    sc.sc_device_status(m)
    got = out.float().cpu().numpy().astype(np.float64)
    m.free()
    rng = np.random.default_rng(35)
    rows = np.unique(np.concatenate([np.arange(0, 256), np.arange(p.n - 2000, p.n),
                                     rng.choice(p.n, size=2000, replace=False)]))
    want = oracle.build_neighbor_table(p.coords, p.res)
    acts = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "silu": oracle.ACT_SILU}
    ref = oracle.epilogue(oracle.conv(want[rows], p.feats, p.weight, p.bias), acts[act], r[rows])
    check_epilogue_out(got[rows], ref, odt, "bf16", "ordered %s %s inplace=%s" % (act, odt,
                                                                                  inplace))


def test_ordered_rows_deterministic_and_shuffled(sc):
    """Shuffled input rows, ordered map, deterministic mode: repeated forwards
    are bit-identical and equal the oracle's within the bars."""
    p = synth.make_problem(2)
    perm = np.random.default_rng(12).permutation(p.n)
    c, f = np.ascontiguousarray(p.coords[perm]), np.ascontiguousarray(p.feats[perm])
    m, _ = gpu_map(sc, c, p.res)
    sc.sc_map_order_rows(m)
    sc.sc_map_order_rows(m)            # a second call keeps the order
    sc.sc_set_deterministic(True)
    try:
        a = gpu_conv(sc, m, f, p.weight, p.bias, "bf16")
        b = gpu_conv(sc, m, f, p.weight, p.bias, "bf16")
    finally:
        sc.sc_set_deterministic(False)
    m.free()
    np.testing.assert_array_equal(a, b)
    assert_close(a, oracle.conv(oracle.build_neighbor_table(c, p.res), f, p.weight, p.bias),
                 "bf16", "ordered shuffled")
