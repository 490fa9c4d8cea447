"""GPU parity of the level changes against oracle/levels.py, through the C ABI.

Subdivision, Channel2Spatial and the way down (parents, child table, each
voxel's parent) must match the oracle bit for bit; the 2x2x2 stride-2
convolutions (down, and its transpose up) must meet the convolution bars
against the oracle's fp64 result over the ORACLE's maps.  The readings are
those of the trellis2mlx README's "Upsample" stage and Channel2Spatial
decoder (the oracle module's docstring states them).
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import levels
from sparse_voxel_convolution_coord_b300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "levels",
                      "one_voxel_three_children.json")
TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def sc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_voxel_convolution_coord_b300 as m
    from sparse_voxel_convolution_coord_b300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(dtype) if dtype is not None else t


def host(t):
    return t.cpu().numpy()


def random_coords(rng, batches, res, density):
    rows = []
    for b in batches:
        xyz = np.argwhere(rng.random((res, res, res)) < density)
        rows.append(np.concatenate([np.full((len(xyz), 1), b), xyz], axis=1))
    return np.ascontiguousarray(np.concatenate(rows), dtype=np.int32)


def assert_bars(got, ref, dtype, what):
    err = got - ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    if dtype == "f32":
        assert rel <= 1e-5, "%s rel L2 %.3e" % (what, rel)
    else:
        rms = np.linalg.norm(ref) / np.sqrt(ref.size)
        assert rel <= 2e-3, "%s rel L2 %.3e" % (what, rel)
        assert np.abs(err).max() <= 1e-2 * rms, "%s max abs over 1e-2 rms" % what


# ---------------------------------------------------------------------------
# subdivision and Channel2Spatial

def oracle_child_of(n, parent, offset):
    t = np.full((n, 8), -1, np.int64)
    t[parent, offset] = np.arange(len(parent))
    return t


@pytest.mark.parametrize("case", ["masks", "all", "none_selected", "shuffled_batches"])
def test_subdivide_bit_exact(sc, case):
    rng = np.random.default_rng(41)
    c = random_coords(rng, [0, 2, 5], 12, 0.2)
    if case == "shuffled_batches":
        c = np.ascontiguousarray(c[rng.permutation(len(c))])
    mask = None
    if case == "masks" or case == "shuffled_batches":
        mask = rng.integers(0, 256, len(c)).astype(np.uint8)
    elif case == "none_selected":
        mask = np.zeros(len(c), np.uint8)
    child, parent, offset, child_of = sc.sc_subdivide(dev(c), 12,
                                                      None if mask is None else dev(mask))
    wc, wp, wo = levels.subdivide(c, mask)
    np.testing.assert_array_equal(host(child), wc)
    np.testing.assert_array_equal(host(parent), wp)
    np.testing.assert_array_equal(host(offset), wo)
    np.testing.assert_array_equal(host(child_of), oracle_child_of(len(c), wp, wo))


def test_subdivide_rejects_out_of_range(sc):
    with pytest.raises(sc.ScError) as e:
        sc.sc_subdivide(dev(np.array([[0, 1, 1, 1], [0, 8, 0, 0]], np.int32)), 8)
    assert e.value.code == sc.SC_ERR_COORD_RANGE


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
def test_channel_to_spatial_bit_exact(sc, dtype):
    rng = np.random.default_rng(43)
    c = random_coords(rng, [0, 1], 10, 0.2)
    mask = rng.integers(0, 256, len(c)).astype(np.uint8)
    C = 24
    f = rng.standard_normal((len(c), 8 * C)).astype(np.float32)
    ft = dev(f, TORCH_DT[dtype])
    f_exact = ft.float().cpu().numpy()          # the values as stored in dtype
    _, parent, offset, _ = sc.sc_subdivide(dev(c), 10, dev(mask))
    got = sc.sc_channel_to_spatial(ft, parent, offset)
    _, wp, wo = levels.subdivide(c, mask)
    want = levels.channel_to_spatial(f_exact, wp, wo)
    np.testing.assert_array_equal(got.float().cpu().numpy(), want)


def test_golden_one_voxel_three_children(sc):
    g = json.load(open(GOLDEN))
    coords = np.array(g["coords"], np.int32)
    child, parent, offset, _ = sc.sc_subdivide(dev(coords), 4,
                                               dev(np.array(g["mask"], np.uint8)))
    assert host(child).tolist() == g["children"]
    assert host(parent).tolist() == g["parent"] and host(offset).tolist() == g["offset"]
    feats = np.arange(16, dtype=np.float32).reshape(1, 16)
    c2s = sc.sc_channel_to_spatial(dev(feats), parent, offset)
    assert host(c2s).tolist() == g["c2s_out"]
    lm = sc.sc_build_level_map(child, 8)
    pc, co, po = sc.sc_get_level_map(lm)
    assert host(pc).tolist() == g["parents_down"] and host(co).tolist() == g["child_of"]
    w = np.stack([(o + 1) * np.eye(2, dtype=np.float32) for o in range(8)])
    bias = np.array(g["bias"], np.float32)
    upo = sc.sc_conv_up(lm, dev(np.array(g["parent_feats"], np.float32)), dev(w), dev(bias))
    dno = sc.sc_conv_down(lm, dev(np.array(g["child_feats"], np.float32)), dev(w), dev(bias))
    sc.sc_level_device_status(lm)
    assert host(upo).tolist() == g["up_out"]
    assert host(dno).tolist() == g["down_out"]
    lm.free()


# ---------------------------------------------------------------------------
# the way down

def check_level_map(sc, c, res, nbatch=None):
    nb = int(c[:, 0].max()) + 1 if nbatch is None else nbatch
    lm = sc.sc_build_level_map(dev(c), res, nb)
    pc, co, po = sc.sc_get_level_map(lm)
    wpc, wco, wpo = levels.downsample_map(c)
    assert lm.parents == len(wpc)
    np.testing.assert_array_equal(host(pc), wpc)
    np.testing.assert_array_equal(host(co), wco)
    np.testing.assert_array_equal(host(po), wpo)
    return lm, wco, wpo


@pytest.mark.parametrize("case", ["config2", "config5", "shuffled", "batches_res13",
                                  "single", "res1"])
def test_level_map_bit_exact(sc, case):
    rng = np.random.default_rng(47)
    if case in ("config2", "config5"):
        p = synth.make_problem(2 if case == "config2" else 5)
        c, res = p.coords, p.res
    elif case == "shuffled":
        p = synth.make_problem(3)
        c, res = np.ascontiguousarray(p.coords[rng.permutation(p.n)]), p.res
    elif case == "batches_res13":          # odd resolution: parents at ceil(13/2) = 7
        c, res = random_coords(rng, [0, 3, 4], 13, 0.15), 13
        c = np.ascontiguousarray(c[rng.permutation(len(c))])
    elif case == "single":
        c, res = np.array([[2, 5, 0, 7]], np.int32), 8
    else:
        c, res = np.array([[b, 0, 0, 0] for b in range(4)], np.int32), 1
    lm, _, _ = check_level_map(sc, c, res)
    lm.free()


def test_level_map_wide_keys(sc):
    """nbatch * (res/2)^3 beyond 2^32: 64-bit parent keys (more sort passes)."""
    rng = np.random.default_rng(48)
    c = random_coords(rng, [0, 40000], 32, 0.02)
    c[:, 1:] *= 31                           # spread over a 1024^3 grid
    c = np.ascontiguousarray(np.unique(c, axis=0)[rng.permutation(len(np.unique(c, axis=0)))])
    lm, _, _ = check_level_map(sc, c.astype(np.int32), 1024, nbatch=40001)
    lm.free()


@pytest.mark.parametrize("coords,res,nbatch,code", [
    ([[0, 1, 1, 1], [0, 1, 1, 1]], 8, 1, 3),       # duplicate
    ([[0, 1, 1, 1], [0, 8, 1, 1]], 8, 1, 2),       # x == res
    ([[0, 1, 1, 1], [2, 1, 1, 1]], 8, 2, 2),       # batch >= nbatch
    ([[-1, 1, 1, 1]], 8, 1, 2),                    # negative batch
])
def test_level_map_errors(sc, coords, res, nbatch, code):
    with pytest.raises(sc.ScError) as e:
        sc.sc_build_level_map(dev(np.array(coords, np.int32)), res, nbatch)
    assert e.value.code == code


# ---------------------------------------------------------------------------
# stride-2 convolutions

def octants(c):
    return (c[:, 1] & 1) * 4 + (c[:, 2] & 1) * 2 + (c[:, 3] & 1)


@pytest.mark.parametrize("dtype,cin,cout", [("bf16", 64, 64), ("bf16", 32, 128),
                                            ("bf16", 128, 256), ("f16", 64, 32),
                                            ("f32", 32, 32), ("f32", 24, 40)])
def test_stride2_convs(sc, dtype, cin, cout):
    rng = np.random.default_rng(cin * 7 + cout)
    c = random_coords(rng, [0, 1], 24, 0.12)      # ~3.3k fine voxels, ragged tiles
    c = np.ascontiguousarray(c[rng.permutation(len(c))])
    lm, wco, wpo = check_level_map(sc, c, 24)
    P = lm.parents
    f_fine = synth.make_tensors(len(c), cin, cout, dtype, 5)[0]
    f_par = synth.make_tensors(P, cin, cout, dtype, 6)[0]
    w = (rng.standard_normal((8, cin, cout)) / np.sqrt(8 * cin)).astype(np.float32)
    if dtype != "f32":
        w = torch.from_numpy(w).to(TORCH_DT[dtype]).float().numpy()
    bias = (0.1 * rng.standard_normal(cout)).astype(np.float32)
    tdt = TORCH_DT[dtype]
    down = sc.sc_conv_down(lm, dev(f_fine, tdt), dev(w, tdt), dev(bias))
    up = sc.sc_conv_up(lm, dev(f_par, tdt), dev(w, tdt), dev(bias))
    sc.sc_level_device_status(lm)
    lm.free()
    want_down = levels.conv_down(wco, f_fine, w, bias)
    want_up = levels.conv_up(wpo, octants(c), f_par, w, bias)
    assert_bars(host(down).astype(np.float64), want_down, dtype, "down %s" % dtype)
    assert_bars(host(up).astype(np.float64), want_up, dtype, "up %s" % dtype)


def test_stride2_convs_fused_epilogue_and_scale(sc):
    """256^3, ~400k fine voxels, C=32 bf16, SiLU + residual + bf16 output:
    sampled rows (the first tile, the ragged tail, 3,000 random rows)."""
    p = synth.make_problem(5)
    lm = sc.sc_build_level_map(dev(p.coords), p.res, 1)
    wpc, wco, wpo = levels.downsample_map(p.coords)
    P = lm.parents
    assert P == len(wpc)
    rng = np.random.default_rng(51)
    w = torch.from_numpy((rng.standard_normal((8, 32, 32)) / 16).astype(np.float32)).to(
        torch.bfloat16)
    f_par = torch.from_numpy(rng.standard_normal((P, 32)).astype(np.float32)).to(torch.bfloat16)
    resid = torch.from_numpy(rng.standard_normal((p.n, 32)).astype(np.float32)).to(torch.bfloat16)
    bias = (0.1 * rng.standard_normal(32)).astype(np.float32)
    up = sc.sc_conv_up(lm, f_par.cuda(), w.cuda(), dev(bias), residual=resid.cuda(), act="silu",
                       out_dtype=torch.bfloat16)
    down = sc.sc_conv_down(lm, dev(p.feats, torch.bfloat16), w.cuda(), dev(bias))
    sc.sc_level_device_status(lm)
    lm.free()
    rows = np.unique(np.concatenate([np.arange(128), np.arange(p.n - 300, p.n),
                                     rng.choice(p.n, 3000, replace=False)]))
    ref = levels.conv_up(wpo[rows], octants(p.coords)[rows], f_par.float().numpy(),
                         w.float().numpy(), bias)
    ref = oracle.round_bf16(oracle.epilogue(ref, oracle.ACT_SILU, resid.float().numpy()[rows]))
    got = up.float().cpu().numpy()[rows].astype(np.float64)
    spacing = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(got - ref) <= spacing + 1e-4)
    prow = np.unique(np.concatenate([np.arange(128), np.arange(P - 100, P),
                                     rng.choice(P, 2000, replace=False)]))
    want_down = levels.conv_down(wco[prow], p.feats, w.float().numpy(), bias)
    assert_bars(down.cpu().numpy()[prow].astype(np.float64), want_down, "bf16", "down 400k")
