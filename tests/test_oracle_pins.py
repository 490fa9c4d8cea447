"""Pins for the CPU oracle, checked without going through the oracle itself.

Each check holds for any correct implementation of the 3x3x3 submanifold
sparse convolution ("Running TRELLIS.2 on a Mac (1/3)", Sparse 3D convolution
paragraph; "Porting TRELLIS.2 From Python to Rust and Metal", section V;
"FABLE_STARTUP_PACKET.md" section 5 for the weight layout):

* neighbour maps against brute-force pairwise search and a dense index volume;
* the closed form sum_k |pairs_k| = (3L-2)^3 for a full L^3 cube, and
  (L-|dx|)(L-|dy|)(L-|dz|) per offset;
* map symmetry nbr[o][k] = i <=> nbr[i][26-k] = o, and nbr[o][13] = o;
* convolution against a dense fp64 Conv3d (padding 1, inactive inputs zero,
  compared at active sites only): a library routine, not this code;
* hand-worked examples under tests/golden/;
* identity centre tap, isolated voxel, permutation equivariance, translation
  invariance and batch independence.

``test_planted_mistakes_are_caught`` compiles mutated copies of the oracle
(a swapped axis, a flipped displacement, a transposed weight, a dropped bias,
a lost border neighbour, an ignored batch index) and checks that at least one
pin fails for each: the pins are sharp enough to catch such slips.
"""
import json
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle import build_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# independent routes (none calls the oracle)

def all_displacements():
    return [(dx, dy, dz) for dx in (-1, 0, 1) for dy in (-1, 0, 1) for dz in (-1, 0, 1)]


def brute_force_table(coords, res):
    """O(N^2) neighbour search: compare every pair of rows."""
    n = len(coords)
    nbr = -np.ones((n, 27), np.int32)
    c = coords.astype(np.int64)
    for o in range(n):
        d = c[:, 1:] - c[o, 1:]                       # displacement of every row
        same_b = c[:, 0] == c[o, 0]
        near = same_b & (np.abs(d).max(axis=1) <= 1)
        for i in np.flatnonzero(near):
            dx, dy, dz = d[i]
            nbr[o, 9 * (dx + 1) + 3 * (dy + 1) + (dz + 1)] = i
    return nbr


def dense_volume_table(coords, res):
    """Dense index volume [B, res+2, res+2, res+2] with a -1 border."""
    nb = int(coords[:, 0].max()) + 1 if len(coords) else 1
    vol = -np.ones((nb, res + 2, res + 2, res + 2), np.int64)
    b, x, y, z = (coords[:, i].astype(np.int64) for i in range(4))
    vol[b, x + 1, y + 1, z + 1] = np.arange(len(coords))
    cols = []
    for dx, dy, dz in all_displacements():
        cols.append(vol[b, x + 1 + dx, y + 1 + dy, z + 1 + dz])
    return np.stack(cols, axis=1).astype(np.int32) if len(coords) else \
        np.zeros((0, 27), np.int32)


def dense_conv3d(coords, res, feats, weight, bias):
    """Dense fp64 Conv3d with padding 1 over the occupancy grids, read at the
    active sites.  W_dense[co, ci, kd, kh, kw] = weight[9kd + 3kh + kw, ci, co]."""
    nb = int(coords[:, 0].max()) + 1
    cin, cout = weight.shape[1], weight.shape[2]
    vol = torch.zeros((nb, cin, res, res, res), dtype=torch.float64)
    cb = torch.from_numpy(coords.astype(np.int64))
    vol[cb[:, 0], :, cb[:, 1], cb[:, 2], cb[:, 3]] = torch.from_numpy(feats.astype(np.float64))
    wd = torch.from_numpy(weight.astype(np.float64)).reshape(3, 3, 3, cin, cout)
    wd = wd.permute(4, 3, 0, 1, 2).contiguous()       # (co, ci, kd, kh, kw)
    b = None if bias is None else torch.from_numpy(bias.astype(np.float64))
    out = torch.nn.functional.conv3d(vol, wd, b, padding=1)
    return out[cb[:, 0], :, cb[:, 1], cb[:, 2], cb[:, 3]].numpy()


def random_coords(rng, n_batches, res, density):
    rows = []
    for b in range(n_batches):
        occ = rng.random((res, res, res)) < density
        xyz = np.argwhere(occ)
        rows.append(np.concatenate([np.full((len(xyz), 1), b), xyz], axis=1))
    c = np.concatenate(rows).astype(np.int32)
    return c[rng.permutation(len(c))]


def random_tensors(rng, n, cin, cout):
    feats = rng.standard_normal((n, cin)).astype(np.float32)
    weight = rng.standard_normal((27, cin, cout)).astype(np.float32)
    bias = rng.standard_normal(cout).astype(np.float32)
    return feats, weight, bias


# ----------------------------------------------------------------------------
# pin checks, parameterised by the oracle build under test

def check_displacements(orc):
    ds = [orc.displacement(k) for k in range(27)]
    assert sorted(ds) == sorted(all_displacements())
    assert ds[13] == (0, 0, 0)
    for k in range(27):
        assert ds[26 - k] == tuple(-v for v in ds[k])
    # the row-major flattening of (Kd, Kh, Kw) with Kd along x
    assert ds == all_displacements()


def check_maps(orc):
    rng = np.random.default_rng(7)
    for res, nbatch, dens in [(1, 2, 1.0), (2, 1, 0.6), (4, 3, 0.35), (6, 2, 0.25), (9, 1, 0.12)]:
        coords = random_coords(rng, nbatch, res, dens)
        got = orc.build_neighbor_table(coords, res)
        np.testing.assert_array_equal(got, brute_force_table(coords, res))
        np.testing.assert_array_equal(got, dense_volume_table(coords, res))


def check_full_cube(orc):
    for L in range(1, 7):
        xyz = np.argwhere(np.ones((L, L, L), bool))
        coords = np.concatenate([np.zeros((len(xyz), 1)), xyz], axis=1).astype(np.int32)
        nbr = orc.build_neighbor_table(coords, L)
        assert int((nbr >= 0).sum()) == (3 * L - 2) ** 3
        for k, (dx, dy, dz) in enumerate(all_displacements()):
            assert int((nbr[:, k] >= 0).sum()) == (L - abs(dx)) * (L - abs(dy)) * (L - abs(dz))


def check_symmetry(orc):
    rng = np.random.default_rng(11)
    coords = random_coords(rng, 2, 8, 0.3)
    nbr = orc.build_neighbor_table(coords, 8)
    n = len(coords)
    assert np.array_equal(nbr[:, 13], np.arange(n))
    o_idx, k_idx = np.nonzero(nbr >= 0)
    i_idx = nbr[o_idx, k_idx]
    assert np.array_equal(nbr[i_idx, 26 - k_idx], o_idx)


def check_golden(orc):
    for name in sorted(os.listdir(GOLDEN)):
        if not name.endswith(".json"):
            continue
        g = json.load(open(os.path.join(GOLDEN, name)))
        coords = np.array(g["coords"], np.int32)
        cin, cout = g["cin"], g["cout"]
        weight = np.zeros((27, cin, cout), np.float32)
        for k in range(27):
            if g["weight_rule"] == "W[k][0][0] = k + 1":
                weight[k, 0, 0] = k + 1
            elif g["weight_rule"] == "W[k] = [[k+1, 1], [0, 2*(k+1)]]":
                weight[k] = [[k + 1, 1], [0, 2 * (k + 1)]]
            else:
                raise AssertionError("unknown weight rule " + g["weight_rule"])
        nbr = orc.build_neighbor_table(coords, g["res"])
        want = -np.ones_like(nbr)
        for o, present in enumerate(g["nbr_present"]):
            for k, i in present:
                want[o, k] = i
        np.testing.assert_array_equal(nbr, want, err_msg=name)
        out = orc.conv(nbr, np.array(g["feats"], np.float32), weight,
                       np.array(g["bias"], np.float32))
        np.testing.assert_array_equal(out, np.array(g["out"]), err_msg=name)


def check_dense_conv(orc):
    rng = np.random.default_rng(5)
    for res, nbatch, dens, cin, cout in [(4, 1, 0.5, 3, 3), (5, 2, 0.3, 4, 6),
                                         (7, 2, 0.2, 5, 5), (6, 1, 0.9, 2, 3)]:
        coords = random_coords(rng, nbatch, res, dens)
        feats, weight, bias = random_tensors(rng, len(coords), cin, cout)
        got = orc.sparse_conv(coords, res, feats, weight, bias)
        want = dense_conv3d(coords, res, feats, weight, bias)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def check_invariants(orc):
    rng = np.random.default_rng(9)
    res, cin = 8, 6
    coords = random_coords(rng, 2, res, 0.3)
    n = len(coords)
    feats, weight, bias = random_tensors(rng, n, cin, cin)
    # identity centre tap returns the input exactly
    w_id = np.zeros((27, cin, cin), np.float32)
    w_id[13] = np.eye(cin)
    np.testing.assert_array_equal(orc.sparse_conv(coords, res, feats, w_id), feats)
    # an isolated voxel gives x W[13] + b
    iso = np.array([[0, 3, 3, 3], [0, 6, 6, 6]], np.int32)
    out = orc.sparse_conv(iso, res, feats[:2], weight, bias)
    want = feats[:2].astype(np.float64) @ weight[13].astype(np.float64) + bias
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-13)
    base = orc.sparse_conv(coords, res, feats, weight, bias)
    # permutation equivariance
    perm = rng.permutation(n)
    outp = orc.sparse_conv(coords[perm], res, feats[perm], weight, bias)
    np.testing.assert_allclose(outp, base[perm], rtol=1e-13, atol=1e-13)
    # translation invariance (inside the grid, so no neighbour is cut off)
    small = coords[(coords[:, 1:] < res - 2).all(axis=1)]
    idx = np.flatnonzero((coords[:, 1:] < res - 2).all(axis=1))
    sub_f = feats[idx]
    out0 = orc.sparse_conv(small, res, sub_f, weight, bias)
    shifted = small.copy()
    shifted[:, 1:] += np.array([2, 1, 2], np.int32)
    out1 = orc.sparse_conv(shifted, res, sub_f, weight, bias)
    np.testing.assert_allclose(out1, out0, rtol=1e-13, atol=1e-13)
    # batch independence: each batch element alone gives the same rows
    for b in range(2):
        rows = np.flatnonzero(coords[:, 0] == b)
        alone = coords[rows].copy()
        alone[:, 0] = 0
        outb = orc.sparse_conv(alone, res, feats[rows], weight, bias)
        np.testing.assert_allclose(outb, base[rows], rtol=1e-13, atol=1e-13)


ALL_CHECKS = [check_displacements, check_maps, check_full_cube, check_symmetry,
              check_golden, check_dense_conv, check_invariants]


# ----------------------------------------------------------------------------
# the pins, on the committed oracle

@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.default())


def test_errors():
    orc = oracle.default()
    with pytest.raises(oracle.OracleError) as e:
        orc.build_neighbor_table(np.array([[0, 0, 0, 4]], np.int32), 4)
    assert e.value.code == oracle.COORD_RANGE
    with pytest.raises(oracle.OracleError) as e:
        orc.build_neighbor_table(np.array([[-1, 0, 0, 0]], np.int32), 4)
    assert e.value.code == oracle.COORD_RANGE
    with pytest.raises(oracle.OracleError) as e:
        orc.build_neighbor_table(np.array([[0, 1, 2, 3], [0, 1, 2, 3]], np.int32), 4)
    assert e.value.code == oracle.DUPLICATE
    # a range error is reported in preference to a duplicate
    with pytest.raises(oracle.OracleError) as e:
        orc.build_neighbor_table(np.array([[0, 1, 2, 3], [0, 1, 2, 3], [0, 0, -1, 0]],
                                          np.int32), 4)
    assert e.value.code == oracle.COORD_RANGE
    assert orc.build_neighbor_table(np.zeros((0, 4), np.int32), 4).shape == (0, 27)


def test_pairs_follow_table():
    orc = oracle.default()
    rng = np.random.default_rng(3)
    coords = random_coords(rng, 2, 7, 0.3)
    nbr = orc.build_neighbor_table(coords, 7)
    off, pin, pout = orc.pairs(nbr)
    assert off[0] == 0 and off[27] == (nbr >= 0).sum() == len(pin) == len(pout)
    for k in range(27):
        o = pout[off[k]:off[k + 1]]
        assert np.all(np.diff(o) > 0)                            # ascending output row
        np.testing.assert_array_equal(o, np.flatnonzero(nbr[:, k] >= 0))
        np.testing.assert_array_equal(pin[off[k]:off[k + 1]], nbr[o, k])
        assert off[k + 1] - off[k] == off[27 - k] - off[26 - k]  # |pairs_k| = |pairs_{26-k}|


def test_row_subset():
    orc = oracle.default()
    rng = np.random.default_rng(4)
    coords = random_coords(rng, 1, 6, 0.4)
    feats, weight, bias = random_tensors(rng, len(coords), 3, 4)
    nbr = orc.build_neighbor_table(coords, 6)
    full = orc.conv(nbr, feats, weight, bias)
    rows = np.array([5, 0, len(coords) - 1])
    np.testing.assert_array_equal(orc.conv(nbr[rows], feats, weight, bias), full[rows])


# ----------------------------------------------------------------------------
# planted mistakes: each mutated oracle must fail at least one pin

MUTATIONS = {
    "swap_x_and_z_taps": [("*dx = k / 9 - 1;", "*dx = k % 3 - 1;"),
                          ("*dz = k % 3 - 1;", "*dz = k / 9 - 1;")],
    "convolution_not_correlation": [("(int64_t)c[1] + dx", "(int64_t)c[1] - dx"),
                                    ("(int64_t)c[2] + dy", "(int64_t)c[2] - dy"),
                                    ("(int64_t)c[3] + dz", "(int64_t)c[3] - dz")],
    "transposed_weight": [("acc[c] += xv * (double)wrow[c];",
                           "acc[c] += xv * (double)wk[(int64_t)c * cin + ci];")],
    "dropped_bias": [("acc[c] + (bias ? (double)bias[c] : 0.0)", "acc[c]")],
    "lost_border_neighbour": [("if (x >= 0 && x < res", "if (x >= 1 && x < res")],
    "batch_ignored": [("where.find(VoxelKey{c[0],", "where.find(VoxelKey{0,")],
    "skipped_last_tap": [("for (int k = 0; k < 27; ++k) {\n      int32_t i = nbr",
                          "for (int k = 0; k < 26; ++k) {\n      int32_t i = nbr")],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src = open(build_oracle.SRC).read()
    for old, new in MUTATIONS[name]:
        assert old in src, (name, old)
        src = src.replace(old, new)
    mpath = os.path.join(str(tmp_path), "mutant.cpp")
    open(mpath, "w").write(src)
    mutant = oracle.Oracle(build_oracle.build(force=True, src=mpath,
                                              lib=os.path.join(str(tmp_path), "libmutant.so")))
    failed = []
    for check in ALL_CHECKS:
        try:
            check(mutant)
        except (AssertionError, oracle.OracleError, IndexError):
            failed.append(check.__name__)
    assert failed, "no pin caught the planted mistake %s" % name


# ----------------------------------------------------------------------------
# the fused epilogue ("Porting TRELLIS.2 From Python to Rust and Metal",
# section V): out = act(conv + bias) + residual, rounded once to the output
# type.  Pinned by closed forms, identities of the activations, the rounding
# rule's worked cases, and an independent bf16 conversion (torch's).

def check_activation(act_fn):
    x = np.array([-3.0, -0.5, 0.0, 0.25, 7.0])
    np.testing.assert_array_equal(act_fn(x, oracle.ACT_NONE), x)
    np.testing.assert_array_equal(act_fn(x, oracle.ACT_RELU), [0.0, 0.0, 0.0, 0.25, 7.0])
    s = lambda v: act_fn(np.asarray(v, np.float64), oracle.ACT_SILU)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    np.testing.assert_allclose(s([np.log(3.0), -np.log(3.0)]),
                               [0.75 * np.log(3.0), -0.25 * np.log(3.0)], rtol=1e-15)
    # silu(x) - silu(-x) = x (sigmoid(x) + sigmoid(-x) = 1), silu(0) = 0
    xs = np.linspace(-40.0, 40.0, 161)
    np.testing.assert_allclose(s(xs) - s(-xs), xs, rtol=1e-14, atol=1e-14)
    assert s([0.0])[0] == 0.0
    # limits, with no overflow at large |x|: silu(x) -> x and -> 0
    big = s([800.0, -800.0])
    assert big[0] == 800.0 and big[1] == 0.0


def check_epilogue(epi_fn):
    v = np.array([[-1.0, 2.0, -0.5]])
    r = np.array([[2.0, -1.0, 0.5]])
    # the residual is added after the activation
    np.testing.assert_array_equal(epi_fn(v, oracle.ACT_RELU, r), [[2.0, 1.0, 0.5]])
    np.testing.assert_array_equal(epi_fn(v, oracle.ACT_NONE, r), v + r)
    np.testing.assert_array_equal(epi_fn(v, oracle.ACT_RELU, None), [[0.0, 2.0, 0.0]])


def check_round_bf16(rnd):
    u = 2.0 ** -7  # bf16 spacing in [1, 2)
    cases = {
        1.0 + u / 2: 1.0,                 # tie -> even (mantissa ...0)
        1.0 + 3 * u / 2: 1.0 + 2 * u,     # tie -> even (mantissa ...10)
        1.0 + u / 2 + 2.0 ** -30: 1.0 + u,  # above the tie
        1.0 + u / 2 - 2.0 ** -30: 1.0,    # below the tie
        -(1.0 + 3 * u / 2): -(1.0 + 2 * u),
        3.0: 3.0,
        1.0 / 3.0: float.fromhex("0x1.560p-2"),  # 0.0101010101 -> 8 significant bits
        2.0 ** -130 * 1.3: 10 * 2.0 ** -133,     # below 2^-126 the spacing is 2^-133
        float.fromhex("0x1.ffp127"): np.inf,     # tie past the largest finite -> inf
        0.0: 0.0,
    }
    got = rnd(np.array(list(cases.keys())))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))


def check_round_bf16_against_torch(rnd):
    # fp32-representable values: rounding them directly to bf16 and torch's
    # fp32 -> bf16 conversion (an independent implementation) must agree
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    x = np.concatenate([x, np.float32([1.00390625, 1.01171875, -2.0078125, 65504.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(rnd(x.astype(np.float64)), want)


def check_round_f16(rnd):
    u = 2.0 ** -10  # binary16 spacing in [1, 2)
    cases = {
        1.0 + u / 2: 1.0,                   # tie -> even
        1.0 + 3 * u / 2: 1.0 + 2 * u,       # tie -> even
        1.0 + u / 2 + 2.0 ** -30: 1.0 + u,
        65504.0: 65504.0,                   # largest finite
        65519.0: 65504.0,                   # below the tie with 2^16
        65520.0: np.inf,                    # the tie goes to 2^16: infinity
        2.0 ** -24: 2.0 ** -24,             # smallest subnormal
        2.0 ** -25: 0.0,                    # tie between 0 and 2^-24 -> 0 (even)
        3 * 2.0 ** -26: 2.0 ** -24,
        -(2.0 ** -14) * 1.5: -(2.0 ** -14) * 1.5,
        1.0 / 3.0: float.fromhex("0x1.554p-2"),
    }
    got = rnd(np.array(list(cases.keys())))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))


def check_round_f16_against_numpy(rnd):
    # numpy's float64 -> float16 conversion rounds to nearest even directly
    # (an independent implementation)
    rng = np.random.default_rng(22)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-20, 12, 20000))
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).astype(np.float64)
    np.testing.assert_array_equal(rnd(x), want)


EPILOGUE_CHECKS = [
    lambda a, e, r, h: check_activation(a),
    lambda a, e, r, h: check_epilogue(e),
    lambda a, e, r, h: check_round_bf16(r),
    lambda a, e, r, h: check_round_bf16_against_torch(r),
    lambda a, e, r, h: check_round_f16(h),
    lambda a, e, r, h: check_round_f16_against_numpy(h),
]


def test_epilogue_pins():
    for chk in EPILOGUE_CHECKS:
        chk(oracle.activation, oracle.epilogue, oracle.round_bf16, oracle.round_f16)


def _mutant_round(mode, sig_bits=8, e_min=-125):
    def rnd(v):
        v = np.asarray(v, np.float64)
        out = np.zeros_like(v)
        nz = (v != 0.0) & np.isfinite(v)
        _, e = np.frexp(v[nz])
        step = np.ldexp(1.0, np.maximum(e, e_min) - sig_bits)
        t = v[nz] / step
        if mode == "truncate":
            q = np.trunc(t)
        elif mode == "even":
            q = np.rint(t)
        else:  # ties away from zero
            q = np.sign(t) * np.floor(np.abs(t) + 0.5)
        out[nz] = q * step
        out[~nz] = v[~nz]
        return out
    return rnd


EPILOGUE_MUTANTS = {
    "residual_before_activation": (
        oracle.activation,
        lambda v, act=0, residual=None: oracle.activation(
            np.asarray(v, np.float64) + (0.0 if residual is None else residual), act),
        oracle.round_bf16, oracle.round_f16),
    "silu_sign_slip": (
        lambda v, act: (np.asarray(v, np.float64) / (1.0 + np.exp(np.asarray(v, np.float64)))
                        if act == oracle.ACT_SILU else oracle.activation(v, act)),
        oracle.epilogue, oracle.round_bf16, oracle.round_f16),
    "round_ties_away": (oracle.activation, oracle.epilogue, _mutant_round("away"),
                        oracle.round_f16),
    "round_truncate": (oracle.activation, oracle.epilogue, _mutant_round("truncate"),
                       oracle.round_f16),
    "f16_ties_away": (oracle.activation, oracle.epilogue, oracle.round_bf16,
                      _mutant_round("away", 11, -13)),
    "f16_wrong_subnormal_spacing": (oracle.activation, oracle.epilogue, oracle.round_bf16,
                                    _mutant_round("even", 11, -14)),
}


@pytest.mark.parametrize("name", sorted(EPILOGUE_MUTANTS))
def test_planted_epilogue_mistakes_are_caught(name):
    fns = EPILOGUE_MUTANTS[name]
    failed = 0
    with np.errstate(over="ignore", invalid="ignore"):
        for chk in EPILOGUE_CHECKS:
            try:
                chk(*fns)
            except AssertionError:
                failed += 1
    assert failed, "no epilogue pin caught %s" % name


def test_golden_epilogue():
    g = json.load(open(os.path.join(GOLDEN, "epilogue", "relu_residual_bf16.json")))
    acts = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "silu": oracle.ACT_SILU}
    y = oracle.epilogue(np.array(g["conv_out"]), acts[g["act"]], np.array(g["residual"]))
    np.testing.assert_allclose(y, np.array(g["out_f32"]), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(oracle.round_bf16(y), np.array(g["out_bf16"]))
