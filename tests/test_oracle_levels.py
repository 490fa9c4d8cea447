"""Pins for the level-change oracle (oracle/levels.py), checked without going
through it: closed forms, brute force, and dense library routines.

* subdivision of a full cube with every child present is the cube at twice
  the resolution, each child's coordinates halved are its parent's, and the
  count is the masks' total popcount (brute force on a small random case);
* the way down inverts subdivision and matches a dictionary brute force;
* Channel2Spatial against a dense 3-D pixel shuffle (reshape and permute of
  a dense [8C, L, L, L] grid into [C, 2L, 2L, 2L]);
* the 2x2x2 stride-2 convolution against torch's dense conv3d and its
  transpose against conv_transpose3d (fp64, inactive sites zero, compared
  at the active sites);
* each of a set of planted mistakes fails at least one pin.
"""
import types

import numpy as np
import pytest
import torch

from oracle import levels


def random_sites(rng, nb, res, density):
    occ = rng.random((nb, res, res, res)) < density
    return np.ascontiguousarray(np.argwhere(occ), dtype=np.int32)


def check_subdivide_full_cube(lv):
    L = 4
    cube = np.argwhere(np.ones((1, L, L, L), bool)).astype(np.int32)
    child, parent, offset = lv.subdivide(cube)
    assert len(child) == 8 * len(cube)
    want = np.argwhere(np.ones((1, 2 * L, 2 * L, 2 * L), bool))
    assert set(map(tuple, child)) == set(map(tuple, want))
    halved = child.astype(np.int64)
    halved[:, 1:] >>= 1
    np.testing.assert_array_equal(halved, cube[parent])
    # parent-major, ascending offset within a parent
    assert np.all(np.diff(parent) >= 0)
    np.testing.assert_array_equal(offset, np.tile(np.arange(8), len(cube)))
    # child o sits at 2 * parent + (o >> 2 & 1, o >> 1 & 1, o & 1)
    d = child[:, 1:].astype(np.int64) - 2 * cube[parent][:, 1:]
    np.testing.assert_array_equal(d, np.stack([(offset >> 2) & 1, (offset >> 1) & 1,
                                               offset & 1], axis=1))


def check_subdivide_masks(lv):
    rng = np.random.default_rng(1)
    coords = random_sites(rng, 2, 5, 0.3)
    mask = rng.integers(0, 256, size=len(coords)).astype(np.uint8)
    child, parent, offset = lv.subdivide(coords, mask)
    assert len(child) == int(sum(bin(int(m)).count("1") for m in mask))
    want = []
    for i, (b, x, y, z) in enumerate(coords):
        for o in range(8):
            if (int(mask[i]) >> o) & 1:
                want.append((b, 2 * x + ((o >> 2) & 1), 2 * y + ((o >> 1) & 1), 2 * z + (o & 1)))
    assert list(map(tuple, child)) == want


def check_downsample(lv):
    rng = np.random.default_rng(2)
    kids = random_sites(rng, 2, 8, 0.25)
    parents, child_of, parent_of = lv.downsample_map(kids)
    # dictionary brute force
    groups = {}
    for r, (b, x, y, z) in enumerate(kids):
        groups.setdefault((b, x // 2, y // 2, z // 2), {})[4 * (x % 2) + 2 * (y % 2) + z % 2] = r
    keys = sorted(groups)
    assert list(map(tuple, parents)) == keys
    for p, k in enumerate(keys):
        for o in range(8):
            assert child_of[p, o] == groups[k].get(o, -1)
    for r in range(len(kids)):
        assert child_of[parent_of[r]].tolist().count(r) == 1
    # inverse of a full subdivision
    base = random_sites(rng, 1, 5, 0.3)
    child, _, _ = lv.subdivide(base)
    par, cof, _ = lv.downsample_map(child)
    np.testing.assert_array_equal(par, base)            # base is in lexicographic order
    assert (cof >= 0).all()
    for p in range(len(par)):
        for o in range(8):
            want = 2 * par[p, 1:] + np.array([(o >> 2) & 1, (o >> 1) & 1, o & 1])
            np.testing.assert_array_equal(child[cof[p, o], 1:], want)


def dense_grid(coords, feats, res):
    """[C, res, res, res] fp64 grid (batch 0) with feats at coords, zeros elsewhere."""
    g = np.zeros((feats.shape[1], res, res, res))
    g[:, coords[:, 1], coords[:, 2], coords[:, 3]] = np.asarray(feats, np.float64).T
    return g


def check_channel_to_spatial(lv):
    rng = np.random.default_rng(3)
    L, C = 4, 3
    coords = random_sites(rng, 1, L, 0.4)
    feats = rng.standard_normal((len(coords), 8 * C))
    mask = rng.integers(1, 256, size=len(coords)).astype(np.uint8)
    child, parent, offset = lv.subdivide(coords, mask)
    got = lv.channel_to_spatial(feats, parent, offset)
    dense = torch.from_numpy(dense_grid(coords, feats, L))          # [8C, L, L, L]
    shuffled = dense.reshape(C, 2, 2, 2, L, L, L).permute(0, 4, 1, 5, 2, 6, 3) \
                    .reshape(C, 2 * L, 2 * L, 2 * L).numpy()
    want = shuffled[:, child[:, 1], child[:, 2], child[:, 3]].T
    np.testing.assert_array_equal(got, want)


def check_conv_down(lv):
    rng = np.random.default_rng(4)
    R, cin, cout = 8, 5, 4
    kids = random_sites(rng, 1, R, 0.3)
    feats = rng.standard_normal((len(kids), cin))
    w = rng.standard_normal((8, cin, cout))
    bias = rng.standard_normal(cout)
    parents, child_of, _ = lv.downsample_map(kids)
    got = lv.conv_down(child_of, feats, w, bias)
    # dense conv3d weight [co, ci, dx, dy, dz] = W[o][ci][co], o = 4dx + 2dy + dz
    wt = torch.from_numpy(w.reshape(2, 2, 2, cin, cout).transpose(4, 3, 0, 1, 2).copy())
    x = torch.from_numpy(dense_grid(kids, feats, R))[None]
    y = torch.nn.functional.conv3d(x, wt, torch.from_numpy(bias), stride=2)[0].numpy()
    want = y[:, parents[:, 1], parents[:, 2], parents[:, 3]].T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def check_conv_up(lv):
    rng = np.random.default_rng(5)
    L, cin, cout = 4, 3, 6
    coords = random_sites(rng, 1, L, 0.4)
    feats = rng.standard_normal((len(coords), cin))
    w = rng.standard_normal((8, cin, cout))
    bias = rng.standard_normal(cout)
    mask = rng.integers(1, 256, size=len(coords)).astype(np.uint8)
    child, parent, offset = lv.subdivide(coords, mask)
    got = lv.conv_up(parent, offset, feats, w, bias)
    # conv_transpose3d weight [ci, co, dx, dy, dz] = W[o][ci][co]
    wt = torch.from_numpy(w.reshape(2, 2, 2, cin, cout).transpose(3, 4, 0, 1, 2).copy())
    x = torch.from_numpy(dense_grid(coords, feats, L))[None]
    y = torch.nn.functional.conv_transpose3d(x, wt, torch.from_numpy(bias), stride=2)[0].numpy()
    want = y[:, child[:, 1], child[:, 2], child[:, 3]].T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


CHECKS = [check_subdivide_full_cube, check_subdivide_masks, check_downsample,
          check_channel_to_spatial, check_conv_down, check_conv_up]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_levels_pin(check):
    check(levels)


def test_downsample_rejects_duplicates():
    with pytest.raises(levels.LevelError):
        levels.downsample_map(np.array([[0, 1, 1, 1], [0, 1, 1, 1]], np.int32))


# ---------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin

def _mutant(**over):
    ns = {k: getattr(levels, k) for k in ("subdivide", "channel_to_spatial", "downsample_map",
                                          "conv_down", "conv_up")}
    ns.update(over)
    return types.SimpleNamespace(**ns)


def _subdivide_xz_swapped(coords, mask=None):
    child, parent, offset = levels.subdivide(coords, mask)
    swapped = ((offset & 1) << 2) | (offset & 2) | ((offset >> 2) & 1)
    c = np.asarray(coords, np.int64).reshape(-1, 4)[parent].copy()
    c[:, 1:] = 2 * c[:, 1:] + levels.CHILD_OFFSETS[swapped]
    return c.astype(np.int32), parent, offset


def _c2s_blocked(feats, parent, offset):
    f = np.asarray(feats)
    n, c8 = f.shape
    f = f.reshape(n, 8, c8 // 8)                   # child o takes channels o*C .. o*C+C-1
    return f[np.asarray(parent), np.asarray(offset), :]


def _downsample_first_seen(coords):
    parents, child_of, parent_of = levels.downsample_map(coords)
    first = np.argsort(np.array([np.flatnonzero(parent_of == p)[0] for p in range(len(parents))]))
    inv = np.empty_like(first)
    inv[first] = np.arange(len(first))
    return parents[first], child_of[first], inv[parent_of]


def _conv_up_transposed(parent, offset, feats, weight, bias=None):
    w = np.asarray(weight)
    return levels.conv_up(parent, 7 - np.asarray(offset), feats, w, bias)


def _conv_down_no_bias(child_of, feats, weight, bias=None):
    return levels.conv_down(child_of, feats, weight, None)


MUTANTS = {
    "child_offset_x_z_swapped": _mutant(subdivide=_subdivide_xz_swapped),
    "channel_groups_blocked": _mutant(channel_to_spatial=_c2s_blocked),
    "parents_in_first_seen_order": _mutant(downsample_map=_downsample_first_seen),
    "up_weights_mirrored": _mutant(conv_up=_conv_up_transposed),
    "down_bias_dropped": _mutant(conv_down=_conv_down_no_bias),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_level_mistakes_are_caught(name):
    failed = []
    for check in CHECKS:
        try:
            check(MUTANTS[name])
        except (AssertionError, IndexError, ValueError):
            failed.append(check.__name__)
    assert failed, "no pin caught %s" % name


def test_golden_levels():
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "levels",
                        "one_voxel_three_children.json")
    g = json.load(open(path))
    child, parent, offset = levels.subdivide(np.array(g["coords"]), np.array(g["mask"]))
    np.testing.assert_array_equal(child, g["children"])
    np.testing.assert_array_equal(parent, g["parent"])
    np.testing.assert_array_equal(offset, g["offset"])
    feats = np.arange(16, dtype=np.float64)[None, :]
    np.testing.assert_array_equal(levels.channel_to_spatial(feats, parent, offset), g["c2s_out"])
    par, child_of, _ = levels.downsample_map(np.array(g["children"]))
    np.testing.assert_array_equal(par, g["parents_down"])
    np.testing.assert_array_equal(child_of, g["child_of"])
    w = np.stack([(o + 1) * np.eye(2) for o in range(8)])
    up = levels.conv_up(parent, offset, np.array(g["parent_feats"]), w, np.array(g["bias"]))
    np.testing.assert_array_equal(up, g["up_out"])
    down = levels.conv_down(child_of, np.array(g["child_feats"]), w, np.array(g["bias"]))
    np.testing.assert_array_equal(down, g["down_out"])
