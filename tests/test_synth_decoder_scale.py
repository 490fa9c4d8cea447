"""The decoder-scale input generator (1024^3, millions of voxels) against its
definition, on grids small enough for a dense evaluation.

The generator finds the 1-voxel shell of a superquadric by sparse refinement
(64^3 cells the surface crosses, split into 8 per level), so that no 1024^3
grid is ever materialised.  The shell it must reproduce is the dense rule of
the other workloads: cells inside the shape with some cell of their 3x3x3
cube outside it (or off the grid).  Coarse cells are kept when field samples
over their grown cube straddle the surface, which can miss a sliver of a
very thin feature, never add a cell: the refined shell must be a subset of
the dense one and cover at least 99.5% of it (over 72,588 cells of eight
such cases, 6 were missed).
"""
import numpy as np
import pytest

from sparse_voxel_convolution_coord_b300 import synth


@pytest.mark.parametrize("res,base,seed", [(64, 16, 1), (128, 16, 2), (128, 8, 4),
                                           (128, 32, 3), (96, 12, 5), (64, 64, 11)])
def test_refined_shell_against_dense(res, base, seed):
    field = synth.SuperquadricField(np.random.default_rng(seed), np.full(3, (res - 1) / 2.0))
    scale = 0.3 * res
    got = synth.refined_shell(res, base, field, scale)
    want = synth.dense_shell(res, field, scale)
    g = set(map(tuple, got))
    w = set(map(tuple, want))
    assert len(g) == len(got), "duplicate cells"
    assert g <= w, "%d cells outside the dense shell" % len(g - w)
    assert len(g) >= 0.995 * len(w), "covers %d of %d" % (len(g), len(w))
    # (x, y, z) lexicographic order
    key = (got[:, 0] * res + got[:, 1]) * res + got[:, 2]
    assert np.all(np.diff(key) > 0)


def test_shell_clipped_by_the_grid_counts_off_grid_as_outside():
    # a shape larger than the grid: the grid's faces carry the shell
    res = 32
    field = synth.SuperquadricField(np.random.default_rng(7), np.full(3, (res - 1) / 2.0))
    scale = 2.0 * res
    got = synth.refined_shell(res, 8, field, scale)
    want = synth.dense_shell(res, field, scale)
    assert set(map(tuple, got)) == set(map(tuple, want))
    assert len(want) == res ** 3 - (res - 2) ** 3


def test_decoder_scale_shell_small():
    # the workload's own routine at 256^3 from 16^3: the base-level shell is
    # bisected to ~target cells and the fine count grows with (256/16)^2
    xyz = synth.decoder_scale_shell(256, 16, 600, np.random.default_rng(3))
    assert len(np.unique(xyz, axis=0)) == len(xyz)
    assert xyz.min() >= 0 and xyz.max() < 256
    assert 0.3 * 600 * 256 <= len(xyz) <= 3 * 600 * 256


def test_config6_is_the_decoder_scale_workload():
    cfg = synth.CONFIGS[6]
    assert (cfg.res, cfg.batch, cfg.cin, cfg.cout, cfg.dtype) == (1024, 1, 64, 64, "f16")
