"""GPU dual-grid mesh extraction against oracle/mesh.py, through the C ABI.

Quads (rows, order, orientation) must equal the oracle's exactly.  The split
of a quad is decided by comparing two fp64 cosines; where they differ by more
than 1e-9 the GPU's split must equal the oracle's, and where they are closer
(a planar quad: both splits give the same normal up to rounding, a tie in
exact arithmetic) either split is a correct result and the test checks that
the GPU's is one of the two.  Shapes are the voxelised closed surfaces the
oracle's pins use (sphere, two spheres, torus), plus random flags over a
dense random voxel set, whose random vertices give no ties.
"""
import numpy as np
import pytest

from oracle import mesh
from test_oracle_mesh import SHAPES, topology, voxelise

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_voxel_convolution_coord_b300 as m
    from sparse_voxel_convolution_coord_b300 import build_lib
    build_lib.build()
    m.load_library()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def cosines(q, v):
    def unit(a, b, c):
        n = np.cross(b - a, c - a)
        ln = np.linalg.norm(n, axis=1, keepdims=True)
        return np.where(ln > 0, n / np.where(ln > 0, ln, 1), n)
    p = [v[q[:, j]] for j in range(4)]
    c02 = np.einsum("ij,ij->i", unit(p[0], p[1], p[2]), unit(p[0], p[2], p[3]))
    c13 = np.einsum("ij,ij->i", unit(p[0], p[1], p[3]), unit(p[1], p[2], p[3]))
    return c02, c13


def check_mesh(sc, coords, flags, verts, res):
    verts32 = np.asarray(verts, np.float32)
    m = sc.sc_build_map(dev(coords.astype(np.int32)), res)
    quads = sc.sc_dual_mesh_quads(m, dev(flags.astype(np.uint8)))
    tris = sc.sc_dual_mesh_triangulate(quads, dev(verts32))
    m.free()
    got_q = quads.cpu().numpy()
    got_t = tris.cpu().numpy().reshape(-1, 2, 3)
    want_q = mesh.quads(coords, flags)
    np.testing.assert_array_equal(got_q, want_q)
    v64 = verts32.astype(np.float64)
    want_t = mesh.triangulate(want_q, v64).reshape(-1, 2, 3)
    c02, c13 = cosines(want_q, v64)
    decided = np.abs(c13 - c02) > 1e-9
    np.testing.assert_array_equal(got_t[decided], want_t[decided])
    q = want_q[~decided]
    alt_a = np.stack([q[:, [0, 1, 2]], q[:, [0, 2, 3]]], axis=1)
    alt_b = np.stack([q[:, [0, 1, 3]], q[:, [1, 2, 3]]], axis=1)
    ok = np.all(got_t[~decided] == alt_a, axis=(1, 2)) | np.all(got_t[~decided] == alt_b,
                                                              axis=(1, 2))
    assert ok.all()
    return got_q, got_t.reshape(-1, 3)


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_closed_shapes(sc, name):
    phi, res, chi, _ = SHAPES[name]
    coords, flags, verts = voxelise(phi, res)
    _, tris = check_mesh(sc, coords, flags, verts, res)
    directed, undirected, euler = topology(tris)
    assert all(c == 2 for c in undirected.values()) and all(c == 1 for c in directed.values())
    assert euler == chi


def test_random_flags_dense_set(sc):
    rng = np.random.default_rng(61)
    occ = rng.random((2, 20, 20, 20)) < 0.6
    coords = np.argwhere(occ).astype(np.int32)            # two batch elements
    coords = np.ascontiguousarray(coords[rng.permutation(len(coords))])
    flags = rng.integers(0, 64, len(coords))
    verts = coords[:, 1:] + rng.random((len(coords), 3))
    q, _ = check_mesh(sc, coords, flags, verts, 20)
    assert len(q) > 1000


def test_no_quads(sc):
    coords = np.array([[0, 1, 1, 1], [0, 5, 5, 5]], np.int32)
    q, t = check_mesh(sc, coords, np.array([7, 63]), np.zeros((2, 3)), 8)
    assert len(q) == 0 and len(t) == 0
