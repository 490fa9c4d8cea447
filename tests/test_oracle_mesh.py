"""Pins for the dual-grid mesh oracle (oracle/mesh.py), by properties any
correct extraction has, not by re-running its steps:

* on voxelised closed shapes (signed distance fields sampled at the grid
  points; active voxels = cells the surface crosses; flags from the corner
  signs; dual vertices = the mean of the cell's edge crossings) the mesh is
  a closed, consistently oriented 2-manifold: every undirected edge lies on
  exactly two triangles and every directed edge on exactly one;
* its Euler characteristic is 2 for a sphere, 4 for two spheres and 0 for
  a torus, and its signed volume is positive (outward normals) and within
  10% of the shape's (mass-point dual vertices shrink convex shapes a
  little);
* a folded quad is split along the diagonal worked out by hand;
* planted mistakes (a wrong neighbour cell, no orientation flip, a fixed
  diagonal, the axes in the wrong cyclic order) each fail a pin.
"""
import types

import numpy as np
import pytest

from oracle import mesh


def voxelise(phi, res):
    """(coords, flags, vertices) of the cells of a res^3 grid that the zero
    set of phi (sampled at the integer points 0..res) crosses."""
    ax = np.arange(res + 1, dtype=np.float64)
    P = np.stack(np.meshgrid(ax, ax, ax, indexing="ij"), axis=-1)
    g = phi(P.reshape(-1, 3)).reshape(res + 1, res + 1, res + 1)
    inside = g < 0
    coords, flags, verts = [], [], []
    corners = [(i, j, k) for i in (0, 1) for j in (0, 1) for k in (0, 1)]
    edges = [((i, j, k), (i + 1, j, k)) for j in (0, 1) for k in (0, 1) for i in (0,)] + \
            [((i, j, k), (i, j + 1, k)) for i in (0, 1) for k in (0, 1) for j in (0,)] + \
            [((i, j, k), (i, j, k + 1)) for i in (0, 1) for j in (0, 1) for k in (0,)]
    for x in range(res):
        for y in range(res):
            for z in range(res):
                s = [inside[x + i, y + j, z + k] for i, j, k in corners]
                if all(s) or not any(s):
                    continue
                pts = []
                for (u, w) in edges:
                    pu = (x + u[0], y + u[1], z + u[2])
                    pw = (x + w[0], y + w[1], z + w[2])
                    if inside[pu] != inside[pw]:
                        t = g[pu] / (g[pu] - g[pw])
                        pts.append(np.array(pu) + t * (np.array(pw) - np.array(pu)))
                f = 0
                for a in range(3):
                    e = [0, 0, 0]
                    e[a] = 1
                    end = (x + e[0], y + e[1], z + e[2])
                    if max(end) <= res and inside[x, y, z] != inside[end]:
                        f |= 1 << a
                    if inside[x, y, z]:
                        f |= 1 << (3 + a)
                coords.append((0, x, y, z))
                flags.append(f)
                verts.append(np.mean(pts, axis=0))
    return np.array(coords, np.int32), np.array(flags, np.int64), np.array(verts)


def topology(tris):
    directed = {}
    for t in tris.tolist():
        for i in range(3):
            e = (t[i], t[(i + 1) % 3])
            directed[e] = directed.get(e, 0) + 1
    undirected = {}
    for (u, w), cnt in directed.items():
        key = (min(u, w), max(u, w))
        undirected[key] = undirected.get(key, 0) + cnt
    nverts = len(np.unique(tris))
    return directed, undirected, nverts - len(undirected) + len(tris)


def signed_volume(v, tris):
    p = v[tris]
    return float(np.einsum("ij,ij->i", p[:, 0], np.cross(p[:, 1], p[:, 2])).sum() / 6.0)


def sphere(c, r):
    return lambda P: np.linalg.norm(P - np.asarray(c), axis=1) - r


def torus(c, R, r):
    def f(P):
        d = P - np.asarray(c)
        q = np.sqrt(d[:, 0] ** 2 + d[:, 1] ** 2) - R
        return np.sqrt(q ** 2 + d[:, 2] ** 2) - r
    return f


SHAPES = {
    "sphere": (sphere((8.2, 7.9, 8.1), 5.3), 16, 2, 4.0 / 3.0 * np.pi * 5.3 ** 3),
    "two_spheres": (lambda P: np.minimum(sphere((7.1, 7.2, 9.0), 4.6)(P),
                                         sphere((17.0, 16.9, 9.1), 4.2)(P)), 24, 4,
                    4.0 / 3.0 * np.pi * (4.6 ** 3 + 4.2 ** 3)),
    "torus": (torus((10.1, 9.9, 7.05), 5.5, 2.2), 20, 0, 2 * np.pi ** 2 * 5.5 * 2.2 ** 2),
}


def check_closed_shapes(m):
    for name, (phi, res, chi, vol) in SHAPES.items():
        coords, flags, verts = voxelise(phi, res)
        v, tris = m.extract(coords, flags, verts)
        directed, undirected, euler = topology(tris)
        assert all(cnt == 2 for cnt in undirected.values()), name + ": not closed"
        assert all(cnt == 1 for cnt in directed.values()), name + ": not consistently oriented"
        assert euler == chi, "%s: Euler characteristic %d, want %d" % (name, euler, chi)
        sv = signed_volume(v, tris)
        # mass-point dual vertices sit inside a convex surface: 4-7% short here
        assert abs(sv - vol) <= 0.10 * vol, "%s: volume %.1f, want %.1f" % (name, sv, vol)


def check_folded_quad(m):
    # normals for the q0-q2 split: (0,-1,1)/sqrt2 and (-1,0,1)/sqrt2, cosine
    # 1/2; for q1-q3: (0,0,1) and (-1,-1,1)/sqrt3, cosine 1/sqrt3 > 1/2
    v = np.array([[0.0, 0, 0], [1, 0, 0], [1, 1, 1], [0, 1, 0]])
    np.testing.assert_array_equal(m.triangulate(np.array([[0, 1, 2, 3]]), v),
                                  [[0, 1, 3], [1, 2, 3]])
    flat = np.array([[0.0, 0, 0], [1, 0, 0], [1, 1, 0], [0, 1, 0]])   # a tie keeps q0-q2
    np.testing.assert_array_equal(m.triangulate(np.array([[0, 1, 2, 3]]), flat),
                                  [[0, 1, 2], [0, 2, 3]])


def check_single_edge(m):
    # four voxels around the x-edge at (1, 1, 1); the owner (1, 1, 1) flags it,
    # start point inside: the quad runs (1,1,1) (1,0,1) (1,0,0) (1,1,0)
    coords = np.array([[0, 1, 1, 1], [0, 1, 0, 1], [0, 1, 0, 0], [0, 1, 1, 0]], np.int32)
    flags = np.array([0b001001, 0, 0, 0])
    np.testing.assert_array_equal(m.quads(coords, flags), [[0, 1, 2, 3]])
    np.testing.assert_array_equal(m.quads(coords, np.array([0b000001, 0, 0, 0])),
                                  [[3, 2, 1, 0]])
    # one of the four missing: no quad
    assert len(m.quads(coords[:3], flags[:3])) == 0


CHECKS = [check_closed_shapes, check_folded_quad, check_single_edge]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_mesh_pin(check):
    check(mesh)


# ---------------------------------------------------------------------------
# planted mistakes

def _with(**over):
    class M:
        pass
    m = M()
    for k in ("quads", "triangulate", "extract"):
        setattr(m, k, getattr(mesh, k))
    for k, fn in over.items():
        setattr(m, k, fn)
    if "extract" not in over:
        m.extract = lambda c, f, v: (np.asarray(v, np.float64),
                                     m.triangulate(m.quads(c, f), v))
    return m


def _quads_wrong_cell(coords, flags):
    orig = mesh._cell_offsets
    try:
        def bad(a):
            offs = orig(a)
            offs[2] = -offs[2]           # +e_b + e_c instead of -e_b - e_c
            return offs
        mesh._cell_offsets = bad
        return mesh.quads(coords, flags)
    finally:
        mesh._cell_offsets = orig


def _quads_no_flip(coords, flags):
    f = np.asarray(flags) | 0b111000    # every start point "inside"
    return mesh.quads(coords, f)


def _triangulate_fixed(q, v):
    q = np.asarray(q, np.int64)
    return np.concatenate([q[:, [0, 1, 2]], q[:, [0, 2, 3]]], axis=1).reshape(-1, 3)


def _quads_anticyclic(coords, flags):
    return mesh.quads(coords, flags)[:, ::-1]


MUTANTS = {
    "wrong_neighbour_cell": _with(quads=_quads_wrong_cell),
    "no_orientation_flip": _with(quads=_quads_no_flip),
    "fixed_diagonal": _with(triangulate=_triangulate_fixed),
    "axes_anticyclic": _with(quads=_quads_anticyclic),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mesh_mistakes_are_caught(name):
    failed = []
    for check in CHECKS:
        try:
            check(MUTANTS[name])
        except (AssertionError, IndexError, ValueError):
            failed.append(check.__name__)
    assert failed, "no pin caught %s" % name
