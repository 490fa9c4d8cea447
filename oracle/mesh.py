"""Dual-grid mesh extraction over active voxels: TEST INFRASTRUCTURE ONLY.

A plain numpy / Python statement of pulling a triangle mesh out of a dual
voxel grid, for checking a GPU version against.  Only tests, the smoke check
and the benchmark's CPU legs may import this module; the library never
does.

What the pages give ("Running TRELLIS.2 on a Mac (1/3)", Mesh extraction
paragraph: the mesh comes out of a dual voxel grid through a hash map --
coordinate-to-index tables, the connected voxels of each edge, and quads
split into triangles by how well their normals align; "Porting TRELLIS.2
From Python to Rust and Metal", results: a compact hash map and a parallel
loop) is the outline.  The readings taken to make it definite:

* voxel (x, y, z) is the cell [x, x+1] x [y, y+1] x [z, z+1]; it carries a
  dual vertex (any point, normally inside its cell) and owns the three
  primal edges that start at its min corner (x, y, z), along +x, +y, +z;
* a 6-bit flag per voxel: bit a (a = 0, 1, 2 for x, y, z) says its edge
  along axis a crosses the surface; bit 3 + a says that edge's start point
  (the voxel's min corner) is inside;
* a crossing edge along axis a is shared by the 4 voxels whose cells touch
  it, at offsets 0, -e_b, -e_b - e_c, -e_c from the owner (b, c the other two
  axes in cyclic order a -> b -> c); when all 4 are active it becomes a quad
  through their dual vertices, in that cyclic order, which for dual vertices
  at cell centres has its right-hand normal along +a.  When the start point
  is outside (the inside lies towards +a) the order is reversed, so that
  normals point away from the inside;
* a quad (q0, q1, q2, q3) becomes two triangles split along q0-q2 or q1-q3,
  whichever gives the two triangles more aligned normals (the larger cosine
  between them); a tie keeps q0-q2;
* triangles are listed by owner voxel row, then axis, two per quad.
Coordinates are looked up in a dictionary (the coordinate-to-index table);
vertices are the voxels' dual vertices, indexed by voxel row.
"""
import numpy as np

_AXES = ((0, 1, 2), (1, 2, 0), (2, 0, 1))   # (a, b, c): cyclic


def _cell_offsets(a):
    _, b, c = _AXES[a]
    eb = np.zeros(3, np.int64)
    ec = np.zeros(3, np.int64)
    eb[b] = 1
    ec[c] = 1
    return [np.zeros(3, np.int64), -eb, -eb - ec, -ec]


def quads(coords, flags):
    """int64 [Q,4] voxel rows of each quad, in the order described above.

    coords int [N,4] (b, x, y, z); flags int [N] (6 bits)."""
    c = np.asarray(coords, np.int64).reshape(-1, 4)
    f = np.asarray(flags, np.int64).reshape(-1)
    index = {tuple(r): i for i, r in enumerate(c.tolist())}
    out = []
    for i in range(len(c)):
        for a in range(3):
            if not (f[i] >> a) & 1:
                continue
            rows = []
            for d in _cell_offsets(a):
                key = (int(c[i, 0]), int(c[i, 1] + d[0]), int(c[i, 2] + d[1]),
                       int(c[i, 3] + d[2]))
                rows.append(index.get(key, -1))
            if min(rows) < 0:
                continue
            if not (f[i] >> (3 + a)) & 1:
                rows = rows[::-1]
            out.append(rows)
    return np.array(out, np.int64).reshape(-1, 4)


def _unit_normal(p0, p1, p2):
    n = np.cross(p1 - p0, p2 - p0)
    ln = np.linalg.norm(n)
    return n / ln if ln > 0 else n


def triangulate(q, vertices):
    """int64 [2Q,3]: each quad split along the diagonal with better-aligned
    triangle normals (q0-q2 on a tie)."""
    v = np.asarray(vertices, np.float64)
    tris = []
    for q0, q1, q2, q3 in np.asarray(q, np.int64).tolist():
        p0, p1, p2, p3 = v[q0], v[q1], v[q2], v[q3]
        cos02 = float(np.dot(_unit_normal(p0, p1, p2), _unit_normal(p0, p2, p3)))
        cos13 = float(np.dot(_unit_normal(p0, p1, p3), _unit_normal(p1, p2, p3)))
        if cos13 > cos02:
            tris += [[q0, q1, q3], [q1, q2, q3]]
        else:
            tris += [[q0, q1, q2], [q0, q2, q3]]
    return np.array(tris, np.int64).reshape(-1, 3)


def extract(coords, flags, vertices):
    """The mesh: (vertices [N,3] fp64, triangles int64 [T,3] into them)."""
    return np.asarray(vertices, np.float64), triangulate(quads(coords, flags), vertices)
