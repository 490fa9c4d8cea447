"""Level changes of a sparse voxel hierarchy: TEST INFRASTRUCTURE ONLY.

Plain numpy statements of the operations that move a structured latent
between resolution levels, for checking GPU kernels against.  Only tests,
the smoke check and the benchmark's CPU legs may import this module; the
library never does.

What the pages give (trellis2mlx README: the pipeline list's "Upsample"
stage, decoder subdivision predictions turned into the high-resolution
coordinate structure; the stage table, 2,977 low-resolution voxels becoming
761,916; the project layout, a sparse UNet decoder with Channel2Spatial
upsampling and a dense Conv3d decoder with pixel-shuffle upsampling) names
the operations but fixes none of their details.  The readings taken:

* subdivision: a voxel (b, x, y, z) at resolution R has 8 children at 2R,
  child o at (b, 2x + dx, 2y + dy, 2z + dz) with (dx, dy, dz) = (o >> 2 & 1,
  o >> 1 & 1, o & 1) -- the same row-major flattening as the convolution's
  27 offsets.  An 8-bit mask per voxel (the decoder's prediction) says which
  children exist; children are listed parent by parent in input order,
  ascending o within a parent;
* Channel2Spatial: a parent's 8*C channels become its children's C, child o
  taking channels c * 8 + o (the dense pixel-shuffle convention: the
  sub-voxel index runs fastest);
* the way down: the parents of a set of voxels at 2R are the distinct
  (b, x >> 1, y >> 1, z >> 1), listed in (b, x, y, z) lexicographic order,
  with an 8-entry table per parent of the row of each child o (or -1);
* the convolutions between levels are the 2x2x2 stride-2 convolution and
  its transpose, weights W[o][ci][co] (the (Kvol, Ci, Co) layout with
  Kvol = 8): down, out[p] = bias + sum_o feats[child_of[p][o]] @ W[o] over
  present children; up, out[child] = bias + feats[parent] @ W[o].
Every product and sum is in fp64.
"""
import numpy as np

#: child o <-> displacement (dx, dy, dz)
CHILD_OFFSETS = np.array([[(o >> 2) & 1, (o >> 1) & 1, o & 1] for o in range(8)], np.int64)


class LevelError(ValueError):
    pass


def subdivide(coords, mask=None):
    """Children of each voxel whose mask bit is set.

    coords int [N,4] (b, x, y, z); mask uint8 [N] (bit o: child o exists) or
    None for all eight.  Returns (child_coords int32 [M,4], parent int64 [M],
    offset int64 [M]), parent-major, ascending offset within a parent."""
    c = np.asarray(coords, dtype=np.int64).reshape(-1, 4)
    n = len(c)
    m = np.full(n, 0xFF, np.int64) if mask is None else np.asarray(mask, np.int64).reshape(n)
    parent = np.repeat(np.arange(n, dtype=np.int64), 8)
    offset = np.tile(np.arange(8, dtype=np.int64), n)
    keep = ((m[parent] >> offset) & 1) == 1
    parent, offset = parent[keep], offset[keep]
    child = c[parent].copy()
    child[:, 1:] = 2 * child[:, 1:] + CHILD_OFFSETS[offset]
    return child.astype(np.int32), parent, offset


def channel_to_spatial(feats, parent, offset):
    """Child features: child (parent i, offset o) takes feats[i, c * 8 + o]
    for c = 0 .. C-1, where feats is [N, 8C]."""
    f = np.asarray(feats)
    n, c8 = f.shape
    if c8 % 8:
        raise LevelError("channel count %d is not a multiple of 8" % c8)
    f = f.reshape(n, c8 // 8, 8)                  # [i, c, o]
    return f[np.asarray(parent), :, np.asarray(offset)]


def downsample_map(coords):
    """Parents of voxels at resolution 2R.

    Returns (parent_coords int32 [P,4] in lexicographic order, child_of int64
    [P,8] = row of child o or -1, parent_of int64 [N]).  Duplicate input
    rows are an error."""
    c = np.asarray(coords, dtype=np.int64).reshape(-1, 4)
    if len(np.unique(c, axis=0)) != len(c):
        raise LevelError("duplicate voxels")
    pc = c.copy()
    pc[:, 1:] >>= 1
    parents, parent_of = np.unique(pc, axis=0, return_inverse=True)
    parent_of = parent_of.reshape(-1)
    off = (c[:, 1] & 1) * 4 + (c[:, 2] & 1) * 2 + (c[:, 3] & 1)
    child_of = np.full((len(parents), 8), -1, np.int64)
    child_of[parent_of, off] = np.arange(len(c))
    return parents.astype(np.int32), child_of, parent_of.astype(np.int64)


def conv_down(child_of, feats, weight, bias=None):
    """fp64 [P,cout]: out[p] = bias + sum_o [child_of[p][o] >= 0]
    feats[child_of[p][o]] @ W[o]; weight [8, cin, cout]."""
    t = np.asarray(child_of, np.int64)
    x = np.asarray(feats, np.float64)
    w = np.asarray(weight, np.float64)
    out = np.zeros((len(t), w.shape[2]))
    for o in range(8):
        rows = t[:, o]
        have = rows >= 0
        out[have] += x[rows[have]] @ w[o]
    if bias is not None:
        out += np.asarray(bias, np.float64)
    return out


def conv_up(parent, offset, feats, weight, bias=None):
    """fp64 [M,cout]: out[m] = bias + feats[parent[m]] @ W[offset[m]];
    weight [8, cin, cout]."""
    x = np.asarray(feats, np.float64)
    w = np.asarray(weight, np.float64)
    p = np.asarray(parent, np.int64)
    o = np.asarray(offset, np.int64)
    out = np.einsum("mi,mio->mo", x[p], w[o])
    if bias is not None:
        out += np.asarray(bias, np.float64)
    return out
