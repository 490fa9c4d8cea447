"""Seeded synthetic voxel sets, features and weights.

This module only draws inputs.  It holds none of the convolution's
arithmetic: no neighbour search, no hash, no gather and no product.  The CUDA
path and the CPU oracle are both fed from it, so that they see the same bits.

The pages measure on private models and a handful of images (structured
latents on 16^3 / 64^3 occupancy grids with thousands to millions of active
voxels: "Porting TRELLIS.2 From Python to Rust and Metal", sections II-III;
the trellis2mlx README stage tables).  No dataset or weights are used here:
seeded surface shells stand in for those voxel sets.

Recipe (the pages fix none of it; this is the reading taken):
  * ball shell: cells p with |p - c|^2 <= r^2 whose 3x3x3 neighbourhood
    reaches a cell outside the ball (or outside the grid);
  * superquadric (Barr) inside-outside function
      F(p) = ((|x'/a|)^(2/e2) + (|y'/b|)^(2/e2))^(e2/e1) + (|z'/c|)^(2/e1),
    p' = R^T (p - centre), R a uniformly random rotation (normalised Gaussian
    quaternion), e1, e2 ~ U[0.5, 3], axes (a, b, c) = U[0.5, 1]^3 * s, with
    the scale s found by bisection so that the voxel count is within 3% of
    the target;
  * t-voxel shell = inside minus its erosion by the 3x3x3 cube repeated t
    times, cells outside the grid counting as outside.  Computed exactly as
    "inside, and some cell of the (2t+1)^3 cube around it is outside";
  * a union of shapes is the union of their individual shells;
  * extra "noise" sites are drawn uniformly from the empty cells;
  * decoder scale (1024^3, millions of voxels, as the pages' shape decoders
    produce from a 64^3 structure by repeated subdivision): the 1-voxel shell
    of one superquadric found by sparse refinement.  The 64^3 cells the
    surface crosses are split into 8 children per level, keeping the
    children whose cube (grown by one fine voxel) straddles the surface by
    the field's values at its corners and centre; at full resolution the
    1-shell rule above is applied exactly, by evaluating the field at each
    candidate's 26 neighbours;
  * rows are listed in (batch, x, y, z) lexicographic order, the order an
    argwhere over an occupancy grid produces;
  * features ~ N(0, 1); weights ~ N(0, 1/sqrt(27 * cin)) (standard deviation);
    bias ~ N(0, 0.1); bf16 values are the round-to-nearest-even of the fp32
    draws.
Seeds: configuration i draws coordinates from 1000+i, features from 2000+i,
weights and bias from 3000+i (numpy PCG64).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
from scipy import ndimage

__all__ = ["CONFIGS", "Problem", "make_problem", "make_coords", "make_tensors",
           "ball_shell", "superquadric_shells", "random_rotation"]


@dataclasses.dataclass(frozen=True)
class Config:
    key: int
    name: str
    batch: int
    res: int
    cin: int
    cout: int
    dtype: str          # "f32", "bf16" or "f16": the dtype of feats and weights
    description: str


CONFIGS = {
    1: Config(1, "ball16_c32_f32", 1, 16, 32, 32, "f32",
              "batch 1, 16^3, shell of a ball r=6 at (8,8,8) plus 50 random sites, "
              "C=32, fp32"),
    2: Config(2, "sq64_20k_c64_bf16", 1, 64, 64, 64, "bf16",
              "batch 1, 64^3, 2-voxel shell of one superquadric, ~20k voxels, "
              "C=64, bf16"),
    3: Config(3, "sq3x64_30k_c256_bf16", 1, 64, 256, 256, "bf16",
              "batch 1, 64^3, union of 3 superquadric 2-voxel shells, ~30k voxels, "
              "C=256, bf16"),
    4: Config(4, "b8_sq64_c128_bf16", 8, 64, 128, 128, "bf16",
              "batch 8, 64^3, one superquadric 2-voxel shell per grid, 8k-40k "
              "voxels each, C=128, bf16"),
    5: Config(5, "sq4x256_400k_c32_bf16", 1, 256, 32, 32, "bf16",
              "batch 1, 256^3, union of 4 superquadric 1-voxel shells (~396k) "
              "plus 1% random sites, C=32, bf16"),
    6: Config(6, "sq1024_dec_c64_f16", 1, 1024, 64, 64, "f16",
              "batch 1, 1024^3, 1-voxel shell of one superquadric refined from "
              "64^3 (millions of voxels, decoder scale), C=64, fp16"),
}


def random_rotation(rng: np.random.Generator) -> np.ndarray:
    """Uniform random rotation matrix from a normalised Gaussian quaternion."""
    q = rng.standard_normal(4)
    q /= np.linalg.norm(q)
    w, x, y, z = q
    return np.array([
        [1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)],
        [2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)],
        [2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)],
    ])


def _grid_points(res: int) -> np.ndarray:
    ax = np.arange(res, dtype=np.float64)
    g = np.stack(np.meshgrid(ax, ax, ax, indexing="ij"), axis=-1)
    return g.reshape(-1, 3)


def _shell_bounds(g: np.ndarray, t: int):
    """For a radius-like field g (inside at scale s iff g <= s), the interval
    [lo, hi) of scales s for which each cell lies in the t-voxel shell:
    lo = g(p), hi = max of g over the (2t+1)^3 cube around p, +inf off-grid."""
    hi = ndimage.maximum_filter(g, size=2 * t + 1, mode="constant", cval=np.inf)
    return g, hi


def _superquadric_field(res: int, rng: np.random.Generator, centre: np.ndarray):
    """Radius-like field G = F^(e1/2) at unit scale: inside at scale s iff G <= s."""
    e1, e2 = rng.uniform(0.5, 3.0, size=2)
    axes = rng.uniform(0.5, 1.0, size=3)
    rot = random_rotation(rng)
    ax = np.arange(res, dtype=np.float64)
    d = [(ax - centre[i]) for i in range(3)]
    # p'_j = sum_i (p_i - c_i) R[i, j], evaluated by broadcasting over the grid.
    pj = []
    for j in range(3):
        v = (d[0][:, None, None] * rot[0, j] + d[1][None, :, None] * rot[1, j]
             + d[2][None, None, :] * rot[2, j])
        pj.append(np.abs(v) / axes[j])
    f = (pj[0] ** (2.0 / e2) + pj[1] ** (2.0 / e2)) ** (e2 / e1) + pj[2] ** (2.0 / e1)
    return (f ** (e1 / 2.0)).astype(np.float32)


def _bisect_scale(bounds, target: int, res: int, tol: float = 0.03, iters: int = 60):
    def occ(s):
        m = np.zeros((res, res, res), dtype=bool)
        for lo, hi in bounds:
            m |= (lo <= s) & (s < hi)
        return m
    lo_s, hi_s = 0.0, 4.0 * res
    best = None
    for _ in range(iters):
        s = 0.5 * (lo_s + hi_s)
        m = occ(s)
        cnt = int(m.sum())
        if best is None or abs(cnt - target) < abs(best[1] - target):
            best = (m, cnt)
        if abs(cnt - target) <= tol * target:
            return m
        if cnt < target:
            lo_s = s
        else:
            hi_s = s
    return best[0]


def superquadric_shells(res: int, n_shapes: int, target: int, t: int,
                        rng: np.random.Generator, jitter: float) -> np.ndarray:
    """Boolean occupancy [res]^3: union of n_shapes superquadric t-shells whose
    common scale is bisected to hit `target` voxels within 3%."""
    bounds = []
    for _ in range(n_shapes):
        centre = (res - 1) / 2.0 + rng.uniform(-jitter, jitter, size=3) * res
        bounds.append(_shell_bounds(_superquadric_field(res, rng, centre), t))
    return _bisect_scale(bounds, target, res)


class SuperquadricField:
    """The radius-like superquadric field G = F^(e1/2) at unit scale,
    evaluated at arbitrary points (inside at scale s iff G <= s)."""

    def __init__(self, rng: np.random.Generator, centre):
        self.e1, self.e2 = rng.uniform(0.5, 3.0, size=2)
        self.axes = rng.uniform(0.5, 1.0, size=3)
        self.rot = random_rotation(rng)
        self.centre = np.asarray(centre, dtype=np.float64)

    def __call__(self, pts: np.ndarray) -> np.ndarray:
        d = np.asarray(pts, dtype=np.float64) - self.centre
        pj = np.abs(d @ self.rot) / self.axes          # p' = R^T (p - c), per axis
        e1, e2 = self.e1, self.e2
        f = (pj[:, 0] ** (2.0 / e2) + pj[:, 1] ** (2.0 / e2)) ** (e2 / e1) + pj[:, 2] ** (2.0 / e1)
        return f ** (e1 / 2.0)


_CUBE = np.array([[i, j, k] for i in (0, 1) for j in (0, 1) for k in (0, 1)], np.int64)
def _lattice(m: int) -> np.ndarray:
    t = np.arange(m, dtype=np.float64) / (m - 1)
    return np.stack(np.meshgrid(t, t, t, indexing="ij"), axis=-1).reshape(-1, 3)


_LATTICE3 = _lattice(3)
_LATTICE5 = _lattice(5)
_NEIGH27 = np.array([[i, j, k] for i in (-1, 0, 1) for j in (-1, 0, 1) for k in (-1, 0, 1)],
                    np.int64)  # index 13 is the cell itself


def _straddles(field, scale, cells: np.ndarray, h: int, res: int) -> np.ndarray:
    """Cells (of side h fine voxels, fine-grid origin h * cell) whose cube,
    grown by 1 + h / 2 fine voxels on every side, has field values on both
    sides of `scale` on an evenly spaced lattice over it (5 x 5 x 5 points
    for h >= 8, else 3 x 3 x 3; points off the grid count as outside, as in
    the shell rule)."""
    lat = _LATTICE5 if h >= 8 else _LATTICE3
    g0 = 1 + h // 2
    lo = (cells * h - g0).astype(np.float64)
    span = float(h - 1 + 2 * g0)
    pts = (lo[:, None, :] + lat[None, :, :] * span).reshape(-1, 3)
    g = field(np.clip(pts, 0, res - 1))
    g[((pts < 0) | (pts > res - 1)).any(axis=1)] = np.inf  # off the grid is outside
    g = g.reshape(len(cells), len(lat))
    return (g.min(axis=1) <= scale) & (g.max(axis=1) > scale)


def _shell_rule(field, scale, cells: np.ndarray, res: int) -> np.ndarray:
    """The exact 1-shell rule on fine cells: inside (G <= scale) with some
    cell of the 3x3x3 cube around it outside (G > scale, or off the grid)."""
    nb = (cells[:, None, :] + _NEIGH27[None, :, :]).reshape(-1, 3)
    off_grid = ((nb < 0) | (nb >= res)).any(axis=1).reshape(len(cells), 27)
    g = field(np.clip(nb, 0, res - 1)).reshape(len(cells), 27)
    return (g[:, 13] <= scale) & (off_grid | (g > scale)).any(axis=1)


_BLOCK4 = np.array([[i, j, k] for i in range(-1, 3) for j in range(-1, 3) for k in range(-1, 3)],
                   np.int64)


def _shell_rule_blocks(field, scale, parents: np.ndarray, res: int) -> np.ndarray:
    """The exact 1-shell rule on the 8 children (2p + {0,1}^3) of each parent
    p, from one evaluation of the field on the parent's 4x4x4 neighbourhood
    (2p + {-1..2}^3) instead of 27 per child.  Returns [nP, 8] booleans in
    _CUBE order."""
    pts = (parents[:, None, :] * 2 + _BLOCK4[None, :, :]).reshape(-1, 3)
    off = ((pts < 0) | (pts >= res)).any(axis=1)
    g = field(np.clip(pts, 0, res - 1))
    out = (off | (g > scale)).reshape(-1, 4, 4, 4)
    g = g.reshape(-1, 4, 4, 4)
    res_ = np.zeros((len(parents), 8), bool)
    for c, (i, j, k) in enumerate(_CUBE):
        win = out[:, i:i + 3, j:j + 3, k:k + 3].reshape(len(parents), 27)
        res_[:, c] = (g[:, i + 1, j + 1, k + 1] <= scale) & win.any(axis=1)
    return res_


def refined_shell(res: int, base: int, field, scale: float) -> np.ndarray:
    """int64 [M,3] fine cells of the 1-voxel shell of {G <= scale} on a res^3
    grid, found from the base^3 cells the surface crosses by splitting each
    kept cell into 8 per level (res / base a power of two): coarse cells are
    kept when they straddle the surface, fine cells by the exact rule.  Cells
    are in (x, y, z) lexicographic order."""
    ax = np.arange(base, dtype=np.int64)
    cells = np.stack(np.meshgrid(ax, ax, ax, indexing="ij"), axis=-1).reshape(-1, 3)
    h = res // base
    chunk = 1 << 18

    def keep_where(test, cs, *args):
        keep = np.zeros(len(cs), bool)
        for a in range(0, len(cs), chunk):
            keep[a:a + chunk] = test(field, scale, cs[a:a + chunk], *args)
        return cs[keep]

    if h == 1:
        cells = keep_where(_shell_rule, cells, res)
    else:
        cells = keep_where(_straddles, cells, h, res)
    while h > 1:
        h //= 2
        if h == 1:  # the children of each kept cell at once
            found = []
            for a in range(0, len(cells), chunk // 8):
                par = cells[a:a + chunk // 8]
                keep = _shell_rule_blocks(field, scale, par, res)
                kids = par[:, None, :] * 2 + _CUBE[None, :, :]
                found.append(kids[keep])
            cells = np.concatenate(found) if found else np.zeros((0, 3), np.int64)
        else:
            kids = (cells[:, None, :] * 2 + _CUBE[None, :, :]).reshape(-1, 3)
            cells = keep_where(_straddles, kids, h, res)
    order = np.lexsort((cells[:, 2], cells[:, 1], cells[:, 0]))
    return cells[order]


def dense_shell(res: int, field, scale: float) -> np.ndarray:
    """The same 1-voxel shell from a dense res^3 evaluation (small res only):
    inside minus its erosion by the 3x3x3 cube, outside the grid counting as
    outside."""
    g = field(_grid_points(res)).reshape(res, res, res)
    inside = g <= scale
    eroded = ndimage.binary_erosion(inside, structure=np.ones((3, 3, 3), bool),
                                    iterations=1, border_value=0)
    return np.argwhere(inside & ~eroded).astype(np.int64)


def decoder_scale_shell(res: int, base: int, target_base: int,
                        rng: np.random.Generator) -> np.ndarray:
    """One superquadric's 1-voxel shell at res^3 by refinement from base^3,
    its scale bisected so that the base^3 1-shell holds ~target_base cells
    (the fine count then grows with (res / base)^2)."""
    centre = np.full(3, (res - 1) / 2.0)
    field = SuperquadricField(rng, centre)
    pts = (_grid_points(base) + 0.5) * (res / base) - 0.5   # base-cell centres, fine units
    g = field(pts).reshape(base, base, base)
    lo_s, hi_s = 0.0, 2.0 * res
    scale = 0.5 * (lo_s + hi_s)
    for _ in range(60):
        scale = 0.5 * (lo_s + hi_s)
        inside = g <= scale
        shell = inside & ~ndimage.binary_erosion(inside, structure=np.ones((3, 3, 3), bool),
                                                  iterations=1, border_value=0)
        cnt = int(shell.sum())
        if abs(cnt - target_base) <= 0.03 * target_base:
            break
        if cnt < target_base:
            lo_s = scale
        else:
            hi_s = scale
    return refined_shell(res, base, field, scale)


def ball_shell(res: int, centre, radius: float) -> np.ndarray:
    p = _grid_points(res) - np.asarray(centre, dtype=np.float64)
    inside = ((p * p).sum(axis=1) <= radius * radius).reshape(res, res, res)
    eroded = ndimage.binary_erosion(inside, structure=np.ones((3, 3, 3), bool),
                                    iterations=1, border_value=0)
    return inside & ~eroded


def _add_random_sites(occ: np.ndarray, count: int, rng: np.random.Generator) -> np.ndarray:
    empty = np.flatnonzero(~occ.ravel())
    pick = rng.choice(empty, size=count, replace=False)
    occ = occ.copy()
    occ.ravel()[pick] = True
    return occ


def _coords_of(occ_list) -> np.ndarray:
    rows = []
    for b, occ in enumerate(occ_list):
        xyz = np.argwhere(occ).astype(np.int32)
        rows.append(np.concatenate([np.full((len(xyz), 1), b, np.int32), xyz], axis=1))
    return np.ascontiguousarray(np.concatenate(rows, axis=0), dtype=np.int32)


_COORD_CACHE: dict = {}


def make_coords(key: int) -> np.ndarray:
    """int32 [N,4] (b,x,y,z) coordinates of configuration `key` (1..6)."""
    if key in _COORD_CACHE:
        return _COORD_CACHE[key]
    cfg = CONFIGS[key]
    rng = np.random.default_rng(1000 + key)
    if key == 1:
        occ = ball_shell(16, (8, 8, 8), 6.0)
        occ = _add_random_sites(occ, 50, rng)
        grids = [occ]
    elif key == 2:
        grids = [superquadric_shells(64, 1, 20000, 2, rng, 0.0)]
    elif key == 3:
        grids = [superquadric_shells(64, 3, 30000, 2, rng, 0.15)]
    elif key == 4:
        targets = rng.integers(8000, 40001, size=cfg.batch)
        grids = [superquadric_shells(64, 1, int(tg), 2, rng, 0.0) for tg in targets]
    elif key == 5:
        occ = superquadric_shells(256, 4, 396000, 1, rng, 0.15)
        occ = _add_random_sites(occ, int(round(0.01 * 396000)), rng)
        grids = [occ]
    elif key == 6:
        xyz = decoder_scale_shell(1024, 64, 12000, rng)
        coords = np.ascontiguousarray(
            np.concatenate([np.zeros((len(xyz), 1), np.int64), xyz], axis=1), dtype=np.int32)
        _COORD_CACHE[key] = coords
        return coords
    else:
        raise KeyError(key)
    coords = _coords_of(grids)
    _COORD_CACHE[key] = coords
    return coords


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returned as fp32."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .to(torch.float32).numpy()


def make_tensors(n: int, cin: int, cout: int, dtype: str, seed_key: int):
    """feats [n,cin], weight [27,cin,cout], bias [cout], all fp32 arrays holding
    values exactly representable in `dtype` (bias always fp32)."""
    rf = np.random.default_rng(2000 + seed_key)
    feats = rf.standard_normal((n, cin), dtype=np.float32)
    rw = np.random.default_rng(3000 + seed_key)
    weight = (rw.standard_normal((27, cin, cout)) / math.sqrt(27 * cin)).astype(np.float32)
    bias = (rw.standard_normal(cout) * 0.1).astype(np.float32)
    if dtype == "bf16":
        feats, weight = round_bf16(feats), round_bf16(weight)
    elif dtype == "f16":
        # numpy's float16 conversion rounds to nearest, ties to even
        feats = feats.astype(np.float16).astype(np.float32)
        weight = weight.astype(np.float16).astype(np.float32)
    elif dtype != "f32":
        raise ValueError(dtype)
    return feats, weight, bias


@dataclasses.dataclass
class Problem:
    config: Config
    res: int
    coords: np.ndarray      # int32 [N,4]
    feats: np.ndarray       # fp32 [N,cin] (bf16-exact for bf16 configs)
    weight: np.ndarray      # fp32 [27,cin,cout]
    bias: np.ndarray        # fp32 [cout]

    @property
    def n(self) -> int:
        return int(self.coords.shape[0])


def make_problem(key: int) -> Problem:
    cfg = CONFIGS[key]
    coords = make_coords(key)
    feats, weight, bias = make_tensors(len(coords), cfg.cin, cfg.cout, cfg.dtype, key)
    return Problem(cfg, cfg.res, coords, feats, weight, bias)
