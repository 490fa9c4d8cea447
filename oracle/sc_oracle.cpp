// sc_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously correct CPU statement of the 3x3x3 submanifold
// sparse convolution over active voxels.  It exists so that the CUDA library
// can be checked against something that shares none of its code: no header,
// no helper, no table and no constant is common to the two.  Only the test
// suite, the package smoke check and the benchmark's CPU-baseline leg load it.
//
// What it follows:
//  * "Running TRELLIS.2 on a Mac (1/3)", section "Swapping out the CUDA
//    libraries one at a time", paragraph "Sparse 3D convolution": a spatial
//    hash of the active voxels; for each kernel position, gather the
//    neighbour's features, multiply by that position's weights, and add the
//    products into the output site.  Outputs are the input sites
//    (submanifold).
//  * "Porting TRELLIS.2 From Python to Rust and Metal", section V "The Kernel
//    That Decided It": a neighbour table built once per resolution level, a
//    gather-GEMM over it with single-precision (here: double) accumulation,
//    bias added in the same pass.
//  * "FABLE_STARTUP_PACKET.md", section 5 (weight-convention table): sparse
//    conv weights are stored (Co, Kd, Kh, Kw, Ci) and reshaped to (Kvol, Ci,
//    Co) for the per-offset gather-GEMM.  Hence W[k][ci][co] with
//    k = 9*kd + 3*kh + kw, kd/kh/kw in {0,1,2}.
//
// Readings where the pages are silent (each also listed in the design notes):
//  * offset k <-> displacement (kd-1, kh-1, kw-1) applied to the (x, y, z)
//    columns of the (batch, x, y, z) coordinates, i.e. the row-major
//    flattening of (Kd, Kh, Kw) with Kd along x;
//  * cross-correlation: tap k reads the voxel AT p + delta_k (the dense
//    Conv3d convention with padding 1);
//  * a neighbour outside [0, res)^3, or in another batch element, is absent;
//  * out-of-range or duplicate input coordinates are errors, never merged;
//    a range error is reported in preference to a duplicate;
//  * output rows are in input row order;
//  * pair lists: for each k, the pairs (nbr[o][k], o) in ascending o;
//  * the bias is added once, after the sum over taps; a NULL bias is zero.
//
// Precision: every product and sum is taken in double.  Inputs arrive as
// float; a bf16 input is first widened to float by the caller, which is exact.

#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

struct VoxelKey {
  int32_t b, x, y, z;
  bool operator==(const VoxelKey& o) const {
    return b == o.b && x == o.x && y == o.y && z == o.z;
  }
};

struct VoxelKeyHash {
  size_t operator()(const VoxelKey& k) const {
    // Any function of the four fields is correct here; equality decides.
    uint64_t h = (uint32_t)k.b;
    h = h * 1000003u + (uint32_t)k.x;
    h = h * 1000003u + (uint32_t)k.y;
    h = h * 1000003u + (uint32_t)k.z;
    return (size_t)(h ^ (h >> 29));
  }
};

// The 27 displacements, k = 9*(dx+1) + 3*(dy+1) + (dz+1).
void displacement(int k, int* dx, int* dy, int* dz) {
  *dx = k / 9 - 1;
  *dy = (k / 3) % 3 - 1;
  *dz = k % 3 - 1;
}

}  // namespace

extern "C" {

// Status codes of this file (independent of the library's own enum).
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_COORD_RANGE = 2, ORACLE_DUPLICATE = 3 };

int oracle_displacement(int k, int* dx, int* dy, int* dz) {
  if (k < 0 || k >= 27) return ORACLE_BAD_ARG;
  displacement(k, dx, dy, dz);
  return ORACLE_OK;
}

// nbr[o*27 + k] = row i with coords[i] == (b_o, x_o+dx_k, y_o+dy_k, z_o+dz_k),
// or -1 when no such row exists.  coords is row-major [n][4] = (b, x, y, z).
int oracle_build_neighbor_table(const int32_t* coords, int64_t n, int32_t res,
                                int32_t* nbr) {
  if (n < 0 || res <= 0 || (n > 0 && (coords == nullptr || nbr == nullptr)))
    return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    const int32_t* c = coords + 4 * i;
    if (c[0] < 0) return ORACLE_COORD_RANGE;
    for (int a = 1; a < 4; ++a)
      if (c[a] < 0 || c[a] >= res) return ORACLE_COORD_RANGE;
  }
  std::unordered_map<VoxelKey, int32_t, VoxelKeyHash> where;
  where.reserve((size_t)n * 2 + 1);
  for (int64_t i = 0; i < n; ++i) {
    const int32_t* c = coords + 4 * i;
    VoxelKey key{c[0], c[1], c[2], c[3]};
    if (!where.emplace(key, (int32_t)i).second) return ORACLE_DUPLICATE;
  }
  for (int64_t o = 0; o < n; ++o) {
    const int32_t* c = coords + 4 * o;
    for (int k = 0; k < 27; ++k) {
      int dx, dy, dz;
      displacement(k, &dx, &dy, &dz);
      int64_t x = (int64_t)c[1] + dx, y = (int64_t)c[2] + dy, z = (int64_t)c[3] + dz;
      int32_t found = -1;
      if (x >= 0 && x < res && y >= 0 && y < res && z >= 0 && z < res) {
        auto it = where.find(VoxelKey{c[0], (int32_t)x, (int32_t)y, (int32_t)z});
        if (it != where.end()) found = it->second;
      }
      nbr[o * 27 + k] = found;
    }
  }
  return ORACLE_OK;
}

// Per-offset pair lists in CSR form.  off[0..27]; for offset k the pairs are
// in[off[k]..off[k+1]) / out[...], listed in ascending output row.  Any of
// in / out may be NULL to only count.  Returns the total pair count.
int64_t oracle_pairs(const int32_t* nbr, int64_t n, int64_t* off, int32_t* in,
                     int32_t* out) {
  int64_t p = 0;
  for (int k = 0; k < 27; ++k) {
    if (off) off[k] = p;
    for (int64_t o = 0; o < n; ++o) {
      int32_t i = nbr[o * 27 + k];
      if (i < 0) continue;
      if (in) in[p] = i;
      if (out) out[p] = (int32_t)o;
      ++p;
    }
  }
  if (off) off[27] = p;
  return p;
}

// out[o][c] = bias[c] + sum_k sum_ci [nbr[o][k] >= 0] feats[nbr[o][k]][ci] * w[k][ci][c]
// for the m output rows whose neighbour rows are given in nbr [m][27] (the
// whole table, or any subset of its rows).  feats: [n][cin], w:
// [27][cin][cout], bias: [cout] or NULL, out: [m][cout].  Every nbr entry
// must lie in [-1, n).  threads <= 0 uses the OpenMP default.
int oracle_conv(const int32_t* nbr, int64_t m, const float* feats, int64_t n,
                int32_t cin, const float* w, int32_t cout, const float* bias,
                double* out, int32_t threads) {
  if (m < 0 || n < 0 || cin <= 0 || cout <= 0) return ORACLE_BAD_ARG;
  if (m == 0) return ORACLE_OK;
  if (!nbr || !w || !out || (n > 0 && !feats)) return ORACLE_BAD_ARG;
  for (int64_t e = 0; e < m * 27; ++e)
    if (nbr[e] < -1 || nbr[e] >= n) return ORACLE_BAD_ARG;
#ifdef _OPENMP
  int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(nt) schedule(dynamic, 64)
#endif
  for (int64_t o = 0; o < m; ++o) {
    std::vector<double> acc((size_t)cout, 0.0);
    for (int k = 0; k < 27; ++k) {
      int32_t i = nbr[o * 27 + k];
      if (i < 0) continue;
      const float* x = feats + (int64_t)i * cin;
      const float* wk = w + (int64_t)k * cin * cout;
      for (int32_t ci = 0; ci < cin; ++ci) {
        double xv = (double)x[ci];
        const float* wrow = wk + (int64_t)ci * cout;
        for (int32_t c = 0; c < cout; ++c) acc[c] += xv * (double)wrow[c];
      }
    }
    for (int32_t c = 0; c < cout; ++c)
      out[o * cout + c] = acc[c] + (bias ? (double)bias[c] : 0.0);
  }
  return ORACLE_OK;
}

// Threads the OpenMP runtime would use (1 when built without OpenMP).
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
