// sc_mesh.cu -- dual-grid mesh extraction over a built map.
//
// "Running TRELLIS.2 on a Mac (1/3)", Mesh extraction paragraph: the mesh
// comes out of a dual voxel grid through a hash map (coordinate-to-index
// tables, the connected voxels of each edge) and quads split into triangles
// by how well their normals align; "Porting TRELLIS.2 From Python to Rust and
// Metal" reports the same step as a compact hash map and a parallel loop.
// The readings taken (they are the oracle's):
//  * voxel (x, y, z) is the cell [x, x+1] x [y, y+1] x [z, z+1]; it carries a
//    dual vertex and owns the three primal edges from its min corner along
//    +x, +y, +z; a 6-bit flag per voxel: bit a says its a-edge crosses the
//    surface, bit 3 + a that the edge's start point is inside;
//  * a crossing a-edge is shared by the voxels at offsets 0, -e_b, -e_b - e_c,
//    -e_c from its owner ((a, b, c) cyclic); when all four are active they
//    form a quad in that order, reversed when the start point is outside;
//  * a quad splits along q0-q2 or q1-q3, whichever gives the two triangles'
//    unit normals the larger dot product; a tie keeps q0-q2;
//  * quads are listed by owner row, then axis; two triangles per quad.
// The four voxels of an edge are all within the owner's 3x3x3 neighbourhood,
// so their rows are read from the map's neighbour table (which the
// coordinate hash built): no probing here.  Kernels: per-voxel quad counts,
// their exclusive scan, the quads, and one thread per quad for the split,
// in fp64 with every product and sum rounded separately (no fused
// multiply-add), the sequence the CPU statement of the same formulas takes.
#include "sc_internal.cuh"

namespace sc {

constexpr int kMeshThreads = 256;

// Offsets k of the cells 0, -e_b, -e_b - e_c, -e_c around an a-edge's owner
// (k = 9 (dx + 1) + 3 (dy + 1) + (dz + 1)).
__constant__ int8_t c_edge_taps[3][4] = {{13, 10, 9, 12}, {13, 12, 3, 4}, {13, 4, 1, 10}};

__device__ __forceinline__ int32_t nbr_at(const int32_t* nbr_t, int64_t o, int k) {
  return __ldg(nbr_t + (o / kTileRows) * (kTileRows * kTaps) + k * kTileRows + (o % kTileRows));
}

// Rows of the quad around voxel o's a-edge, in output order; false if the
// edge is not flagged or a cell is inactive.
__device__ __forceinline__ bool edge_quad(const int32_t* nbr_t, int64_t o, uint32_t f, int a,
                                          int4& q) {
  if (!((f >> a) & 1u)) return false;
  int32_t r[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = nbr_at(nbr_t, o, c_edge_taps[a][j]);
  if (r[0] < 0 || r[1] < 0 || r[2] < 0 || r[3] < 0) return false;
  q = ((f >> (3 + a)) & 1u) ? make_int4(r[0], r[1], r[2], r[3]) : make_int4(r[3], r[2], r[1], r[0]);
  return true;
}

__global__ void __launch_bounds__(kMeshThreads) k_quad_counts(const int32_t* __restrict__ nbr_t,
                                                              int64_t n,
                                                              const uint8_t* __restrict__ flags,
                                                              int32_t* __restrict__ counts) {
  const int64_t o = (int64_t)blockIdx.x * kMeshThreads + threadIdx.x;
  if (o >= n) return;
  const uint32_t f = __ldg(flags + o);
  int c = 0;
  int4 q;
#pragma unroll
  for (int a = 0; a < 3; ++a) c += edge_quad(nbr_t, o, f, a, q) ? 1 : 0;
  counts[o] = c;
}

__global__ void __launch_bounds__(kMeshThreads) k_quads(const int32_t* __restrict__ nbr_t,
                                                        int64_t n,
                                                        const uint8_t* __restrict__ flags,
                                                        const int32_t* __restrict__ first,
                                                        int4* __restrict__ quads) {
  const int64_t o = (int64_t)blockIdx.x * kMeshThreads + threadIdx.x;
  if (o >= n) return;
  const uint32_t f = __ldg(flags + o);
  int64_t at = __ldg(first + o);
  int4 q;
#pragma unroll
  for (int a = 0; a < 3; ++a)
    if (edge_quad(nbr_t, o, f, a, q)) quads[at++] = q;
}

struct D3 {
  double x, y, z;
};
__device__ __forceinline__ D3 sub3(D3 a, D3 b) {
  return {__dsub_rn(a.x, b.x), __dsub_rn(a.y, b.y), __dsub_rn(a.z, b.z)};
}
__device__ __forceinline__ D3 cross3(D3 a, D3 b) {
  return {__dsub_rn(__dmul_rn(a.y, b.z), __dmul_rn(a.z, b.y)),
          __dsub_rn(__dmul_rn(a.z, b.x), __dmul_rn(a.x, b.z)),
          __dsub_rn(__dmul_rn(a.x, b.y), __dmul_rn(a.y, b.x))};
}
__device__ __forceinline__ double dot3(D3 a, D3 b) {
  return __dadd_rn(__dadd_rn(__dmul_rn(a.x, b.x), __dmul_rn(a.y, b.y)), __dmul_rn(a.z, b.z));
}
// Unit normal of triangle (p0, p1, p2); the zero vector stays zero.
__device__ __forceinline__ D3 unit_normal(D3 p0, D3 p1, D3 p2) {
  const D3 nrm = cross3(sub3(p1, p0), sub3(p2, p0));
  const double len = __dsqrt_rn(dot3(nrm, nrm));
  if (!(len > 0.0)) return nrm;
  return {__ddiv_rn(nrm.x, len), __ddiv_rn(nrm.y, len), __ddiv_rn(nrm.z, len)};
}

__global__ void __launch_bounds__(kMeshThreads) k_triangulate(const int4* __restrict__ quads,
                                                              int64_t nq,
                                                              const float* __restrict__ verts,
                                                              int32_t* __restrict__ tris) {
  const int64_t i = (int64_t)blockIdx.x * kMeshThreads + threadIdx.x;
  if (i >= nq) return;
  const int4 q = __ldg(quads + i);
  auto vtx = [&](int32_t r) -> D3 {
    const float* v = verts + (int64_t)r * 3;
    return {(double)__ldg(v), (double)__ldg(v + 1), (double)__ldg(v + 2)};
  };
  const D3 p0 = vtx(q.x), p1 = vtx(q.y), p2 = vtx(q.z), p3 = vtx(q.w);
  const double cos02 = dot3(unit_normal(p0, p1, p2), unit_normal(p0, p2, p3));
  const double cos13 = dot3(unit_normal(p0, p1, p3), unit_normal(p1, p2, p3));
  int32_t* t = tris + i * 6;
  if (cos13 > cos02) {
    t[0] = q.x; t[1] = q.y; t[2] = q.w;
    t[3] = q.y; t[4] = q.z; t[5] = q.w;
  } else {
    t[0] = q.x; t[1] = q.y; t[2] = q.z;
    t[3] = q.x; t[4] = q.z; t[5] = q.w;
  }
}

namespace {
unsigned mesh_blocks(int64_t n) { return (unsigned)((n + kMeshThreads - 1) / kMeshThreads); }
}  // namespace

cudaError_t launch_quad_counts(const sc_map* m, const uint8_t* flags, int32_t* counts,
                               cudaStream_t s) {
  k_quad_counts<<<mesh_blocks(m->n), kMeshThreads, 0, s>>>(m->nbr, m->n, flags, counts);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quads(const sc_map* m, const uint8_t* flags, const int32_t* first,
                         int32_t* quads, cudaStream_t s) {
  k_quads<<<mesh_blocks(m->n), kMeshThreads, 0, s>>>(m->nbr, m->n, flags, first,
                                                     reinterpret_cast<int4*>(quads));
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_triangulate(const int32_t* quads, int64_t nq, const float* verts,
                               int32_t* tris, cudaStream_t s) {
  if (nq == 0) return cudaSuccess;
  k_triangulate<<<mesh_blocks(nq), kMeshThreads, 0, s>>>(reinterpret_cast<const int4*>(quads),
                                                         nq, verts, tris);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace sc
