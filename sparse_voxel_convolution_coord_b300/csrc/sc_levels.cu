// sc_levels.cu -- moving a sparse voxel set between resolution levels.
//
// The trellis2mlx README names the operations (its pipeline list's
// "Upsample" stage: the decoder's subdivision predictions become the
// high-resolution coordinates; its project layout: a sparse UNet decoder
// upsampling by Channel2Spatial) without fixing their details; the library
// takes these readings:
//
//  subdivision     voxel (b, x, y, z) at resolution R has 8 children at 2R,
//                  child o at (b, 2x + (o >> 2 & 1), 2y + (o >> 1 & 1),
//                  2z + (o & 1)) (the row-major flattening the 27 offsets
//                  use); an 8-bit mask per voxel selects them; children are
//                  listed parent by parent in input order, ascending o.
//                  Kernels: per-parent child counts, their exclusive scan,
//                  a scatter of the children.
//  Channel2Spatial child o of parent i takes channels c * 8 + o of the
//                  parent's 8C (the sub-voxel index runs fastest, as in the
//                  dense pixel shuffle).  One warp per parent reads its row
//                  once and writes each present child's row.
//  the way down    the parents of a voxel set at 2R are the distinct
//                  (b, x >> 1, y >> 1, z >> 1), in (b, x, y, z) order, each
//                  with the row of its child o (or -1).  The parents' packed
//                  keys are radix-sorted with the rows (9-bit stable passes,
//                  sc_sort.cu); the first of each run of equal keys starts a
//                  parent, an exclusive scan of those starts numbers them,
//                  and a scatter fills the child table (tile-major, as the
//                  convolutions read it) and each child's parent.  Two rows
//                  with one parent and one octant are duplicates: an error.
//  2x2x2 stride-2  down: out[p] = bias + sum_o feats[child_of[p][o]] @ W[o];
//  convolutions    up:   out[child] = bias + feats[parent] @ W[octant].
//                  Both run on the gather-GEMM kernels of sc_conv_tc.cu /
//                  sc_conv_simt.cu with 8 taps.  Down reads the child table
//                  as its neighbour table.  Up reads, for each child, its
//                  parent at the child's own octant only; its positions are
//                  the child rows grouped by octant (a stable 3-bit counting
//                  sort), so that a 128-position tile spans one or two
//                  octants and the kernel skips the rest, and the epilogue
//                  writes each position to its child row.
#include <algorithm>
#include <cstring>

#include "sc_internal.cuh"

namespace sc {

constexpr int kLevelThreads = 256;

__device__ __forceinline__ int octant_of(const int4 c) {
  return ((c.y & 1) << 2) | ((c.z & 1) << 1) | (c.w & 1);
}

// ---------------------------------------------------------------------------
// subdivision

__global__ void __launch_bounds__(kLevelThreads) k_child_counts(const int4* __restrict__ coords,
                                                                const uint8_t* __restrict__ mask,
                                                                int64_t n, int res,
                                                                int32_t* __restrict__ counts,
                                                                uint32_t* status) {
  const int64_t i = (int64_t)blockIdx.x * kLevelThreads + threadIdx.x;
  uint32_t err = 0;
  if (i < n) {
    const int4 c = __ldg(coords + i);
    const bool ok = c.x >= 0 && (unsigned)c.y < (unsigned)res && (unsigned)c.z < (unsigned)res &&
                    (unsigned)c.w < (unsigned)res;
    if (!ok) err = kStatRange;
    counts[i] = mask ? __popc((uint32_t)__ldg(mask + i)) : 8;
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (err && (threadIdx.x & 31) == 0) atomicOr(status, err);
}

__global__ void __launch_bounds__(kLevelThreads) k_subdivide(
    const int4* __restrict__ coords, const uint8_t* __restrict__ mask, int64_t n,
    const int32_t* __restrict__ first, int4* __restrict__ child_coords,
    int32_t* __restrict__ parent, int32_t* __restrict__ offset, int32_t* __restrict__ child_of) {
  const int64_t i = (int64_t)blockIdx.x * kLevelThreads + threadIdx.x;
  if (i >= n) return;
  const int4 c = __ldg(coords + i);
  const uint32_t m = mask ? (uint32_t)__ldg(mask + i) : 0xffu;
  int32_t row = __ldg(first + i);
#pragma unroll
  for (int o = 0; o < 8; ++o) {
    const bool has = (m >> o) & 1u;
    if (child_of) child_of[i * 8 + o] = has ? row : -1;
    if (has) {
      child_coords[row] =
          make_int4(c.x, 2 * c.y + ((o >> 2) & 1), 2 * c.z + ((o >> 1) & 1), 2 * c.w + (o & 1));
      if (parent) parent[row] = (int32_t)i;
      if (offset) offset[row] = o;
      ++row;
    }
  }
}

// One warp per parent: the parent's 8C values (esz-byte elements) are read
// once, in order, and child o's C values (channels c * 8 + o) written.
template <typename T>
__global__ void __launch_bounds__(kLevelThreads) k_channel_to_spatial(
    const T* __restrict__ feats, const int32_t* __restrict__ parent,
    const int32_t* __restrict__ offset, int64_t m, int c, T* __restrict__ out) {
  const int64_t child = (int64_t)blockIdx.x * (kLevelThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (child >= m) return;
  const int64_t p = __ldg(parent + child);
  const int o = __ldg(offset + child);
  const T* src = feats + p * (int64_t)c * 8 + o;
  T* dst = out + child * (int64_t)c;
  for (int j = lane; j < c; j += 32) dst[j] = src[(int64_t)j * 8];
}

// ---------------------------------------------------------------------------
// the way down

template <typename K>
__global__ void __launch_bounds__(kLevelThreads) k_parent_keys(const int4* __restrict__ coords,
                                                               int64_t n, int res, int nbatch,
                                                               K* __restrict__ keys,
                                                               uint32_t* __restrict__ octs,
                                                               uint32_t* status) {
  const int64_t i = (int64_t)blockIdx.x * kLevelThreads + threadIdx.x;
  uint32_t err = 0;
  if (i < n) {
    const int4 c = __ldg(coords + i);
    const bool ok = c.x >= 0 && c.x < nbatch && (unsigned)c.y < (unsigned)res &&
                    (unsigned)c.z < (unsigned)res && (unsigned)c.w < (unsigned)res;
    if (!ok) err = kStatRange;
    const K pr = (K)((res + 1) / 2);
    // out-of-range rows still get a key (the build fails; nothing is read
    // out of bounds on the way)
    keys[i] = ok ? (((K)c.x * pr + (K)(c.y >> 1)) * pr + (K)(c.z >> 1)) * pr + (K)(c.w >> 1)
                 : (K)0;
    octs[i] = (uint32_t)octant_of(c);
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (err && (threadIdx.x & 31) == 0) atomicOr(status, err);
}

// A sorted position starts a parent where its key differs from the one before.
template <typename K>
__global__ void __launch_bounds__(kLevelThreads) k_run_starts(const K* __restrict__ keys, int64_t n,
                                                              int32_t* __restrict__ starts) {
  const int64_t j = (int64_t)blockIdx.x * kLevelThreads + threadIdx.x;
  if (j < n) starts[j] = (j == 0 || keys[j] != keys[j - 1]) ? 1 : 0;
}

// Sorted position j (row i = rows[j]) belongs to parent p = (parents
// started before j) + start[j] - 1.
__global__ void __launch_bounds__(kLevelThreads) k_assign_parents(
    const int4* __restrict__ coords, const int32_t* __restrict__ rows,
    const int32_t* __restrict__ starts, const int32_t* __restrict__ excl, int64_t n,
    int32_t* __restrict__ down_nbr, uint32_t* __restrict__ down_mask,
    int32_t* __restrict__ parent_of, int4* __restrict__ parent_coords, uint32_t* status) {
  const int64_t j = (int64_t)blockIdx.x * kLevelThreads + threadIdx.x;
  uint32_t err = 0;
  if (j < n) {
    const int32_t i = __ldg(rows + j);
    const int32_t p = __ldg(excl + j) + __ldg(starts + j) - 1;
    const int4 c = __ldg(coords + i);
    const int o = octant_of(c);
    parent_of[i] = p;
    int32_t* slot = down_nbr + ((int64_t)(p / kTileRows) * 8 + o) * kTileRows + (p % kTileRows);
    if (atomicCAS(slot, -1, i) != -1) err = kStatDuplicate;
    atomicOr(down_mask + p / kTileRows, 1u << o);
    if (__ldg(starts + j)) parent_coords[p] = make_int4(c.x, c.y >> 1, c.z >> 1, c.w >> 1);
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (err && (threadIdx.x & 31) == 0) atomicOr(status, err);
}

// Position q of the octant-grouped order: child row i = rows[q]; its only
// tap is its own octant (the parent's row), the others absent.  Pad
// positions of the last tile have no row.  One block per tile.
__global__ void __launch_bounds__(kTileRows) k_up_table(const int32_t* __restrict__ rows,
                                                       const uint32_t* __restrict__ octs,
                                                       const int32_t* __restrict__ parent_of,
                                                       int64_t n, int32_t* __restrict__ up_nbr,
                                                       int32_t* __restrict__ up_row,
                                                       uint32_t* __restrict__ up_mask) {
  __shared__ uint32_t s_or[kTileRows / 32];
  const int64_t q = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
  int32_t i = -1, par = -1;
  int o = 0;
  if (q < n) {
    i = __ldg(rows + q);
    o = (int)__ldg(octs + i);
    par = __ldg(parent_of + i);
  }
  int32_t* blk = up_nbr + (int64_t)blockIdx.x * 8 * kTileRows + threadIdx.x;
#pragma unroll
  for (int t = 0; t < 8; ++t) blk[t * kTileRows] = (i >= 0 && t == o) ? par : -1;
  up_row[q] = i;
  const uint32_t w = __reduce_or_sync(0xffffffffu, i >= 0 ? 1u << o : 0u);
  if ((threadIdx.x & 31) == 0) s_or[threadIdx.x >> 5] = w;
  __syncthreads();
  if (threadIdx.x == 0) up_mask[blockIdx.x] = s_or[0] | s_or[1] | s_or[2] | s_or[3];
}

// Row-major child table [np][8] from the tile-major one.
__global__ void __launch_bounds__(kLevelThreads) k_child_table(const int32_t* __restrict__ down_nbr,
                                                               int64_t np,
                                                               int32_t* __restrict__ out) {
  const int64_t e = (int64_t)blockIdx.x * kLevelThreads + threadIdx.x;
  if (e >= np * 8) return;
  const int64_t p = e >> 3;
  const int o = (int)(e & 7);
  out[e] = __ldg(down_nbr + ((p / kTileRows) * 8 + o) * kTileRows + (p % kTileRows));
}

namespace {
unsigned blocks_for(int64_t n, int per) { return (unsigned)((n + per - 1) / per); }
}  // namespace

cudaError_t launch_child_counts(const int32_t* coords, const uint8_t* mask, int64_t n, int res,
                                int32_t* counts, uint32_t* status, cudaStream_t s) {
  k_child_counts<<<blocks_for(n, kLevelThreads), kLevelThreads, 0, s>>>(
      reinterpret_cast<const int4*>(coords), mask, n, res, counts, status);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_subdivide(const int32_t* coords, const uint8_t* mask, int64_t n,
                             const int32_t* first, int32_t* child_coords, int32_t* parent,
                             int32_t* offset, int32_t* child_of, cudaStream_t s) {
  k_subdivide<<<blocks_for(n, kLevelThreads), kLevelThreads, 0, s>>>(
      reinterpret_cast<const int4*>(coords), mask, n, first, reinterpret_cast<int4*>(child_coords),
      parent, offset, child_of);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_channel_to_spatial(const void* feats, const int32_t* parent,
                                      const int32_t* offset, int64_t m, int c, int esize,
                                      void* out, cudaStream_t s) {
  const unsigned blocks = blocks_for(m, kLevelThreads / 32);
  if (esize == 4)
    k_channel_to_spatial<float><<<blocks, kLevelThreads, 0, s>>>(
        static_cast<const float*>(feats), parent, offset, m, c, static_cast<float*>(out));
  else
    k_channel_to_spatial<uint16_t><<<blocks, kLevelThreads, 0, s>>>(
        static_cast<const uint16_t*>(feats), parent, offset, m, c, static_cast<uint16_t*>(out));
  note_launches(1);
  return cudaGetLastError();
}

// Scratch of a level-map build over n rows with `kbytes`-byte keys.
size_t level_scratch_bytes(int64_t n, int kbytes) {
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t nn = (size_t)std::max<int64_t>(n, 1);
  return 2 * up(nn * kbytes) + 2 * up(nn * 4)  // keys, rows (two buffers each)
         + up(nn * 4)                          // octants
         + 2 * up(nn * 4)                      // run starts, their scan
         + up(std::max(sort_scratch_bytes(n, 512), scan_scratch_bytes(n))) + up(16);
}

// The way down: fills h's tables from n fine rows; the number of parents is
// left in *np_dev (device int64).
template <typename K>
cudaError_t build_level_tables(const int32_t* coords, int64_t n, int res, int nbatch, int key_bits,
                               void* scratch, int32_t* down_nbr, uint32_t* down_mask,
                               int32_t* parent_of, int32_t* parent_coords, int32_t* up_nbr,
                               int32_t* up_row, uint32_t* up_mask, int64_t* np_dev,
                               uint32_t* status, cudaStream_t s) {
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t nn = (size_t)std::max<int64_t>(n, 1);
  uint8_t* p = static_cast<uint8_t*>(scratch);
  K* keys[2];
  int32_t* rows[2];
  keys[0] = reinterpret_cast<K*>(p);
  p += up(nn * sizeof(K));
  keys[1] = reinterpret_cast<K*>(p);
  p += up(nn * sizeof(K));
  rows[0] = reinterpret_cast<int32_t*>(p);
  p += up(nn * 4);
  rows[1] = reinterpret_cast<int32_t*>(p);
  p += up(nn * 4);
  uint32_t* octs = reinterpret_cast<uint32_t*>(p);
  p += up(nn * 4);
  int32_t* starts = reinterpret_cast<int32_t*>(p);
  p += up(nn * 4);
  int32_t* excl = reinterpret_cast<int32_t*>(p);
  p += up(nn * 4);
  void* work = p;

  const int4* c4 = reinterpret_cast<const int4*>(coords);
  const int64_t ntiles = (n + kTileRows - 1) / kTileRows;
  cudaError_t e = cudaMemsetAsync(down_nbr, 0xff, (size_t)ntiles * 8 * kTileRows * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(down_mask, 0, (size_t)ntiles * 4, s);
  if (e != cudaSuccess) return e;
  k_parent_keys<K><<<blocks_for(n, kLevelThreads), kLevelThreads, 0, s>>>(c4, n, res, nbatch,
                                                                          keys[0], octs, status);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // Radix sort of (parent key, row), 9 bits a pass, least significant first
  // (key_bits >= 1, so the rows are always written by a pass).
  int cur = 0;
  for (int shift = 0; shift < key_bits; shift += 9) {
    const int bits = std::min(9, key_bits - shift);
    e = sort_pass<K>(keys[cur], shift == 0 ? nullptr : rows[cur], keys[cur ^ 1], rows[cur ^ 1],
                     n, shift, bits, work, s);
    if (e != cudaSuccess) return e;
    cur ^= 1;
  }
  k_run_starts<K><<<blocks_for(n, kLevelThreads), kLevelThreads, 0, s>>>(keys[cur], n, starts);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = scan_exclusive(starts, excl, n, np_dev, work, s);
  if (e != cudaSuccess) return e;
  k_assign_parents<<<blocks_for(n, kLevelThreads), kLevelThreads, 0, s>>>(
      c4, rows[cur], starts, excl, n, down_nbr, down_mask, parent_of,
      reinterpret_cast<int4*>(parent_coords), status);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // The transposed convolution's positions: child rows grouped by octant.
  e = sort_pass<uint32_t>(octs, nullptr, reinterpret_cast<uint32_t*>(keys[cur ^ 1]),
                          rows[cur ^ 1], n, 0, 3, work, s);
  if (e != cudaSuccess) return e;
  k_up_table<<<(unsigned)ntiles, kTileRows, 0, s>>>(rows[cur ^ 1], octs, parent_of, n, up_nbr,
                                                   up_row, up_mask);
  note_launches(1);
  return cudaGetLastError();
}

template cudaError_t build_level_tables<uint32_t>(const int32_t*, int64_t, int, int, int, void*,
                                                  int32_t*, uint32_t*, int32_t*, int32_t*,
                                                  int32_t*, int32_t*, uint32_t*, int64_t*,
                                                  uint32_t*, cudaStream_t);
template cudaError_t build_level_tables<unsigned long long>(const int32_t*, int64_t, int, int, int,
                                                            void*, int32_t*, uint32_t*, int32_t*,
                                                            int32_t*, int32_t*, int32_t*,
                                                            uint32_t*, int64_t*, uint32_t*,
                                                            cudaStream_t);

cudaError_t launch_child_table(const int32_t* down_nbr, int64_t np, int32_t* out, cudaStream_t s) {
  if (np == 0) return cudaSuccess;
  k_child_table<<<blocks_for(np * 8, kLevelThreads), kLevelThreads, 0, s>>>(down_nbr, np, out);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace sc
