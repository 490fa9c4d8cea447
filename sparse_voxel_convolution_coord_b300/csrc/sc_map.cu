// sc_map.cu -- coordinate hash table and neighbour map on the GPU.
//
// The method ("Running TRELLIS.2 on a Mac (1/3)", Sparse 3D convolution
// paragraph: a spatial hash of the active voxels; "Porting TRELLIS.2 From
// Python to Rust and Metal", section V: a neighbour table built once per
// resolution level) needs, for every active voxel and each of the 27 offsets,
// the row of the neighbour voxel or -1.  Here:
//
//  k_hash_insert     open addressing over a power-of-two table of packed
//                    64-bit slots (key << vbits | row).  A group of kWindow
//                    lanes cooperates on one key: it reads a window of
//                    kWindow consecutive slots in one coalesced load, finds a
//                    duplicate or the first empty slot with one ballot, and
//                    claims it with a 64-bit CAS; windows follow linearly.
//  k_neighbor_query  one thread per voxel; its 26 probes (the centre is the
//                    voxel itself) are issued together, then resolved.  The
//                    block's 128 rows x 27 results are staged in shared memory
//                    and written with coalesced 16-byte stores.  The block
//                    also ORs its rows' presence masks into the tile mask the
//                    convolution uses to skip absent offsets, and adds its
//                    pair count to a global counter.
//  k_pairs_*         CSR pair lists per offset (ascending output row),
//                    built on demand: count, scan, scatter.
#include <algorithm>

#include "sc_internal.cuh"

namespace sc {

constexpr int kWindow = 8;  // lanes (and slots) per cooperative probe window

// ---------------------------------------------------------------------------
// insert

__global__ void __launch_bounds__(256) k_hash_insert(const int4* __restrict__ coords,
                                                     HashParams hp, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int glane = lane % kWindow;
  const int gbase = lane - glane;
  const unsigned gmask = (kWindow == 32) ? 0xffffffffu : (((1u << kWindow) - 1u) << gbase);
  const int64_t group = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kWindow;
  const int64_t ngroups = ((int64_t)gridDim.x * blockDim.x) / kWindow;
  const uint64_t res = (uint64_t)hp.res;
  uint32_t err = 0;

  for (int64_t i = group; i < hp.n; i += ngroups) {
    const int4 c = __ldg(coords + i);
    const bool ok = c.x >= 0 && (unsigned)c.y < (unsigned)hp.res &&
                    (unsigned)c.z < (unsigned)hp.res && (unsigned)c.w < (unsigned)hp.res;
    if (!ok) {
      err |= kStatRange;
      continue;
    }
    if ((uint64_t)c.x >= hp.bmax) {
      err |= kStatKeySpace;
      continue;
    }
    const uint64_t key = (((uint64_t)c.x * res + (uint64_t)c.y) * res + (uint64_t)c.z) * res +
                         (uint64_t)c.w;
    const uint64_t mine = (key << hp.vbits) | (uint64_t)i;
    uint64_t pos = hash_home(key, hp.log2cap) & ~(uint64_t)(kWindow - 1);
    bool done = false;
    for (uint64_t w = 0; w <= hp.cap_mask / kWindow && !done; ++w) {
      const uint64_t s = __ldcg(reinterpret_cast<const unsigned long long*>(hp.slots) + pos + glane);
      const unsigned same = __ballot_sync(gmask, s != kEmptySlot && (s >> hp.vbits) == key) & gmask;
      if (same) {
        err |= kStatDuplicate;
        done = true;
        break;
      }
      unsigned empty = __ballot_sync(gmask, s == kEmptySlot) & gmask;
      while (empty) {
        const int leader = __ffs(empty) - 1;
        unsigned long long old = 0;
        if (lane == leader)
          old = atomicCAS(reinterpret_cast<unsigned long long*>(hp.slots) + pos + (leader - gbase),
                          (unsigned long long)kEmptySlot, (unsigned long long)mine);
        old = __shfl_sync(gmask, old, leader);
        if (old == kEmptySlot) {
          done = true;
          break;
        }
        if ((old >> hp.vbits) == key) {
          err |= kStatDuplicate;
          done = true;
          break;
        }
        empty &= ~(1u << leader);
      }
      pos = (pos + kWindow) & hp.cap_mask;
    }
    if (!done) err |= kStatTableFull;
  }
  if (err && glane == 0) atomicOr(status, err);
}

// ---------------------------------------------------------------------------
// query

// Resolve a key whose first probe (the window start) returned `s`.
__device__ __forceinline__ int32_t finish_probe(const HashParams& hp, uint64_t key, uint64_t pos,
                                                uint64_t s) {
  const uint64_t vmask = (1ull << hp.vbits) - 1ull;
  for (uint64_t it = 0; it <= hp.cap_mask; ++it) {
    if (s == kEmptySlot) return -1;
    if ((s >> hp.vbits) == key) return (int32_t)(s & vmask);
    pos = (pos + 1) & hp.cap_mask;
    s = __ldg(reinterpret_cast<const unsigned long long*>(hp.slots) + pos);
  }
  return -1;
}

__global__ void __launch_bounds__(kTileRows) k_neighbor_query(
    const int4* __restrict__ coords, HashParams hp, int32_t* __restrict__ nbr,
    uint32_t* __restrict__ tile_mask, unsigned long long* pair_count, uint32_t* status,
    bool pad_tiles) {
  __shared__ __align__(16) int32_t s_nbr[kTileRows * kTaps];
  __shared__ uint32_t s_or[kTileRows / 32];
  __shared__ uint32_t s_cnt[kTileRows / 32];
  const int64_t row0 = (int64_t)blockIdx.x * kTileRows;
  const int64_t o = row0 + threadIdx.x;
  uint32_t mask = 0;
  if (o < hp.n) {
    const int4 c = __ldg(coords + o);
    const int64_t res = hp.res;
    const uint64_t key0 = (((uint64_t)c.x * res + (uint64_t)c.y) * res + (uint64_t)c.z) * res +
                          (uint64_t)c.w;
    uint64_t pos[kTaps], s[kTaps];
    bool inside[kTaps];
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
      const int dx = k / 9 - 1, dy = (k / 3) % 3 - 1, dz = k % 3 - 1;
      inside[k] = (unsigned)(c.y + dx) < (unsigned)hp.res &&
                  (unsigned)(c.z + dy) < (unsigned)hp.res && (unsigned)(c.w + dz) < (unsigned)hp.res;
      const uint64_t key = key0 + (uint64_t)((int64_t)dx * res * res + (int64_t)dy * res + dz);
      pos[k] = hash_home(key, hp.log2cap) & ~(uint64_t)(kWindow - 1);
      s[k] = (inside[k] && k != kCentre)
                 ? __ldg(reinterpret_cast<const unsigned long long*>(hp.slots) + pos[k])
                 : kEmptySlot;
    }
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
      const int dx = k / 9 - 1, dy = (k / 3) % 3 - 1, dz = k % 3 - 1;
      int32_t r;
      if (k == kCentre) {
        r = (int32_t)o;
      } else {
        const uint64_t key = key0 + (uint64_t)((int64_t)dx * res * res + (int64_t)dy * res + dz);
        r = inside[k] ? finish_probe(hp, key, pos[k], s[k]) : -1;
      }
      s_nbr[threadIdx.x * kTaps + k] = r;
      mask |= (r >= 0 ? 1u : 0u) << k;
    }
  } else {
#pragma unroll
    for (int k = 0; k < kTaps; ++k) s_nbr[threadIdx.x * kTaps + k] = -1;
  }
  const uint32_t wor = __reduce_or_sync(0xffffffffu, mask);
  const uint32_t wcnt = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(mask));
  if ((threadIdx.x & 31) == 0) {
    s_or[threadIdx.x >> 5] = wor;
    s_cnt[threadIdx.x >> 5] = wcnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0, cnt = 0;
    for (int w = 0; w < kTileRows / 32; ++w) {
      m |= s_or[w];
      cnt += s_cnt[w];
    }
    tile_mask[blockIdx.x] = m;
    atomicAdd(pair_count, (unsigned long long)cnt);
  }
  const int64_t rows = pad_tiles ? (int64_t)kTileRows : min((int64_t)kTileRows, hp.n - row0);
  const int total = (int)rows * kTaps;
  int32_t* dst = nbr + row0 * kTaps;  // 16-byte aligned: row0 * 27 * 4 = blockIdx * 13824
  const int nvec = total >> 2;
  for (int i = threadIdx.x; i < nvec; i += kTileRows)
    reinterpret_cast<int4*>(dst)[i] = reinterpret_cast<const int4*>(s_nbr)[i];
  for (int i = (nvec << 2) + threadIdx.x; i < total; i += kTileRows) dst[i] = s_nbr[i];
  (void)status;
}

cudaError_t launch_hash_insert(const int32_t* coords, const HashParams& hp, uint32_t* status,
                               cudaStream_t s) {
  if (hp.n == 0) return cudaSuccess;
  const int64_t threads = hp.n * kWindow;
  const int64_t blocks = std::min<int64_t>((threads + 255) / 256, 148LL * 64);
  k_hash_insert<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const int4*>(coords), hp,
                                                  status);
  return cudaGetLastError();
}

cudaError_t launch_neighbor_query(const int32_t* coords, const HashParams& hp, int32_t* nbr,
                                  uint32_t* tile_mask, unsigned long long* pair_count,
                                  uint32_t* status, bool pad_tiles, cudaStream_t s) {
  if (hp.n == 0) return cudaSuccess;
  const int64_t blocks = (hp.n + kTileRows - 1) / kTileRows;
  k_neighbor_query<<<(unsigned)blocks, kTileRows, 0, s>>>(
      reinterpret_cast<const int4*>(coords), hp, nbr, tile_mask, pair_count, status, pad_tiles);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// pair lists (CSR per offset, ascending output row within an offset)

__global__ void __launch_bounds__(kTileRows) k_pairs_count(const int32_t* __restrict__ nbr,
                                                           int64_t n, int64_t nblocks,
                                                           int64_t* __restrict__ counts) {
  const int64_t o = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
  for (int k = 0; k < kTaps; ++k) {
    const bool p = o < n && nbr[o * kTaps + k] >= 0;
    const int c = __syncthreads_count(p);
    if (threadIdx.x == 0) counts[(int64_t)k * nblocks + blockIdx.x] = c;
  }
}

// Exclusive scan of `len` counts in place by one block of 1024 threads;
// total[0] receives the sum.
__global__ void __launch_bounds__(1024) k_scan_exclusive(int64_t* data, int64_t len,
                                                         int64_t* total) {
  __shared__ int64_t s_warp[32];
  __shared__ int64_t s_carry;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t base = 0; base < len; base += 1024) {
    const int64_t i = base + threadIdx.x;
    const int64_t v = i < len ? data[i] : 0;
    int64_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int64_t w = s_warp[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += y;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int64_t incl = x + (warp > 0 ? s_warp[warp - 1] : 0) + s_carry;
    if (i < len) data[i] = incl - v;
    __syncthreads();
    if (threadIdx.x == 1023) s_carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) total[0] = s_carry;
}

__global__ void __launch_bounds__(kTileRows) k_pairs_write(const int32_t* __restrict__ nbr,
                                                           int64_t n, int64_t nblocks,
                                                           const int64_t* __restrict__ offs,
                                                           int32_t* pin, int32_t* pout) {
  __shared__ int s_warp[kTileRows / 32];
  const int64_t o = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int k = 0; k < kTaps; ++k) {
    const int32_t i = o < n ? nbr[o * kTaps + k] : -1;
    const bool p = i >= 0;
    const unsigned b = __ballot_sync(0xffffffffu, p);
    if (lane == 0) s_warp[warp] = __popc(b);
    __syncthreads();
    int before = __popc(b & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    if (p) {
      const int64_t at = offs[(int64_t)k * nblocks + blockIdx.x] + before;
      if (pin) pin[at] = i;
      if (pout) pout[at] = (int32_t)o;
    }
    __syncthreads();
  }
}

__global__ void k_pairs_offsets(const int64_t* offs, int64_t nblocks, const int64_t* total,
                                int64_t* off28) {
  const int k = threadIdx.x;
  if (k < kTaps) off28[k] = offs[(int64_t)k * nblocks];
  if (k == kTaps) off28[kTaps] = total[0];
}

size_t pairs_scratch_bytes(int64_t n) {
  const int64_t nblocks = (n + kTileRows - 1) / kTileRows;
  return (size_t)(kTaps * nblocks + 1 + 28) * sizeof(int64_t);
}

cudaError_t launch_pairs(const sc_map* m, int64_t* off_host, int32_t* in, int32_t* out,
                         void* scratch, cudaStream_t s) {
  const int64_t n = m->n;
  const int64_t nblocks = (n + kTileRows - 1) / kTileRows;
  int64_t* counts = static_cast<int64_t*>(scratch);
  int64_t* total = counts + kTaps * nblocks;
  int64_t* off28 = total + 1;
  k_pairs_count<<<(unsigned)nblocks, kTileRows, 0, s>>>(m->nbr, n, nblocks, counts);
  k_scan_exclusive<<<1, 1024, 0, s>>>(counts, kTaps * nblocks, total);
  if (in || out)
    k_pairs_write<<<(unsigned)nblocks, kTileRows, 0, s>>>(m->nbr, n, nblocks, counts, in, out);
  k_pairs_offsets<<<1, 32, 0, s>>>(counts, nblocks, total, off28);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(off_host, off28, 28 * sizeof(int64_t), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

}  // namespace sc
