// sc_map.cu -- coordinate hash table and neighbour map on the GPU.
//
// The method ("Running TRELLIS.2 on a Mac (1/3)", Sparse 3D convolution
// paragraph: a spatial hash of the active voxels; "Porting TRELLIS.2 From
// Python to Rust and Metal", section V: a neighbour table built once per
// resolution level) needs, for every active voxel and each of the 27 offsets,
// the row of the neighbour voxel or -1.  Here:
//
//  k_hash_insert     open addressing over a power-of-two table of packed
//                    64-bit slots (32-bit keys: key << 32 | moved flag << 31 |
//                    row; otherwise key << vbits | row) with brick-local home
//                    slots and double-hashing probes (sc_internal.cuh).  The
//                    warp inserts its 32 keys in synchronous probing rounds:
//                    in each round every lane whose key is still pending
//                    claims its next probe slot with one 64-bit CAS, and a
//                    ballot ends the rounds once no lane is pending.  The CAS
//                    returns the occupant, so a duplicate key is seen when
//                    its twin's slot is reached.  Errors are OR-reduced per
//                    warp.
//  k_neighbor_query  one thread per (voxel, neighbour column dx, dy): the
//                    three neighbours dz = -1, 0, 1 of the column are probed
//                    with three independent loads (brick-local homes put a
//                    warp's loads, 32 consecutive voxels on one column, on
//                    few cache lines), collisions followed along the probe
//                    sequence.  With 32-bit keys a lookup stops at its home
//                    slot on its key, an empty slot, or another key whose
//                    moved flag is clear.  The tile-major output
//                    [tile][27][128] is written coalesced (a warp writes 32
//                    consecutive rows of one offset).  Each block ORs its
//                    rows' presence bits into the tile mask the convolution
//                    uses to skip absent offsets, and adds its pair count to
//                    one of 32 global counters.  Used up to 2^20 voxels;
//                    from 2^18 voxels each thread takes three columns.
//  k_neighbor_query32  (32-bit keys, 2^20 voxels and more) one thread per
//                    voxel: the 27 cells around it fall in 2 x 2 x 2 bricks
//                    whose group hashes follow from one by additions, so all
//                    26 home-slot loads are issued before any is resolved; a
//                    block is one tile, so it stores the tile's mask.
//  The insert, and the per-voxel query, are launched as programmatic
//  dependents of the kernel before them: they start while it finishes, read
//  their coordinates, and wait for it (griddepcontrol.wait) before touching
//  the table.
//  k_pairs_*         CSR pair lists per offset (ascending output row),
//                    built on demand: count, scan, scatter.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "sc_internal.cuh"

namespace sc {

constexpr int kInsertThreads = 256;

// ---------------------------------------------------------------------------
// insert

// Key of a live slot.
template <bool K32>
__device__ __forceinline__ uint64_t slot_key(const HashParams& hp, unsigned long long s) {
  if constexpr (K32)
    return s >> 32;
  else
    return s >> hp.vbits;
}

// Voxels per thread of the insert (build-time SC_INSERT_VPT, default 1):
// more gives each warp independent CAS chains in flight.
#ifndef SC_INSERT_VPT
#define SC_INSERT_VPT 1
#endif
constexpr int kInsertVpt = SC_INSERT_VPT;

template <bool K32, int VPT = 1>
__global__ void __launch_bounds__(kInsertThreads) k_hash_insert(const int4* __restrict__ coords,
                                                                HashParams hp, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  unsigned long long* slots = reinterpret_cast<unsigned long long*>(hp.slots);
  uint32_t err = 0;
  bool pending[VPT];
  uint64_t key[VPT], mine[VPT], pos[VPT], step[VPT], home[VPT];
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    // voxel v of this thread: blocks cover VPT * kInsertThreads consecutive rows
    const int64_t i =
        ((int64_t)blockIdx.x * VPT + v) * kInsertThreads + threadIdx.x;
    pending[v] = false;
    key[v] = mine[v] = pos[v] = step[v] = 0;
    if (i < hp.n) {
      const int4 c = __ldg(coords + i);
      const bool in_range = c.x >= 0 && (unsigned)c.y < (unsigned)hp.res &&
                            (unsigned)c.z < (unsigned)hp.res && (unsigned)c.w < (unsigned)hp.res;
      if (!in_range) {
        err |= kStatRange;
      } else if ((uint64_t)c.x >= hp.bmax) {
        err |= kStatKeySpace;
      } else if constexpr (K32) {
        const uint32_t k32 = cell_key32(hp, c.x, c.y, c.z, c.w);
        key[v] = k32;
        mine[v] = ((uint64_t)k32 << 32) | (uint64_t)i;
        pos[v] = home_slot32(hp, c.x, c.y, c.z, c.w);
        step[v] = probe_step32(hp, k32);
        pending[v] = true;
      } else {
        key[v] = cell_key(hp, c.x, c.y, c.z, c.w);
        mine[v] = (key[v] << hp.vbits) | (uint64_t)i;
        pos[v] = home_slot(hp, c.x, c.y, c.z, c.w);
        step[v] = probe_step(hp, key[v]);
        pending[v] = true;
      }
    }
    home[v] = pos[v];
  }
  // Everything above read only the coordinates; the table is cleared by the
  // kernel launched before this one (a programmatic dependency when launched
  // with that attribute: wait for its completion here).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Synchronous probing rounds; at most hp.probe_limit rounds (every slot,
  // unless sc_set_probe_limit set a smaller cap).  A thread's voxels take
  // their CAS of a round together.
  auto any_pending = [&]() {
    bool a = false;
#pragma unroll
    for (int v = 0; v < VPT; ++v) a |= pending[v];
    return a;
  };
  for (uint64_t round = 0; __any_sync(0xffffffffu, any_pending()); ++round) {
    unsigned long long old[VPT];
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (pending[v] && round >= hp.probe_limit) {
        err |= kStatTableFull;
        pending[v] = false;
      }
      old[v] = pending[v] ? atomicCAS(slots + pos[v], kEmptySlot, mine[v]) : 0ull;
    }
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      if (!pending[v]) continue;
      if (old[v] == kEmptySlot) {
        pending[v] = false;
      } else if (slot_key<K32>(hp, old[v]) == key[v]) {
        err |= kStatDuplicate;
        pending[v] = false;
      } else {
        // 32-bit keys: mark the home slot, whose key moved on.
        if (K32 && round == 0) atomicOr(slots + home[v], (unsigned long long)kMovedFlag);
        pos[v] = (pos[v] + step[v]) & hp.cap_mask;
      }
    }
  }
  err = __reduce_or_sync(0xffffffffu, err);
  if (err && lane == 0) atomicOr(status, err);
}

// ---------------------------------------------------------------------------
// query

// Row of `key` whose home slot `home` held `s`, continuing its probe
// sequence; -1 if absent.
__device__ __forceinline__ int32_t finish_probe(const HashParams& hp, uint64_t key, uint64_t home,
                                                unsigned long long s) {
  const uint64_t vmask = (1ull << hp.vbits) - 1ull;
  const unsigned long long* slots = reinterpret_cast<const unsigned long long*>(hp.slots);
  if (s == kEmptySlot) return -1;
  if ((s >> hp.vbits) == key) return (int32_t)(s & vmask);
  const uint64_t step = probe_step(hp, key);
  uint64_t pos = home;
  for (uint64_t it = 0; it < hp.cap_mask; ++it) {
    pos = (pos + step) & hp.cap_mask;
    s = __ldg(slots + pos);
    if (s == kEmptySlot) return -1;
    if ((s >> hp.vbits) == key) return (int32_t)(s & vmask);
  }
  return -1;
}

// Grid (tiles, 9): block (t, col) resolves, for the 128 voxels of tile t,
// the three neighbours (dz = -1, 0, 1) of neighbour column
// col = 3 * (dx + 1) + (dy + 1), i.e. offsets k = 3 * col + {0, 1, 2}.
// Grid (tiles, 9 / NCOL): block (t, y) resolves, for the 128 voxels of tile
// t, the three neighbours (dz = -1, 0, 1) of each of its NCOL neighbour
// columns col = y * NCOL + i, col = 3 * (dx + 1) + (dy + 1), i.e. offsets
// k = 3 * col + {0, 1, 2}.  (NCOL > 1 only with 32-bit keys.)
#ifndef SC_QUERY_NCOL
#define SC_QUERY_NCOL 1
#endif
constexpr int kQueryCols = SC_QUERY_NCOL;

template <NbrLayout L, bool K32, int NCOL = 1>
__global__ void __launch_bounds__(kTileRows) k_neighbor_query(
    const int4* __restrict__ coords, HashParams hp, int32_t* __restrict__ nbr,
    uint32_t* __restrict__ tile_mask, unsigned long long* pair_count) {
  __shared__ uint32_t s_or[kTileRows / 32];
  __shared__ uint32_t s_cnt[kTileRows / 32];
  const unsigned long long* slots = reinterpret_cast<const unsigned long long*>(hp.slots);
  const int64_t row0 = (int64_t)blockIdx.x * kTileRows;
  const int64_t o = row0 + threadIdx.x;
  const bool valid = o < hp.n;
  const int4 c = valid ? __ldg(coords + o) : make_int4(0, 0, 0, 0);
  // The table is written by the insert kernel launched before this one (a
  // programmatic dependency: this grid may start while that one finishes).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint32_t bits = 0;
#pragma unroll
  for (int ci = 0; ci < NCOL; ++ci) {
  const int col = blockIdx.y * NCOL + ci;
  const int dx = col / 3 - 1, dy = col % 3 - 1;
  const int x = c.y + dx, y = c.z + dy;
  const bool colin =
      valid && (unsigned)x < (unsigned)hp.res && (unsigned)y < (unsigned)hp.res;
  // Shared arithmetic of the column: the key of (x, y, z - 1) (the other two
  // are +1, +2) and the groups of the two bricks along z that the three
  // cells fall in (bricks zb and zb + 1, zb = (z - 1) >> 1).
  const int zb = (c.w - 1) >> 1;
  int32_t r[3];
  if constexpr (K32) {
    const uint32_t key_lo = cell_key32(hp, c.x, x, y, c.w - 1);
    uint32_t pos[3];
    uint32_t pend = 0;  // lookups the home slot did not settle
    const uint32_t BR = (uint32_t)hp.bres;
    const uint32_t brick_lo =
        (((uint32_t)c.x * BR + (uint32_t)(x >> 1)) * BR + (uint32_t)(y >> 1)) * BR + (uint32_t)zb;
    const uint32_t g_lo = group32(hp, brick_lo), g_hi = group32(hp, brick_lo + 1u);
    const uint32_t cellxy = (uint32_t)(((x & 1) << 2) | ((y & 1) << 1));
    unsigned long long sl[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int z = c.w + j - 1;
      const bool in = colin && (unsigned)z < (unsigned)hp.res && !(col == 4 && j == 1);
      pos[j] = (((z >> 1) != zb ? g_hi : g_lo) << 3) | cellxy | (uint32_t)(z & 1);
      sl[j] = in ? __ldg(slots + pos[j]) : kEmptySlot;
    }
    // Home slots: the key, an empty slot, or another key with the moved
    // flag clear all settle the lookup; otherwise it follows the probe
    // sequence, the column's open lookups advancing together.
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      r[j] = -1;
      if (sl[j] != kEmptySlot) {
        if ((uint32_t)(sl[j] >> 32) == key_lo + (uint32_t)j)
          r[j] = (int32_t)((uint32_t)sl[j] & kRowMask32);
        else if (sl[j] & kMovedFlag)
          pend |= 1u << j;
      }
    }
    const uint32_t cmask = (uint32_t)hp.cap_mask;
    for (uint32_t it = 0; pend != 0 && it < cmask; ++it) {
#pragma unroll
      for (int j = 0; j < 3; ++j)
        if (pend & (1u << j)) {
          pos[j] = (pos[j] + probe_step32(hp, key_lo + (uint32_t)j)) & cmask;
          sl[j] = __ldg(slots + pos[j]);
        }
#pragma unroll
      for (int j = 0; j < 3; ++j)
        if (pend & (1u << j)) {
          if (sl[j] == kEmptySlot) {
            pend &= ~(1u << j);
          } else if ((uint32_t)(sl[j] >> 32) == key_lo + (uint32_t)j) {
            r[j] = (int32_t)((uint32_t)sl[j] & kRowMask32);
            pend &= ~(1u << j);
          }
        }
    }
  } else {
    const uint64_t key_lo = cell_key(hp, c.x, x, y, c.w - 1);
    const int64_t BR = hp.bres;
    const int64_t brick_lo = (((int64_t)c.x * BR + (x >> 1)) * BR + (y >> 1)) * BR + zb;
    const int gshift = 64 - (hp.log2cap - 3);
    const uint64_t g_lo = ((uint64_t)brick_lo * 0x9E3779B97F4A7C15ull) >> gshift;
    const uint64_t g_hi = ((uint64_t)(brick_lo + 1) * 0x9E3779B97F4A7C15ull) >> gshift;
    const uint64_t cellxy = (uint64_t)(((x & 1) << 2) | ((y & 1) << 1));
    unsigned long long sl[3];
    uint64_t home[3];
    bool in[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int z = c.w + j - 1;
      in[j] = colin && (unsigned)z < (unsigned)hp.res && !(col == 4 && j == 1);
      home[j] = ((((z >> 1) != zb) ? g_hi : g_lo) << 3) | cellxy | (uint64_t)(z & 1);
      sl[j] = in[j] ? __ldg(slots + home[j]) : kEmptySlot;
    }
#pragma unroll
    for (int j = 0; j < 3; ++j)
      r[j] = in[j] ? finish_probe(hp, key_lo + (uint64_t)j, home[j], sl[j]) : -1;
  }
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const int k = 3 * col + j;
    if (k == kCentre) r[j] = valid ? (int32_t)o : -1;
    bits |= (r[j] >= 0 ? 1u : 0u) << k;
    if constexpr (L == kNbrTileMajor)
      nbr[row0 * kTaps + k * kTileRows + threadIdx.x] = r[j];
    else if (valid)
      nbr[o * kTaps + k] = r[j];
  }
  }
  const uint32_t cnt = (uint32_t)__popc(bits);
  const int lane = threadIdx.x & 31;
  // Per block: the offsets present in its rows into the tile mask (zeroed
  // before the launch), its pair count into one of the counters (one
  // atomic of each per block: per warp, the counters' L2 slice saturates).
  const uint32_t wor = __reduce_or_sync(0xffffffffu, bits);
  const uint32_t wcnt = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) {
    s_or[threadIdx.x >> 5] = wor;
    s_cnt[threadIdx.x >> 5] = wcnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0, bc = 0;
    for (int w = 0; w < kTileRows / 32; ++w) {
      m |= s_or[w];
      bc += s_cnt[w];
    }
    if (m) atomicOr(tile_mask + blockIdx.x, m);
    if (bc)
      atomicAdd(pair_count + (blockIdx.x * 9u + blockIdx.y) % kPairCounters,
                (unsigned long long)bc);
  }
}

// 32-bit keys: one thread per voxel resolves all 26 neighbours.  The 27
// cells around a voxel lie in 2 x 2 x 2 bricks (along each axis the bricks
// (v - 1) >> 1 and the next), and the brick hash is linear in the brick
// index, so the eight group hashes cost an add each; every neighbour's home
// slot is its cell within its brick's group.  All 26 home loads are
// independent, so a thread keeps many in flight; a lookup the home slot
// does not settle (the moved flag of another key) continues after the main
// pass along its probe sequence.  Rows of a 128-row tile are one block, so
// the tile's offset mask is a plain store.  Tile-major output is written
// straight out (a warp's stores of one offset are 32 consecutive rows);
// row-major output is staged in shared memory and written out contiguously.
template <NbrLayout L>
__global__ void __launch_bounds__(kTileRows, 4) k_neighbor_query32(
    const int4* __restrict__ coords, HashParams hp, int32_t* __restrict__ nbr,
    uint32_t* __restrict__ tile_mask, unsigned long long* pair_count) {
  __shared__ uint32_t s_or[kTileRows / 32];
  __shared__ uint32_t s_cnt[kTileRows / 32];
  __shared__ __align__(16) int32_t s_rows[L == kNbrRowMajor ? kTileRows * kTaps : 4];
  const unsigned long long* slots = reinterpret_cast<const unsigned long long*>(hp.slots);
  const int64_t row0 = (int64_t)blockIdx.x * kTileRows;
  const int64_t o = row0 + threadIdx.x;
  const bool valid = o < hp.n;
  // A pad row sits far outside the grid, so that every neighbour is absent.
  const int4 c = valid ? __ldg(coords + o) : make_int4(0, -4, -4, -4);
  const uint32_t R = (uint32_t)hp.res, BR = (uint32_t)hp.bres;
  const int x = c.y, y = c.z, z = c.w;
  const uint32_t key0 = cell_key32(hp, c.x, x, y, z);
  const int bx = (x - 1) >> 1, by = (y - 1) >> 1, bz = (z - 1) >> 1;
  // brick(bx + i, by + j, bz + l) = brick000 + i BR^2 + j BR + l (mod 2^32),
  // and so is its hash times the multiplier.
  const uint32_t brick000 = (((uint32_t)c.x * BR + (uint32_t)bx) * BR + (uint32_t)by) * BR +
                            (uint32_t)bz;
  constexpr uint32_t kPhi = 0x9E3779B9u;
  const uint32_t h000 = brick000 * kPhi, hA = BR * BR * kPhi, hB = BR * kPhi;
  const int gshift = 32 - (hp.log2cap - 3);
  const uint32_t RR = R * R;
  int32_t* out_t = nbr + row0 * kTaps + threadIdx.x;  // tile-major: [k * 128]
  int32_t* out_s = s_rows + threadIdx.x * kTaps;      // row-major staging: [k]
  auto put = [&](int k, int32_t r) {
    if constexpr (L == kNbrTileMajor)
      out_t[k * kTileRows] = r;
    else
      out_s[k] = r;
  };
  // The table is written by the insert kernel launched before this one.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // All 26 home slots are loaded before any is looked at, so that the
  // thread has them all in flight at once.
  unsigned long long sl[kTaps];
#pragma unroll
  for (int k = 0; k < kTaps; ++k) {
    const int dx = k / 9 - 1, dy = (k / 3) % 3 - 1, dz = k % 3 - 1;
    const int xx = x + dx, yy = y + dy, zz = z + dz;
    const bool in = k != kCentre && (unsigned)xx < R && (unsigned)yy < R && (unsigned)zz < R;
    const uint32_t slot =
        (((h000 + (uint32_t)((xx >> 1) - bx) * hA + (uint32_t)((yy >> 1) - by) * hB +
           (uint32_t)((zz >> 1) - bz) * kPhi) >>
          gshift)
         << 3) |
        (uint32_t)(((xx & 1) << 2) | ((yy & 1) << 1) | (zz & 1));
    sl[k] = in ? __ldg(slots + slot) : kEmptySlot;
  }
  uint32_t bits = 0, pend = 0;
#pragma unroll
  for (int k = 0; k < kTaps; ++k) {
    if (k == kCentre) continue;
    const int dx = k / 9 - 1, dy = (k / 3) % 3 - 1, dz = k % 3 - 1;
    const uint32_t key = key0 + (uint32_t)dx * RR + (uint32_t)dy * R + (uint32_t)dz;
    int32_t r = -1;
    if (sl[k] != kEmptySlot) {
      if ((uint32_t)(sl[k] >> 32) == key)
        r = (int32_t)((uint32_t)sl[k] & kRowMask32);
      else if (sl[k] & kMovedFlag)
        pend |= 1u << k;
    }
    bits |= (r >= 0 ? 1u : 0u) << k;
    put(k, r);
  }
  // Lookups that left their home slot: follow the probe sequence.
  const uint32_t cmask = (uint32_t)hp.cap_mask;
  while (pend) {
    const int k = __ffs(pend) - 1;
    pend &= pend - 1u;
    const int dx = k / 9 - 1, dy = (k / 3) % 3 - 1, dz = k % 3 - 1;
    const int xx = x + dx, yy = y + dy, zz = z + dz;
    const uint32_t key = key0 + (uint32_t)dx * RR + (uint32_t)dy * R + (uint32_t)dz;
    uint32_t pos = (((h000 + (uint32_t)((xx >> 1) - bx) * hA + (uint32_t)((yy >> 1) - by) * hB +
                      (uint32_t)((zz >> 1) - bz) * kPhi) >>
                     gshift)
                    << 3) |
                   (uint32_t)(((xx & 1) << 2) | ((yy & 1) << 1) | (zz & 1));
    const uint32_t step = probe_step32(hp, key);
    for (uint32_t it = 0; it < cmask; ++it) {
      pos = (pos + step) & cmask;
      const unsigned long long sl = __ldg(slots + pos);
      if (sl == kEmptySlot) break;
      if ((uint32_t)(sl >> 32) == key) {
        put(k, (int32_t)((uint32_t)sl & kRowMask32));
        bits |= 1u << k;
        break;
      }
    }
  }
  put(kCentre, valid ? (int32_t)o : -1);
  if (valid) bits |= 1u << kCentre;
  // The tile's offsets present in any row (this block is the whole tile) and
  // its pair count into one of the counters.
  const int lane = threadIdx.x & 31;
  const uint32_t wor = __reduce_or_sync(0xffffffffu, bits);
  const uint32_t wcnt = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(bits));
  if (lane == 0) {
    s_or[threadIdx.x >> 5] = wor;
    s_cnt[threadIdx.x >> 5] = wcnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t m = 0, bc = 0;
#pragma unroll
    for (int w = 0; w < kTileRows / 32; ++w) {
      m |= s_or[w];
      bc += s_cnt[w];
    }
    tile_mask[blockIdx.x] = m;
    if (bc) atomicAdd(pair_count + blockIdx.x % kPairCounters, (unsigned long long)bc);
  }
  if constexpr (L == kNbrRowMajor) {
    // The block's rows [row0, row0 + rows) are one contiguous range of
    // rows * 27 ints: copy it out with 16-byte stores where aligned.
    const int total = (int)min((int64_t)kTileRows, hp.n - row0) * kTaps;
    int32_t* dst = nbr + row0 * kTaps;
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
      const int nvec = total >> 2;
      for (int i = threadIdx.x; i < nvec; i += kTileRows)
        reinterpret_cast<int4*>(dst)[i] = reinterpret_cast<const int4*>(s_rows)[i];
      for (int i = (nvec << 2) + threadIdx.x; i < total; i += kTileRows) dst[i] = s_rows[i];
    } else {
      for (int i = threadIdx.x; i < total; i += kTileRows) dst[i] = s_rows[i];
    }
  }
}

// nbr_out[n][27] from the tile-major table: one block per tile, staged in
// shared memory so that both sides are coalesced.
__global__ void __launch_bounds__(kTileRows) k_nbr_to_row_major(const int32_t* __restrict__ nbr_t,
                                                                int64_t n,
                                                                int32_t* __restrict__ out) {
  __shared__ __align__(16) int32_t s[kTileRows * kTaps];
  const int64_t row0 = (int64_t)blockIdx.x * kTileRows;
  const int32_t* src = nbr_t + row0 * kTaps;
#pragma unroll 3
  for (int k = 0; k < kTaps; ++k) s[threadIdx.x * kTaps + k] = src[k * kTileRows + threadIdx.x];
  __syncthreads();
  const int total = (int)min((int64_t)kTileRows, n - row0) * kTaps;
  int32_t* dst = out + row0 * kTaps;
  const int nvec = total >> 2;
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    for (int i = threadIdx.x; i < nvec; i += kTileRows)
      reinterpret_cast<int4*>(dst)[i] = reinterpret_cast<const int4*>(s)[i];
    for (int i = (nvec << 2) + threadIdx.x; i < total; i += kTileRows) dst[i] = s[i];
  } else {
    for (int i = threadIdx.x; i < total; i += kTileRows) dst[i] = s[i];
  }
}

// One launch instead of three memsets: every slot empty (all ones), the
// tile masks and the status / pair-counter block zero.
__global__ void __launch_bounds__(256) k_map_init(ulonglong2* __restrict__ slots, int64_t npairs2,
                                                  uint32_t* __restrict__ tile_mask, int64_t ntiles,
                                                  uint32_t* __restrict__ status) {
  // The insert kernel launched after this one may start at once: it reads
  // coordinates first and waits for this grid before touching the table.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const ulonglong2 ones = make_ulonglong2(kEmptySlot, kEmptySlot);
  for (int64_t i = t; i < npairs2; i += stride) slots[i] = ones;
  for (int64_t i = t; i < ntiles; i += stride) tile_mask[i] = 0u;
  if (t < kStatusBlockBytes / 4) status[t] = 0u;
}

cudaError_t launch_map_init(const HashParams& hp, uint32_t* tile_mask, int64_t ntiles,
                            uint32_t* status, cudaStream_t s) {
  const int64_t npairs2 = (int64_t)(hp.cap_mask + 1) / 2;  // 16-byte stores
  const int64_t work = std::max<int64_t>(npairs2, ntiles);
  const int64_t blocks = std::min<int64_t>((work + 255) / 256, 148LL * 8);
  static_assert(kStatusBlockBytes / 4 <= 256, "status block cleared by the first block");
  k_map_init<<<(unsigned)std::max<int64_t>(blocks, 1), 256, 0, s>>>(
      reinterpret_cast<ulonglong2*>(hp.slots), npairs2, tile_mask, ntiles, status);
  note_launches(1);
  return cudaGetLastError();
}

// A launch with the programmatic-dependency attribute: the kernel may start
// while the one before it in the stream finishes, and waits for it
// (griddepcontrol.wait) before it reads that kernel's output.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), unsigned blocks, unsigned threads,
                             size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

// The same with a two-dimensional grid.
template <typename... Params, typename... Args>
cudaError_t launch_dependent2(void (*kern)(Params...), dim3 grid, unsigned threads,
                              cudaStream_t s, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

cudaError_t launch_hash_insert(const int32_t* coords, const HashParams& hp, uint32_t* status,
                               cudaStream_t s) {
  if (hp.n == 0) return cudaSuccess;
  const int64_t per_block = (int64_t)kInsertThreads * kInsertVpt;
  const unsigned blocks = (unsigned)((hp.n + per_block - 1) / per_block);
  const int4* c4 = reinterpret_cast<const int4*>(coords);
  cudaError_t e = hp.k32 ? launch_dependent(k_hash_insert<true, kInsertVpt>, blocks,
                                            kInsertThreads, 0, s, c4, hp, status)
                         : launch_dependent(k_hash_insert<false, kInsertVpt>, blocks,
                                            kInsertThreads, 0, s, c4, hp, status);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

cudaError_t launch_neighbor_query(const int32_t* coords, const HashParams& hp, int32_t* nbr,
                                  uint32_t* tile_mask, unsigned long long* pair_count,
                                  uint32_t* status, NbrLayout layout, cudaStream_t s) {
  (void)status;
  if (hp.n == 0) return cudaSuccess;
  const int64_t tiles = (hp.n + kTileRows - 1) / kTileRows;
  const int4* c4 = reinterpret_cast<const int4*>(coords);
  if (hp.k32) {
    // Up to ~1M voxels the nine-threads-per-voxel kernel keeps more loads in
    // flight across the GPU (measured on B300: 17.5 against 20.5 us for a
    // 30k-voxel build, 49 against 54 us at 400k); beyond, the kernel with
    // one thread per voxel and all 26 loads in flight is faster (386 against
    // 457 us at 3.3M).
    // From 2^18 voxels three columns per thread (fewer threads, their setup
    // shared) beat one (measured: 46.1 against 48.1 us at 400k; 17.3 against
    // 15.3 us at 30k and 25.5 against 23.5 us at 144k the other way).
    cudaError_t e;
    if (kQueryCols == 1 && hp.n >= (int64_t(1) << 18) && hp.n < (int64_t(1) << 20)) {
      const dim3 grid((unsigned)tiles, 3);
      e = layout == kNbrTileMajor
              ? launch_dependent2(k_neighbor_query<kNbrTileMajor, true, 3>, grid, kTileRows, s,
                                  c4, hp, nbr, tile_mask, pair_count)
              : launch_dependent2(k_neighbor_query<kNbrRowMajor, true, 3>, grid, kTileRows, s,
                                  c4, hp, nbr, tile_mask, pair_count);
    } else if (hp.n < (int64_t(1) << 20)) {
      const dim3 grid((unsigned)tiles, 9 / kQueryCols);
      e = layout == kNbrTileMajor
              ? launch_dependent2(k_neighbor_query<kNbrTileMajor, true, kQueryCols>, grid,
                                  kTileRows, s, c4, hp, nbr, tile_mask, pair_count)
              : launch_dependent2(k_neighbor_query<kNbrRowMajor, true, kQueryCols>, grid,
                                  kTileRows, s, c4, hp, nbr, tile_mask, pair_count);
    } else {
      e = layout == kNbrTileMajor
              ? launch_dependent(k_neighbor_query32<kNbrTileMajor>, (unsigned)tiles, kTileRows,
                                 0, s, c4, hp, nbr, tile_mask, pair_count)
              : launch_dependent(k_neighbor_query32<kNbrRowMajor>, (unsigned)tiles, kTileRows,
                                 0, s, c4, hp, nbr, tile_mask, pair_count);
    }
    if (e == cudaSuccess) note_launches(1);
    return e;
  }
  const dim3 grid((unsigned)tiles, 9);
  if (layout == kNbrTileMajor) {
    if (hp.k32)
      k_neighbor_query<kNbrTileMajor, true><<<grid, kTileRows, 0, s>>>(c4, hp, nbr, tile_mask,
                                                                       pair_count);
    else
      k_neighbor_query<kNbrTileMajor, false><<<grid, kTileRows, 0, s>>>(c4, hp, nbr, tile_mask,
                                                                        pair_count);
  } else {
    if (hp.k32)
      k_neighbor_query<kNbrRowMajor, true><<<grid, kTileRows, 0, s>>>(c4, hp, nbr, tile_mask,
                                                                      pair_count);
    else
      k_neighbor_query<kNbrRowMajor, false><<<grid, kTileRows, 0, s>>>(c4, hp, nbr, tile_mask,
                                                                       pair_count);
  }
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_nbr_to_row_major(const sc_map* m, int32_t* nbr_out, cudaStream_t s) {
  if (m->n == 0) return cudaSuccess;
  k_nbr_to_row_major<<<(unsigned)m->ntiles, kTileRows, 0, s>>>(m->nbr, m->n, nbr_out);
  note_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// row order for the convolution
//
// A 128-row tile of the convolution skips an offset only when no row of the
// tile has that neighbour.  In input order nearly every tile holds every
// offset (27 per tile against ~15-22 per row on thin shells), so the kernel
// gathers zero rows for the rest.  Sorting the rows by their 27-bit presence
// masks (a stable radix sort, least significant 9 bits first) puts rows with
// the same neighbourhood shape into the same tiles; the permuted tile-major
// table, its tile masks and each position's original row drive the
// convolution, whose epilogue writes every position to its row.

__global__ void __launch_bounds__(kTileRows) k_row_masks(const int32_t* __restrict__ nbr_t,
                                                        int64_t n, uint32_t* __restrict__ masks) {
  const int64_t o = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
  if (o >= n) return;
  const int32_t* col = nbr_t + (int64_t)blockIdx.x * kTileRows * kTaps + threadIdx.x;
  uint32_t m = 0;
#pragma unroll
  for (int k = 0; k < kTaps; ++k) m |= (__ldg(col + k * kTileRows) >= 0 ? 1u : 0u) << k;
  masks[o] = m;
}

// One block per output tile: position q takes row perm[q], whose 27 entries
// are read from a row-major copy of the table (108 contiguous bytes per row;
// in the tile-major table they would be 27 scattered words) by the lanes of
// one warp, staged in shared memory, and written out tile-major.
__global__ void __launch_bounds__(kTileRows) k_permute_table(const int32_t* __restrict__ nbr_rm,
                                                            const int32_t* __restrict__ perm,
                                                            int64_t n, int32_t* __restrict__ out_t,
                                                            uint32_t* __restrict__ out_mask,
                                                            int32_t* __restrict__ row_of) {
  __shared__ uint32_t s_or[kTileRows / 32];
  __shared__ int32_t s_t[kTaps][kTileRows + 1];
  const int64_t q0 = (int64_t)blockIdx.x * kTileRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // warp w copies positions 32w .. 32w + 31, one row (27 lanes) at a time
  for (int r = 0; r < 32; ++r) {
    const int pos = warp * 32 + r;
    const int64_t q = q0 + pos;
    const int32_t row = q < n ? __ldg(perm + q) : -1;
    if (lane < kTaps)
      s_t[lane][pos] = row >= 0 ? __ldg(nbr_rm + (int64_t)row * kTaps + lane) : -1;
  }
  __syncthreads();
  const int64_t q = q0 + threadIdx.x;
  int32_t* dst = out_t + q0 * kTaps + threadIdx.x;
  uint32_t bits = 0;
#pragma unroll
  for (int k = 0; k < kTaps; ++k) {
    const int32_t v = s_t[k][threadIdx.x];
    dst[k * kTileRows] = v;
    bits |= (v >= 0 ? 1u : 0u) << k;
  }
  const int32_t row = q < n ? __ldg(perm + q) : -1;
  row_of[q] = row;
  const uint32_t w = __reduce_or_sync(0xffffffffu, bits);
  if ((threadIdx.x & 31) == 0) s_or[threadIdx.x >> 5] = w;
  __syncthreads();
  if (threadIdx.x == 0) out_mask[blockIdx.x] = s_or[0] | s_or[1] | s_or[2] | s_or[3];
}

// Per tile of the mask-sorted order: 27 - (offsets present in the tile), the
// key that puts the costliest tiles first.
__global__ void __launch_bounds__(kTileRows) k_tile_keys(const uint32_t* __restrict__ masks,
                                                        int64_t n, uint32_t* __restrict__ tkey) {
  __shared__ uint32_t s_or[kTileRows / 32];
  const int64_t q = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
  const uint32_t w = __reduce_or_sync(0xffffffffu, q < n ? __ldg(masks + q) : 0u);
  if ((threadIdx.x & 31) == 0) s_or[threadIdx.x >> 5] = w;
  __syncthreads();
  if (threadIdx.x == 0)
    tkey[blockIdx.x] = (uint32_t)(kTaps - __popc(s_or[0] | s_or[1] | s_or[2] | s_or[3]));
}

// Tile j of the final order is tile torder[j] of the mask-sorted one.
__global__ void __launch_bounds__(kTileRows) k_tile_gather(const int32_t* __restrict__ perm,
                                                          int64_t n,
                                                          const int32_t* __restrict__ torder,
                                                          int32_t* __restrict__ perm2) {
  const int64_t old = (int64_t)__ldg(torder + blockIdx.x) * kTileRows + threadIdx.x;
  perm2[(int64_t)blockIdx.x * kTileRows + threadIdx.x] = old < n ? __ldg(perm + old) : -1;
}

size_t order_scratch_bytes(int64_t n) {
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t ntiles = (size_t)((n + kTileRows - 1) / kTileRows);
  return 4 * up((size_t)n * 4) + 3 * up(ntiles * 4) + up(ntiles * kTileRows * 4) +
         std::max(up(sort_scratch_bytes(n, 512)), up((size_t)n * kTaps * 4));
}

cudaError_t launch_order_rows(const sc_map* m, void* scratch, cudaStream_t s) {
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const int64_t n = m->n;
  uint8_t* p = static_cast<uint8_t*>(scratch);
  uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(p),
                       reinterpret_cast<uint32_t*>(p + up((size_t)n * 4))};
  int32_t* vals[2] = {reinterpret_cast<int32_t*>(p + 2 * up((size_t)n * 4)),
                      reinterpret_cast<int32_t*>(p + 3 * up((size_t)n * 4))};
  const int64_t nt = m->ntiles;
  uint8_t* p2 = p + 4 * up((size_t)n * 4);
  uint32_t* tkey = reinterpret_cast<uint32_t*>(p2);
  uint32_t* tkey_out = reinterpret_cast<uint32_t*>(p2 + up((size_t)nt * 4));
  int32_t* torder = reinterpret_cast<int32_t*>(p2 + 2 * up((size_t)nt * 4));
  int32_t* perm2 = reinterpret_cast<int32_t*>(p2 + 3 * up((size_t)nt * 4));
  void* work = p2 + 3 * up((size_t)nt * 4) + up((size_t)nt * kTileRows * 4);
  k_row_masks<<<(unsigned)m->ntiles, kTileRows, 0, s>>>(m->nbr, n, keys[0]);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  int cur = 0;
  for (int shift = 0; shift < kTaps && e == cudaSuccess; shift += 9) {
    e = sort_pass<uint32_t>(keys[cur], shift == 0 ? nullptr : vals[cur], keys[cur ^ 1],
                            vals[cur ^ 1], n, shift, std::min(9, kTaps - shift), work, s);
    cur ^= 1;
  }
  if (e != cudaSuccess) return e;
  // Tiles with the most offsets first (stable: tiles of one count keep their
  // mask order), so that the persistent grid's round-robin hands out work
  // longest first and the last round is made of the cheapest tiles.
  k_tile_keys<<<(unsigned)nt, kTileRows, 0, s>>>(keys[cur], n, tkey);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = sort_pass<uint32_t>(tkey, nullptr, tkey_out, torder, nt, 0, 5, work, s);
  if (e != cudaSuccess) return e;
  k_tile_gather<<<(unsigned)nt, kTileRows, 0, s>>>(vals[cur], n, torder, perm2);
  note_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // The sort's work space is free again: the row-major table goes there.
  int32_t* nbr_rm = static_cast<int32_t*>(work);
  e = launch_nbr_to_row_major(m, nbr_rm, s);
  if (e != cudaSuccess) return e;
  k_permute_table<<<(unsigned)nt, kTileRows, 0, s>>>(nbr_rm, perm2, nt * kTileRows, m->ord_nbr,
                                                    m->ord_mask, m->ord_row);
  note_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// pair lists (CSR per offset, ascending output row within an offset)

__global__ void __launch_bounds__(kTileRows) k_pairs_count(const int32_t* __restrict__ nbr_t,
                                                           int64_t nblocks,
                                                           int64_t* __restrict__ counts) {
  const int32_t* col = nbr_t + (int64_t)blockIdx.x * kTileRows * kTaps + threadIdx.x;
  for (int k = 0; k < kTaps; ++k) {
    const int c = __syncthreads_count(col[k * kTileRows] >= 0);  // pad rows are -1
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

__global__ void __launch_bounds__(kTileRows) k_pairs_write(const int32_t* __restrict__ nbr_t,
                                                           int64_t nblocks,
                                                           const int64_t* __restrict__ offs,
                                                           int32_t* pin, int32_t* pout) {
  __shared__ int s_warp[kTileRows / 32];
  const int64_t o = (int64_t)blockIdx.x * kTileRows + threadIdx.x;
  const int32_t* col = nbr_t + (int64_t)blockIdx.x * kTileRows * kTaps + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int k = 0; k < kTaps; ++k) {
    const int32_t i = col[k * kTileRows];
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
  const int64_t nblocks = m->ntiles;
  int64_t* counts = static_cast<int64_t*>(scratch);
  int64_t* total = counts + kTaps * nblocks;
  int64_t* off28 = total + 1;
  k_pairs_count<<<(unsigned)nblocks, kTileRows, 0, s>>>(m->nbr, nblocks, counts);
  k_scan_exclusive<<<1, 1024, 0, s>>>(counts, kTaps * nblocks, total);
  if (in || out)
    k_pairs_write<<<(unsigned)nblocks, kTileRows, 0, s>>>(m->nbr, nblocks, counts, in, out);
  k_pairs_offsets<<<1, 32, 0, s>>>(counts, nblocks, total, off28);
  note_launches((in || out) ? 4 : 3);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(off_host, off28, 28 * sizeof(int64_t), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

}  // namespace sc
