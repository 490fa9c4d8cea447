// sc_internal.cuh -- shared definitions of the sm_103a sparse-conv library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sc.h"

namespace sc {

// Rows per output tile: one tcgen05 accumulator tile (M = 128, one TMEM lane
// per row) and one CTA of the neighbour-query kernel.
constexpr int kTileRows = 128;
constexpr int kTaps = 27;
constexpr int kCentre = 13;
constexpr uint64_t kEmptySlot = ~0ull;

// Status block of a map (16-byte aligned): four status words, then
// kPairCounters 64-bit pair counters.  Each query block adds its pair count
// to one counter (a counter per block-index residue, not one global counter:
// tens of thousands of same-address atomics would serialise in one L2
// slice); the host sums them.
constexpr int kPairCounters = 32;
constexpr int kStatusBlockBytes = 16 + 8 * kPairCounters;

// Device status word bits (the map's `d_status`).
enum : uint32_t {
  kStatRange = 1u,
  kStatDuplicate = 2u,
  kStatTableFull = 4u,
  kStatTimeout = 8u,
  kStatKeySpace = 16u,  // (batch+1) * res^3 does not fit the packed key field
};

// ---------------------------------------------------------------------------
// Coordinate hash: packed 64-bit slots, empty = all ones, over the key
// key = ((b * res + x) * res + y) * res + z.  Two packings:
//   32-bit keys (k32, whenever batch x res^3 fits below 2^32 - 1 and the
//     table has at most 2^32 slots): slot = key << 32 | flag << 31 | row.
//     The flag of a slot is set when a key whose home it is had to move on
//     (its home was taken), so a lookup that finds another key at its home
//     slot with the flag clear knows at once that its key is absent.  All
//     hashing is 32-bit arithmetic.
//   64-bit keys otherwise: slot = key << vbits | row, vbits = bit length of
//     n, so a row index never fills its field and a live slot is never all
//     ones; lookups probe until their key or an empty slot.
//
// Home slots preserve locality: the grid is cut into 2x2x2 bricks, a brick
// hashes to a group of 8 consecutive slots (64 bytes) and a voxel's home is
// the slot of its cell within the group.  The 26 neighbours of a voxel then
// live in the groups of at most 8 bricks, which neighbouring voxels (threads
// of a warp) share, so a warp's probe loads touch few cache lines.
// Collisions continue by double hashing: probe i of a key is
// home + i * step(key) (mod capacity), step odd so the sequence visits every
// slot.  Linear probing from brick-local homes builds long clusters (runs of
// tens of occupied slots at load 0.4); an independent stride does not.

struct HashParams {
  uint64_t* slots;
  uint64_t cap_mask;   // capacity - 1 (capacity a power of two, >= 64)
  int log2cap;
  int k32;             // 32-bit keys (see above)
  int vbits;           // 64-bit keys: bits of the row field
  int res;
  int bres;            // bricks per axis: (res + 1) / 2
  uint64_t bmax;       // batch indices must be < bmax
  int64_t n;
  uint64_t probe_limit;  // slots an insertion may probe before reporting a full table
};

// Process-wide cap on an insertion's probes (sc_set_probe_limit); 0 = none
// beyond the table's capacity.
uint32_t probe_limit_setting();

__device__ __forceinline__ uint64_t cell_key(const HashParams& hp, int b, int x, int y, int z) {
  const uint64_t r = (uint64_t)hp.res;
  return (((uint64_t)b * r + (uint64_t)x) * r + (uint64_t)y) * r + (uint64_t)z;
}

__device__ __forceinline__ uint64_t home_slot(const HashParams& hp, int b, int x, int y, int z) {
  const uint64_t br = (uint64_t)hp.bres;
  const uint64_t brick =
      (((uint64_t)b * br + (uint64_t)(x >> 1)) * br + (uint64_t)(y >> 1)) * br + (uint64_t)(z >> 1);
  // Fibonacci hashing of the brick onto one of capacity / 8 groups.
  const uint64_t group = (brick * 0x9E3779B97F4A7C15ull) >> (64 - (hp.log2cap - 3));
  return (group << 3) | (uint64_t)(((x & 1) << 2) | ((y & 1) << 1) | (z & 1));
}

// Odd probe stride of a key (a second multiplicative hash).
__device__ __forceinline__ uint64_t probe_step(const HashParams& hp, uint64_t key) {
  return ((key * 0xC2B2AE3D27D4EB4Full) >> (64 - hp.log2cap)) | 1ull;
}

// The same three functions with 32-bit keys (32-bit multiplicative hashes).
__device__ __forceinline__ uint32_t cell_key32(const HashParams& hp, int b, int x, int y, int z) {
  const uint32_t r = (uint32_t)hp.res;
  return (((uint32_t)b * r + (uint32_t)x) * r + (uint32_t)y) * r + (uint32_t)z;
}
__device__ __forceinline__ uint32_t group32(const HashParams& hp, uint32_t brick) {
  return (brick * 0x9E3779B9u) >> (32 - (hp.log2cap - 3));
}
__device__ __forceinline__ uint32_t home_slot32(const HashParams& hp, int b, int x, int y, int z) {
  const uint32_t br = (uint32_t)hp.bres;
  const uint32_t brick =
      (((uint32_t)b * br + (uint32_t)(x >> 1)) * br + (uint32_t)(y >> 1)) * br + (uint32_t)(z >> 1);
  return (group32(hp, brick) << 3) | (uint32_t)(((x & 1) << 2) | ((y & 1) << 1) | (z & 1));
}
__device__ __forceinline__ uint32_t probe_step32(const HashParams& hp, uint32_t key) {
  return ((key * 0xC2B2AE35u) >> (32 - hp.log2cap)) | 1u;
}
constexpr uint64_t kMovedFlag = 1ull << 31;  // 32-bit keys: a key homed here moved on
constexpr uint32_t kRowMask32 = 0x7fffffffu;

// Host: hash parameters for n >= 1 rows at resolution res in 2^log2cap slots
// (6 <= log2cap), with 32-bit keys when they fit (and k32_allowed).  Returns
// false when not even batch 0 fits the key.
inline bool make_hash_params(HashParams& hp, uint64_t* slots, int64_t n, int res, int log2cap,
                             bool k32_allowed) {
  const uint64_t res3 = (uint64_t)res * res * res;
  const int vbits = 64 - __builtin_clzll((unsigned long long)n);
  hp.slots = slots;
  hp.cap_mask = (1ull << log2cap) - 1ull;
  hp.log2cap = log2cap;
  hp.vbits = vbits;
  hp.res = res;
  hp.bres = (res + 1) / 2;
  hp.n = n;
  const uint64_t lim = probe_limit_setting();
  hp.probe_limit = (lim && lim < (1ull << log2cap)) ? lim : (1ull << log2cap);
  hp.k32 = k32_allowed && log2cap <= 32 && res3 <= 0xffffffffull;
  if (hp.k32) {
    hp.bmax = 0xffffffffull / res3;  // keys <= 2^32 - 2: a live slot is never all ones
    return true;
  }
  hp.bmax = (1ull << (64 - vbits)) / res3;
  return hp.bmax > 0;
}

// Host: log2 of the table capacity for n rows, load factor <= 1/4 (a
// brick's cells share a group of 8 slots; at load 1/2 a third of the
// lookups of absent neighbours met another key at home).  The build-time
// SC_HASH_SLOTS_PER_ROW (default 4) sets the bound.
#ifndef SC_HASH_SLOTS_PER_ROW
#define SC_HASH_SLOTS_PER_ROW 4
#endif
inline int hash_log2cap(int64_t n) {
  int l = 6;
  while ((1ull << l) < (uint64_t)SC_HASH_SLOTS_PER_ROW * (uint64_t)n) ++l;
  return l;
}

// Neighbour tables: row-major nbr[n][27], or tile-major nbr[tile][27][128]
// (rows of a 128-row tile contiguous per offset; pad rows -1), the layout
// the map handle keeps for the convolution kernels.
enum NbrLayout { kNbrRowMajor = 0, kNbrTileMajor = 1 };

// ---------------------------------------------------------------------------
// mbarrier / TMA / tcgen05 wrappers (inline PTX, sm_100+ family).

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// SC_TRY_WAIT_HINT_NS (build time): how long a try_wait may suspend the
// thread before it returns false (0: the hardware's own limit).  20 us
// (a waiting thread is woken when the phase completes, so a long hint only
// cuts the spinning that steals issue slots from the working warps):
// measured 3-5% faster convolutions than the default limit.
#ifndef SC_TRY_WAIT_HINT_NS
#define SC_TRY_WAIT_HINT_NS 20000
#endif
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
#if SC_TRY_WAIT_HINT_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"((uint32_t)SC_TRY_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: returns false if the phase did not complete within ~2 s or
// another role of the CTA has already given up (*abort != 0).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > 2000000000ull) return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Four rows r0..r3 (each one box of the 2-D map, box height 1) at column x.
// Rows outside the tensor are filled with zeros and still count in bytes.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int4 rows) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(rows.x), "r"(rows.y), "r"(rows.z), "r"(rows.w), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 2-D load delivered to the same shared-memory offset (data and
// mbarrier complete_tx) in every CTA of the cluster named in cta_mask.
__device__ __forceinline__ void tma_load_2d_multicast(void* dst, const CUtensorMap* map,
                                                      uint64_t* bar, int32_t x, int32_t y,
                                                      uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(cta_mask)
      : "memory");
}

// Contiguous global -> shared copy (16-byte aligned addresses, size a
// multiple of 16), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Brings a contiguous global range (16-byte aligned, size a multiple of 16)
// into L2 without waiting for it.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives, then waits for all.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// 16-byte global -> shared copy through L2 (not L1); src_bytes = 0 writes
// zeros without reading.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Arrive on `bar` (without raising its expected count) once every cp.async
// this thread has issued so far has completed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's completed generic-proxy shared-memory writes visible to
// the async proxy (tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// TMEM allocation (whole warp), address written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// As tc_commit, arriving on the mbarrier at the same offset in every CTA of
// cta_mask.
__device__ __forceinline__ void tc_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t gets row (lane base + t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 layout, version 1).
//   layout: 0 none, 2 = 128B swizzle, 4 = 64B swizzle, 6 = 32B swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for sm_100 family
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16 (or both fp16), D = fp32,
// A K-major, B MN-major (row-major W[k][ci][co] has co contiguous), M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool f16 = false) {
  return (1u << 4)                      // D format fp32
         | ((f16 ? 0u : 1u) << 7)       // A format: 0 fp16, 1 bf16
         | ((f16 ? 0u : 1u) << 10)      // B format: the same as A
         | (0u << 15)                   // A K-major
         | (1u << 16)                   // B MN-major
         | ((uint32_t)(n >> 3) << 17)   // N / 8
         | ((uint32_t)(m >> 4) << 24);  // M / 16
}

}  // namespace sc

// ---------------------------------------------------------------------------
// Host-side launch entry points implemented in the kernel files.

struct sc_map {
  uint64_t magic;
  int device;
  int64_t n;
  int32_t res;
  int64_t ntiles;
  int64_t npairs;
  sc::HashParams hash;
  int32_t* nbr;          // tile-major [ntiles][27][128], pad rows -1
  uint32_t* tile_mask;   // [ntiles] OR of the 27-bit presence masks of a tile's rows
  uint32_t* d_status;    // device status word + pair counter scratch
  void* block;           // the one device allocation the buffers above are carved from
  unsigned long long* d_pairs;  // kPairCounters counters after the status words
  void* (*alloc)(size_t, void*, void*);
  void (*free_fn)(void*, void*, void*);
  void* alloc_ctx;
  // Builds that did not synchronise (sc_build_map_async): until `pending` is
  // cleared by the first call that needs the result, the status words and
  // the pair count are only on the device; `built` is recorded after the
  // build's kernels.  build_word keeps the build's status bits once read.
  int pending;
  cudaEvent_t built;
  uint32_t build_word;
  // Row order for the convolution (sc_map_order_rows): the tile-major table
  // over rows sorted by their 27-bit neighbour masks, its tile masks, and
  // each position's row; nullptr until ordered.
  void* ord_block;
  int32_t* ord_nbr;
  uint32_t* ord_mask;
  int32_t* ord_row;
};

namespace sc {

// Clear a map's scratch: all slots empty, tile masks and the status block
// zero (slots 16-byte aligned).
cudaError_t launch_map_init(const HashParams& hp, uint32_t* tile_mask, int64_t ntiles,
                            uint32_t* status, cudaStream_t s);
cudaError_t launch_hash_insert(const int32_t* coords, const HashParams& hp, uint32_t* status,
                               cudaStream_t s);
cudaError_t launch_neighbor_query(const int32_t* coords, const HashParams& hp, int32_t* nbr,
                                  uint32_t* tile_mask, unsigned long long* pair_count,
                                  uint32_t* status, NbrLayout layout, cudaStream_t s);
// Row-major copy nbr_out[n][27] of the map's tile-major table.
cudaError_t launch_nbr_to_row_major(const sc_map* m, int32_t* nbr_out, cudaStream_t s);
cudaError_t launch_pairs(const sc_map* m, int64_t* off_host, int32_t* in, int32_t* out,
                         void* scratch, cudaStream_t s);
size_t pairs_scratch_bytes(int64_t n);
// The convolution's fused epilogue ("Porting TRELLIS.2 From Python to Rust
// and Metal", section V: bias, rounding, activation and the residual add in
// the same pass): out = act(acc + bias) + residual, in fp32, then stored as
// fp32 or rounded to bf16 / fp16 (nearest, ties to even).
struct Epilogue {
  const float* bias;     // [cout] or nullptr
  const void* residual;  // [n][cout] in the output dtype, or nullptr
  void* out;             // [n][cout]
  int act;               // SC_ACT_NONE / SC_ACT_RELU / SC_ACT_SILU
  int out_half;          // output: 0 fp32, kOutBf16, kOutF16
};
constexpr int kOutBf16 = 1;
constexpr int kOutF16 = 2;

__device__ __forceinline__ float apply_act(float v, int act) {
  if (act == SC_ACT_RELU) return fmaxf(v, 0.f);
  // v * sigmoid(v) = v / (1 + e^-v), by the fast divide (2 ulp); as v -> -inf
  // the denominator passes 2^126 and the quotient is -0, the function's limit.
  if (act == SC_ACT_SILU) return __fdividef(v, 1.f + __expf(-v));
  return v;
}

// What the convolution kernels read of a map: per 128-position tile, a
// tile-major block of `taps` input rows per position (-1: absent), the
// tile's offset mask, and optionally the output row of each position.
struct ConvMap {
  const int32_t* nbr;         // [ntiles][taps][128]
  const uint32_t* tile_mask;  // [ntiles]
  const int32_t* row_of;      // [ntiles * 128] output row (-1: none), or nullptr: identity
  int64_t n;                  // positions 0 .. n-1 hold an output row
  int64_t ntiles;
  int taps;                   // 27 (3x3x3) or 8 (2x2x2 between levels)
  uint32_t* status;           // device status word for bounded waits
};
inline ConvMap conv_map_of(const sc_map* m) {
  // Ordered: pad positions (row -1) may sit in any tile, so every position
  // of every tile is looked at.
  if (m->ord_nbr)
    return ConvMap{m->ord_nbr,        m->ord_mask, m->ord_row, m->ntiles * kTileRows,
                   m->ntiles,         kTaps,       m->d_status};
  return ConvMap{m->nbr, m->tile_mask, nullptr, m->n, m->ntiles, kTaps, m->d_status};
}

cudaError_t launch_conv_simt_f32(const ConvMap& m, const float* feats, const float* w,
                                 const Epilogue& ep, int cin, int cout, cudaStream_t s);
// bf16 or fp16 operands (f16 = true); returns cudaErrorNotSupported for
// shapes outside the tensor-core envelope.
cudaError_t launch_conv_tc(const ConvMap& m, const void* feats, const void* w, bool f16,
                           const Epilogue& ep, int cin, int cout, cudaStream_t s);
bool conv_tc_supported(int cin, int cout);
// Level changes (sc_levels.cu).
cudaError_t launch_child_counts(const int32_t* coords, const uint8_t* mask, int64_t n, int res,
                                int32_t* counts, uint32_t* status, cudaStream_t s);
cudaError_t launch_subdivide(const int32_t* coords, const uint8_t* mask, int64_t n,
                             const int32_t* first, int32_t* child_coords, int32_t* parent,
                             int32_t* offset, int32_t* child_of, cudaStream_t s);
cudaError_t launch_channel_to_spatial(const void* feats, const int32_t* parent,
                                      const int32_t* offset, int64_t m, int c, int esize,
                                      void* out, cudaStream_t s);
size_t level_scratch_bytes(int64_t n, int kbytes);
template <typename K>
cudaError_t build_level_tables(const int32_t* coords, int64_t n, int res, int nbatch, int key_bits,
                               void* scratch, int32_t* down_nbr, uint32_t* down_mask,
                               int32_t* parent_of, int32_t* parent_coords, int32_t* up_nbr,
                               int32_t* up_row, uint32_t* up_mask, int64_t* np_dev,
                               uint32_t* status, cudaStream_t s);
cudaError_t launch_child_table(const int32_t* down_nbr, int64_t np, int32_t* out, cudaStream_t s);
// Dual-grid mesh (sc_mesh.cu).
cudaError_t launch_quad_counts(const sc_map* m, const uint8_t* flags, int32_t* counts,
                               cudaStream_t s);
cudaError_t launch_quads(const sc_map* m, const uint8_t* flags, const int32_t* first,
                         int32_t* quads, cudaStream_t s);
cudaError_t launch_triangulate(const int32_t* quads, int64_t nq, const float* verts,
                               int32_t* tris, cudaStream_t s);
// sc_sort.cu
cudaError_t scan_exclusive(const int32_t* in, int32_t* out, int64_t len, int64_t* total,
                           void* scratch, cudaStream_t s);
size_t scan_scratch_bytes(int64_t len);
template <typename K>
cudaError_t sort_pass(const K* keys_in, const int32_t* vals_in, K* keys_out, int32_t* vals_out,
                      int64_t n, int shift, int bits, void* scratch, cudaStream_t s);
size_t sort_scratch_bytes(int64_t n, int bins);
// Row order for the convolution (sc_map.cu): scratch bytes, and the build
// of m's ord_* tables (allocated by the caller) from its neighbour table.
size_t order_scratch_bytes(int64_t n);
cudaError_t launch_order_rows(const sc_map* m, void* scratch, cudaStream_t s);

// Process-wide count of the kernels this library has launched (host side).
void note_launches(int k);
uint32_t* status_readback_buffer();  // pinned, kStatusBlockBytes, per host thread
uint64_t launches();
// Deterministic mode: the tensor-core kernel splits a unit in at most two
// parts (a + b == b + a in fp32), so repeated calls are bit-identical.
void set_deterministic(bool on);
// Record a failure (or SC_OK with an empty message) as the calling thread's
// last error; returns st.
sc_status set_last_error(sc_status st, const char* msg);

}  // namespace sc
