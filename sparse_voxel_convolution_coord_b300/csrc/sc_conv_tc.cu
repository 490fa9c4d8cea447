// sc_conv_tc.cu -- bf16 / fp16 submanifold convolution on the sm_103a tensor
// cores.
//
// What it computes ("Porting TRELLIS.2 From Python to Rust and Metal",
// section V: a gather-GEMM over the neighbour table with half-precision
// inputs, single-precision accumulation and the bias fused into the same
// pass; "Running TRELLIS.2 on a Mac (1/3)", Sparse 3D convolution paragraph):
//
//   out[o][:] = bias + sum_{k : nbr[o][k] >= 0} feats[nbr[o][k]][:] @ W[k]
//
// and, in the FUSED instantiation, the rest of the epilogue in the same pass
// (the same section: bias, rounding, activation and the residual add):
// out = act(out) + residual, stored as fp32, bf16 or fp16.
//
// How: an output-stationary implicit GEMM.  A CTA owns a tile of 128 output
// rows; the GEMM's K dimension is (offset, input channel).  For each offset
// present in the tile (its 27-bit OR mask), the 128 neighbour rows are
// gathered straight from the feature matrix by cp.async (absent neighbours
// zero-filled) and W[k] arrives by tiled TMA; a single thread issues
// tcgen05.mma (M = 128, N = cout padded to 64, or 32 when cout <= 32, K = 16,
// bf16 x bf16 or fp16 x fp16 -> fp32; the instruction descriptor is a launch
// argument) into a TMEM accumulator.  A pipeline stage holds K = 64 or 128
// channels: one offset's 64-channel block (or two, for wide inputs with
// cout <= 128), or the whole rows of several offsets (cin <= 64).  Each output row belongs to exactly one tile, so the epilogue
// (TMEM -> registers -> shared staging -> coalesced stores) needs no atomics,
// except in the tail split below.
//
// Tail split: the grid is persistent (one cluster per pair of SMs), so when
// the units do not divide evenly over the clusters the last, partial wave
// would leave most SMs idle.  The host then splits each unit of that wave
// into S parts by ranges of its K stages; parts are spread over all
// clusters, and each adds its partial accumulator into the output (zeroed
// beforehand) with 16-byte float atomics, the last part adding the bias.
// Those rows' sums are then taken in an order that can vary between runs.
// The parts run first, so that their atomic epilogues overlap other CTAs'
// main loops and the kernel ends on plain stores.  The rows are zeroed by a
// small kernel launched just before, with this one as its programmatic
// dependent: both run at once, and only the epilogue waits for the zeroing
// (griddepcontrol.wait) before its first atomic add.
//
// Clusters: with CL = 2 the two CTAs of a cluster work on adjacent tiles in
// lock step (the union of their offset masks) and share each W slice: every
// CTA loads half of the slice's 64-column boxes and multicasts them to both,
// halving the L2 -> SM traffic of the weights, which at cin = cout = 256 is
// two thirds of all operand traffic.  A stage is released only when both
// CTAs' MMAs have consumed it (each MMA warp commits to the "empty" barrier
// of both CTAs).
//
// CTA = 14 warps, persistent over units of CL tiles:
//   warps 0-3  epilogue (warp q reads TMEM lanes 32q..32q+31 = rows of the tile)
//   warp 4     loader: the tile's 128 x 27 neighbour block by one bulk copy
//              (two buffers, one unit ahead, for cout <= 64; one buffer,
//              refilled after a unit's stages, above) and, per stage, this
//              CTA's W boxes by tiled TMA
//   warps 5-12 A producers, in 2 or 4 groups that take the stages in turn:
//              per stage the group's threads gather the A rows with 16-byte
//              cp.async copies (consecutive threads take consecutive 16-byte
//              chunks of a row, so a warp instruction moves whole lines;
//              absent neighbours are zero-filled) straight into the swizzled
//              operand layout; each thread's mbarrier arrival fires when its
//              copies land.  (TMA gather4 moves only
//              four 64-128 byte rows per operation; its per-operation cost,
//              not bandwidth, bounded the gather.)
//   warp 13    TMEM allocation; lane 0 issues the MMAs and the commits
// Two TMEM accumulators let the epilogue of one tile overlap the next tile's
// main loop.  Every wait is bounded (~2 s): a CTA that gives up records
// SC_ERR_DEVICE_TIMEOUT in the map's status word and leaves cleanly.
//
// Shared-memory operand layouts (A written swizzled by the producers'
// cp.async addresses, B by TMA swizzling):
//   A (gathered rows, K-major): per stage SEGS segments, each 128 rows x CS
//     16-bit values, rows of 2*CS bytes with the matching 128/64/32-byte
//     swizzle;
//   B (W[k] rows, MN-major): per stage [column blocks][K rows][128 B] with
//     the 128-byte swizzle (64-column blocks; LBO = K x 128 B between
//     blocks, SBO = 1 KB between 8-row groups), or [K rows][64 B] with the
//     64-byte swizzle at N = 32 (SBO = 512 B).
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "sc_internal.cuh"

namespace sc {

#ifndef SC_PRODUCER_WARPS
#define SC_PRODUCER_WARPS 8
#endif
constexpr int kLoaderWarp = 4;                          // W boxes + neighbour blocks
constexpr int kProducerWarps = SC_PRODUCER_WARPS;       // A gathers: warps 5 .. 4 + kProducerWarps
constexpr int kProducerThreads = 32 * kProducerWarps;
// The producers form groups that take the pipeline stages in turn (stage g
// of the CTA's sequence goes to group g mod groups), so a thread issues
// `groups` times the copies of one stage per wait and arrival, with that
// many stage times to do it.  Four groups where the MMAs of a stage are
// short (NPAD <= 64), two otherwise (measured on B300); build-time
// SC_PRODUCER_GROUPS overrides.
#ifndef SC_PRODUCER_GROUPS
#define SC_PRODUCER_GROUPS 0
#endif
template <int NPAD>
constexpr int producer_groups(int stages, int stage_copies) {
  // Four groups only where each thread's share of a stage stays at 16
  // copies or fewer (its per-copy registers), two otherwise.
  return SC_PRODUCER_GROUPS > 0
             ? SC_PRODUCER_GROUPS
             : (NPAD <= 64 && stages >= 4 && stage_copies <= 16 * (kProducerThreads / 4) ? 4 : 2);
}
constexpr int kMmaWarp = 5 + kProducerWarps;
constexpr int kTcThreads = 32 * (kMmaWarp + 1);

constexpr int kSmemLimit = 227 * 1024;                  // opt-in dynamic shared memory per CTA
constexpr int kNbrBytes = kTileRows * kTaps * 4;        // a tile's neighbour block, <= 13,824 B
// Epilogue staging: each epilogue warp transposes its 32 rows x 32 columns
// through shared memory (row stride 36 floats: 16-byte aligned, and both the
// row-wise writes and the column-group reads are bank-conflict-free).
constexpr int kStageRow = 36;
constexpr int kEpiBytes = 4 * 32 * kStageRow * 4;       // 18,432 B
constexpr uint64_t kWaitNs = 2000000000ull;             // bounded waits: 2 s
constexpr uint64_t kDrainNs = 50000000ull;              // final drain after an abort: 50 ms

// Ring depth cap (build-time SC_MAX_STAGES); the shared-memory budget sets
// the depth below it.
#ifndef SC_MAX_STAGES
#define SC_MAX_STAGES 8
#endif

// SEGS segments of CS channels per stage: one segment (CS = 64) is one
// offset's 64-channel block of a wide input; several (cin == CS) are that
// many offsets' whole rows.  64 / CS by default (K = 64 per stage); twice
// that for the narrow layers, whose stages are otherwise too short for the
// per-stage synchronisation.
template <int NPAD, int CS, int SEGS = 64 / CS>
struct TcCfg {
  static constexpr int kSegs = SEGS;                    // segments per stage
  static constexpr int kKst = SEGS * CS;                // K (channels) per stage
  static constexpr int kRowBytes = CS * 2;              // one gathered row segment
  static constexpr int kChunks = kRowBytes / 16;        // 16-byte copies per row segment
  static constexpr int kSegCopies = kTileRows * kChunks;        // 16-byte copies per segment
  static constexpr int kASeg = kTileRows * kRowBytes;   // bytes per A segment
  static constexpr int kABytes = kTileRows * kKst * 2;  // 16 or 32 KB per stage
  // B blocks: 64 columns (128-byte rows, 128-byte swizzle), or all of a
  // 32-column B (64-byte rows, 64-byte swizzle).
  static constexpr int kBCols = NPAD < 64 ? NPAD : 64;  // columns per B block
  static constexpr int kBRow = kBCols * 2;              // bytes per K row of a block
  static constexpr int kBlocksN = NPAD / kBCols;        // column blocks of B
  static constexpr uint32_t kLayoutB = kBRow == 128 ? 2u : 4u;
  static_assert(kBRow == 128 || kBRow == 64, "B blocks of 64 or 32 columns");
  static constexpr int kBBytes = kKst * NPAD * 2;       // kKst K rows x NPAD bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  // Neighbour blocks: two (the next unit's prefetched during this one) for
  // cout <= 64, whose short units would expose the refill; one otherwise,
  // refilled after a unit's stages while the MMA drains the ring.
  static constexpr int kNbrBufs = NPAD <= 64 ? 2 : 1;
  // Fixed: neighbour block(s), the epilogue's staging (4 warps x 32 rows x
  // kStageRow floats), bias, barriers.
  static constexpr int kFixed = kNbrBufs * kNbrBytes + kEpiBytes + NPAD * 4 + 256;
  static constexpr int kStages0 = (kSmemLimit - 1024 - kFixed) / kStageBytes;
  static constexpr int kStages = kStages0 > SC_MAX_STAGES ? SC_MAX_STAGES : kStages0;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kFixed;
  static constexpr int kGroups = producer_groups<NPAD>(kStages, kSegs * kSegCopies);
  static constexpr int kGroupThreads = kProducerThreads / kGroups;
  static_assert(kGroupThreads * kGroups == kProducerThreads && kGroupThreads % 32 == 0,
                "producer groups are whole warps");
  static constexpr int kPerThread = kSegs * kSegCopies / kGroupThreads;
  static_assert(kPerThread * kGroupThreads == kSegs * kSegCopies &&
                    kGroupThreads % kChunks == 0,
                "producer threads must tile the stage's copies");
  static constexpr uint32_t kTmemCols = (2 * NPAD <= 128) ? 128 : (2 * NPAD <= 256 ? 256 : 512);
  static constexpr uint32_t kLayoutA = CS == 64 ? 2u : (CS == 32 ? 4u : 6u);
  static constexpr uint32_t kSboA = 8 * kRowBytes;
  static_assert(kStages >= 2, "pipeline needs two stages");
  static_assert(SEGS > 1 || CS == 64, "a one-segment stage is a 64-channel block");
  // A group waits on a slot's empty barrier by phase parity for the stage
  // kStages before its own; it has issued its previous stage, kGroups
  // earlier, so every stage up to kGroups + kStages back has been consumed.
  // The stage 2 kStages back must be among them, or the slot's barrier may
  // still be a phase behind and the parity test would pass early.
  static_assert(kStages >= kGroups, "producer groups need at least one ring slot each");
  static_assert(kSmemBytes <= kSmemLimit, "shared memory budget");
};

struct TcArgs {
  const __nv_bfloat16* feats;  // [n][cin]
  const int32_t* nbr;          // tile-major [ntiles][taps][128], pad rows -1
  const uint32_t* tile_mask;   // [ntiles]
  const int32_t* row_of;       // output row of each tile position (-1: none), or nullptr: the
                               // position itself
  int taps;                    // 27 (3x3x3) or 8 (2x2x2 between levels)
  const float* bias;
  const void* residual;  // [n][cout] in the output dtype, or nullptr
  void* out;             // fp32 or bf16 [n][cout]
  int act;               // fused activation (SC_ACT_*)
  int out_half;          // 16-bit output (kOutBf16 / kOutF16, nearest even), 0: fp32
  uint32_t idesc;        // MMA instruction descriptor (bf16 or fp16 operands)
  uint32_t* status;
  int64_t n;       // tile positions that hold an output row
  int64_t ntiles;
  int64_t whole;   // units 0 .. whole-1 are one work item each
  int64_t tail;    // units whole .. whole+tail-1 are `split` items each
  int64_t nparts;  // tail * split
  int64_t nitems;  // nparts + whole
  int split;
  int sv;          // virtual stages per unit (work items are ranges of them)
  int cin;
  int cout;
};

// A work item: unit `unit`, virtual stage range [a, b) of [0, sv) (the whole
// unit when a == 0 and b == sv).  A unit of nst real stages runs stages
// [a nst / sv, b nst / sv): the parts of one unit partition its stages
// whatever nst is, and the part that ends the unit (b == sv) adds the bias.
struct WorkItem {
  int64_t unit;
  int a, b;
};

// The items of cluster cid, in order: items cid, cid + ncl, ... of the
// sequence (tail parts, numbered part-major so that a unit's parts go to
// different clusters and run concurrently, then the whole units).
struct ItemIter {
  int64_t k;
  __device__ __forceinline__ ItemIter(const TcArgs& p, int64_t cid) : k(cid) {}
  __device__ __forceinline__ bool next(const TcArgs& p, int64_t ncl, WorkItem& w) {
    if (k >= p.nitems) return false;
    if (k >= p.nparts) {
      w = {k - p.nparts, 0, p.sv};
    } else {
      // k < nparts = tail x split and part < split <= 8: 32-bit arithmetic.
      const uint32_t kk = (uint32_t)k, tail = (uint32_t)p.tail;
      const int part = (int)(kk / tail);
      w = {p.whole + (int64_t)(kk - (uint32_t)part * tail),
           (int)((uint32_t)(part * p.sv) / (uint32_t)p.split),
           (int)((uint32_t)((part + 1) * p.sv) / (uint32_t)p.split)};
    }
    k += ncl;
    return true;
  }
};

// Stage range [s0, s1) of an item of a unit with nst stages.
__device__ __forceinline__ void item_range(const WorkItem& w, int sv, int nst, int& s0, int& s1) {
  if (w.a == 0 && w.b == sv) {  // a whole unit
    s0 = 0;
    s1 = nst;
    return;
  }
  // a, b <= sv and nst <= sv, with sv at most taps x (1024 / 64): 32 bits hold
  // the products.
  s0 = (int)((uint32_t)(w.a * nst) / (uint32_t)sv);
  s1 = (int)((uint32_t)(w.b * nst) / (uint32_t)sv);
}

// Bounded wait with its own limit; ignores the abort flag (used to drain).
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > limit_ns) return false;
  return true;
}

// OR of the offset masks of the CL tiles of a unit.
template <int CL>
__device__ __forceinline__ uint32_t unit_mask(const uint32_t* tile_mask, int64_t unit,
                                              int64_t ntiles) {
  uint32_t m = 0;
#pragma unroll
  for (int r = 0; r < CL; ++r) {
    const int64_t t = unit * CL + r;
    if (t < ntiles) m |= __ldg(tile_mask + t);
  }
  return m;
}

// Stages of a unit.  Block stages (GRP false): each present offset's cin/64
// channel blocks, SEGS consecutive blocks per stage.  Group stages (GRP
// true, cin == CS): the present offsets taken SEGS at a time.
template <int CS, int SEGS, bool GRP>
__device__ __forceinline__ int unit_stages(uint32_t mask, int cin) {
  const int np = __popc(mask);
  if constexpr (!GRP) {
    return np * (cin >> 6) / SEGS;
  } else {
    return (np + SEGS - 1) / SEGS;
  }
}

// Walks the K slices of a unit in order.  Block stages: each present offset
// k (ascending) with its cin/64 channel blocks, SEGS blocks per stage (all
// segments of a stage take offset k; segment j starts at channel c0 + 64 j).
// Group stages: the present offsets SEGS at a time (k = taps, one past the
// last offset, pads the last stage: its W box lies past the end of W and is
// zero-filled).  next() fills the stage's offsets and returns its first
// channel.
template <int CS, int SEGS, bool GRP>
struct OffsetIter {
  uint32_t rem;
  int cblk = 0, cblocks, taps;
  __device__ __forceinline__ OffsetIter(uint32_t mask, int cin, int taps_)
      : rem(mask), cblocks(cin >> 6), taps(taps_) {}
  // Step over the first `n` stages.
  __device__ __forceinline__ void skip(int n) {
    if constexpr (!GRP) {
      cblk += n * SEGS;
      while (cblk >= cblocks) {
        cblk -= cblocks;
        rem &= rem - 1u;
      }
    } else {
      for (int i = 0; i < n * SEGS; ++i) rem &= rem - 1u;
    }
  }
  __device__ __forceinline__ int next(int (&ks)[SEGS]) {
    if constexpr (!GRP) {
      const int k = __ffs(rem) - 1;
#pragma unroll
      for (int j = 0; j < SEGS; ++j) ks[j] = k;
      const int c0 = cblk * 64;
      cblk += SEGS;
      if (cblk == cblocks) {
        cblk = 0;
        rem &= rem - 1u;
      }
      return c0;
    } else {
#pragma unroll
      for (int j = 0; j < SEGS; ++j) {
        ks[j] = rem ? __ffs(rem) - 1 : taps;
        rem &= rem - 1u;
      }
      return 0;
    }
  }
};

// Zeroes the rows the split units add into.  It lets its dependent (the
// convolution) launch at once; the dependent waits for this grid's
// completion only where it reads these rows.
__global__ void __launch_bounds__(256) k_zero_rows(float4* __restrict__ p, int64_t n4) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// The same for the rows of positions [pos0, n) through a row indirection
// (c4 = cout / 4 float4 per row): a warp per position, its lanes over the
// row's float4 columns.
__global__ void __launch_bounds__(256) k_zero_rows_of(float4* __restrict__ out,
                                                      const int32_t* __restrict__ row_of,
                                                      int64_t pos0, int64_t n, int c4) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t pos = pos0 + (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pos < n;
       pos += wstride) {
    const int32_t row = __ldg(row_of + pos);
    if (row < 0) continue;
    float4* dst = out + (int64_t)row * c4;
    for (int c = lane; c < c4; c += 32) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// FUSED: the epilogue applies an activation, adds a residual or rounds to
// bf16 (the plain variant only adds the bias and stores fp32).
template <int NPAD, int CS, int SEGS, bool GRP, int CL, bool FUSED>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_conv_tc(const __grid_constant__ CUtensorMap tm_b, const TcArgs p) {
  using C = TcCfg<NPAD, CS, SEGS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::kStages * C::kABytes;
  int32_t* s_nbr = reinterpret_cast<int32_t*>(sB + C::kStages * C::kBBytes);  // [bufs][27][128]
  float* s_epi =
      reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(s_nbr) + C::kNbrBufs * kNbrBytes);
  float* s_bias = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(s_epi) + kEpiBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(s_bias + NPAD);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* nbr_full = acc_empty + 2;
  uint64_t* nbr_empty = nbr_full + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(nbr_empty + 2);
  int* s_abort = reinterpret_cast<int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int64_t cid = blockIdx.x / CL;
  const int64_t ncl = gridDim.x / CL;
  constexpr uint16_t kAllCtas = (uint16_t)((1u << CL) - 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], C::kGroupThreads + 1);  // one per thread of a producer group + the loader
      mbar_init(&empty[s], CL);  // one commit from the MMA warp of every CTA of the cluster
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kTileRows);
      mbar_init(&nbr_full[a], 1);
      mbar_init(&nbr_empty[a], kProducerThreads);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(s_tmem, C::kTmemCols);
  for (int i = threadIdx.x; i < NPAD; i += kTcThreads)
    s_bias[i] = (p.bias != nullptr && i < p.cout) ? p.bias[i] : 0.f;
  if (warp == kLoaderWarp && lane == 0) prefetch_tensormap(&tm_b);
  tc_fence_before();
  __syncthreads();
  if constexpr (CL > 1) cluster_sync_all();  // peers' barriers exist before any multicast
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  volatile int* abort_flag = s_abort;

  if (warp == kLoaderWarp) {
    // ------------------------------------------------------------ loader
    // Lane 0: per stage, this CTA's W boxes by tiled TMA and, once the
    // producers have released a neighbour-block buffer, the next unit's
    // block (one bulk copy).
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, fills = 0;
      int buf = 0;
      bool ok = true;
      // Refill buffer b with item w's block once every A producer has
      // released its contents (nothing when there is no such item).
      auto issue_nbr = [&](bool have, const WorkItem& w, int b) -> bool {
        if (!have) return true;
        const int64_t t = w.unit * CL + rank;
        if (t >= p.ntiles) return true;
        if ((fills >> (2 + b)) & 1u) {  // used before: wait for the release
          if (!mbar_wait_bounded(&nbr_empty[b], ((fills >> b) & 1u) ^ 1u, abort_flag))
            return false;
        }
        const uint32_t nbytes = (uint32_t)(p.taps * kTileRows * 4);
        mbar_arrive_expect_tx(&nbr_full[b], nbytes);
        bulk_copy_g2s(s_nbr + b * kTileRows * kTaps, p.nbr + t * (kTileRows * p.taps), nbytes,
                      &nbr_full[b]);
        fills ^= 1u << b;        // parity of the fills of buffer b
        fills |= 1u << (2 + b);  // buffer b used at least once
        return true;
      };
      ItemIter items(p, cid), ahead(p, cid);
      WorkItem wi, wn;
      bool have_next = ahead.next(p, ncl, wn);
      ok = issue_nbr(have_next, wn, 0);
      while (ok && items.next(p, ncl, wi)) {
        have_next = ahead.next(p, ncl, wn);  // the item after wi
        if constexpr (C::kNbrBufs == 1) {
          // One buffer: the next unit's block is copied in only once this
          // unit's gathers are issued; bring it into L2 now, so that the
          // copy then does not wait on DRAM.
          const int64_t tn = wn.unit * CL + rank;
          if (have_next && tn < p.ntiles)
            bulk_prefetch_l2(p.nbr + tn * (kTileRows * p.taps), (uint32_t)(p.taps * kTileRows * 4));
        }
        const uint32_t mask = unit_mask<CL>(p.tile_mask, wi.unit, p.ntiles);
        int s0, s1;
        item_range(wi, p.sv, unit_stages<CS, SEGS, GRP>(mask, p.cin), s0, s1);
        if constexpr (C::kNbrBufs == 2) {
          if (!issue_nbr(have_next, wn, buf ^ 1)) {
            ok = false;
            break;
          }
        }
        OffsetIter<CS, SEGS, GRP> it(mask, p.cin, p.taps);
        it.skip(s0);
        for (int s = s0; s < s1; ++s) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          // The expect_tx covers every box of the stage, including those the
          // peer CTA multicasts here.
          mbar_arrive_expect_tx(&full[stage], C::kBBytes);
          uint8_t* b_st = sB + stage * C::kBBytes;
          int ks[C::kSegs];
          const int c0 = it.next(ks);
#pragma unroll
          for (int j = 0; j < C::kSegs; ++j) {
#pragma unroll
            for (int nb2 = 0; nb2 < C::kBlocksN; ++nb2) {
              const int b = j * C::kBlocksN + nb2;
              if ((uint32_t)(b % CL) == rank) {
                // k == 27 addresses rows past W's end: the box is zero-filled.
                uint8_t* dst = b_st + nb2 * (C::kKst * C::kBRow) + j * CS * C::kBRow;
                const int32_t y = ks[j] * p.cin + c0 + (GRP ? 0 : 64 * j);
                if constexpr (CL > 1)
                  tma_load_2d_multicast(dst, &tm_b, &full[stage], nb2 * C::kBCols, y, kAllCtas);
                else
                  tma_load_2d(dst, &tm_b, &full[stage], nb2 * C::kBCols, y);
              }
            }
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        // One buffer: the next unit's block as soon as every producer is
        // done with this one (the MMA still holds up to kStages stages).
        if constexpr (C::kNbrBufs == 1) {
          if (ok && !issue_nbr(have_next, wn, 0)) ok = false;
        }
        buf ^= C::kNbrBufs - 1;
      }
      if (!ok) {
        *s_abort = 1;
        atomicOr(p.status, kStatTimeout);
      }
      // Drain: wait until every stage armed here has been released by the MMA
      // warps of all CTAs of the cluster, so that no copy or commit aimed at
      // this CTA's shared memory is still in flight when it exits.
      for (int i = 0; i < C::kStages; ++i) {
        if (!mbar_wait_for(&empty[stage], phase ^ 1u, ok ? kWaitNs : kDrainNs)) {
          atomicOr(p.status, kStatTimeout);
          break;
        }
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp > kLoaderWarp && warp < kMmaWarp) {
    // ------------------------------------------------------------ A producers
    const int pt0 = threadIdx.x - 32 * (kLoaderWarp + 1);  // 0 .. kProducerThreads - 1
    const int grp = pt0 / C::kGroupThreads;     // this thread's producer group
    const int pt = pt0 % C::kGroupThreads;      // its place in the group
    const int chunk_id = pt % C::kChunks;       // which 16 bytes of a row segment
    // The stage's kSegs x 128 rows x kChunks 16-byte copies, thread pt of the
    // group taking copies q = pt + i * kGroupThreads (consecutive threads:
    // consecutive chunks of one row).  Copy i reads row r_i of segment i *
    // kGroupThreads / kSegCopies (the segment does not depend on pt, as
    // kSegCopies is a multiple of kGroupThreads) and lands at byte dst_i
    // of the stage: row r of a segment starts at r * kRowBytes, and its chunk
    // c sits at c ^ ((r * kRowBytes >> 7) & (kChunks - 1)) (the 128/64/32-byte
    // swizzle of the operand descriptors).  All of this is fixed per thread;
    // a stage only looks up its rows and issues the copies.
    static_assert(C::kSegCopies % C::kGroupThreads == 0, "a pass of copies stays in one segment");
    int r_i[C::kPerThread];
    uint32_t dst_i[C::kPerThread];
#pragma unroll
    for (int i = 0; i < C::kPerThread; ++i) {
      const int q = pt + i * C::kGroupThreads;
      const int r = (q / C::kChunks) % kTileRows;
      const int sw = (r * C::kRowBytes >> 7) & (C::kChunks - 1);
      r_i[i] = r;
      dst_i[i] = (uint32_t)((i * C::kGroupThreads / C::kSegCopies) * C::kASeg + r * C::kRowBytes +
                            ((chunk_id ^ sw) << 4));
    }
    const char* const fbase = reinterpret_cast<const char*>(p.feats) + chunk_id * 16;
    const int rstride = p.cin * 2;  // bytes per feature row
    uint32_t stage = 0, phase = 0, nbr_phase = 0;
    uint32_t gst = 0;  // stages of the CTA's sequence so far (all items)
    int buf = 0;
    bool ok = true;
    ItemIter items(p, cid);
    WorkItem wi;
    while (ok && items.next(p, ncl, wi)) {
      const int64_t tile = wi.unit * CL + rank;
      const bool has_rows = tile < p.ntiles;
      const uint32_t mask = unit_mask<CL>(p.tile_mask, wi.unit, p.ntiles);
      int s0, s1;
      item_range(wi, p.sv, unit_stages<CS, SEGS, GRP>(mask, p.cin), s0, s1);
      if (has_rows) {
        if (!mbar_wait_bounded(&nbr_full[buf], (nbr_phase >> buf) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        nbr_phase ^= 1u << buf;
      }
      const int32_t* nb = s_nbr + buf * (kTileRows * kTaps);
      OffsetIter<CS, SEGS, GRP> it(mask, p.cin, p.taps);
      it.skip(s0);
      for (int s = s0; s < s1; ++s, ++gst) {
        int ks[C::kSegs];
        const int c0 = it.next(ks);
        if ((int)(gst % C::kGroups) != grp) {  // another group's stage
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* a_st = sA + stage * C::kABytes;
        // Segment j's offset as a row base in the neighbour block, -1 where
        // the segment pads the last stage (k == taps) or the tile is past
        // the end; absent neighbours (-1 in the block) copy zeros (source
        // size 0 reads nothing: a shared zero row would make every SM hit
        // the same L2 line).
        int kb[C::kSegs];
#pragma unroll
        for (int jj = 0; jj < C::kSegs; ++jj)
          kb[jj] = (has_rows && ks[jj] < p.taps) ? ks[jj] * kTileRows : -1;
        const char* const fsrc = fbase + c0 * 2;
        // All rows first (their shared-memory loads overlap), then the copies.
        int row[C::kPerThread];
#pragma unroll
        for (int i = 0; i < C::kPerThread; ++i) {
          const int j = i * C::kGroupThreads / C::kSegCopies;
          row[i] = nb[max(kb[j], 0) + r_i[i]];
          if (kb[j] < 0) row[i] = -1;
        }
#pragma unroll
        for (int i = 0; i < C::kPerThread; ++i) {
          // Block stages: segment j is the next 64-channel block of the row.
          const int j = i * C::kGroupThreads / C::kSegCopies;
          const char* const fseg = fsrc + (GRP ? 0 : j * 128);
          cp_async_16(a_st + dst_i[i], row[i] >= 0 ? fseg + (int64_t)row[i] * rstride : fbase,
                      row[i] >= 0 ? 16u : 0u);
        }
        cp_async_arrive_noinc(&full[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (has_rows) mbar_arrive(&nbr_empty[buf]);  // this thread is done with the block
      buf ^= C::kNbrBufs - 1;
    }
    if (!ok) {
      *s_abort = 1;
      if (pt0 == 0) atomicOr(p.status, kStatTimeout);
    }
    cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      // Operand descriptors of stage 0, segment 0, K step 0.
      const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, C::kSboA, C::kLayoutA);
      const uint64_t b_desc0 = smem_desc(smem_u32(sB), C::kKst * C::kBRow, 8 * C::kBRow, C::kLayoutB);
      ItemIter items(p, cid);
      WorkItem wi;
      while (ok && items.next(p, ncl, wi)) {
        int s0, s1;
        item_range(wi, p.sv, unit_stages<CS, SEGS, GRP>(unit_mask<CL>(p.tile_mask, wi.unit, p.ntiles), p.cin),
                   s0, s1);
        if (s0 == s1) continue;  // an empty part: no accumulator, no epilogue
        const int nst = s1 - s0;
        if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * NPAD;
        for (int s = 0; s < nst; ++s) {
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          fence_proxy_async_smem();  // the A rows were written by cp.async (generic proxy)
          // The stage's descriptors differ from stage 0's only in the start
          // address field (bits 0-13, address / 16; every operand address
          // stays below 256 KB, so the field never carries).
          const uint64_t ad_s = a_desc0 + (uint64_t)((stage * C::kABytes) >> 4);
          const uint64_t bd_s = b_desc0 + (uint64_t)((stage * C::kBBytes) >> 4);
#pragma unroll
          for (int j = 0; j < C::kSegs; ++j) {
#pragma unroll
            for (int kk = 0; kk < CS / 16; ++kk) {
              const uint64_t ad = ad_s + (uint64_t)((j * C::kASeg + kk * 32) >> 4);
              const uint64_t bd = bd_s + (uint64_t)(((j * CS + kk * 16) * C::kBRow) >> 4);
              tc_mma_bf16(d_tmem, ad, bd, p.idesc, (s | j | kk) != 0 ? 1u : 0u);
            }
          }
          if constexpr (CL > 1)
            tc_commit_multicast(&empty[stage], kAllCtas);
          else
            tc_commit(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        *s_abort = 1;
        atomicOr(p.status, kStatTimeout);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    bool rows_zeroed = false;  // the zeroing grid is complete and visible
    const int nchunks = (p.cout + 31) >> 5;
    ItemIter items(p, cid);
    WorkItem wi;
    while (ok && items.next(p, ncl, wi)) {
      // Whole units store; parts add into the zeroed rows, the one that ends
      // the unit with the bias and the residual.  (The host never splits
      // with an activation or a 16-bit output.)  A whole unit has rows, so
      // its centre offset: it is never empty; an empty part is skipped, as
      // the MMA issuer skips it.
      const bool add = !(wi.a == 0 && wi.b == p.sv);
      const bool last = wi.b == p.sv;
      if (add) {
        int s0, s1;
        item_range(wi, p.sv,
                   unit_stages<CS, SEGS, GRP>(unit_mask<CL>(p.tile_mask, wi.unit, p.ntiles), p.cin), s0, s1);
        if (s0 == s1) continue;
      }
      const float bscale = last ? 1.f : 0.f;
      const bool resid = FUSED && p.residual != nullptr && last;
      const int64_t wrow0 = (wi.unit * CL + rank) * kTileRows + warp * 32;  // this warp's rows
      // Output row of this lane's position (-1: a pad position); the stores
      // below take the rows of other lanes by shuffle.
      const int64_t my_pos = wrow0 + lane;
      const int32_t my_row =
          my_pos < p.n ? (p.row_of ? __ldg(p.row_of + my_pos) : (int32_t)my_pos) : -1;
      if (resid && my_row >= 0) {
        // This thread's row of the residual into L2 while the main loop runs
        // (128-byte lines); the column-group loads below then hit L2.
        const int rbytes = p.cout * (p.out_half ? 2 : 4);
        const char* rrow = static_cast<const char*>(p.residual) + (int64_t)my_row * rbytes;
        for (int off = 0; off < rbytes; off += 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(rrow + off));
      }
      if (add && !rows_zeroed) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        rows_zeroed = true;
      }
      if (!mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + acc * NPAD;
      float* stg = s_epi + warp * (32 * kStageRow);
      // Column-group q of a chunk: rows 4q + lane / 8, columns 4 (lane % 8)
      // of the chunk's 32.  Residual values of half h (groups 4h .. 4h + 3).
      auto load_resid = [&](int ch, int h, float4 (&rv)[4]) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int q = 4 * h + qq;
          const int c = ch * 32 + 4 * (lane & 7);
          const int32_t row = __shfl_sync(0xffffffffu, my_row, 4 * q + (lane >> 3));
          rv[qq] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (resid && row >= 0 && c < p.cout) {
            const int64_t e = (int64_t)row * p.cout + c;
            if (p.out_half) {
              const uint2 rb = __ldg(reinterpret_cast<const uint2*>(
                  static_cast<const __nv_bfloat16*>(p.residual) + e));
              if (p.out_half == kOutBf16) {
                rv[qq].x = __uint_as_float(rb.x << 16);  // bf16 -> fp32 is exact: the high half
                rv[qq].y = __uint_as_float(rb.x & 0xffff0000u);
                rv[qq].z = __uint_as_float(rb.y << 16);
                rv[qq].w = __uint_as_float(rb.y & 0xffff0000u);
              } else {
                const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&rb.x));
                const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&rb.y));
                rv[qq] = make_float4(f01.x, f01.y, f23.x, f23.y);
              }
            } else {
              rv[qq] = __ldg(
                  reinterpret_cast<const float4*>(static_cast<const float*>(p.residual) + e));
            }
          }
        }
      };
      // Half h of the chunk from the staging block out to global memory:
      // activation, residual, rounding; each store covers four rows x 128
      // contiguous bytes (64 for bf16).
      auto store_half = [&](int ch, int h, const float4 (&rv)[4]) {
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int q = 4 * h + qq;
          const int r = 4 * q + (lane >> 3), g = lane & 7;
          const int c = ch * 32 + 4 * g;
          const int32_t row = __shfl_sync(0xffffffffu, my_row, r);
          float4 o = *reinterpret_cast<const float4*>(stg + r * kStageRow + 4 * g);
          if (row >= 0 && c < p.cout) {
            const int64_t e = (int64_t)row * p.cout + c;
            if (p.act) {
              o.x = apply_act(o.x, p.act);
              o.y = apply_act(o.y, p.act);
              o.z = apply_act(o.z, p.act);
              o.w = apply_act(o.w, p.act);
            }
            o.x += rv[qq].x;
            o.y += rv[qq].y;
            o.z += rv[qq].z;
            o.w += rv[qq].w;
            if (p.out_half) {
              uint2 pk;
              if (p.out_half == kOutBf16) {
                const __nv_bfloat162 b01 = __float22bfloat162_rn(make_float2(o.x, o.y));
                const __nv_bfloat162 b23 = __float22bfloat162_rn(make_float2(o.z, o.w));
                pk.x = *reinterpret_cast<const uint32_t*>(&b01);
                pk.y = *reinterpret_cast<const uint32_t*>(&b23);
              } else {
                const __half2 h01 = __float22half2_rn(make_float2(o.x, o.y));
                const __half2 h23 = __float22half2_rn(make_float2(o.z, o.w));
                pk.x = *reinterpret_cast<const uint32_t*>(&h01);
                pk.y = *reinterpret_cast<const uint32_t*>(&h23);
              }
              __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + e), pk);
            } else {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + e);
              if (add)
                atomicAdd(dst, o);
              else
                __stcs(dst, o);
            }
          }
        }
      };
      for (int ch = 0; ch < nchunks; ++ch) {
        // Residual loads are issued early (the first half before the TMEM
        // load, the second before the first half is stored), so their L2
        // latency overlaps work; out and residual may be one buffer (in
        // place: each element is read, then written, by this thread), so no
        // load can move past a store by itself.
        float4 ra[4], rb[4];
        if constexpr (FUSED) load_resid(ch, 0, ra);
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + ch * 32, v);
        tmem_ld_wait();
        // Row `lane` (+ bias) into the staging block, 16 bytes at a time ...
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int c = ch * 32 + 4 * q;
          float4 o;
          o.x = __uint_as_float(v[4 * q + 0]) + bscale * s_bias[c + 0];
          o.y = __uint_as_float(v[4 * q + 1]) + bscale * s_bias[c + 1];
          o.z = __uint_as_float(v[4 * q + 2]) + bscale * s_bias[c + 2];
          o.w = __uint_as_float(v[4 * q + 3]) + bscale * s_bias[c + 3];
          *reinterpret_cast<float4*>(stg + lane * kStageRow + 4 * q) = o;
        }
        __syncwarp();
        // ... and out again by column groups.
        if constexpr (FUSED) {
          load_resid(ch, 1, rb);
          store_half(ch, 0, ra);
          store_half(ch, 1, rb);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int r = 4 * q + (lane >> 3), g = lane & 7;
            const int c = ch * 32 + 4 * g;
            const int32_t row = __shfl_sync(0xffffffffu, my_row, r);
            const float4 o = *reinterpret_cast<const float4*>(stg + r * kStageRow + 4 * g);
            if (row >= 0 && c < p.cout) {
              float4* dst =
                  reinterpret_cast<float4*>(static_cast<float*>(p.out) + (int64_t)row * p.cout + c);
              if (add)
                atomicAdd(dst, o);
              else
                __stcs(dst, o);
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
      *s_abort = 1;
      atomicOr(p.status, kStatTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CL > 1) cluster_sync_all();  // no peer traffic is aimed at this CTA any more
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side

namespace {

// cuTensorMapEncodeTiled from the CUDA driver API, looked up once
// (thread-safe static initialisation).
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    cudaGetLastError();
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz, CUtensorMapDataType dt) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr int kMaxDev = 64;

// Per device and kernel instantiation: the shared-memory attribute is set
// once and the number of co-resident clusters is queried once.
struct LaunchCache {
  std::mutex mu;
  int max_clusters[kMaxDev] = {};
};

// Cluster size for the weight multicast.  Default: pairs when a W slice has
// at least two 64-column boxes to split (cout > 64), single CTAs otherwise.
// SC_CONV_CLUSTER=1|2|4 overrides it (4 only where a slice has four boxes).
int cluster_size(int npad) {
  static int forced = [] {
    const char* e = std::getenv("SC_CONV_CLUSTER");
    const int v = e ? std::atoi(e) : 0;
    return (v == 1 || v == 2 || v == 4) ? v : 0;
  }();
  if (forced == 4) return npad >= 256 ? 4 : 2;
  if (forced) return forced;
  return npad > 64 ? 2 : 1;
}

// Parts per unit of the last, partial round of units (1 = no split).  With
// G clusters, `waves` full rounds and `rem` units left over, the leftover
// round takes ceil(rem * S / G) / S of a unit's time when each of its units
// is split S ways.  A split costs a zeroing pass and atomic adds (charged as
// 0.05 + 0.04 S of a unit), each part should keep at least six K stages, and
// a predicted gain under 5% is not taken (a split of 563 units over 74
// clusters, predicted 2%, measured 1% slower).
std::atomic<bool> g_deterministic{false};

int tail_split(int64_t nunits, int64_t G, int max_stages) {
  static const int forced = [] {
    const char* e = std::getenv("SC_CONV_SPLIT");
    return e ? std::atoi(e) : 0;
  }();
  const int64_t rem = nunits >= G ? nunits % G : nunits;
  if (rem == 0 || G <= 0) return 1;
  const double waves = (double)(nunits / G);
  const double t1 = waves + 1.0;
  // Two addends into a zeroed row sum the same in either order; three do not.
  const int cap = std::max(1, std::min(g_deterministic.load() ? 2 : 8, max_stages / 6));
  if (forced > 0) return std::min(forced, cap);
  int best = 1;
  double best_t = t1;
  for (int S = 2; S <= cap; ++S) {
    const double t = waves + (double)((rem * S + G - 1) / G) / S + 0.05 + 0.04 * S;
    if (t < best_t - 1e-9) {
      best_t = t;
      best = S;
    }
  }
  return best_t < 0.95 * t1 ? best : 1;
}

template <int NPAD, int CS, int SEGS, bool GRP, int CL, bool FUSED>
cudaError_t launch_typed(const ConvMap& m, const void* feats, const void* w, bool f16,
                         const Epilogue& ep, int cin, int cout, cudaStream_t s) {
  using C = TcCfg<NPAD, CS, SEGS>;
  auto kern = k_conv_tc<NPAD, CS, SEGS, GRP, CL, FUSED>;
  static LaunchCache cache;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;

  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;

  int max_clusters;
  {
    std::lock_guard<std::mutex> lk(cache.mu);
    if (cache.max_clusters[dev] == 0) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
      if (e != cudaSuccess) return e;
      int sms = 148;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      cfg.gridDim = dim3(CL * (sms / CL), 1, 1);
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess || nc <= 0) {
        cudaGetLastError();
        nc = sms / CL;
      }
      cache.max_clusters[dev] = nc;
    }
    max_clusters = cache.max_clusters[dev];
  }

  alignas(64) CUtensorMap tm_b;
  if (!encode_2d(&tm_b, w, (uint64_t)cout, (uint64_t)m.taps * cin, (uint64_t)cout * 2, C::kBCols,
                 CS, C::kBRow == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                 f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
    return cudaErrorInvalidValue;
  TcArgs a;
  a.feats = static_cast<const __nv_bfloat16*>(feats);
  a.nbr = m.nbr;
  a.tile_mask = m.tile_mask;
  a.row_of = m.row_of;
  a.taps = m.taps;
  a.bias = ep.bias;
  a.residual = ep.residual;
  a.out = ep.out;
  a.act = ep.act;
  a.out_half = ep.out_half;
  a.idesc = idesc_bf16_f32(kTileRows, NPAD, f16);
  a.status = m.status;
  a.n = m.n;
  a.ntiles = m.ntiles;
  a.cin = cin;
  a.cout = cout;
  const int64_t nunits = (m.ntiles + CL - 1) / CL;
  if (nunits == 0) return cudaSuccess;
  const int max_stages = !GRP ? m.taps * (cin / 64) / SEGS : (m.taps + SEGS - 1) / SEGS;
  // An activation or a 16-bit output cannot be applied to partial sums.  In
  // place (residual == out), the split rows would be zeroed, and other parts'
  // sums added, before the last part reads the residual from them.
  const bool unsplit = ep.act || ep.out_half || (ep.residual && ep.residual == ep.out);
  const int split = unsplit ? 1 : tail_split(nunits, max_clusters, max_stages);
  a.split = split;
  a.tail = split > 1 ? (nunits >= max_clusters ? nunits % max_clusters : nunits) : 0;
  a.whole = nunits - a.tail;
  a.nparts = a.tail * split;
  a.nitems = a.nparts + a.whole;
  a.sv = max_stages;
  if (a.tail > 0) {
    // The split units' rows start at zero; their parts add into them.  The
    // convolution is this launch's programmatic dependent (attribute 1).
    const int64_t row0 = a.whole * CL * kTileRows;  // first position of the split units
    const int64_t n4 = (m.n - row0) * cout / 4;     // cout is a multiple of 16
    const int64_t zb = std::min<int64_t>((n4 + 255) / 256, 2 * 148);
    if (m.row_of)
      k_zero_rows_of<<<(unsigned)zb, 256, 0, s>>>(static_cast<float4*>(ep.out), m.row_of, row0,
                                                   m.n, cout / 4);
    else
      k_zero_rows<<<(unsigned)zb, 256, 0, s>>>(
          reinterpret_cast<float4*>(static_cast<float*>(ep.out) + row0 * cout), n4);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    note_launches(1);
    cfg.numAttrs = 2;
  }
  cfg.gridDim = dim3((unsigned)(CL * std::min<int64_t>(a.nitems, max_clusters)), 1, 1);
  void* args[2] = {&tm_b, &a};
  e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kern), args);
  if (e == cudaSuccess) note_launches(1);
  return e;
}

template <int NPAD, int CS, int SEGS, bool GRP>
cudaError_t launch_cl(const ConvMap& m, const void* feats, const void* w, bool f16,
                      const Epilogue& ep, int cin, int cout, cudaStream_t s) {
  const bool fused = ep.act || ep.residual || ep.out_half;
  if constexpr (NPAD >= 256) {
    if (cluster_size(NPAD) == 4)
      return fused ? launch_typed<NPAD, CS, SEGS, GRP, 4, true>(m, feats, w, f16, ep, cin, cout, s)
                   : launch_typed<NPAD, CS, SEGS, GRP, 4, false>(m, feats, w, f16, ep, cin, cout, s);
  }
  if (cluster_size(NPAD) == 2)
    return fused ? launch_typed<NPAD, CS, SEGS, GRP, 2, true>(m, feats, w, f16, ep, cin, cout, s)
                 : launch_typed<NPAD, CS, SEGS, GRP, 2, false>(m, feats, w, f16, ep, cin, cout, s);
  return fused ? launch_typed<NPAD, CS, SEGS, GRP, 1, true>(m, feats, w, f16, ep, cin, cout, s)
               : launch_typed<NPAD, CS, SEGS, GRP, 1, false>(m, feats, w, f16, ep, cin, cout, s);
}

// Wide stages for narrow layers (build-time SC_NARROW_K128, default on).
#ifndef SC_NARROW_K128
#define SC_NARROW_K128 1
#endif
constexpr bool kNarrowStages = SC_NARROW_K128 != 0;
// Two-block stages for wide inputs with cout <= 128 (build-time
// SC_WIDE_K128, default on).
#ifndef SC_WIDE_K128
#define SC_WIDE_K128 1
#endif
constexpr bool kWideStages = SC_WIDE_K128 != 0;

template <int NPAD>
cudaError_t launch_npad(const ConvMap& m, const void* feats, const void* w, bool f16,
                        const Epilogue& ep, int cin, int cout, cudaStream_t s) {
  // Narrow layers (cout <= 64, cin <= 64): K = 128 per stage, so that each
  // stage's fixed synchronisation cost is spread over eight MMAs.
  constexpr int W = (NPAD <= 64 && kNarrowStages) ? 2 : 1;
  if (cin == 16) return launch_cl<NPAD, 16, 4 * W, true>(m, feats, w, f16, ep, cin, cout, s);
  if (cin == 32) return launch_cl<NPAD, 32, 2 * W, true>(m, feats, w, f16, ep, cin, cout, s);
  if (cin == 64) {
    if constexpr (W == 2) return launch_cl<NPAD, 64, 2, true>(m, feats, w, f16, ep, cin, cout, s);
    return launch_cl<NPAD, 64, 1, false>(m, feats, w, f16, ep, cin, cout, s);
  }
  // Wide inputs with cout <= 128: two 64-channel blocks of an offset per
  // stage (K = 128), where the blocks pair up.
  if constexpr (NPAD <= 128 && kWideStages) {
    if ((cin / 64) % 2 == 0)
      return launch_cl<NPAD, 64, 2, false>(m, feats, w, f16, ep, cin, cout, s);
  }
  return launch_cl<NPAD, 64, 1, false>(m, feats, w, f16, ep, cin, cout, s);
}

}  // namespace

void set_deterministic(bool on) { g_deterministic.store(on); }

bool conv_tc_supported(int cin, int cout) {
  const bool cin_ok = cin == 16 || cin == 32 || (cin % 64 == 0 && cin >= 64 && cin <= 1024);
  const bool cout_ok = cout >= 16 && cout <= 256 && cout % 16 == 0;
  return cin_ok && cout_ok;
}

cudaError_t launch_conv_tc(const ConvMap& m, const void* feats, const void* w, bool f16,
                           const Epilogue& ep, int cin, int cout, cudaStream_t s) {
  if (!conv_tc_supported(cin, cout)) return cudaErrorNotSupported;
  // cout <= 32 runs as N = 32 (an M = 128 MMA takes N in steps of 16; the
  // narrower B halves the shared-memory bytes of W per stage), otherwise
  // cout rounded up to 64.
  const int npad = cout <= 32 ? 32 : (cout + 63) / 64 * 64;
  switch (npad) {
    case 32: return launch_npad<32>(m, feats, w, f16, ep, cin, cout, s);
    case 64: return launch_npad<64>(m, feats, w, f16, ep, cin, cout, s);
    case 128: return launch_npad<128>(m, feats, w, f16, ep, cin, cout, s);
    case 192: return launch_npad<192>(m, feats, w, f16, ep, cin, cout, s);
    default: return launch_npad<256>(m, feats, w, f16, ep, cin, cout, s);
  }
}

}  // namespace sc
