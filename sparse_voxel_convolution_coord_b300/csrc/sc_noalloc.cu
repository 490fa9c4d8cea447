// sc_noalloc.cu -- neighbour-table build that allocates no device memory.
//
// sc_build_map allocates its hash table, neighbour table and tile masks.
// Some callers cannot let a library allocate: runtimes that hand a plugin a
// fixed memory budget and forbid allocation while work is being enqueued,
// latency-critical loops where cudaMalloc's implicit device synchronisation
// is not acceptable, or embedded deployments that reserve all device memory
// up front.  For them this file provides one entry point that runs the same
// hash-insert and neighbour-query kernels, with their scratch (the hash table,
// the per-tile masks and the status/pair-count words) in one file-scope
// static device array instead of allocated buffers.  The caller passes the
// coordinates and the output table; the scratch is held by every device that
// loads the library until the process exits.
#include <cstdio>
#include <mutex>

#include "sc_internal.cuh"

namespace {

constexpr int64_t kNoAllocMaxVoxels = int64_t(1) << 19;           // 524,288 voxels
constexpr uint64_t kNoAllocSlots = uint64_t(1) << 20;             // table at load <= 1/2
constexpr int64_t kNoAllocMaxTiles = kNoAllocMaxVoxels / sc::kTileRows;  // 4,096
// Layout in 64-bit words: [slots | tile masks (2 per word) | status, pairs].
constexpr uint64_t kMaskWordOffset = kNoAllocSlots;
constexpr uint64_t kStatusWordOffset = kMaskWordOffset + kNoAllocMaxTiles / 2;
constexpr uint64_t kScratchWords = kStatusWordOffset + sc::kStatusBlockBytes / 8;

static __device__ __align__(256) uint64_t g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint64_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device, looked up once
// per device (the array's name is only a host-side stand-in).
cudaError_t scratch_on_current_device(uint64_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<uint64_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

sc_status report(sc_status st, const char* fmt, long long a = 0, long long b = 0) {
  char msg[256];
  snprintf(msg, sizeof(msg), fmt, a, b);
  return sc::set_last_error(st, msg);
}

}  // namespace

extern "C" SC_API sc_status sc_build_neighbor_table_noalloc(const int32_t* coords, int64_t n,
                                                            int32_t res, int32_t* nbr_out,
                                                            int64_t* pairs_out, void* stream) {
  if (n < 0) return report(SC_ERR_INVALID_ARG, "sc_build_neighbor_table_noalloc: n=%lld < 0", n);
  if (n > kNoAllocMaxVoxels)
    return report(SC_ERR_UNSUPPORTED,
                  "sc_build_neighbor_table_noalloc: n=%lld exceeds the static scratch limit of "
                  "%lld voxels; use sc_build_map",
                  n, kNoAllocMaxVoxels);
  if (res < 1 || res > (1 << 20))
    return report(SC_ERR_INVALID_ARG, "sc_build_neighbor_table_noalloc: res=%lld outside [1, 2^20]",
                  res);
  if (pairs_out) *pairs_out = 0;
  if (n == 0) return sc::set_last_error(SC_OK, "");
  if (!coords || !nbr_out || (reinterpret_cast<uintptr_t>(coords) & 15u) ||
      (reinterpret_cast<uintptr_t>(nbr_out) & 15u))
    return report(SC_ERR_INVALID_ARG,
                  "sc_build_neighbor_table_noalloc: coords and nbr_out must be 16-byte aligned "
                  "device pointers");
  uint64_t* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess)
    return report(SC_ERR_CUDA, "sc_build_neighbor_table_noalloc: scratch lookup failed (%lld)",
                  (long long)e);
  // Load factor <= 1/4 where the static table allows, <= 1/2 always.
  int log2cap = sc::hash_log2cap(n);
  while ((1ull << log2cap) > kNoAllocSlots) --log2cap;
  sc::HashParams hp;
  if (!sc::make_hash_params(hp, scratch, n, res, log2cap, true))
    return report(SC_ERR_UNSUPPORTED,
                  "sc_build_neighbor_table_noalloc: res=%lld too large for the hash key", res);
  uint32_t* tile_mask = reinterpret_cast<uint32_t*>(scratch + kMaskWordOffset);
  uint32_t* status = reinterpret_cast<uint32_t*>(scratch + kStatusWordOffset);
  unsigned long long* pair_count = reinterpret_cast<unsigned long long*>(status + 4);

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The scratch keeps the previous call's contents: clear the slots in use and
  // the status / pair-count words.
  const int64_t ntiles = (n + sc::kTileRows - 1) / sc::kTileRows;
  // As sc_build_map: a batch index beyond the 32-bit key space is retried
  // once with 64-bit keys.
  // The status block comes back into this stack array: pageable memory, so
  // nothing is allocated (a pinned buffer would need cudaHostAlloc, and the
  // call synchronises anyway).
  uint32_t host[sc::kStatusBlockBytes / 4] = {};
  for (int attempt = 0; attempt < 2; ++attempt) {
    e = sc::launch_map_init(hp, tile_mask, ntiles, status, s);
    if (e == cudaSuccess) e = sc::launch_hash_insert(coords, hp, status, s);
    if (e == cudaSuccess)
      e = sc::launch_neighbor_query(coords, hp, nbr_out, tile_mask, pair_count, status,
                                    sc::kNbrRowMajor, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(host, status, sc::kStatusBlockBytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess || !hp.k32 || !(host[0] & sc::kStatKeySpace) ||
        (host[0] & sc::kStatRange))
      break;
    if (!sc::make_hash_params(hp, scratch, n, res, log2cap, false)) break;
  }
  const uint64_t bmax = hp.bmax;
  if (e != cudaSuccess)
    return report(SC_ERR_CUDA, "sc_build_neighbor_table_noalloc: CUDA error %lld", (long long)e);
  const uint32_t st = host[0];
  if (st & sc::kStatRange)
    return report(SC_ERR_COORD_RANGE,
                  "sc_build_neighbor_table_noalloc: a coordinate lies outside [0,%lld)^3 or has "
                  "a negative batch index",
                  res);
  if (st & sc::kStatKeySpace)
    return report(SC_ERR_UNSUPPORTED,
                  "sc_build_neighbor_table_noalloc: batch index >= %lld does not fit the hash key",
                  (long long)bmax);
  if (st & sc::kStatDuplicate)
    return report(SC_ERR_DUPLICATE, "sc_build_neighbor_table_noalloc: duplicate (batch,x,y,z) rows");
  if (st) return report(SC_ERR_TABLE_FULL, "sc_build_neighbor_table_noalloc: probe bound exceeded");
  if (pairs_out) {
    unsigned long long pc;
    pc = 0;
    for (int c = 0; c < sc::kPairCounters; ++c) {
      unsigned long long v;
      memcpy(&v, host + 4 + 2 * c, sizeof(v));
      pc += v;
    }
    *pairs_out = (int64_t)pc;
  }
  return sc::set_last_error(SC_OK, "");
}
