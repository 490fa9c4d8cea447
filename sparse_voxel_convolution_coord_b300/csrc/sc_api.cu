// sc_api.cu -- the C ABI declared in include/sc.h.
//
// Host-side argument checking, handle lifetime, device allocation and error
// reporting.  All arithmetic of the method runs in the kernels of sc_map.cu,
// sc_conv_tc.cu and sc_conv_simt.cu; nothing here computes on the host.
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>
#include <unordered_set>

#include "sc_internal.cuh"

namespace {

constexpr uint64_t kMagicLive = 0x53434d41504c4956ull;  // "SCMAPLIV"

thread_local sc_status t_status = SC_OK;
thread_local char t_msg[512] = "";

std::mutex g_mu;
std::unordered_set<sc_map*>* g_live = nullptr;  // never destroyed (safe at exit)

struct AllocCfg {
  void* (*alloc)(size_t, void*, void*) = nullptr;
  void (*free_fn)(void*, void*, void*) = nullptr;
  void* ctx = nullptr;
} g_alloc;

sc_status fail(sc_status st, const char* fmt, ...) {
  t_status = st;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return st;
}

sc_status ok() {
  t_status = SC_OK;
  t_msg[0] = 0;
  return SC_OK;
}

sc_status fail_cuda(cudaError_t e, const char* what) {
  return fail(SC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool is_live(sc_map* m) {
  if (!m) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_live && g_live->count(m) && m->magic == kMagicLive;
}

// The library's own stream-ordered pool on `dev`.  Its release threshold is
// unlimited, so memory freed by sc_free_map stays reserved for the next map
// instead of being unmapped at the next synchronisation (re-mapping tens of
// MB costs more than building the map); sc_release_cached_memory trims it.
constexpr int kMaxPoolDevices = 64;
std::mutex g_pool_mu;
cudaMemPool_t g_pools[kMaxPoolDevices] = {};

cudaMemPool_t lib_pool(int dev) {
  if (dev < 0 || dev >= kMaxPoolDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_pool_mu);
  if (!g_pools[dev]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    uint64_t keep = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    g_pools[dev] = pool;
  }
  return g_pools[dev];
}

void* dev_alloc(sc_map* m, size_t bytes, cudaStream_t s) {
  if (bytes == 0) bytes = 16;
  if (m->alloc) return m->alloc(bytes, s, m->alloc_ctx);
  cudaMemPool_t pool = lib_pool(m->device);
  void* p = nullptr;
  if (!pool || cudaMallocFromPoolAsync(&p, bytes, pool, s) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return p;
}

void dev_free(sc_map* m, void* p, cudaStream_t s) {
  if (!p) return;
  if (m->free_fn)
    m->free_fn(p, s, m->alloc_ctx);
  else
    cudaFreeAsync(p, s);
}

void release_buffers(sc_map* m, cudaStream_t s) {
  dev_free(m, m->block, s);
  m->block = nullptr;
  m->hash.slots = nullptr;
  m->nbr = nullptr;
  m->tile_mask = nullptr;
  m->d_status = nullptr;
  m->d_pairs = nullptr;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int bit_length(uint64_t v) { return v ? 64 - __builtin_clzll(v) : 0; }

}  // namespace

namespace sc {
sc_status set_last_error(sc_status st, const char* msg) {
  return st == SC_OK ? ok() : fail(st, "%s", msg);
}
}  // namespace sc

namespace sc {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launches(int k) { g_launches.fetch_add((uint64_t)k, std::memory_order_relaxed); }

// Pinned host block for a build's status read-back, one per host thread
// (a copy into pageable memory goes through a driver staging buffer).
// nullptr if pinned memory cannot be had; callers then use their own.
uint32_t* status_readback_buffer() {
  struct Block {
    uint32_t* p = nullptr;
    ~Block() {
      if (p) cudaFreeHost(p);
    }
  };
  thread_local Block b;
  if (!b.p) {
    void* q = nullptr;
    if (cudaHostAlloc(&q, kStatusBlockBytes, cudaHostAllocPortable) == cudaSuccess)
      b.p = static_cast<uint32_t*>(q);
    else
      cudaGetLastError();
  }
  return b.p;
}
uint64_t launches() { return g_launches.load(std::memory_order_relaxed); }
}  // namespace sc

extern "C" {

sc_status sc_last_error(void) { return t_status; }
const char* sc_last_error_msg(void) { return t_msg; }
const char* sc_version(void) { return "sc-b300 0.1 (sm_103a)"; }

sc_status sc_set_allocator(void* (*alloc)(size_t, void*, void*),
                           void (*free_fn)(void*, void*, void*), void* ctx) {
  if ((alloc == nullptr) != (free_fn == nullptr))
    return fail(SC_ERR_INVALID_ARG, "sc_set_allocator: alloc and free must both be set or NULL");
  g_alloc.alloc = alloc;
  g_alloc.free_fn = free_fn;
  g_alloc.ctx = ctx;
  return ok();
}

uint64_t sc_kernel_launches(void) { return sc::launches(); }

sc_status sc_release_cached_memory(void) {
  std::lock_guard<std::mutex> lk(g_pool_mu);
  for (int d = 0; d < kMaxPoolDevices; ++d) {
    if (!g_pools[d]) continue;
    const cudaError_t e = cudaMemPoolTrimTo(g_pools[d], 0);
    if (e != cudaSuccess) return fail_cuda(e, "sc_release_cached_memory");
  }
  return ok();
}

sc_status sc_set_deterministic(int32_t enable) {
  if (enable != 0 && enable != 1)
    return fail(SC_ERR_INVALID_ARG, "sc_set_deterministic: enable must be 0 or 1");
  sc::set_deterministic(enable != 0);
  return ok();
}

sc_handle sc_build_map(const int32_t* coords, int64_t n, int32_t res, void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n < 0 || n >= (int64_t(1) << 31)) {
    fail(SC_ERR_INVALID_ARG, "sc_build_map: n=%lld outside [0, 2^31)", (long long)n);
    return nullptr;
  }
  if (res < 1 || res > (1 << 20)) {
    fail(SC_ERR_INVALID_ARG, "sc_build_map: res=%d outside [1, 2^20]", res);
    return nullptr;
  }
  if (n > 0 && (coords == nullptr || !aligned(coords, 16))) {
    fail(SC_ERR_INVALID_ARG, "sc_build_map: coords must be a 16-byte aligned device pointer");
    return nullptr;
  }
  sc_map* m = new sc_map();
  std::memset(m, 0, sizeof(*m));
  m->magic = kMagicLive;
  cudaGetDevice(&m->device);
  m->n = n;
  m->res = res;
  m->alloc = g_alloc.alloc;
  m->free_fn = g_alloc.free_fn;
  m->alloc_ctx = g_alloc.ctx;
  m->ntiles = (n + sc::kTileRows - 1) / sc::kTileRows;

  if (n > 0) {
    const int log2cap = sc::hash_log2cap(n);
    const uint64_t cap = 1ull << log2cap;
    if (!sc::make_hash_params(m->hash, nullptr, n, res, log2cap, true)) {
      delete m;
      fail(SC_ERR_UNSUPPORTED, "sc_build_map: res^3 exceeds the 2^%d key space for n=%lld",
           64 - bit_length((uint64_t)n), (long long)n);
      return nullptr;
    }
    // One allocation, carved (every piece 256-byte aligned): the hash table,
    // the tile-major neighbour table [ntiles][27][128] (pad rows -1: a
    // tile's rows are contiguous per offset, and a tile's whole 13,824-byte
    // block is one contiguous range for the convolution), the tile masks and
    // the status / pair-counter block (sc::kStatusBlockBytes).
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t b_slots = up(cap * sizeof(uint64_t));
    const size_t b_nbr = up((size_t)m->ntiles * sc::kTileRows * sc::kTaps * sizeof(int32_t));
    const size_t b_mask = up((size_t)m->ntiles * sizeof(uint32_t));
    m->block = dev_alloc(m, b_slots + b_nbr + b_mask + up(sc::kStatusBlockBytes), s);
    if (!m->block) {
      delete m;
      fail(SC_ERR_ALLOC, "sc_build_map: device allocation failed (n=%lld)", (long long)n);
      return nullptr;
    }
    uint8_t* base = static_cast<uint8_t*>(m->block);
    m->hash.slots = reinterpret_cast<uint64_t*>(base);
    m->nbr = reinterpret_cast<int32_t*>(base + b_slots);
    m->tile_mask = reinterpret_cast<uint32_t*>(base + b_slots + b_nbr);
    m->d_status = reinterpret_cast<uint32_t*>(base + b_slots + b_nbr + b_mask);
    m->d_pairs = reinterpret_cast<unsigned long long*>(m->d_status + 4);
    // The three kernels, then one synchronisation for the status and the
    // pair count.  A batch index beyond the 32-bit key space (rare: more
    // than (2^32 - 1) / res^3 batch elements) is retried once with 64-bit
    // keys in the same buffers.
    uint32_t host_local[sc::kStatusBlockBytes / 4] = {};
    uint32_t* host = sc::status_readback_buffer();
    if (!host) host = host_local;
    cudaError_t e = cudaSuccess;
    for (int attempt = 0; attempt < 2; ++attempt) {
      e = sc::launch_map_init(m->hash, m->tile_mask, m->ntiles, m->d_status, s);
      if (e == cudaSuccess) e = sc::launch_hash_insert(coords, m->hash, m->d_status, s);
      if (e == cudaSuccess)
        e = sc::launch_neighbor_query(coords, m->hash, m->nbr, m->tile_mask, m->d_pairs,
                                      m->d_status, sc::kNbrTileMajor, s);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(host, m->d_status, sc::kStatusBlockBytes, cudaMemcpyDeviceToHost, s);
      if (e == cudaSuccess) e = cudaStreamSynchronize(s);
      if (e != cudaSuccess || !m->hash.k32 || !(host[0] & sc::kStatKeySpace) ||
          (host[0] & sc::kStatRange))
        break;
      if (!sc::make_hash_params(m->hash, m->hash.slots, n, res, log2cap, false)) break;
    }
    if (e != cudaSuccess) {
      release_buffers(m, s);
      delete m;
      fail_cuda(e, "sc_build_map");
      return nullptr;
    }
    const uint64_t bmax = m->hash.bmax;
    const uint32_t st = host[0];
    if (st) {
      release_buffers(m, s);
      delete m;
      if (st & sc::kStatRange)
        fail(SC_ERR_COORD_RANGE,
             "sc_build_map: a coordinate lies outside [0,%d)^3 or has a negative batch index",
             res);
      else if (st & sc::kStatKeySpace)
        fail(SC_ERR_UNSUPPORTED,
             "sc_build_map: batch index >= %llu does not fit the hash key for res=%d, n=%lld",
             (unsigned long long)bmax, res, (long long)n);
      else if (st & sc::kStatDuplicate)
        fail(SC_ERR_DUPLICATE, "sc_build_map: duplicate (batch,x,y,z) rows");
      else
        fail(SC_ERR_TABLE_FULL, "sc_build_map: hash probe bound exceeded");
      return nullptr;
    }
    uint64_t pairs;
    pairs = 0;
    for (int c = 0; c < sc::kPairCounters; ++c) {
      uint64_t v;
      std::memcpy(&v, host + 4 + 2 * c, sizeof(v));
      pairs += v;
    }
    m->npairs = (int64_t)pairs;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live) g_live = new std::unordered_set<sc_map*>();
    g_live->insert(m);
  }
  ok();
  return m;
}

sc_status sc_free_map(sc_handle h, void* stream) {
  if (h == nullptr) return ok();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live || !g_live->count(h) || h->magic != kMagicLive)
      return fail(SC_ERR_BAD_HANDLE, "sc_free_map: handle is not live");
    g_live->erase(h);
  }
  release_buffers(h, static_cast<cudaStream_t>(stream));
  h->magic = 0;
  delete h;
  return ok();
}

int64_t sc_map_size(sc_handle h) {
  if (!is_live(h)) {
    fail(SC_ERR_BAD_HANDLE, "sc_map_size: handle is not live");
    return -1;
  }
  ok();
  return h->n;
}

int64_t sc_map_pairs(sc_handle h) {
  if (!is_live(h)) {
    fail(SC_ERR_BAD_HANDLE, "sc_map_pairs: handle is not live");
    return -1;
  }
  ok();
  return h->npairs;
}

sc_status sc_get_neighbor_table(sc_handle h, int32_t* nbr_out, void* stream) {
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_get_neighbor_table: handle is not live");
  if (h->n == 0) return ok();
  if (!nbr_out) return fail(SC_ERR_INVALID_ARG, "sc_get_neighbor_table: nbr_out is NULL");
  cudaError_t e = sc::launch_nbr_to_row_major(h, nbr_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "sc_get_neighbor_table");
  return ok();
}

sc_status sc_get_pairs(sc_handle h, int64_t* off_host, int32_t* in, int32_t* out, void* stream) {
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_get_pairs: handle is not live");
  if (!off_host) return fail(SC_ERR_INVALID_ARG, "sc_get_pairs: off_host is NULL");
  if (h->n == 0) {
    for (int k = 0; k < 28; ++k) off_host[k] = 0;
    return ok();
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* scratch = dev_alloc(h, sc::pairs_scratch_bytes(h->n), s);
  if (!scratch) return fail(SC_ERR_ALLOC, "sc_get_pairs: scratch allocation failed");
  cudaError_t e = sc::launch_pairs(h, off_host, in, out, scratch, s);
  dev_free(h, scratch, s);
  if (e != cudaSuccess) return fail_cuda(e, "sc_get_pairs");
  return ok();
}

sc_status sc_forward(sc_handle h, const void* feats, const void* weight, const float* bias,
                     float* out, int32_t cin, int32_t cout, sc_dtype dtype, void* stream) {
  return sc_forward_ex(h, feats, weight, bias, nullptr, out, cin, cout, dtype, SC_ACT_NONE, SC_F32,
                       stream);
}

sc_status sc_forward_ex(sc_handle h, const void* feats, const void* weight, const float* bias,
                        const void* residual, void* out, int32_t cin, int32_t cout,
                        sc_dtype dtype, sc_activation act, sc_dtype out_dtype, void* stream) {
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_forward: handle is not live");
  if (cin < 1 || cout < 1) return fail(SC_ERR_INVALID_ARG, "sc_forward: cin/cout must be >= 1");
  if (dtype != SC_F32 && dtype != SC_BF16 && dtype != SC_F16)
    return fail(SC_ERR_UNSUPPORTED, "sc_forward: dtype %d not supported", (int)dtype);
  if (out_dtype != SC_F32 && out_dtype != SC_BF16 && out_dtype != SC_F16)
    return fail(SC_ERR_INVALID_ARG, "sc_forward_ex: out_dtype %d not supported", (int)out_dtype);
  if (act != SC_ACT_NONE && act != SC_ACT_RELU && act != SC_ACT_SILU)
    return fail(SC_ERR_INVALID_ARG, "sc_forward_ex: activation %d not supported", (int)act);
  if (dtype != SC_F32 && !sc::conv_tc_supported(cin, cout))
    return fail(SC_ERR_UNSUPPORTED,
                "sc_forward: bf16/fp16 need cin in {16,32} or a multiple of 64 <= 1024 and cout "
                "a multiple of 16 <= 256 (got cin=%d cout=%d)",
                cin, cout);
  if (dtype == SC_F32 && cout > 256)
    return fail(SC_ERR_UNSUPPORTED, "sc_forward: fp32 path supports cout <= 256 (got %d)", cout);
  if (h->n == 0) return ok();
  if (!feats || !weight || !out)
    return fail(SC_ERR_INVALID_ARG, "sc_forward: feats, weight and out must be non-NULL");
  if (!aligned(feats, 16) || !aligned(weight, 16) || !aligned(out, 16) ||
      (residual && !aligned(residual, 16)) || (bias && !aligned(bias, 4)))
    return fail(SC_ERR_INVALID_ARG,
                "sc_forward: feats/weight/out/residual must be 16-byte aligned");
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != h->device)
    return fail(SC_ERR_INVALID_ARG, "sc_forward: map lives on device %d, current is %d",
                h->device, dev);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  sc::Epilogue ep;
  ep.bias = bias;
  ep.residual = residual;
  ep.out = out;
  ep.act = (int)act;
  ep.out_half = out_dtype == SC_BF16 ? sc::kOutBf16 : (out_dtype == SC_F16 ? sc::kOutF16 : 0);
  cudaError_t e;
  if (dtype != SC_F32)
    e = sc::launch_conv_tc(h, feats, weight, dtype == SC_F16, ep, cin, cout, s);
  else
    e = sc::launch_conv_simt_f32(h, static_cast<const float*>(feats),
                                 static_cast<const float*>(weight), ep, cin, cout, s);
  if (e != cudaSuccess) return fail_cuda(e, "sc_forward");
  return ok();
}

sc_status sc_device_status(sc_handle h, void* stream) {
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_device_status: handle is not live");
  if (h->n == 0) return ok();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t st = 0;
  cudaError_t e = cudaMemcpyAsync(&st, h->d_status, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->d_status, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e, "sc_device_status");
  if (st & sc::kStatTimeout)
    return fail(SC_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (device status 0x%x)", st);
  if (st & sc::kStatTableFull) return fail(SC_ERR_TABLE_FULL, "hash probe bound exceeded");
  if (st) return fail(SC_ERR_CUDA, "device status 0x%x", st);
  return ok();
}

}  // extern "C"
