// sc_api.cu -- the C ABI declared in include/sc.h.
//
// Host-side argument checking, handle lifetime, device allocation and error
// reporting.  All arithmetic of the method runs in the kernels of sc_map.cu,
// sc_conv_tc.cu and sc_conv_simt.cu; nothing here computes on the host.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>
#include <unordered_set>

#include "sc_internal.cuh"

// A level-change map (the way down from a voxel set at resolution res to
// its parents at res / 2, and back up); see sc_levels.cu.
struct sc_level {
  uint64_t magic;
  int device;
  int64_t n;        // fine rows
  int64_t np;       // parents
  int32_t res;
  int64_t ntiles;   // ceil(n / 128): tiles of both tables (np <= n)
  void* block;
  int32_t* parent_coords;  // [n][4], the first np used
  int32_t* down_nbr;       // [ntiles][8][128] child rows per parent, tile-major
  uint32_t* down_mask;     // [ntiles]
  int32_t* parent_of;      // [n]
  int32_t* up_nbr;         // [ntiles][8][128] parent at each position's octant
  int32_t* up_row;         // [ntiles * 128] child row of each position
  uint32_t* up_mask;       // [ntiles]
  uint32_t* d_status;
  int64_t* d_np;
  void* (*alloc)(size_t, void*, void*);
  void (*free_fn)(void*, void*, void*);
  void* alloc_ctx;
};

namespace {

constexpr uint64_t kMagicLive = 0x53434d41504c4956ull;  // "SCMAPLIV"

thread_local sc_status t_status = SC_OK;
thread_local char t_msg[512] = "";

std::mutex g_mu;
std::unordered_set<sc_map*>* g_live = nullptr;  // never destroyed (safe at exit)

constexpr uint64_t kMagicLevel = 0x53434c4556454c53ull;  // "SCLEVELS"
std::unordered_set<sc_level*>* g_live_levels = nullptr;   // guarded by g_mu

bool level_live(sc_level* m) {
  if (!m) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_live_levels && g_live_levels->count(m) && m->magic == kMagicLevel;
}

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

// Device memory for a handle (a map or a level map): its allocator, or the
// library pool of its device.
template <typename H>
void* dev_alloc(H* m, size_t bytes, cudaStream_t s) {
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

template <typename H>
void dev_free(H* m, void* p, cudaStream_t s) {
  if (!p) return;
  if (m->free_fn)
    m->free_fn(p, s, m->alloc_ctx);
  else
    cudaFreeAsync(p, s);
}

void release_buffers(sc_map* m, cudaStream_t s) {
  dev_free(m, m->ord_block, s);
  m->ord_block = nullptr;
  m->ord_nbr = nullptr;
  m->ord_mask = nullptr;
  m->ord_row = nullptr;
  dev_free(m, m->block, s);
  m->block = nullptr;
  m->hash.slots = nullptr;
  m->nbr = nullptr;
  m->tile_mask = nullptr;
  m->d_status = nullptr;
  m->d_pairs = nullptr;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// True when p is ordinary device memory of device `dev` (cudaMalloc,
// stream-ordered pools, VMM mappings).  Host memory (pageable, pinned or
// mapped), managed memory and another GPU's memory are not: the convolution
// reads W through a tensor map whose loads may be multicast to the two CTAs
// of a cluster, which must only ever read this GPU's own memory.
bool on_device(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

// [a, a + na) and [b, b + nb) share a byte.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

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

namespace {
std::atomic<uint32_t> g_probe_limit{0};
}
uint32_t probe_limit_setting() { return g_probe_limit.load(std::memory_order_relaxed); }
}  // namespace sc

namespace {

// Library-owned non-blocking stream per device, for reading back an
// asynchronous build's status block without ordering against the caller's
// streams (the build's event is waited on first).
std::mutex g_rb_mu;
cudaStream_t g_rb_stream[kMaxPoolDevices] = {};

cudaStream_t readback_stream(int dev) {
  if (dev < 0 || dev >= kMaxPoolDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_rb_mu);
  if (!g_rb_stream[dev]) {
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_rb_stream[dev] = st;
  }
  return g_rb_stream[dev];
}

// Sum of the per-block pair counters of a status block read back to the host.
int64_t sum_pairs(const uint32_t* host) {
  uint64_t pairs = 0;
  for (int c = 0; c < sc::kPairCounters; ++c) {
    uint64_t v;
    std::memcpy(&v, host + 4 + 2 * c, sizeof(v));
    pairs += v;
  }
  return (int64_t)pairs;
}

// The error a build's status bits stand for (the message names `who`).
sc_status build_error(uint32_t st, const sc_map* m, bool async, const char* who) {
  if (st & sc::kStatRange)
    return fail(SC_ERR_COORD_RANGE,
                "%s: a coordinate lies outside [0,%d)^3 or has a negative batch index", who,
                m->res);
  if (st & sc::kStatKeySpace)
    return async ? fail(SC_ERR_COORD_RANGE, "%s: a batch index is >= nbatch = %llu", who,
                        (unsigned long long)m->hash.bmax)
                 : fail(SC_ERR_UNSUPPORTED,
                        "%s: batch index >= %llu does not fit the hash key for res=%d, n=%lld",
                        who, (unsigned long long)m->hash.bmax, m->res, (long long)m->n);
  if (st & sc::kStatDuplicate) return fail(SC_ERR_DUPLICATE, "%s: duplicate (batch,x,y,z) rows", who);
  if (st & sc::kStatTableFull) return fail(SC_ERR_TABLE_FULL, "%s: hash probe bound exceeded", who);
  return ok();
}

constexpr uint32_t kBuildBits =
    sc::kStatRange | sc::kStatDuplicate | sc::kStatTableFull | sc::kStatKeySpace;

// Wait for an asynchronous build and read its status and pair count (once);
// then report the build's error, or SC_OK.
sc_status resolve(sc_map* m, const char* who) {
  if (m->pending) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != m->device) cudaSetDevice(m->device);
    uint32_t host[sc::kStatusBlockBytes / 4] = {};
    cudaError_t e = cudaEventSynchronize(m->built);
    cudaStream_t rs = e == cudaSuccess ? readback_stream(m->device) : nullptr;
    if (e == cudaSuccess && !rs) e = cudaErrorUnknown;
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(host, m->d_status, sc::kStatusBlockBytes, cudaMemcpyDeviceToHost, rs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(rs);
    if (cur != m->device && cur >= 0) cudaSetDevice(cur);
    if (e != cudaSuccess) return fail_cuda(e, who);
    m->build_word = host[0] & kBuildBits;
    m->npairs = m->build_word ? -1 : sum_pairs(host);
    cudaEventDestroy(m->built);
    m->built = nullptr;
    m->pending = 0;
  }
  return build_error(m->build_word, m, true, who);
}

// sc_build_map (sync: one synchronisation, errors returned as NULL) and
// sc_build_map_async (no synchronisation; nbatch fixes the key width).
sc_handle build_map(const int32_t* coords, int64_t n, int32_t res, int32_t nbatch, void* stream,
                    bool async) {
  const char* who = async ? "sc_build_map_async" : "sc_build_map";
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n < 0 || n >= (int64_t(1) << 31)) {
    fail(SC_ERR_INVALID_ARG, "%s: n=%lld outside [0, 2^31)", who, (long long)n);
    return nullptr;
  }
  if (res < 1 || res > (1 << 20)) {
    fail(SC_ERR_INVALID_ARG, "%s: res=%d outside [1, 2^20]", who, res);
    return nullptr;
  }
  if (n > 0 && (coords == nullptr || !aligned(coords, 16))) {
    fail(SC_ERR_INVALID_ARG, "%s: coords must be a 16-byte aligned device pointer", who);
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
    bool key_ok = sc::make_hash_params(m->hash, nullptr, n, res, log2cap, true);
    if (async) {
      // The caller's batch count fixes the key width up front: 32-bit keys
      // when nbatch * res^3 fits them, else 64-bit; a batch index >= nbatch
      // is then a range error found on the device.
      if (key_ok && m->hash.k32 && (uint64_t)nbatch > m->hash.bmax)
        key_ok = sc::make_hash_params(m->hash, nullptr, n, res, log2cap, false);
      key_ok = key_ok && (uint64_t)nbatch <= m->hash.bmax;
      if (key_ok) m->hash.bmax = (uint64_t)nbatch;
    }
    if (!key_ok) {
      delete m;
      fail(SC_ERR_UNSUPPORTED, "%s: (batch + 1) * res^3 exceeds the 2^%d key space for n=%lld",
           who, 64 - bit_length((uint64_t)n), (long long)n);
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
      fail(SC_ERR_ALLOC, "%s: device allocation failed (n=%lld)", who, (long long)n);
      return nullptr;
    }
    uint8_t* base = static_cast<uint8_t*>(m->block);
    m->hash.slots = reinterpret_cast<uint64_t*>(base);
    m->nbr = reinterpret_cast<int32_t*>(base + b_slots);
    m->tile_mask = reinterpret_cast<uint32_t*>(base + b_slots + b_nbr);
    m->d_status = reinterpret_cast<uint32_t*>(base + b_slots + b_nbr + b_mask);
    m->d_pairs = reinterpret_cast<unsigned long long*>(m->d_status + 4);
    auto launch_build = [&]() {
      cudaError_t e = sc::launch_map_init(m->hash, m->tile_mask, m->ntiles, m->d_status, s);
      if (e == cudaSuccess) e = sc::launch_hash_insert(coords, m->hash, m->d_status, s);
      if (e == cudaSuccess)
        e = sc::launch_neighbor_query(coords, m->hash, m->nbr, m->tile_mask, m->d_pairs,
                                      m->d_status, sc::kNbrTileMajor, s);
      return e;
    };
    cudaError_t e = cudaSuccess;
    if (async) {
      // The three kernels and an event; the status is read on first need.
      e = cudaEventCreateWithFlags(&m->built, cudaEventDisableTiming);
      if (e == cudaSuccess) e = launch_build();
      if (e == cudaSuccess) e = cudaEventRecord(m->built, s);
      m->pending = 1;
      m->npairs = -1;
    } else {
      // The three kernels, then one synchronisation for the status and the
      // pair count.  A batch index beyond the 32-bit key space (rare: more
      // than (2^32 - 1) / res^3 batch elements) is retried once with 64-bit
      // keys in the same buffers.
      uint32_t host_local[sc::kStatusBlockBytes / 4] = {};
      uint32_t* host = sc::status_readback_buffer();
      if (!host) host = host_local;
      for (int attempt = 0; attempt < 2; ++attempt) {
        e = launch_build();
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(host, m->d_status, sc::kStatusBlockBytes, cudaMemcpyDeviceToHost,
                              s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess || !m->hash.k32 || !(host[0] & sc::kStatKeySpace) ||
            (host[0] & sc::kStatRange))
          break;
        if (!sc::make_hash_params(m->hash, m->hash.slots, n, res, log2cap, false)) break;
      }
      if (e == cudaSuccess && host[0]) {
        release_buffers(m, s);
        build_error(host[0], m, false, who);
        delete m;
        return nullptr;
      }
      m->npairs = sum_pairs(host);
    }
    if (e != cudaSuccess) {
      if (m->built) cudaEventDestroy(m->built);
      release_buffers(m, s);
      delete m;
      fail_cuda(e, who);
      return nullptr;
    }
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live) g_live = new std::unordered_set<sc_map*>();
    g_live->insert(m);
  }
  ok();
  return m;
}

// Operand checks shared by every convolution entry point, then the launch.
// n_in: rows of feats; n_out: rows of out (and residual); taps from cm.
sc_status run_conv(const sc::ConvMap& cm, int map_dev, int64_t n_in, int64_t n_out,
                   const void* feats, const void* weight, const float* bias, const void* residual,
                   void* out, int32_t cin, int32_t cout, sc_dtype dtype, sc_activation act,
                   sc_dtype out_dtype, void* stream, const char* who) {
  if (cin < 1 || cout < 1) return fail(SC_ERR_INVALID_ARG, "%s: cin/cout must be >= 1", who);
  if (dtype != SC_F32 && dtype != SC_BF16 && dtype != SC_F16)
    return fail(SC_ERR_UNSUPPORTED, "%s: dtype %d not supported", who, (int)dtype);
  if (out_dtype != SC_F32 && out_dtype != SC_BF16 && out_dtype != SC_F16)
    return fail(SC_ERR_INVALID_ARG, "%s: out_dtype %d not supported", who, (int)out_dtype);
  if (act != SC_ACT_NONE && act != SC_ACT_RELU && act != SC_ACT_SILU)
    return fail(SC_ERR_INVALID_ARG, "%s: activation %d not supported", who, (int)act);
  if (dtype != SC_F32 && !sc::conv_tc_supported(cin, cout))
    return fail(SC_ERR_UNSUPPORTED,
                "%s: bf16/fp16 need cin in {16,32} or a multiple of 64 <= 1024 and cout "
                "a multiple of 16 <= 256 (got cin=%d cout=%d)",
                who, cin, cout);
  if (dtype == SC_F32 && cout > 256)
    return fail(SC_ERR_UNSUPPORTED, "%s: fp32 path supports cout <= 256 (got %d)", who, cout);
  if (n_out == 0) return ok();
  if (!feats || !weight || !out)
    return fail(SC_ERR_INVALID_ARG, "%s: feats, weight and out must be non-NULL", who);
  if (!aligned(feats, 16) || !aligned(weight, 16) || !aligned(out, 16) ||
      (residual && !aligned(residual, 16)) || (bias && !aligned(bias, 4)))
    return fail(SC_ERR_INVALID_ARG, "%s: feats/weight/out/residual must be 16-byte aligned", who);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != map_dev)
    return fail(SC_ERR_INVALID_ARG, "%s: map lives on device %d, current is %d", who, map_dev,
                dev);
  if (!on_device(feats, dev) || !on_device(weight, dev) || !on_device(out, dev) ||
      (residual && !on_device(residual, dev)) || (bias && !on_device(bias, dev)))
    return fail(SC_ERR_INVALID_ARG,
                "%s: feats, weight, bias, residual and out must be device memory of "
                "device %d (not host, mapped, managed or another GPU's memory)",
                who, dev);
  {
    const size_t in_es = dtype == SC_F32 ? 4 : 2, out_es = out_dtype == SC_F32 ? 4 : 2;
    const size_t out_b = (size_t)n_out * cout * out_es;
    if (overlap(out, out_b, feats, (size_t)n_in * cin * in_es) ||
        overlap(out, out_b, weight, (size_t)cm.taps * cin * cout * in_es) ||
        (bias && overlap(out, out_b, bias, (size_t)cout * 4)))
      return fail(SC_ERR_INVALID_ARG, "%s: out overlaps feats, weight or bias", who);
    // In place (residual == out) is allowed: each element is read and then
    // written by one thread.  A partial overlap is not.
    if (residual && residual != out && overlap(out, out_b, residual, out_b))
      return fail(SC_ERR_INVALID_ARG, "%s: residual must be out itself or not overlap it", who);
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  sc::Epilogue ep;
  ep.bias = bias;
  ep.residual = residual;
  ep.out = out;
  ep.act = (int)act;
  ep.out_half = out_dtype == SC_BF16 ? sc::kOutBf16 : (out_dtype == SC_F16 ? sc::kOutF16 : 0);
  cudaError_t e;
  if (dtype != SC_F32)
    e = sc::launch_conv_tc(cm, feats, weight, dtype == SC_F16, ep, cin, cout, s);
  else
    e = sc::launch_conv_simt_f32(cm, static_cast<const float*>(feats),
                                 static_cast<const float*>(weight), ep, cin, cout, s);
  if (e != cudaSuccess) return fail_cuda(e, who);
  return ok();
}

}  // namespace

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

sc_status sc_set_probe_limit(int32_t limit) {
  if (limit < 0) return fail(SC_ERR_INVALID_ARG, "sc_set_probe_limit: limit %d < 0", limit);
  sc::g_probe_limit.store((uint32_t)limit, std::memory_order_relaxed);
  return ok();
}

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
  return build_map(coords, n, res, 0, stream, false);
}

sc_handle sc_build_map_async(const int32_t* coords, int64_t n, int32_t res, int32_t nbatch,
                             void* stream) {
  if (nbatch < 1) {
    fail(SC_ERR_INVALID_ARG, "sc_build_map_async: nbatch=%d < 1", nbatch);
    return nullptr;
  }
  return build_map(coords, n, res, nbatch, stream, true);
}

sc_status sc_map_status(sc_handle h) {
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_map_status: handle is not live");
  return resolve(h, "sc_map_status");
}

sc_status sc_free_map(sc_handle h, void* stream) {
  if (h == nullptr) return ok();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live || !g_live->count(h) || h->magic != kMagicLive)
      return fail(SC_ERR_BAD_HANDLE, "sc_free_map: handle is not live");
    g_live->erase(h);
  }
  // An unread build's event is released once the build has run (destroying
  // a recorded event does not wait).
  if (h->built) cudaEventDestroy(h->built);
  release_buffers(h, static_cast<cudaStream_t>(stream));
  h->magic = 0;
  delete h;
  return ok();
}

sc_status sc_map_order_rows(sc_handle h, void* stream) {
  const char* who = "sc_map_order_rows";
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "%s: handle is not live", who);
  if (h->n == 0 || h->ord_block) return ok();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t b_nbr = up((size_t)h->ntiles * sc::kTileRows * sc::kTaps * 4);
  const size_t b_mask = up((size_t)h->ntiles * 4);
  const size_t b_row = up((size_t)h->ntiles * sc::kTileRows * 4);
  void* blk = dev_alloc(h, b_nbr + b_mask + b_row, s);
  void* scratch = blk ? dev_alloc(h, sc::order_scratch_bytes(h->n), s) : nullptr;
  if (!scratch) {
    if (blk) dev_free(h, blk, s);
    return fail(SC_ERR_ALLOC, "%s: device allocation failed", who);
  }
  uint8_t* b = static_cast<uint8_t*>(blk);
  h->ord_block = blk;
  h->ord_nbr = reinterpret_cast<int32_t*>(b);
  h->ord_mask = reinterpret_cast<uint32_t*>(b + b_nbr);
  h->ord_row = reinterpret_cast<int32_t*>(b + b_nbr + b_mask);
  const cudaError_t e = sc::launch_order_rows(h, scratch, s);
  dev_free(h, scratch, s);
  if (e != cudaSuccess) {
    dev_free(h, blk, s);
    h->ord_block = nullptr;
    h->ord_nbr = nullptr;
    h->ord_mask = nullptr;
    h->ord_row = nullptr;
    return fail_cuda(e, who);
  }
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
  if (resolve(h, "sc_map_pairs") != SC_OK) return -1;
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
  return run_conv(sc::conv_map_of(h), h->device, h->n, h->n, feats, weight, bias, residual, out,
                  cin, cout, dtype, act, out_dtype, stream, "sc_forward");
}

// ---------------------------------------------------------------------------
// level changes

sc_status sc_subdivide(const int32_t* coords, const uint8_t* mask, int64_t n, int32_t res,
                       int32_t* child_coords, int32_t* parent, int32_t* offset, int32_t* child_of,
                       int64_t* m_out, void* stream) {
  const char* who = "sc_subdivide";
  if (!m_out) return fail(SC_ERR_INVALID_ARG, "%s: m_out is NULL", who);
  *m_out = 0;
  if (n < 0 || n >= (int64_t(1) << 28))
    return fail(SC_ERR_INVALID_ARG, "%s: n=%lld outside [0, 2^28)", who, (long long)n);
  if (res < 1 || res > (1 << 19))
    return fail(SC_ERR_INVALID_ARG, "%s: res=%d outside [1, 2^19]", who, res);
  if (n == 0) return ok();
  if (!coords || !child_coords || !aligned(coords, 16) || !aligned(child_coords, 16))
    return fail(SC_ERR_INVALID_ARG, "%s: coords and child_coords must be 16-byte aligned", who);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  sc_map tmp;
  std::memset(&tmp, 0, sizeof(tmp));
  cudaGetDevice(&tmp.device);
  tmp.alloc = g_alloc.alloc;
  tmp.free_fn = g_alloc.free_fn;
  tmp.alloc_ctx = g_alloc.ctx;
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t b_cnt = up((size_t)n * 4);
  void* blk = dev_alloc(&tmp, 2 * b_cnt + up(sc::scan_scratch_bytes(n)) + 256, s);
  if (!blk) return fail(SC_ERR_ALLOC, "%s: scratch allocation failed", who);
  uint8_t* b = static_cast<uint8_t*>(blk);
  int32_t* counts = reinterpret_cast<int32_t*>(b);
  int32_t* first = reinterpret_cast<int32_t*>(b + b_cnt);
  void* scan_work = b + 2 * b_cnt;
  uint8_t* tail = b + 2 * b_cnt + up(sc::scan_scratch_bytes(n));
  int64_t* total = reinterpret_cast<int64_t*>(tail);
  uint32_t* status = reinterpret_cast<uint32_t*>(tail + 8);
  struct {
    int64_t total;
    uint32_t status;
    uint32_t pad;
  } host = {0, 0, 0};
  cudaError_t e = cudaMemsetAsync(status, 0, 4, s);
  if (e == cudaSuccess) e = sc::launch_child_counts(coords, mask, n, res, counts, status, s);
  if (e == cudaSuccess) e = sc::scan_exclusive(counts, first, n, total, scan_work, s);
  if (e == cudaSuccess)
    e = sc::launch_subdivide(coords, mask, n, first, child_coords, parent, offset, child_of, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&host, tail, 12, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  dev_free(&tmp, blk, s);
  if (e != cudaSuccess) return fail_cuda(e, who);
  if (host.status & sc::kStatRange)
    return fail(SC_ERR_COORD_RANGE,
                "%s: a coordinate lies outside [0,%d)^3 or has a negative batch index", who, res);
  *m_out = host.total;
  return ok();
}

sc_status sc_channel_to_spatial(const void* feats, const int32_t* parent, const int32_t* offset,
                                int64_t m, int32_t c, sc_dtype dtype, void* out, void* stream) {
  const char* who = "sc_channel_to_spatial";
  if (m < 0 || c < 1) return fail(SC_ERR_INVALID_ARG, "%s: m < 0 or c < 1", who);
  if (dtype != SC_F32 && dtype != SC_BF16 && dtype != SC_F16)
    return fail(SC_ERR_UNSUPPORTED, "%s: dtype %d not supported", who, (int)dtype);
  if (m == 0) return ok();
  if (!feats || !parent || !offset || !out)
    return fail(SC_ERR_INVALID_ARG, "%s: NULL argument", who);
  const cudaError_t e = sc::launch_channel_to_spatial(feats, parent, offset, m, c,
                                                      dtype == SC_F32 ? 4 : 2, out,
                                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, who);
  return ok();
}

sc_level_handle sc_build_level_map(const int32_t* coords, int64_t n, int32_t res, int32_t nbatch,
                                   void* stream) {
  const char* who = "sc_build_level_map";
  if (n < 0 || n >= (int64_t(1) << 31)) {
    fail(SC_ERR_INVALID_ARG, "%s: n=%lld outside [0, 2^31)", who, (long long)n);
    return nullptr;
  }
  if (res < 1 || res > (1 << 20) || nbatch < 1) {
    fail(SC_ERR_INVALID_ARG, "%s: res=%d outside [1, 2^20] or nbatch=%d < 1", who, res, nbatch);
    return nullptr;
  }
  if (n > 0 && (!coords || !aligned(coords, 16))) {
    fail(SC_ERR_INVALID_ARG, "%s: coords must be a 16-byte aligned device pointer", who);
    return nullptr;
  }
  // Parent keys ((b * pr + x) * pr + y) * pr + z, pr = ceil(res / 2).
  const uint64_t pr = (uint64_t)(res + 1) / 2;
  const int bits_b = bit_length((uint64_t)nbatch - 1), bits_p = bit_length(pr - 1);
  if (bits_b + 3 * bits_p > 63) {
    fail(SC_ERR_UNSUPPORTED, "%s: nbatch * (res/2)^3 does not fit a 63-bit key", who);
    return nullptr;
  }
  const uint64_t kmax = ((uint64_t)nbatch * pr * pr * pr) - 1;
  const int key_bits = std::max(1, bit_length(kmax));
  const bool k32 = key_bits <= 32;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  sc_level* h = new sc_level();
  std::memset(h, 0, sizeof(*h));
  h->magic = kMagicLevel;
  cudaGetDevice(&h->device);
  h->n = n;
  h->res = res;
  h->alloc = g_alloc.alloc;
  h->free_fn = g_alloc.free_fn;
  h->alloc_ctx = g_alloc.ctx;
  h->ntiles = (n + sc::kTileRows - 1) / sc::kTileRows;
  if (n > 0) {
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t nt = (size_t)h->ntiles;
    const size_t b_pc = up((size_t)n * 16), b_tab = up(nt * 8 * sc::kTileRows * 4),
                 b_mask = up(nt * 4), b_rows = up((size_t)n * 4),
                 b_uprow = up(nt * sc::kTileRows * 4);
    h->block = dev_alloc(h, b_pc + 2 * b_tab + 2 * b_mask + b_rows + b_uprow + 256, s);
    void* scratch = h->block ? dev_alloc(h, sc::level_scratch_bytes(n, k32 ? 4 : 8), s) : nullptr;
    if (!scratch) {
      if (h->block) dev_free(h, h->block, s);
      delete h;
      fail(SC_ERR_ALLOC, "%s: device allocation failed (n=%lld)", who, (long long)n);
      return nullptr;
    }
    uint8_t* b = static_cast<uint8_t*>(h->block);
    h->parent_coords = reinterpret_cast<int32_t*>(b);
    b += b_pc;
    h->down_nbr = reinterpret_cast<int32_t*>(b);
    b += b_tab;
    h->up_nbr = reinterpret_cast<int32_t*>(b);
    b += b_tab;
    h->down_mask = reinterpret_cast<uint32_t*>(b);
    b += b_mask;
    h->up_mask = reinterpret_cast<uint32_t*>(b);
    b += b_mask;
    h->parent_of = reinterpret_cast<int32_t*>(b);
    b += b_rows;
    h->up_row = reinterpret_cast<int32_t*>(b);
    b += b_uprow;
    h->d_np = reinterpret_cast<int64_t*>(b);
    h->d_status = reinterpret_cast<uint32_t*>(b + 8);
    struct {
      int64_t np;
      uint32_t status;
      uint32_t pad;
    } host = {0, 0, 0};
    cudaError_t e = cudaMemsetAsync(h->d_status, 0, 4, s);
    if (e == cudaSuccess)
      e = k32 ? sc::build_level_tables<uint32_t>(coords, n, res, nbatch, key_bits, scratch,
                                                 h->down_nbr, h->down_mask, h->parent_of,
                                                 h->parent_coords, h->up_nbr, h->up_row,
                                                 h->up_mask, h->d_np, h->d_status, s)
              : sc::build_level_tables<unsigned long long>(
                    coords, n, res, nbatch, key_bits, scratch, h->down_nbr, h->down_mask,
                    h->parent_of, h->parent_coords, h->up_nbr, h->up_row, h->up_mask, h->d_np,
                    h->d_status, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&host, h->d_np, 12, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    dev_free(h, scratch, s);
    if (e != cudaSuccess || host.status) {
      dev_free(h, h->block, s);
      delete h;
      if (e != cudaSuccess)
        fail_cuda(e, who);
      else if (host.status & sc::kStatRange)
        fail(SC_ERR_COORD_RANGE,
             "%s: a coordinate lies outside [0,%d)^3 or a batch index outside [0,%d)", who, res,
             nbatch);
      else
        fail(SC_ERR_DUPLICATE, "%s: duplicate (batch,x,y,z) rows", who);
      return nullptr;
    }
    h->np = host.np;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live_levels) g_live_levels = new std::unordered_set<sc_level*>();
    g_live_levels->insert(h);
  }
  ok();
  return h;
}

int64_t sc_level_parents(sc_level_handle h) {
  if (!level_live(h)) {
    fail(SC_ERR_BAD_HANDLE, "sc_level_parents: handle is not live");
    return -1;
  }
  ok();
  return h->np;
}

sc_status sc_get_level_map(sc_level_handle h, int32_t* parent_coords, int32_t* child_of,
                           int32_t* parent_of, void* stream) {
  const char* who = "sc_get_level_map";
  if (!level_live(h)) return fail(SC_ERR_BAD_HANDLE, "%s: handle is not live", who);
  if (h->n == 0) return ok();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (parent_coords)
    e = cudaMemcpyAsync(parent_coords, h->parent_coords, (size_t)h->np * 16,
                        cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && parent_of)
    e = cudaMemcpyAsync(parent_of, h->parent_of, (size_t)h->n * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && child_of) e = sc::launch_child_table(h->down_nbr, h->np, child_of, s);
  if (e != cudaSuccess) return fail_cuda(e, who);
  return ok();
}

sc_status sc_conv_down(sc_level_handle h, const void* feats, const void* weight,
                       const float* bias, const void* residual, void* out, int32_t cin,
                       int32_t cout, sc_dtype dtype, sc_activation act, sc_dtype out_dtype,
                       void* stream) {
  if (!level_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_conv_down: handle is not live");
  const sc::ConvMap cm{h->down_nbr, h->down_mask, nullptr, h->np,
                       (h->np + sc::kTileRows - 1) / sc::kTileRows, 8, h->d_status};
  return run_conv(cm, h->device, h->n, h->np, feats, weight, bias, residual, out, cin, cout,
                  dtype, act, out_dtype, stream, "sc_conv_down");
}

sc_status sc_conv_up(sc_level_handle h, const void* feats, const void* weight, const float* bias,
                     const void* residual, void* out, int32_t cin, int32_t cout, sc_dtype dtype,
                     sc_activation act, sc_dtype out_dtype, void* stream) {
  if (!level_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_conv_up: handle is not live");
  const sc::ConvMap cm{h->up_nbr, h->up_mask, h->up_row, h->n, h->ntiles, 8, h->d_status};
  return run_conv(cm, h->device, h->np, h->n, feats, weight, bias, residual, out, cin, cout,
                  dtype, act, out_dtype, stream, "sc_conv_up");
}

sc_status sc_level_device_status(sc_level_handle h, void* stream) {
  if (!level_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_level_device_status: handle is not live");
  if (h->n == 0) return ok();
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t st = 0;
  cudaError_t e = cudaMemcpyAsync(&st, h->d_status, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->d_status, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e, "sc_level_device_status");
  if (st & sc::kStatTimeout)
    return fail(SC_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (device status 0x%x)", st);
  if (st) return fail(SC_ERR_CUDA, "device status 0x%x", st);
  return ok();
}

sc_status sc_free_level_map(sc_level_handle h, void* stream) {
  if (h == nullptr) return ok();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live_levels || !g_live_levels->count(h) || h->magic != kMagicLevel)
      return fail(SC_ERR_BAD_HANDLE, "sc_free_level_map: handle is not live");
    g_live_levels->erase(h);
  }
  if (h->block) dev_free(h, h->block, static_cast<cudaStream_t>(stream));
  h->magic = 0;
  delete h;
  return ok();
}

// ---------------------------------------------------------------------------
// dual-grid mesh

sc_status sc_dual_mesh_quads(sc_handle h, const uint8_t* flags, int32_t* quads, int64_t* q_out,
                             void* stream) {
  const char* who = "sc_dual_mesh_quads";
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "%s: handle is not live", who);
  if (!q_out) return fail(SC_ERR_INVALID_ARG, "%s: q_out is NULL", who);
  *q_out = 0;
  if (h->n == 0) return ok();
  if (!flags || !quads || !aligned(quads, 16))
    return fail(SC_ERR_INVALID_ARG, "%s: flags and a 16-byte aligned quads are required", who);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t b_cnt = up((size_t)h->n * 4);
  void* blk = dev_alloc(h, 2 * b_cnt + up(sc::scan_scratch_bytes(h->n)) + 256, s);
  if (!blk) return fail(SC_ERR_ALLOC, "%s: scratch allocation failed", who);
  uint8_t* b = static_cast<uint8_t*>(blk);
  int32_t* counts = reinterpret_cast<int32_t*>(b);
  int32_t* first = reinterpret_cast<int32_t*>(b + b_cnt);
  int64_t* total = reinterpret_cast<int64_t*>(b + 2 * b_cnt + up(sc::scan_scratch_bytes(h->n)));
  int64_t nq = 0;
  cudaError_t e = sc::launch_quad_counts(h, flags, counts, s);
  if (e == cudaSuccess)
    e = sc::scan_exclusive(counts, first, h->n, total, b + 2 * b_cnt, s);
  if (e == cudaSuccess) e = sc::launch_quads(h, flags, first, quads, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&nq, total, 8, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  dev_free(h, blk, s);
  if (e != cudaSuccess) return fail_cuda(e, who);
  *q_out = nq;
  return ok();
}

sc_status sc_dual_mesh_triangulate(const int32_t* quads, int64_t nq, const float* vertices,
                                   int32_t* tris, void* stream) {
  const char* who = "sc_dual_mesh_triangulate";
  if (nq < 0) return fail(SC_ERR_INVALID_ARG, "%s: nq < 0", who);
  if (nq == 0) return ok();
  if (!quads || !vertices || !tris || !aligned(quads, 16))
    return fail(SC_ERR_INVALID_ARG, "%s: NULL or unaligned argument", who);
  const cudaError_t e =
      sc::launch_triangulate(quads, nq, vertices, tris, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, who);
  return ok();
}

sc_status sc_device_status(sc_handle h, void* stream) {
  if (!is_live(h)) return fail(SC_ERR_BAD_HANDLE, "sc_device_status: handle is not live");
  if (h->n == 0) return ok();
  // An asynchronous build's own error first (it stays with the map).
  if (resolve(h, "sc_device_status") != SC_OK) return sc_last_error();
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
