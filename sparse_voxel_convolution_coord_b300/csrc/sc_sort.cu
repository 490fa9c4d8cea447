// sc_sort.cu -- device-wide exclusive scan and stable counting-sort passes.
//
// Building blocks of the level-change maps (sc_levels.cu): subdivision needs
// each parent's first child row (a scan of child counts), the way down needs
// the distinct parents in (batch, x, y, z) order (a least-significant-digit
// radix sort of the parents' packed keys, 9 bits per stable pass), and the
// transposed convolution groups child rows by their octant (one 3-bit pass).
//
// Scan: three launches -- per-chunk sums (4096 elements a block), a scan of
// the chunk sums in one block, and the chunks' own scans with their carry.
//
// Counting-sort pass over the digit d = (key >> shift) & (bins - 1), bins <=
// 512: per-block digit counts [d][block] (digit-major, so that their
// exclusive scan is each (digit, block)'s first output position), the scan,
// and a scatter in which every block ranks its elements stably: elements are
// taken 256 at a time in index order; within a warp __match_any_sync gives
// each element the number of earlier lanes with its digit, and per-warp
// digit counts in shared memory, prefixed across warps and carried across
// the block's rounds, give the rest.
#include <cstring>

#include "sc_internal.cuh"

namespace sc {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
constexpr int kScanChunk = kScanThreads * kScanItems;

constexpr int kSortThreads = 256;
constexpr int kMaxBins = 512;  // digits of up to 9 bits
constexpr int kSortItems = 8;
constexpr int kSortTile = kSortThreads * kSortItems;  // elements per block

// Exclusive prefix of v over the block (1024 threads); the block's total in
// *total.
__device__ __forceinline__ int64_t block_exclusive_1024(int64_t v, int64_t* s_warp,
                                                        int64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  const int64_t excl = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
  *total = s_warp[31];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(const int32_t* __restrict__ in,
                                                              int64_t len,
                                                              int64_t* __restrict__ partial) {
  __shared__ int64_t s_warp[32];
  const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanItems;
  int64_t v = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < len) v += in[base + i];
  int64_t total;
  block_exclusive_1024(v, s_warp, &total);
  if (threadIdx.x == 0) partial[blockIdx.x] = total;
}

// One block: exclusive scan of the chunk sums in place; the grand total into
// *total (device).
__global__ void __launch_bounds__(kScanThreads) k_scan_partials(int64_t* partial, int64_t nchunks,
                                                                int64_t* total) {
  __shared__ int64_t s_warp[32];
  int64_t carry = 0;
  for (int64_t base = 0; base < nchunks; base += kScanThreads) {
    const int64_t i = base + threadIdx.x;
    const int64_t v = i < nchunks ? partial[i] : 0;
    int64_t t;
    const int64_t e = block_exclusive_1024(v, s_warp, &t);
    if (i < nchunks) partial[i] = carry + e;
    carry += t;
  }
  if (threadIdx.x == 0) *total = carry;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_apply(const int32_t* __restrict__ in,
                                                             int32_t* __restrict__ out,
                                                             int64_t len,
                                                             const int64_t* __restrict__ partial) {
  __shared__ int64_t s_warp[32];
  const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanItems;
  int32_t v[kScanItems];
  int64_t sum = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    v[i] = base + i < len ? in[base + i] : 0;
    sum += v[i];
  }
  int64_t total;
  int64_t run = block_exclusive_1024(sum, s_warp, &total) + partial[blockIdx.x];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    if (base + i < len) out[base + i] = (int32_t)run;
    run += v[i];
  }
}

size_t scan_scratch_bytes(int64_t len) {
  return (size_t)((len + kScanChunk - 1) / kScanChunk + 1) * sizeof(int64_t);
}

cudaError_t scan_exclusive(const int32_t* in, int32_t* out, int64_t len, int64_t* total,
                           void* scratch, cudaStream_t s) {
  const int64_t nchunks = (len + kScanChunk - 1) / kScanChunk;
  int64_t* partial = static_cast<int64_t*>(scratch);
  if (len == 0) return cudaMemsetAsync(total, 0, sizeof(int64_t), s);
  k_scan_reduce<<<(unsigned)nchunks, kScanThreads, 0, s>>>(in, len, partial);
  k_scan_partials<<<1, kScanThreads, 0, s>>>(partial, nchunks, total);
  k_scan_apply<<<(unsigned)nchunks, kScanThreads, 0, s>>>(in, out, len, partial);
  note_launches(3);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// counting-sort pass

template <typename K>
__device__ __forceinline__ int digit_of(K key, int shift, int bins) {
  return (int)((key >> shift) & (K)(bins - 1));
}

template <typename K>
__global__ void __launch_bounds__(kSortThreads) k_digit_counts(const K* __restrict__ keys,
                                                               int64_t n, int shift, int bins,
                                                               int32_t* __restrict__ counts) {
  __shared__ int32_t s_cnt[kMaxBins];
  for (int d = threadIdx.x; d < bins; d += kSortThreads) s_cnt[d] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
#pragma unroll
  for (int j = 0; j < kSortItems; ++j) {
    const int64_t i = base + j * kSortThreads + threadIdx.x;
    if (i < n) atomicAdd(&s_cnt[digit_of(keys[i], shift, bins)], 1);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < bins; d += kSortThreads)
    counts[(int64_t)d * gridDim.x + blockIdx.x] = s_cnt[d];
}

template <typename K>
__global__ void __launch_bounds__(kSortThreads) k_digit_scatter(
    const K* __restrict__ keys_in, const int32_t* __restrict__ vals_in, int64_t n, int shift,
    int bins, const int32_t* __restrict__ offsets, K* __restrict__ keys_out,
    int32_t* __restrict__ vals_out) {
  __shared__ int32_t s_wcnt[kSortThreads / 32][kMaxBins];
  __shared__ int32_t s_base[kMaxBins];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int d = threadIdx.x; d < kMaxBins; d += kSortThreads) {
    s_base[d] = d < bins ? offsets[(int64_t)d * gridDim.x + blockIdx.x] : 0;
#pragma unroll
    for (int w = 0; w < kSortThreads / 32; ++w) s_wcnt[w][d] = 0;
  }
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
  const uint32_t lt = (1u << lane) - 1u;
  for (int j = 0; j < kSortItems; ++j) {
    const int64_t i = base + j * kSortThreads + threadIdx.x;
    const bool valid = i < n;
    K key = 0;
    int32_t val = 0;
    int d = bins;  // out-of-range elements form their own (unwritten) group
    if (valid) {
      key = keys_in[i];
      val = vals_in ? vals_in[i] : (int32_t)i;
      d = digit_of(key, shift, bins);
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const int wrank = __popc(peers & lt);
    if (valid && wrank == 0) s_wcnt[warp][d] = __popc(peers);
    __syncthreads();
    // Per digit: the warps' counts become their first positions.
    for (int dd = threadIdx.x; dd < bins; dd += kSortThreads) {
      int32_t run = s_base[dd];
#pragma unroll
      for (int w = 0; w < kSortThreads / 32; ++w) {
        const int32_t c = s_wcnt[w][dd];
        s_wcnt[w][dd] = run;
        run += c;
      }
      s_base[dd] = run;
    }
    __syncthreads();
    if (valid) {
      const int32_t pos = s_wcnt[warp][d] + wrank;
      keys_out[pos] = key;
      vals_out[pos] = val;
    }
    __syncthreads();
    for (int dd = threadIdx.x; dd < bins; dd += kSortThreads) {
#pragma unroll
      for (int w = 0; w < kSortThreads / 32; ++w) s_wcnt[w][dd] = 0;
    }
    __syncthreads();
  }
}

size_t sort_scratch_bytes(int64_t n, int bins) {
  const int64_t nblocks = (n + kSortTile - 1) / kSortTile;
  const int64_t len = nblocks * bins;
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  return up((size_t)len * sizeof(int32_t)) + up(scan_scratch_bytes(len)) + up(sizeof(int64_t));
}

template <typename K>
cudaError_t sort_pass(const K* keys_in, const int32_t* vals_in, K* keys_out, int32_t* vals_out,
                      int64_t n, int shift, int bits, void* scratch, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int bins = 1 << bits;
  const int64_t nblocks = (n + kSortTile - 1) / kSortTile;
  const int64_t len = nblocks * bins;
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  uint8_t* p = static_cast<uint8_t*>(scratch);
  int32_t* counts = reinterpret_cast<int32_t*>(p);
  void* scan_scratch = p + up((size_t)len * sizeof(int32_t));
  int64_t* total = reinterpret_cast<int64_t*>(p + up((size_t)len * sizeof(int32_t)) +
                                              up(scan_scratch_bytes(len)));
  k_digit_counts<K><<<(unsigned)nblocks, kSortThreads, 0, s>>>(keys_in, n, shift, bins, counts);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = scan_exclusive(counts, counts, len, total, scan_scratch, s);
  if (e != cudaSuccess) return e;
  k_digit_scatter<K><<<(unsigned)nblocks, kSortThreads, 0, s>>>(keys_in, vals_in, n, shift, bins,
                                                                counts, keys_out, vals_out);
  note_launches(1);
  return cudaGetLastError();
}

template cudaError_t sort_pass<uint32_t>(const uint32_t*, const int32_t*, uint32_t*, int32_t*,
                                         int64_t, int, int, void*, cudaStream_t);
template cudaError_t sort_pass<unsigned long long>(const unsigned long long*, const int32_t*,
                                                   unsigned long long*, int32_t*, int64_t, int,
                                                   int, void*, cudaStream_t);

}  // namespace sc
