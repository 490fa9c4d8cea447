// sc_conv_simt.cu -- fp32 submanifold convolution on CUDA cores.
//
// out[o][c] = bias[c] + sum_k sum_ci feats[nbr[o][k]][ci] * W[k][ci][c], every
// product and sum in fp32 FFMA ("Porting TRELLIS.2 From Python to Rust and
// Metal", section V: gather-GEMM over the neighbour table, single-precision
// accumulation, bias in the same pass).  Used for fp32 inputs, where a
// tensor-core tf32 product would round the inputs to 10 mantissa bits.
//
// One CTA owns 32 output rows and all cout columns; for each offset present
// in the rows' 128-row tile, 32-wide chunks of the gathered rows and of W[k]
// are staged in shared memory.  Each output row is written once, no atomics.
#include "sc_internal.cuh"

namespace sc {

constexpr int kSimtRows = 32;
constexpr int kSimtChunk = 32;
constexpr int kSimtThreads = 256;
constexpr int kSimtColsPerThread = 32;  // cout <= 8 * 32 = 256

__global__ void __launch_bounds__(kSimtThreads) k_conv_simt_f32(
    const int32_t* __restrict__ nbr, const uint32_t* __restrict__ tile_mask, int64_t n,
    const float* __restrict__ feats, const float* __restrict__ w, const float* __restrict__ bias,
    float* __restrict__ out, int cin, int cout) {
  __shared__ float sA[kSimtRows][kSimtChunk + 1];
  extern __shared__ float sW[];  // [kSimtChunk][cout]
  const int64_t row0 = (int64_t)blockIdx.x * kSimtRows;
  const int r = threadIdx.x >> 3;   // output row within the block
  const int cg = threadIdx.x & 7;   // column group: columns cg, cg+8, ...
  float acc[kSimtColsPerThread];
#pragma unroll
  for (int j = 0; j < kSimtColsPerThread; ++j) acc[j] = 0.f;
  const uint32_t mask = tile_mask[row0 / kTileRows];

  for (int k = 0; k < kTaps; ++k) {
    if (!((mask >> k) & 1u)) continue;
    for (int c0 = 0; c0 < cin; c0 += kSimtChunk) {
      for (int e = threadIdx.x; e < kSimtRows * kSimtChunk; e += kSimtThreads) {
        const int rr = e / kSimtChunk, cc = e % kSimtChunk;
        const int64_t row = row0 + rr;
        const int32_t i = row < n ? nbr[row * kTaps + k] : -1;
        sA[rr][cc] = (i >= 0 && c0 + cc < cin) ? feats[(int64_t)i * cin + c0 + cc] : 0.f;
      }
      for (int e = threadIdx.x; e < kSimtChunk * cout; e += kSimtThreads) {
        const int cc = e / cout, c = e % cout;
        sW[e] = (c0 + cc < cin) ? w[((int64_t)k * cin + c0 + cc) * cout + c] : 0.f;
      }
      __syncthreads();
#pragma unroll 4
      for (int cc = 0; cc < kSimtChunk; ++cc) {
        const float a = sA[r][cc];
#pragma unroll
        for (int j = 0; j < kSimtColsPerThread; ++j) {
          const int c = cg + 8 * j;
          if (c < cout) acc[j] = fmaf(a, sW[cc * cout + c], acc[j]);
        }
      }
      __syncthreads();
    }
  }
  const int64_t row = row0 + r;
  if (row < n) {
#pragma unroll
    for (int j = 0; j < kSimtColsPerThread; ++j) {
      const int c = cg + 8 * j;
      if (c < cout) out[row * cout + c] = acc[j] + (bias ? bias[c] : 0.f);
    }
  }
}

cudaError_t launch_conv_simt_f32(const sc_map* m, const float* feats, const float* w,
                                 const float* bias, float* out, int cin, int cout,
                                 cudaStream_t s) {
  const int64_t blocks = (m->n + kSimtRows - 1) / kSimtRows;
  const size_t smem = (size_t)kSimtChunk * cout * sizeof(float);
  k_conv_simt_f32<<<(unsigned)blocks, kSimtThreads, smem, s>>>(m->nbr, m->tile_mask, m->n, feats,
                                                               w, bias, out, cin, cout);
  return cudaGetLastError();
}

}  // namespace sc
