// sc_conv_simt.cu -- fp32 submanifold convolution on CUDA cores.
//
// out[o][c] = bias[c] + sum_k sum_ci feats[nbr[o][k]][ci] * W[k][ci][c], every
// product and sum in fp32 FFMA ("Porting TRELLIS.2 From Python to Rust and
// Metal", section V: gather-GEMM over the neighbour table, single-precision
// accumulation, bias in the same pass).  Used for fp32 inputs, where a
// tensor-core tf32 product would round the inputs to 10 mantissa bits.
//
// One warp owns one output row and all cout columns (lane l holds columns
// l, l+32, ...).  Per 32-channel slice of the input, the warp first issues
// the 27 gathers of its neighbour rows together (independent loads, one
// coalesced 128-byte row slice each) into shared memory, then accumulates
// over the present offsets with W read through L1 (every warp of the grid
// reads the same W).  Each output row is written once, no atomics.
#include "sc_internal.cuh"

namespace sc {

constexpr int kSimtWarps = 8;  // output rows per block

template <int J>  // columns per lane = J, cout <= 32 * J
__global__ void __launch_bounds__(kSimtWarps * 32) k_conv_simt_f32(
    const int32_t* __restrict__ nbr, int64_t n, const float* __restrict__ feats,
    const float* __restrict__ w, const float* __restrict__ bias, float* __restrict__ out, int cin,
    int cout) {
  __shared__ float s_a[kSimtWarps][kTaps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t o = (int64_t)blockIdx.x * kSimtWarps + warp;
  if (o >= n) return;  // no block-wide synchronisation below
  // tile-major table: row o of tile o / 128, offset k at [tile][k][o % 128]
  const int32_t nb =
      lane < kTaps ? __ldg(nbr + (o / kTileRows) * (kTileRows * kTaps) + lane * kTileRows +
                           (o % kTileRows))
                   : -1;
  const uint32_t present = __ballot_sync(0xffffffffu, nb >= 0);
  float acc[J];
#pragma unroll
  for (int j = 0; j < J; ++j) acc[j] = 0.f;

  for (int ci0 = 0; ci0 < cin; ci0 += 32) {
    const int width = min(32, cin - ci0);
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
      const int32_t i = __shfl_sync(0xffffffffu, nb, k);
      s_a[warp][k][lane] =
          (i >= 0 && lane < width) ? __ldg(feats + (int64_t)i * cin + ci0 + lane) : 0.f;
    }
    __syncwarp();
    for (uint32_t rem = present; rem; rem &= rem - 1u) {
      const int k = __ffs(rem) - 1;
      const float* wk = w + ((int64_t)k * cin + ci0) * cout + lane;
#pragma unroll 4
      for (int cc = 0; cc < width; ++cc) {
        const float a = s_a[warp][k][cc];
        const float* wr = wk + (int64_t)cc * cout;
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (lane + 32 * j < cout) acc[j] = fmaf(a, __ldg(wr + 32 * j), acc[j]);
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int c = lane + 32 * j;
    if (c < cout) out[o * cout + c] = acc[j] + (bias ? __ldg(bias + c) : 0.f);
  }
}

cudaError_t launch_conv_simt_f32(const sc_map* m, const float* feats, const float* w,
                                 const float* bias, float* out, int cin, int cout,
                                 cudaStream_t s) {
  const unsigned blocks = (unsigned)((m->n + kSimtWarps - 1) / kSimtWarps);
  const int J = (cout + 31) / 32;
  const dim3 block(kSimtWarps * 32);
  if (J <= 1)
    k_conv_simt_f32<1><<<blocks, block, 0, s>>>(m->nbr, m->n, feats, w, bias, out, cin, cout);
  else if (J <= 2)
    k_conv_simt_f32<2><<<blocks, block, 0, s>>>(m->nbr, m->n, feats, w, bias, out, cin, cout);
  else if (J <= 4)
    k_conv_simt_f32<4><<<blocks, block, 0, s>>>(m->nbr, m->n, feats, w, bias, out, cin, cout);
  else
    k_conv_simt_f32<8><<<blocks, block, 0, s>>>(m->nbr, m->n, feats, w, bias, out, cin, cout);
  return cudaGetLastError();
}

}  // namespace sc
