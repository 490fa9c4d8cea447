// sc_conv_simt.cu -- fp32 submanifold convolution on CUDA cores.
//
// out[o][c] = bias[c] + sum_k sum_ci feats[nbr[o][k]][ci] * W[k][ci][c], every
// product and sum in fp32 FFMA ("Porting TRELLIS.2 From Python to Rust and
// Metal", section V: gather-GEMM over the neighbour table, single-precision
// accumulation, bias in the same pass).  Used for fp32 inputs, where a
// tensor-core tf32 product would round the inputs to 10 mantissa bits.
//
// A block owns 8 output rows (one warp each; lane l holds columns l, l+32,
// ...).  Per 32-channel slice of the input: every warp gathers its row's 27
// neighbour slices at once (independent coalesced loads) into shared memory;
// then, for each offset present in any of the block's rows, the W[k] slice
// (32 rows x cout) is staged in shared memory by cp.async, double-buffered one
// offset ahead, and shared by the 8 warps.  Each output row is written once,
// no atomics, through the fused epilogue (activation, residual, fp32, bf16 or
// fp16 output).
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sc_internal.cuh"

namespace sc {

constexpr int kSimtWarps = 8;  // output rows per block

__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_16_ca(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

template <int J>  // columns per lane = J, cout <= 32 * J
__global__ void __launch_bounds__(kSimtWarps * 32) k_conv_simt_f32(
    const int32_t* __restrict__ nbr, const int32_t* __restrict__ row_of, int64_t n, int taps,
    const float* __restrict__ feats, const float* __restrict__ w, const Epilogue ep, int cin,
    int cout) {
  __shared__ float s_a[kSimtWarps][kTaps][32];
  __shared__ uint32_t s_mask[kSimtWarps];
  extern __shared__ __align__(16) float s_w[];  // [2][32][32 * J]
  constexpr int kWStride = 32 * J;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t o = (int64_t)blockIdx.x * kSimtWarps + warp;  // tile position
  // output row of the position (-1: none)
  const int32_t orow = o < n ? (row_of ? __ldg(row_of + o) : (int32_t)o) : -1;
  const bool valid = orow >= 0;
  // tile-major table: position o of tile o / 128, offset k at [tile][k][o % 128]
  const int32_t nb =
      (valid && lane < taps)
          ? __ldg(nbr + (o / kTileRows) * (kTileRows * taps) + lane * kTileRows + (o % kTileRows))
          : -1;
  const uint32_t present = __ballot_sync(0xffffffffu, nb >= 0);
  if (lane == 0) s_mask[warp] = present;
  __syncthreads();
  uint32_t bmask = 0;
#pragma unroll
  for (int q = 0; q < kSimtWarps; ++q) bmask |= s_mask[q];
  const bool vec = (cout & 3) == 0;  // 16-byte copies of W rows

  float acc[J];
#pragma unroll
  for (int j = 0; j < J; ++j) acc[j] = 0.f;

  // Stage W[k][ci0 .. ci0 + width)[0 .. cout) into buffer b.
  auto stage_w = [&](int k, int ci0, int width, int b) {
    float* dst = s_w + b * 32 * kWStride;
    const float* src = w + ((int64_t)k * cin + ci0) * cout;
    if (vec) {
      const int per_row = cout >> 2;
      for (int e = threadIdx.x; e < width * per_row; e += kSimtWarps * 32) {
        const int r = e / per_row, c4 = e - r * per_row;
        cp_async_16_ca(dst + r * kWStride + 4 * c4, src + (int64_t)r * cout + 4 * c4);
      }
    } else {
      for (int e = threadIdx.x; e < width * cout; e += kSimtWarps * 32) {
        const int r = e / cout, c = e - r * cout;
        cp_async_4(dst + r * kWStride + c, src + (int64_t)r * cout + c);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  for (int ci0 = 0; ci0 < cin; ci0 += 32) {
    const int width = min(32, cin - ci0);
    uint32_t rem = bmask;
    if (rem) stage_w(__ffs(rem) - 1, ci0, width, 0);
#pragma unroll
    for (int k = 0; k < kTaps; ++k) {
      if (k >= taps) break;
      const int32_t i = __shfl_sync(0xffffffffu, nb, k);
      s_a[warp][k][lane] =
          (i >= 0 && lane < width) ? __ldg(feats + (int64_t)i * cin + ci0 + lane) : 0.f;
    }
    int buf = 0;
    while (rem) {
      const int k = __ffs(rem) - 1;
      rem &= rem - 1u;
      if (rem) {
        stage_w(__ffs(rem) - 1, ci0, width, buf ^ 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      __syncthreads();  // W slice k and every warp's gathered rows are in place
      const float* ws = s_w + buf * 32 * kWStride + lane;
#pragma unroll 8
      for (int cc = 0; cc < width; ++cc) {
        const float a = s_a[warp][k][cc];
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (lane + 32 * j < cout) acc[j] = fmaf(a, ws[cc * kWStride + 32 * j], acc[j]);
      }
      __syncthreads();  // buffer buf is free for the offset after next
      buf ^= 1;
    }
    __syncthreads();  // s_a is rewritten for the next slice
  }
  if (valid) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = lane + 32 * j;
      if (c >= cout) continue;
      const int64_t e = (int64_t)orow * cout + c;
      float v = apply_act(acc[j] + (ep.bias ? __ldg(ep.bias + c) : 0.f), ep.act);
      if (ep.out_half == kOutBf16) {
        if (ep.residual)
          v += __bfloat162float(static_cast<const __nv_bfloat16*>(ep.residual)[e]);
        static_cast<__nv_bfloat16*>(ep.out)[e] = __float2bfloat16_rn(v);
      } else if (ep.out_half == kOutF16) {
        if (ep.residual) v += __half2float(static_cast<const __half*>(ep.residual)[e]);
        static_cast<__half*>(ep.out)[e] = __float2half_rn(v);
      } else {
        if (ep.residual) v += __ldg(static_cast<const float*>(ep.residual) + e);
        static_cast<float*>(ep.out)[e] = v;
      }
    }
  }
}

template <int J>
cudaError_t launch_simt(const ConvMap& m, const float* feats, const float* w, const Epilogue& ep,
                        int cin, int cout, cudaStream_t s) {
  const size_t smem = 2ull * 32 * 32 * J * sizeof(float);
  // Opt-in above 48 KB of dynamic shared memory, once per device (function
  // attributes are per device; setting one twice is harmless).
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_set[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(k_conv_simt_f32<J>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const unsigned blocks = (unsigned)((m.n + kSimtWarps - 1) / kSimtWarps);
  k_conv_simt_f32<J><<<blocks, kSimtWarps * 32, smem, s>>>(m.nbr, m.row_of, m.n, m.taps, feats, w,
                                                           ep, cin, cout);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_conv_simt_f32(const ConvMap& m, const float* feats, const float* w,
                                 const Epilogue& ep, int cin, int cout, cudaStream_t s) {
  const int J = (cout + 31) / 32;
  if (J <= 1) return launch_simt<1>(m, feats, w, ep, cin, cout, s);
  if (J <= 2) return launch_simt<2>(m, feats, w, ep, cin, cout, s);
  if (J <= 4) return launch_simt<4>(m, feats, w, ep, cin, cout, s);
  return launch_simt<8>(m, feats, w, ep, cin, cout, s);
}

}  // namespace sc
