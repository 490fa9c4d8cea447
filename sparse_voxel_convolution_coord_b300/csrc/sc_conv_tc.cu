// sc_conv_tc.cu -- bf16 submanifold convolution on the sm_103a tensor cores.
//
// What it computes ("Porting TRELLIS.2 From Python to Rust and Metal",
// section V: a gather-GEMM over the neighbour table with half-precision
// inputs, single-precision accumulation and the bias fused into the same
// pass; "Running TRELLIS.2 on a Mac (1/3)", Sparse 3D convolution paragraph):
//
//   out[o][:] = bias + sum_{k : nbr[o][k] >= 0} feats[nbr[o][k]][:] @ W[k]
//
// How: an output-stationary implicit GEMM.  A CTA owns a tile of 128 output
// rows; the GEMM's K dimension is (offset, input channel).  For each offset
// present in the tile (its 27-bit OR mask), the 128 neighbour rows are
// gathered straight from the feature matrix by TMA (tile::gather4, four rows
// per instruction, absent neighbours given an out-of-range row so the copy
// fills zeros) and W[k] arrives by tiled TMA; a single thread issues
// tcgen05.mma (M = 128, N = cout padded to 64, K = 16, bf16 x bf16 -> fp32)
// into a TMEM accumulator.  Each output row belongs to exactly one tile, so
// the epilogue (TMEM -> registers, + bias, fp32 store) needs no atomics.
//
// CTA = 6 warps, persistent over tiles:
//   warps 0-3  epilogue (warp q reads TMEM lanes 32q..32q+31 = rows of the tile)
//   warp 4     producer: stages the tile's neighbour rows in shared memory,
//              then per pipeline stage one lane arms the stage barrier and
//              issues W's boxes, and all 32 lanes issue one gather4 each
//   warp 5     TMEM allocation; lane 0 issues the MMAs and the commits
// Two TMEM accumulators let the epilogue of one tile overlap the next tile's
// main loop.  Every wait is bounded (~2 s): a CTA that gives up records
// SC_ERR_DEVICE_TIMEOUT in the map's status word and leaves cleanly.
//
// Shared-memory operand layouts (both built by TMA swizzling):
//   A (gathered rows, K-major): per stage 64/CS segments, each 128 rows x CS
//     bf16, rows of 2*CS bytes with the matching 128/64/32-byte swizzle;
//   B (W[k] rows, MN-major): per stage [cout/64 blocks][64 K rows][128 B],
//     128-byte swizzle; LBO = 8 KB between 64-column blocks, SBO = 1 KB
//     between 8-row groups.
#include <algorithm>
#include <cstring>
#include <cudaTypedefs.h>

#include "sc_internal.cuh"

namespace sc {

constexpr int kTcThreads = 192;
constexpr int kSmemBudget = 212 * 1024;

template <int NPAD, int CS>
struct TcCfg {
  static constexpr int kSegs = 64 / CS;                 // offset segments per stage
  static constexpr int kRowBytes = CS * 2;               // one gathered row segment
  static constexpr int kASeg = kTileRows * kRowBytes;    // bytes per A segment
  static constexpr int kABytes = kTileRows * 128;        // 16 KB per stage
  static constexpr int kBBytes = 64 * NPAD * 2;          // 64 K rows x NPAD bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kFixed = kTaps * kTileRows * 4 + NPAD * 4 + 1024;  // nbr, bias, bars
  static constexpr int kStages0 = (kSmemBudget - kFixed - 1024) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kFixed;
  static constexpr uint32_t kTmemCols = (2 * NPAD <= 128) ? 128 : (2 * NPAD <= 256 ? 256 : 512);
  static constexpr uint32_t kLayoutA = CS == 64 ? 2u : (CS == 32 ? 4u : 6u);
  static constexpr uint32_t kSboA = 8 * kRowBytes;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kTileRows, NPAD);
  static_assert(kStages >= 2, "pipeline needs two stages");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct TcArgs {
  const int32_t* nbr;
  const uint32_t* tile_mask;
  const float* bias;
  float* out;
  uint32_t* status;
  int64_t n;
  int64_t ntiles;
  int cin;
  int cout;
};

// Stages of a tile: (present offsets) x (cin / 64) when CS == 64, else the
// present offsets taken 64/CS at a time.
template <int CS>
__device__ __forceinline__ int tile_stages(uint32_t mask, int cin) {
  const int np = __popc(mask);
  if constexpr (CS == 64) {
    return np * (cin >> 6);
  } else {
    constexpr int g = 64 / CS;
    return (np + g - 1) / g;
  }
}

// Position of the j-th (0-based) set bit of mask, or 27 when there is none.
__device__ __forceinline__ int nth_bit(uint32_t mask, int j) {
  for (int i = 0; i < j && mask; ++i) mask &= mask - 1;
  return mask ? __ffs(mask) - 1 : kTaps;
}

template <int NPAD, int CS>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_conv_tc(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              const TcArgs p) {
  using C = TcCfg<NPAD, CS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::kStages * C::kABytes;
  int32_t* s_nbr = reinterpret_cast<int32_t*>(sB + C::kStages * C::kBBytes);  // [27][128]
  float* s_bias = reinterpret_cast<float*>(s_nbr + kTaps * kTileRows);
  uint64_t* full = reinterpret_cast<uint64_t*>(s_bias + NPAD);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_empty + 2);
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kTileRows);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(s_tmem, C::kTmemCols);
  for (int i = threadIdx.x; i < NPAD; i += kTcThreads)
    s_bias[i] = (p.bias != nullptr && i < p.cout) ? p.bias[i] : 0.f;
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  volatile int* abort_flag = &s_abort;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int32_t oob = (int32_t)p.n;  // a row index past the end: TMA fills zeros
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
      const int64_t row0 = tile * kTileRows;
      const uint32_t mask = p.tile_mask[tile];
      const int nst = tile_stages<CS>(mask, p.cin);
      __syncwarp();
      for (int e = lane; e < kTileRows * kTaps; e += 32) {
        const int r = e / kTaps, k = e - r * kTaps;
        const int64_t row = row0 + r;
        const int32_t v = row < p.n ? __ldg(p.nbr + row0 * kTaps + e) : -1;
        s_nbr[k * kTileRows + r] = v < 0 ? oob : v;
      }
      __syncwarp();
      for (int s = 0; s < nst; ++s) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
        __syncwarp();
        uint8_t* a_st = sA + stage * C::kABytes;
        uint8_t* b_st = sB + stage * C::kBBytes;
#pragma unroll
        for (int j = 0; j < C::kSegs; ++j) {
          int k, c0;
          if constexpr (CS == 64) {
            const int chunks = p.cin >> 6;
            k = nth_bit(mask, s / chunks);
            c0 = (s % chunks) * 64;
          } else {
            k = nth_bit(mask, s * C::kSegs + j);
            c0 = 0;
          }
          int4 rows;
          if (k < kTaps)
            rows = *reinterpret_cast<const int4*>(&s_nbr[k * kTileRows + 4 * lane]);
          else
            rows = make_int4(oob, oob, oob, oob);
          tma_gather4(a_st + j * C::kASeg + lane * 4 * C::kRowBytes, &tm_a, &full[stage], c0,
                      rows);
          if (lane == 0) {
            // k == 27 addresses rows past W's end: the box is zero-filled.
#pragma unroll
            for (int nb = 0; nb < NPAD / 64; ++nb)
              tma_load_2d(b_st + nb * (64 * 128) + j * CS * 128, &tm_b, &full[stage], nb * 64,
                          k * p.cin + c0);
          }
        }
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      s_abort = 1;
      atomicOr(p.status, kStatTimeout);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
        const int nst = tile_stages<CS>(p.tile_mask[tile], p.cin);
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
          const uint32_t a_base = smem_u32(sA + stage * C::kABytes);
          const uint32_t b_base = smem_u32(sB + stage * C::kBBytes);
#pragma unroll
          for (int j = 0; j < C::kSegs; ++j) {
#pragma unroll
            for (int kk = 0; kk < CS / 16; ++kk) {
              const uint64_t ad =
                  smem_desc(a_base + j * C::kASeg + kk * 32, 16, C::kSboA, C::kLayoutA);
              const uint64_t bd = smem_desc(b_base + (j * CS + kk * 16) * 128, 64 * 128, 1024, 2u);
              tc_mma_bf16(d_tmem, ad, bd, C::kIdesc, (s | j | kk) != 0 ? 1u : 0u);
            }
          }
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
        s_abort = 1;
        atomicOr(p.status, kStatTimeout);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    const int nchunks = (p.cout + 31) >> 5;
    for (int64_t tile = blockIdx.x; tile < p.ntiles && ok; tile += gridDim.x) {
      if (!mbar_wait_bounded(&acc_full[acc], acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t row = tile * kTileRows + warp * 32 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + acc * NPAD;
      float* orow = p.out + row * p.cout;
      for (int ch = 0; ch < nchunks; ++ch) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + ch * 32, v);
        tmem_ld_wait();
        if (row < p.n) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int c = ch * 32 + 4 * q;
            if (c < p.cout) {
              float4 o;
              o.x = __uint_as_float(v[4 * q + 0]) + s_bias[c + 0];
              o.y = __uint_as_float(v[4 * q + 1]) + s_bias[c + 1];
              o.z = __uint_as_float(v[4 * q + 2]) + s_bias[c + 2];
              o.w = __uint_as_float(v[4 * q + 3]) + s_bias[c + 3];
              __stcs(reinterpret_cast<float4*>(orow + c), o);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && lane == 0) {
      s_abort = 1;
      atomicOr(p.status, kStatTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz) {
  auto fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  return sms;
}

template <int NPAD, int CS>
cudaError_t launch_typed(const sc_map* m, const void* feats, const void* w, const float* bias,
                         float* out, int cin, int cout, cudaStream_t s) {
  using C = TcCfg<NPAD, CS>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_conv_tc<NPAD, CS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  alignas(64) CUtensorMap tm_a, tm_b;
  const CUtensorMapSwizzle swz_a = CS == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : CS == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  if (!encode_2d(&tm_a, feats, (uint64_t)cin, (uint64_t)m->n, (uint64_t)cin * 2, CS, 1, swz_a))
    return cudaErrorInvalidValue;
  if (!encode_2d(&tm_b, w, (uint64_t)cout, (uint64_t)kTaps * cin, (uint64_t)cout * 2, 64, CS,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  TcArgs a;
  a.nbr = m->nbr;
  a.tile_mask = m->tile_mask;
  a.bias = bias;
  a.out = out;
  a.status = m->d_status;
  a.n = m->n;
  a.ntiles = m->ntiles;
  a.cin = cin;
  a.cout = cout;
  const int grid = (int)std::min<int64_t>(m->ntiles, num_sms());
  k_conv_tc<NPAD, CS><<<grid, kTcThreads, C::kSmemBytes, s>>>(tm_a, tm_b, a);
  return cudaGetLastError();
}

template <int NPAD>
cudaError_t launch_npad(const sc_map* m, const void* feats, const void* w, const float* bias,
                        float* out, int cin, int cout, cudaStream_t s) {
  if (cin == 16) return launch_typed<NPAD, 16>(m, feats, w, bias, out, cin, cout, s);
  if (cin == 32) return launch_typed<NPAD, 32>(m, feats, w, bias, out, cin, cout, s);
  return launch_typed<NPAD, 64>(m, feats, w, bias, out, cin, cout, s);
}

}  // namespace

bool conv_tc_supported(int cin, int cout) {
  const bool cin_ok = cin == 16 || cin == 32 || (cin % 64 == 0 && cin >= 64 && cin <= 1024);
  const bool cout_ok = cout >= 16 && cout <= 256 && cout % 16 == 0;
  return cin_ok && cout_ok;
}

cudaError_t launch_conv_tc_bf16(const sc_map* m, const void* feats, const void* w,
                                const float* bias, float* out, int cin, int cout,
                                cudaStream_t s) {
  if (!conv_tc_supported(cin, cout)) return cudaErrorNotSupported;
  const int npad = (cout + 63) / 64 * 64;
  switch (npad) {
    case 64: return launch_npad<64>(m, feats, w, bias, out, cin, cout, s);
    case 128: return launch_npad<128>(m, feats, w, bias, out, cin, cout, s);
    case 192: return launch_npad<192>(m, feats, w, bias, out, cin, cout, s);
    default: return launch_npad<256>(m, feats, w, bias, out, cin, cout, s);
  }
}

}  // namespace sc
