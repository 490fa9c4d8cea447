/*
 * sc.h -- C ABI of the B300 (sm_103a) 3x3x3 submanifold sparse convolution.
 *
 * The operation (from "Running TRELLIS.2 on a Mac (1/3)", section "Swapping
 * out the CUDA libraries one at a time", paragraph "Sparse 3D convolution",
 * and "Porting TRELLIS.2 From Python to Rust and Metal", section V "The
 * Kernel That Decided It"):
 *
 *   active voxels p_i = (b_i, x_i, y_i, z_i), i = 0..N-1, features F[N][Cin];
 *   27 offsets k = 9*(dx+1) + 3*(dy+1) + (dz+1), dx,dy,dz in {-1,0,1};
 *   nbr[o][k] = the row i with p_i = (b_o, x_o+dx, y_o+dy, z_o+dz), else -1;
 *   out[o][c] = bias[c] + sum_k sum_ci [nbr[o][k] >= 0] F[nbr[o][k]][ci] * W[k][ci][c].
 *
 * Output sites are the input sites (submanifold), in input row order.  The
 * weight layout W[27][Cin][Cout] is the (Kvol, Ci, Co) view of the on-disk
 * (Co, Kd, Kh, Kw, Ci) sparse-conv weights ("FABLE_STARTUP_PACKET.md",
 * section 5, weight-convention table), i.e. k is the row-major flattening of
 * (Kd, Kh, Kw) with Kd along x.  A neighbour outside [0,res)^3 or in another
 * batch element is absent (zero padding).
 *
 * Conventions for every call below:
 *  - Pointers are DEVICE pointers unless the argument says "host".
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Calls return a status (or NULL / -1 for handle and size getters) and set
 *    a thread-local error readable with sc_last_error()/sc_last_error_msg().
 *    Invalid arguments are rejected on the host before anything is launched.
 *  - There is no CPU fallback: every step runs in this library's CUDA
 *    kernels on the device that owns the pointers (the current device).
 *  - Device loops are bounded; a kernel that gives up sets a device status
 *    word that sc_device_status() reports.  No call traps or asserts on the
 *    device.
 */
#ifndef SC_H_
#define SC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SC_API __attribute__((visibility("default")))
#else
#define SC_API
#endif

typedef struct sc_map* sc_handle; /* opaque neighbour-map handle owned by the library */

typedef enum {
  SC_OK = 0,
  SC_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, bad alignment, ... */
  SC_ERR_COORD_RANGE = 2,  /* a coordinate outside [0,res) or a negative batch  */
  SC_ERR_DUPLICATE = 3,    /* two rows with the same (b,x,y,z)                  */
  SC_ERR_TABLE_FULL = 4,   /* hash probe bound exceeded (cannot happen: the
                              table's load factor is at most 1/2)               */
  SC_ERR_UNSUPPORTED = 5,  /* shape/dtype outside the kernels' envelope         */
  SC_ERR_ALLOC = 6,        /* device allocation failed                          */
  SC_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed                 */
  SC_ERR_BAD_HANDLE = 8,   /* handle not live (double free, use after free)     */
  SC_ERR_DEVICE_TIMEOUT = 9 /* a bounded device wait ran out (see sc_device_status) */
} sc_status;

typedef enum { SC_F32 = 0, SC_BF16 = 1, SC_F16 = 2 } sc_dtype;

/* Activation of the fused epilogue (sc_forward_ex). */
typedef enum {
  SC_ACT_NONE = 0,
  SC_ACT_RELU = 1, /* max(v, 0)                  */
  SC_ACT_SILU = 2  /* v * sigmoid(v) = v / (1 + e^-v) */
} sc_activation;

/*
 * Build the coordinate hash table and the neighbour map of N active voxels
 * ("Porting TRELLIS.2 ...", section V: the neighbour table is built once per
 * resolution level and reused by every convolution at that level; the
 * trellis2mlx README feature list reports the cache-hit win of doing so).
 *
 *   coords  device int32 [n][4] row-major (batch, x, y, z); 16-byte aligned.
 *           0 <= x,y,z < res, 0 <= batch.  Read only during the call; it may
 *           be freed afterwards.
 *   n       number of active voxels, 0 <= n < 2^31.  n == 0 gives an empty
 *           map on which sc_forward is a no-op.
 *   res     grid side, 1 <= res <= 2^20.
 *   stream  stream on which the build runs.
 *
 * Returns a handle, or NULL with sc_last_error() set to SC_ERR_COORD_RANGE
 * (a coordinate outside [0,res) or a negative batch), SC_ERR_DUPLICATE (two
 * equal rows; a range error is reported in preference), SC_ERR_UNSUPPORTED
 * (the packed hash key does not fit: keys use 64 - bitlen(n) bits, so
 * (max batch + 1) * res^3 must be <= 2^(64 - bitlen(n)); e.g. res = 1024
 * with n < 2^24 allows 512 batch elements), SC_ERR_INVALID_ARG,
 * SC_ERR_ALLOC or SC_ERR_CUDA.
 * Keys are 32-bit whenever batch * res^3 stays below 2^32 - 1 (at res = 64,
 * batch indices below 16,383); a batch index beyond that makes the build
 * run a second time with 64-bit keys.
 * The call synchronises `stream` once (twice in that retry), to read the
 * device status word and the pair count; when it returns, every buffer of
 * the map is ready for use on any stream.  The handle owns its device memory (hash table,
 * neighbour table nbr[n][27], per-tile offset masks) until sc_free_map.
 */
SC_API sc_handle sc_build_map(const int32_t* coords, int64_t n, int32_t res, void* stream);

/*
 * Run the convolution over a built map: for each output row o (input order)
 *   out[o][:] = bias[:] + sum_k feats[nbr[o][k]][:] @ W[k]   (k with nbr >= 0)
 * ("Porting TRELLIS.2 ...", section V: gather-GEMM over the neighbour table,
 * half-precision inputs, single-precision accumulation, bias fused into the
 * same pass).  On the SC_BF16 path each 128-row tile has one owner, except
 * the tiles of a last, partial round over the SMs: their K range may be
 * split over several CTAs that add into the (zeroed) rows with float atomics,
 * so those rows' sums are taken in an order that can vary from run to run
 * (differences at fp32 rounding level).  sc_set_deterministic(1) limits the
 * split to two parts, whose sum is order-independent, making repeated calls
 * bit-identical.
 *
 *   feats   device [n][cin], dtype `dtype`, row-major, 16-byte aligned.
 *   weight  device [27][cin][cout], dtype `dtype`, row-major, 16-byte aligned.
 *   bias    device fp32 [cout], or NULL for zero bias.
 *   out     device fp32 [n][cout], row-major, 16-byte aligned; fully written.
 *   dtype   SC_BF16 / SC_F16: tensor-core path (tcgen05, bf16 x bf16 or
 *           fp16 x fp16 -> fp32 in TMEM); cin in {16, 32} or a multiple of
 *           64 up to 1024; cout a multiple of 16 up to 256.
 *           SC_F32: fp32 FFMA path (no reduced-precision products); any
 *           cin >= 1 and 1 <= cout <= 256.
 * Asynchronous on `stream`; never synchronises.  Returns SC_ERR_UNSUPPORTED
 * for shapes outside the envelope above, SC_ERR_BAD_HANDLE for a dead handle.
 */
SC_API sc_status sc_forward(sc_handle h, const void* feats, const void* weight, const float* bias,
                     float* out, int32_t cin, int32_t cout, sc_dtype dtype, void* stream);

/*
 * sc_forward with the whole epilogue fused into the same pass ("Porting
 * TRELLIS.2 ...", section V: bias, rounding, activation and the residual add
 * fused into the convolution's output pass):
 *   out[o][:] = act(acc[o][:] + bias[:]) + residual[o][:]
 * computed in fp32 (acc = the sum over offsets above) and stored once in
 * out_dtype, bf16 by rounding to nearest, ties to even.  The pages fix
 * neither the activation nor the order; the activation is applied to the
 * convolution's output and the residual (a skip connection) added after it.
 *
 *   residual  device [n][cout] in out_dtype, 16-byte aligned, or NULL.
 *   out       device [n][cout] in out_dtype, 16-byte aligned; fully written.
 *   act       SC_ACT_NONE, SC_ACT_RELU or SC_ACT_SILU.
 *   out_dtype SC_F32, SC_BF16 or SC_F16 (any with any input dtype); bf16
 *             and fp16 by rounding to nearest, ties to even (fp16 overflows
 *             to infinity past 65,504).
 * sc_forward(...) is sc_forward_ex(..., NULL residual, SC_ACT_NONE, SC_F32).
 * On the tensor-core path an activation or a 16-bit output turns the tail split
 * (see sc_forward) off, since neither can be applied to a partial sum; a
 * residual alone keeps it (the last part adds it).
 * Errors as sc_forward, plus SC_ERR_INVALID_ARG for a bad act or out_dtype.
 */
SC_API sc_status sc_forward_ex(sc_handle h, const void* feats, const void* weight,
                               const float* bias, const void* residual, void* out, int32_t cin,
                               int32_t cout, sc_dtype dtype, sc_activation act, sc_dtype out_dtype,
                               void* stream);

/*
 * Release a map.  Its device memory is freed in stream order on `stream`:
 * the caller must order every other stream that used the map before that
 * stream.  A handle that is not live (freed already, or never returned by
 * sc_build_map) gives SC_ERR_BAD_HANDLE and is not touched.  NULL is a no-op.
 */
SC_API sc_status sc_free_map(sc_handle h, void* stream);

/*
 * Deterministic mode for sc_forward (process-wide; default 0).  With 1, every
 * call on the same inputs returns bit-identical outputs, at the cost of the
 * tail split described under sc_forward (a last partial round of tiles then
 * runs as fewer, longer parts).  Returns SC_OK, or SC_ERR_INVALID_ARG for a
 * value other than 0 or 1.
 */
SC_API sc_status sc_set_deterministic(int32_t enable);

/*
 * Number of GPU kernels this library has launched in this process, counted on
 * the host at each launch (map build: 3 per sc_build_map, 6 when it retries
 * with 64-bit keys; sc_forward: 1, or 2 when the tensor-core path zeroes
 * split rows first; 1 per sc_get_neighbor_table; 3 or 4 per sc_get_pairs).
 * For measuring launches over a region of code.
 */
SC_API uint64_t sc_kernel_launches(void);

/*
 * Return to the device the memory the library keeps cached for later maps.
 * Map buffers come from a library-owned stream-ordered pool that keeps freed
 * memory reserved, since unmapping and remapping it costs more than a build.
 * Live maps' memory is untouched, and so is memory whose stream-ordered free
 * has not executed yet; synchronise those streams first to release
 * everything.  Does nothing when sc_set_allocator routes allocations
 * elsewhere.  SC_OK, or SC_ERR_CUDA.
 */
SC_API sc_status sc_release_cached_memory(void);

/* Number of rows n of the map, or -1 (and SC_ERR_BAD_HANDLE) for a dead handle. */
SC_API int64_t sc_map_size(sc_handle h);

/* Total pair count P = sum_k |{o : nbr[o][k] >= 0}|, or -1 for a dead handle. */
SC_API int64_t sc_map_pairs(sc_handle h);

/*
 * Copy the neighbour table to nbr_out, device int32 [n][27] row-major
 * (nbr[o][k] as defined above, -1 = absent).  Asynchronous on `stream`.
 */
SC_API sc_status sc_get_neighbor_table(sc_handle h, int32_t* nbr_out, void* stream);

/*
 * Per-offset pair lists in CSR form ("Running TRELLIS.2 on a Mac (1/3)",
 * Sparse 3D convolution: for each kernel position the (input, output) pairs
 * that are gathered, multiplied and added).
 *   off_host  host int64 [28]: pairs of offset k are [off[k], off[k+1]).
 *   in, out   device int32 [P] (P = sc_map_pairs): input row and output row of
 *             each pair; within one offset, pairs are in ascending output row.
 * Either of in/out may be NULL.  Synchronises `stream` once (to fill off_host).
 */
SC_API sc_status sc_get_pairs(sc_handle h, int64_t* off_host, int32_t* in, int32_t* out, void* stream);

/*
 * Install a device allocator for the map's buffers (e.g. a framework's
 * caching allocator).  alloc(bytes, stream, ctx) returns a device pointer or
 * NULL; free(ptr, stream, ctx) releases it in stream order.  Passing NULL for
 * both restores the default (cudaMallocAsync / cudaFreeAsync).  Maps keep the
 * allocator they were built with.  Not thread-safe against concurrent builds.
 */
SC_API sc_status sc_set_allocator(void* (*alloc)(size_t bytes, void* stream, void* ctx),
                           void (*free_fn)(void* ptr, void* stream, void* ctx), void* ctx);

/*
 * Synchronise `stream` and report the map's device status word: SC_OK, or the
 * first error a bounded device loop of a kernel using this map recorded since
 * the last call (SC_ERR_DEVICE_TIMEOUT, SC_ERR_TABLE_FULL).  Clears the word.
 */
SC_API sc_status sc_device_status(sc_handle h, void* stream);

/*
 * Neighbour table without any device allocation.  The pages have no
 * counterpart to this call; it exists for callers that cannot let a library
 * allocate device memory: runtimes that give a plugin a fixed memory budget
 * and forbid allocation while work is enqueued, loops where the implicit
 * device synchronisation of cudaMalloc is unacceptable, and deployments that
 * reserve all device memory up front.
 *
 * It writes the same table as sc_build_map + sc_get_neighbor_table:
 *   coords     device int32 [n][4] (batch, x, y, z), 16-byte aligned.
 *   n          0 <= n <= 524288 (2^19); larger n gives SC_ERR_UNSUPPORTED.
 *   res        grid side, 1 <= res <= 2^20 (same key-space rule as sc_build_map).
 *   nbr_out    device int32 [n][27], 16-byte aligned, owned by the caller.
 *   pairs_out  host int64, receives the pair count P; may be NULL.
 * Errors as sc_build_map (SC_ERR_COORD_RANGE, SC_ERR_DUPLICATE, ...).
 * Synchronises `stream` once, to read the status and pair count.
 *
 * Scratch: the hash table (2^20 slots, 8 MiB) and 16 KiB of tile masks and
 * status words live in one static device array that every device which loads
 * the library holds until the process exits.  The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress); make that
 * first call before any stream capture.  All calls share the one array and
 * each clears what it needs, so calls that overlap on the GPU (other streams,
 * other host threads) race and must be serialised by the caller.  The call
 * itself allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.
 */
SC_API sc_status sc_build_neighbor_table_noalloc(const int32_t* coords, int64_t n, int32_t res,
                                                 int32_t* nbr_out, int64_t* pairs_out,
                                                 void* stream);

/* Thread-local status and message of the last failing call on this thread. */
SC_API sc_status sc_last_error(void);
SC_API const char* sc_last_error_msg(void);

/* Library version string. */
SC_API const char* sc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SC_H_ */
