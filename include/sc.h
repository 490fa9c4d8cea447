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
  SC_ERR_TABLE_FULL = 4,   /* hash probe bound exceeded (at the table's load
                              factor of at most 1/2 only under a probe limit
                              set by sc_set_probe_limit)                        */
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
 * sc_build_map without any host synchronisation: the hash build and the
 * neighbour map are enqueued on `stream` and the handle is returned at once,
 * so that the build overlaps host work and the convolutions enqueued after
 * it (same definition and citations as sc_build_map).
 *
 *   nbatch  batch indices must lie in [0, nbatch), nbatch >= 1.  It fixes the
 *           hash key width up front (32-bit keys when nbatch * res^3 < 2^32),
 *           so there is no retry; SC_ERR_UNSUPPORTED when even 64-bit keys
 *           cannot hold nbatch * res^3 (see sc_build_map).
 * The map's buffers are ready in stream order on `stream`: sc_forward on the
 * same stream (or one ordered after it) can follow at once.  Errors the
 * device finds (a coordinate outside [0,res), a batch index outside
 * [0,nbatch), duplicate rows) are not returned here: the first call that
 * needs the build's result -- sc_map_status, sc_map_pairs, sc_device_status
 * -- waits for the build and reports them (SC_ERR_COORD_RANGE,
 * SC_ERR_DUPLICATE, SC_ERR_TABLE_FULL), and they stay with the map.  A
 * convolution over a map whose build failed computes garbage but never
 * reads or writes outside its buffers.  Returns NULL only for errors found
 * on the host (SC_ERR_INVALID_ARG, SC_ERR_UNSUPPORTED, SC_ERR_ALLOC,
 * SC_ERR_CUDA).  No counterpart on the pages beyond sc_build_map's.
 */
SC_API sc_handle sc_build_map_async(const int32_t* coords, int64_t n, int32_t res, int32_t nbatch,
                                    void* stream);

/*
 * Wait for the map's build (if sc_build_map_async left it unread) and return
 * its outcome: SC_OK or the build's error (see above).  Synchronises with
 * the build only, not with later work on its stream.  Error plumbing with no
 * counterpart on the pages.
 */
SC_API sc_status sc_map_status(sc_handle h);

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
 *           It must not overlap feats, weight or bias.
 * Every pointer must be ordinary device memory of the map's device
 * (cudaMalloc, a stream-ordered pool or a VMM mapping); host memory (even
 * pinned or mapped), managed memory and another GPU's memory give
 * SC_ERR_INVALID_ARG before anything is launched.  (The tensor-core kernel
 * reads W through a tensor map whose loads are shared by the two CTAs of a
 * cluster on this GPU.)
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
 *   residual  device [n][cout] in out_dtype, 16-byte aligned, or NULL.  It
 *             may be out itself (an in-place skip connection: each element
 *             is read before it is written); any other overlap with out is
 *             SC_ERR_INVALID_ARG.
 *   out       device [n][cout] in out_dtype, 16-byte aligned; fully written.
 *   act       SC_ACT_NONE, SC_ACT_RELU or SC_ACT_SILU.
 *   out_dtype SC_F32, SC_BF16 or SC_F16 (any with any input dtype); bf16
 *             and fp16 by rounding to nearest, ties to even (fp16 overflows
 *             to infinity past 65,504).
 * sc_forward(...) is sc_forward_ex(..., NULL residual, SC_ACT_NONE, SC_F32).
 * On the tensor-core path an activation or a 16-bit output turns the tail split
 * (see sc_forward) off, since neither can be applied to a partial sum; so
 * does residual == out, since the split rows are zeroed and summed into
 * before the last part would read the residual from them.  A separate
 * residual keeps the split (the last part adds it).
 * Errors as sc_forward, plus SC_ERR_INVALID_ARG for a bad act or out_dtype
 * or a residual that partly overlaps out.
 */
SC_API sc_status sc_forward_ex(sc_handle h, const void* feats, const void* weight,
                               const float* bias, const void* residual, void* out, int32_t cin,
                               int32_t cout, sc_dtype dtype, sc_activation act, sc_dtype out_dtype,
                               void* stream);

/*
 * Reorder the map's rows for the convolutions that follow (call once after
 * the build, on a stream ordered after it; asynchronous).  A 128-row tile
 * skips an offset only when none of its rows has that neighbour, and in
 * input order almost every tile holds all 27.  This call sorts the rows by
 * their 27-bit neighbour-presence masks (stable) and keeps a permuted copy
 * of the neighbour table with each position's original row, so that tiles
 * group rows of one neighbourhood shape and skip more offsets (fewer
 * gathered rows and tensor-core stages); the convolution still writes every
 * output to its own row, so results are those of the unordered map up to
 * fp32 summation order.  Costs 112 bytes a row of device memory and a few
 * kernels; sc_get_neighbor_table and sc_get_pairs are unaffected.  The
 * pages build the table once per level and reuse it across that level's
 * convolutions; this is a one-off cost of the same kind (no counterpart on
 * the pages).  SC_OK, SC_ERR_BAD_HANDLE, SC_ERR_ALLOC or SC_ERR_CUDA.
 */
SC_API sc_status sc_map_order_rows(sc_handle h, void* stream);

/*
 * Release a map (library plumbing: the pages have no counterpart; they keep
 * maps in a per-tensor cache).  Its device memory is freed in stream order on `stream`:
 * the caller must order every other stream that used the map before that
 * stream.  A handle that is not live (freed already, or never returned by
 * sc_build_map) gives SC_ERR_BAD_HANDLE and is not touched.  NULL is a no-op.
 */
SC_API sc_status sc_free_map(sc_handle h, void* stream);

/*
 * Deterministic mode for sc_forward (process-wide; default 0; no counterpart
 * on the pages, whose reference layer is compared bit for bit against one
 * run of their own kernel).  With 1, every
 * call on the same inputs returns bit-identical outputs, at the cost of the
 * tail split described under sc_forward (a last partial round of tiles then
 * runs as fewer, longer parts).  Returns SC_OK, or SC_ERR_INVALID_ARG for a
 * value other than 0 or 1.
 */
SC_API sc_status sc_set_deterministic(int32_t enable);

/*
 * Instrumentation with no counterpart on the pages.
 * Number of GPU kernels this library has launched in this process, counted on
 * the host at each launch (map build: 3 per sc_build_map, 6 when it retries
 * with 64-bit keys; sc_forward: 1, or 2 when the tensor-core path zeroes
 * split rows first; 1 per sc_get_neighbor_table; 3 or 4 per sc_get_pairs).
 * For measuring launches over a region of code.
 */
SC_API uint64_t sc_kernel_launches(void);

/*
 * Memory plumbing with no counterpart on the pages.
 * Return to the device the memory the library keeps cached for later maps.
 * Map buffers come from a library-owned stream-ordered pool that keeps freed
 * memory reserved, since unmapping and remapping it costs more than a build.
 * Live maps' memory is untouched, and so is memory whose stream-ordered free
 * has not executed yet; synchronise those streams first to release
 * everything.  Does nothing when sc_set_allocator routes allocations
 * elsewhere.  SC_OK, or SC_ERR_CUDA.
 */
SC_API sc_status sc_release_cached_memory(void);

/* Number of rows n of the map, or -1 (and SC_ERR_BAD_HANDLE) for a dead handle
 * (an accessor with no counterpart on the pages). */
SC_API int64_t sc_map_size(sc_handle h);

/* Total pair count P = sum_k |{o : nbr[o][k] >= 0}|, or -1 for a dead handle
 * or a failed asynchronous build (whose build it waits for first):
 * the number of (input, output) pairs that "Running TRELLIS.2 on a Mac (1/3)",
 * Sparse 3D convolution, gathers and multiplies, which sets the layer's
 * effective work 2 * P * cin * cout. */
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
 * Allocation plumbing with no counterpart on the pages.
 * Install a device allocator for the map's buffers (e.g. a framework's
 * caching allocator).  alloc(bytes, stream, ctx) returns a device pointer or
 * NULL; free(ptr, stream, ctx) releases it in stream order.  Passing NULL for
 * both restores the default (cudaMallocAsync / cudaFreeAsync).  Maps keep the
 * allocator they were built with.  Not thread-safe against concurrent builds.
 */
SC_API sc_status sc_set_allocator(void* (*alloc)(size_t bytes, void* stream, void* ctx),
                           void (*free_fn)(void* ptr, void* stream, void* ctx), void* ctx);

/*
 * Error plumbing with no counterpart on the pages.
 * Synchronise `stream` and report the map's device status word: SC_OK, or the
 * first error a bounded device loop of a kernel using this map recorded since
 * the last call (SC_ERR_DEVICE_TIMEOUT, SC_ERR_TABLE_FULL).  Clears the word.
 * An asynchronous build's own error (see sc_build_map_async) is reported
 * first, and on every call.
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
 * itself allocates nothing: no cudaMalloc, cudaFree, cudaHostAlloc or
 * allocating library routine; the status words come back into a buffer on
 * the calling thread's stack.
 */
SC_API sc_status sc_build_neighbor_table_noalloc(const int32_t* coords, int64_t n, int32_t res,
                                                 int32_t* nbr_out, int64_t* pairs_out,
                                                 void* stream);

/* ------------------------------------------------------------------------
 * Level changes: moving a sparse voxel set between resolution levels.
 * The trellis2mlx README names these operations -- its pipeline list's
 * "Upsample" stage (the decoder's subdivision predictions become the
 * high-resolution coordinates), its stage table (2,977 low-resolution voxels
 * become 761,916) and its project layout (a sparse UNet decoder upsampling
 * by Channel2Spatial) -- without fixing their details; the readings taken
 * are stated at each call.
 */
typedef struct sc_level* sc_level_handle; /* opaque level map owned by the library */

/*
 * Children of each voxel whose mask bit is set: child o (0..7) of (b, x, y,
 * z) is (b, 2x + (o >> 2 & 1), 2y + (o >> 1 & 1), 2z + (o & 1)) -- the same
 * row-major flattening as the 27 offsets.  Children are listed parent by
 * parent in input order, ascending o within a parent.
 *   coords        device int32 [n][4] at resolution res, 16-byte aligned.
 *   mask          device uint8 [n] (bit o: child o exists), or NULL for all 8.
 *   n             0 <= n < 2^28;  res  1 <= res <= 2^19 (children at 2 res).
 *   child_coords  device int32 [capacity][4], 16-byte aligned: room for every
 *                 selected child (8n always suffices).
 *   parent, offset  device int32 [capacity] or NULL: each child's parent row
 *                 and o.
 *   child_of      device int32 [n][8] or NULL: row of child o of each voxel,
 *                 or -1.
 *   m_out         host: receives the number of children M.
 * Synchronises `stream` once (to return M).  SC_ERR_COORD_RANGE for a
 * coordinate outside [0,res) or a negative batch, SC_ERR_INVALID_ARG,
 * SC_ERR_ALLOC, SC_ERR_CUDA.
 */
SC_API sc_status sc_subdivide(const int32_t* coords, const uint8_t* mask, int64_t n, int32_t res,
                              int32_t* child_coords, int32_t* parent, int32_t* offset,
                              int32_t* child_of, int64_t* m_out, void* stream);

/*
 * Channel2Spatial: each child takes C of its parent's 8C channels, child o
 * channel c = parent channel c * 8 + o (the sub-voxel index runs fastest, as
 * in the dense pixel shuffle).
 *   feats   device [n_parents][8c] in dtype.
 *   parent, offset  device int32 [m] (as sc_subdivide returns them).
 *   out     device [m][c] in dtype.
 * Asynchronous on `stream`.
 */
SC_API sc_status sc_channel_to_spatial(const void* feats, const int32_t* parent,
                                       const int32_t* offset, int64_t m, int32_t c, sc_dtype dtype,
                                       void* out, void* stream);

/*
 * The way down: the parents of n voxels at resolution res are the distinct
 * (b, x >> 1, y >> 1, z >> 1), listed in (b, x, y, z) order, each with the
 * row of its child o (o as in sc_subdivide) or -1.  The returned map also
 * drives the 2x2x2 stride-2 convolutions between the two levels.
 *   coords  device int32 [n][4] (the fine voxels), 16-byte aligned.
 *   res     1 <= res <= 2^20;  nbatch: batch indices lie in [0, nbatch).
 * Synchronises `stream` once.  NULL with SC_ERR_COORD_RANGE (a coordinate
 * outside [0,res) or a batch index outside [0,nbatch)), SC_ERR_DUPLICATE,
 * SC_ERR_UNSUPPORTED (nbatch * ceil(res/2)^3 beyond 2^63), SC_ERR_INVALID_ARG,
 * SC_ERR_ALLOC or SC_ERR_CUDA.
 */
SC_API sc_level_handle sc_build_level_map(const int32_t* coords, int64_t n, int32_t res,
                                          int32_t nbatch, void* stream);

/* Number of parents P, or -1 (SC_ERR_BAD_HANDLE) for a dead handle. */
SC_API int64_t sc_level_parents(sc_level_handle h);

/*
 * Copy the map out (any output may be NULL): parent_coords device int32
 * [P][4]; child_of device int32 [P][8] (row of child o, -1 if absent);
 * parent_of device int32 [n] (each fine voxel's parent).  Asynchronous.
 */
SC_API sc_status sc_get_level_map(sc_level_handle h, int32_t* parent_coords, int32_t* child_of,
                                  int32_t* parent_of, void* stream);

/*
 * 2x2x2 stride-2 convolution down a level, weights W[8][cin][cout] (the
 * (Kvol, Ci, Co) layout with Kvol = 8, o as above):
 *   out[p] = act(bias + sum_o feats[child_of[p][o]] @ W[o]) + residual[p]
 * over present children; feats [n][cin] (fine rows), out [P][cout].  The
 * epilogue, dtypes, shape envelope and pointer rules are those of
 * sc_forward_ex.  Asynchronous on `stream`.
 */
SC_API sc_status sc_conv_down(sc_level_handle h, const void* feats, const void* weight,
                              const float* bias, const void* residual, void* out, int32_t cin,
                              int32_t cout, sc_dtype dtype, sc_activation act, sc_dtype out_dtype,
                              void* stream);

/*
 * Its transpose, up a level:
 *   out[i] = act(bias + feats[parent_of[i]] @ W[octant of i]) + residual[i]
 * for every fine voxel i; feats [P][cin] (parent rows), out [n][cout].
 * Otherwise as sc_conv_down.
 */
SC_API sc_status sc_conv_up(sc_level_handle h, const void* feats, const void* weight,
                            const float* bias, const void* residual, void* out, int32_t cin,
                            int32_t cout, sc_dtype dtype, sc_activation act, sc_dtype out_dtype,
                            void* stream);

/* As sc_device_status, for the convolutions over a level map. */
SC_API sc_status sc_level_device_status(sc_level_handle h, void* stream);

/* Release a level map (stream-ordered, as sc_free_map). */
SC_API sc_status sc_free_level_map(sc_level_handle h, void* stream);

/* ------------------------------------------------------------------------
 * Dual-grid mesh extraction over a built map ("Running TRELLIS.2 on a Mac
 * (1/3)", Mesh extraction paragraph: a dual voxel grid, coordinate-to-index
 * tables, the connected voxels of each edge, quads split into triangles by
 * how well their normals align; "Porting TRELLIS.2 From Python to Rust and
 * Metal", results: a compact hash map and a parallel loop).  Readings:
 * voxel (x, y, z) is the cell [x, x+1] x [y, y+1] x [z, z+1] and owns the
 * three primal edges from its min corner along +x, +y, +z; flag bit a (0..2)
 * says its a-edge crosses the surface, bit 3 + a that the edge's start point
 * is inside.
 */

/*
 * Quads of the crossing edges: the voxels at offsets 0, -e_b, -e_b - e_c,
 * -e_c from the edge's owner ((a, b, c) cyclic), when all four are active,
 * in that order (right-hand normal along +a for cell-centre vertices),
 * reversed when the start point is outside.  Listed by owner row, then axis.
 *   flags   device uint8 [n] (6 bits per voxel, n = sc_map_size).
 *   quads   device int32 [capacity][4] of voxel rows, 16-byte aligned;
 *           capacity 3n always suffices.
 *   q_out   host: receives the number of quads Q.
 * The four rows of each edge come from the map's neighbour table.
 * Synchronises `stream` once.
 */
SC_API sc_status sc_dual_mesh_quads(sc_handle h, const uint8_t* flags, int32_t* quads,
                                    int64_t* q_out, void* stream);

/*
 * Two triangles per quad (q0, q1, q2, q3): (q0, q1, q2), (q0, q2, q3) when
 * that split's unit normals have the larger dot product, else (q0, q1, q3),
 * (q1, q2, q3); a tie keeps the first.  Computed in fp64, each product and
 * sum rounded separately.
 *   quads     device int32 [nq][4] (16-byte aligned), rows into vertices.
 *   vertices  device fp32 [n][3]: each voxel's dual vertex.
 *   tris      device int32 [2 nq][3].
 * Asynchronous on `stream`.
 */
SC_API sc_status sc_dual_mesh_triangulate(const int32_t* quads, int64_t nq, const float* vertices,
                                          int32_t* tris, void* stream);

/*
 * Cap, for testing the hash's bounded probe loop, on the slots one key's
 * insertion may probe (process-wide; 0, the default, = the table's
 * capacity).  Builds whose insertion needs more probes fail with
 * SC_ERR_TABLE_FULL (sc_build_map, sc_build_neighbor_table_noalloc).  With
 * 1, any key whose home slot is taken by another key fails the build.  No
 * counterpart on the pages.  SC_OK, or SC_ERR_INVALID_ARG for limit < 0.
 */
SC_API sc_status sc_set_probe_limit(int32_t limit);

/* Thread-local status and message of the last failing call on this thread
 * (error plumbing with no counterpart on the pages). */
SC_API sc_status sc_last_error(void);
SC_API const char* sc_last_error_msg(void);

/* Library version string (no counterpart on the pages). */
SC_API const char* sc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SC_H_ */
