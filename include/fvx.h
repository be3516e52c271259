/*
 * fvx — sparse-voxel IndexGrid build, 3x3x3 kernel map and sparse convolution
 * on one GB300 (sm_103a).  Plain C ABI: opaque handles, plain pointers and
 * sizes; no C++ or torch types cross this boundary.
 *
 * Sources (page title, section):
 *   [fVDB-notes]  "fVDB: A Deep-Learning Framework for Sparse, Large Scale, and
 *                 High Performance Spatial Intelligence" (reading notes):
 *                 "Core method", "IndexGrid", "GPU-accelerated IndexGrid
 *                 build", "Sparse-convolution operators", "Limitations and
 *                 future work".
 *   [fVDB-ONNX]   "Proposal: ONNX Runtime support for fVDB operations",
 *                 §1.1 Tensor Representations, §1.2 Custom Operator Schemas.
 *   [DriveRT]     "DriveRT": "Shared neighbour maps", "Counts kept on the GPU",
 *                 "Kernels selected per GPU", "Compilation and deployment"
 *                 (C ABI; dynamic sizes are never truncated), "Inspection and
 *                 debugging" (errors name what failed).
 *
 * Conventions shared by every call
 *   - Device pointers are CUDA global-memory addresses on the current device;
 *     host pointers are ordinary process memory.  Every argument says which.
 *   - Every call is asynchronous on the given stream unless it says it
 *     synchronises.  fvx_stream is a cudaStream_t (NULL = legacy default).
 *   - The library owns grids and kernel maps (their sizes depend on the data)
 *     and frees them in *_destroy.  The caller owns coordinates, features,
 *     weights and outputs.
 *   - Every call returns an fvx_status; nothing throws across the ABI.
 *     fvx_last_error() gives a message naming the call, argument or kernel.
 *   - Coordinates are signed int32 voxel indices (i, j, k).  Active indices are
 *     0-based ranks in the canonical tree order: batch, then root tile
 *     (floor(c/4096), signed), then upper-node child, lower-node child and
 *     voxel-in-leaf, each child position in x-major order.  Absent -> -1.
 */
#ifndef FVX_H
#define FVX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fvx_grid_s* fvx_grid;
typedef struct fvx_kmap_s* fvx_kmap;
typedef struct fvx_hits_s* fvx_hits; /* voxels along rays (library-owned) */
typedef void* fvx_stream; /* cudaStream_t */

typedef enum {
  FVX_OK = 0,
  FVX_ERR_INVALID_ARG = 1,    /* malformed argument (sizes, offsets, dtype) */
  FVX_ERR_RANGE = 2,          /* data outside the supported range (see call) */
  FVX_ERR_CAPACITY = 3,       /* a caller buffer is too small; required size reported */
  FVX_ERR_ALLOC = 4,          /* the allocator returned NULL */
  FVX_ERR_CUDA = 5,           /* a CUDA runtime call or kernel launch failed */
  FVX_ERR_DEVICE_TIMEOUT = 6, /* a bounded device-side wait gave up */
  FVX_ERR_CHECK = 7           /* a device-side check failed (see fvx_last_error) */
} fvx_status;

/* Conv arithmetic / storage types.
 *   FVX_F32            fp32 feats, weights and output; exact fp32 FFMA.
 *   FVX_BF16           bf16 feats and weights, fp32 accumulation, fp32 output.
 *   FVX_BF16_OUT_BF16  bf16 feats and weights, fp32 accumulation, output rounded
 *                      to bf16 (nearest even): adds up to 2^-8 |y| of error. */
typedef enum { FVX_F32 = 0, FVX_BF16 = 1, FVX_BF16_OUT_BF16 = 2 } fvx_dtype;

/* Device memory the library allocates for grids, kernel maps and temporary
 * buffers goes through these callbacks (stream-ordered).  Default (or after
 * passing NULLs): cudaMallocAsync / cudaFreeAsync on the call's stream.
 * alloc returns NULL on failure; the call then returns FVX_ERR_ALLOC. */
typedef void* (*fvx_alloc_fn)(size_t bytes, fvx_stream stream, void* ctx);
typedef void (*fvx_free_fn)(void* ptr, fvx_stream stream, void* ctx);
fvx_status fvx_set_allocator(fvx_alloc_fn alloc, fvx_free_fn free_fn, void* ctx);

/* ---------------------------------------------------------------------------
 * IndexGrid build  [fVDB-notes, "GPU-accelerated IndexGrid build", steps 1-12;
 * "IndexGrid"; fVDB-ONNX §1.2 GridFromIJK]
 *
 * coords        device int32 [n_rows, 3], row-major; rows need not be sorted or
 *               unique (duplicates collapse to one active voxel).
 * n_rows        >= 0; at most 2^31 - 2.  n_rows == 0 gives an empty grid.
 * batch_offsets HOST int64 [B + 1], CSR over rows: batch b owns rows
 *               [batch_offsets[b], batch_offsets[b+1]); monotone, starts at 0,
 *               ends at n_rows.  [fVDB-ONNX §1.1: joffsets]
 * B             >= 1.
 * out           receives the new grid handle (library-owned).
 *
 * Topology: the root is the sorted list of (batch, tile) upper nodes; an upper
 * node holds a 32^3-bit child mask, a lower node 16^3 bits, a leaf 8^3 bits in
 * an 80-byte record: 8 mask words, the index of its first active voxel and the
 * popcounts of words 0..w-1 (w = 1..7) in 9-bit fields.  [fVDB-notes, "Core
 * method": fanout 32/16/8; "IndexGrid": 80 bytes per leaf]
 *
 * Synchronises the stream twice (to size the sort keys and to size the
 * topology).  Errors: FVX_ERR_INVALID_ARG (NULL pointers, bad offsets),
 * FVX_ERR_RANGE (the packed sort keys would need more than 64 bits: only
 * possible with very many batches spread over the full int32 range),
 * FVX_ERR_ALLOC, FVX_ERR_CUDA. */
fvx_status fvx_build_grid(const int32_t* coords, int64_t n_rows, const int64_t* batch_offsets, int32_t B,
                          fvx_stream stream, fvx_grid* out);

/* Counts of a built grid (host values, no device work). */
fvx_status fvx_grid_counts(fvx_grid g, int64_t* n_upper, int64_t* n_lower, int64_t* n_leaf, int64_t* n_active);

/* Device pointers into the grid's topology, owned by the grid (valid until
 * fvx_grid_destroy).  All arrays are in canonical order.  32-byte aligned. */
typedef struct {
  int32_t batch_size;
  int64_t n_rows, n_upper, n_lower, n_leaf, n_active;
  const int32_t* ijk;                 /* [n_active, 3]  coordinate of each index (sidecar order) */
  const int32_t* row_to_index;        /* [n_rows]       active index of each input row */
  const int64_t* voxel_batch_offsets; /* [B + 1]        CSR of active indices per batch */
  const int32_t* leaf_origin;         /* [n_leaf, 3] */
  const int32_t* leaf_batch;          /* [n_leaf] */
  const uint64_t* leaf_records;       /* [n_leaf, 10]: mask[8], first index, packed 9-bit prefix */
  const int32_t* lower_origin;        /* [n_lower, 3] */
  const int32_t* lower_batch;         /* [n_lower] */
  const uint64_t* lower_mask;         /* [n_lower, 64]  child leaves, bit n = (x*16+y)*16+z */
  const uint32_t* lower_prefix;       /* [n_lower, 64]  popcount of mask words before w */
  const uint32_t* lower_first;        /* [n_lower]      index of the first child leaf */
  const int32_t* upper_origin;        /* [n_upper, 3] */
  const int32_t* upper_batch;         /* [n_upper] */
  const uint64_t* upper_mask;         /* [n_upper, 512] child lower nodes, bit n = (x*32+y)*32+z */
  const uint32_t* upper_prefix;       /* [n_upper, 512] */
  const uint32_t* upper_first;        /* [n_upper]      index of the first child lower node */
} fvx_grid_view_t;
fvx_status fvx_grid_view(fvx_grid g, fvx_grid_view_t* view);

/* Host copy of the per-batch voxel offsets [B + 1] (synchronises the grid's
 * last stream on first call). */
fvx_status fvx_grid_batch_offsets(fvx_grid g, int64_t* host_out);

/* Coordinate -> active index or -1, by tree walk: root search, then upper and
 * lower child masks with prefix counts, then the leaf's packed prefix plus the
 * popcount of the mask word below the voxel (two branches).
 * [fVDB-notes, "IndexGrid"; fVDB-ONNX §1.2 IJKToIndex / CoordsInGrid]
 * coords device int32 [n, 3]; batch_idx device int32 [n] or NULL (all batch 0);
 * out_idx device int32 [n]. */
fvx_status fvx_lookup(fvx_grid g, const int32_t* coords, const int32_t* batch_idx, int64_t n, int32_t* out_idx,
                      fvx_stream stream);

/* Output grid of a strided conv: the unique floor(ijk / stride) per batch,
 * built by the same GPU build.  stride >= 1.  [fVDB-ONNX §1.2 CoarsenedGrid /
 * ConvGrid]  Synchronises like fvx_build_grid. */
fvx_status fvx_coarsen(fvx_grid g, int32_t stride, fvx_stream stream, fvx_grid* out);

/* Refined grid: every voxel ijk of g replaced by its factor^3 children
 * factor*ijk + {0..factor-1}^3, same batch; the output grid of a transposed
 * strided conv whose kernel covers one stride cell.  factor 1..1024 and
 * n_active * factor^3 <= 2^31 - 2 (FVX_ERR_RANGE otherwise); a child
 * coordinate outside int32 is found on the device and reported as
 * FVX_ERR_CHECK.  Voxels in the output are ordered like any built grid.
 * [fVDB-ONNX §1.2 RefinedGrid]  Synchronises like fvx_build_grid. */
fvx_status fvx_refine(fvx_grid g, int32_t factor, fvx_stream stream, fvx_grid* out);

/* ---------------------------------------------------------------------------
 * Kernel map  [DriveRT, "Shared neighbour maps"; "Kernels selected per GPU"]
 *
 * For every output voxel q of gout and offset slot s = (di+1)*9 + (dj+1)*3 +
 * (dk+1), d in {-1,0,1}^3, the input voxel p of gin at stride*ijk(q) + d in
 * the same batch.  Pairs are grouped by s, and inside a group ordered by q.
 * ksize must be 3; stride 1 (submanifold: pass gout == gin) or 2 (gout is
 * usually fvx_coarsen(gin, 2)).  gin and gout must have the same batch size.
 * Does not synchronise: the pair lists are sized for every output having all
 * 27 neighbours (216 bytes per output voxel of device memory) and the list
 * offsets stay on the device until fvx_kmap_view is asked for them.  Maps
 * whose worst case exceeds 8 GiB (environment FVX_KMAP_CAP_BYTES, read once)
 * or the int32 pair index range synchronise once to size the lists exactly.
 * Never truncated.
 * [DriveRT, "Counts kept on the GPU"; "Compilation and deployment": dynamic
 * sizes, no truncation] */
fvx_status fvx_kernel_map(fvx_grid gin, fvx_grid gout, int32_t ksize, int32_t stride, fvx_stream stream,
                          fvx_kmap* out);

/* offsets_host: HOST int64 [28] (list s is [offsets[s], offsets[s+1]));
 * in_idx / out_idx: device int32 [n_pairs]; out_mask: device uint32 [n_out],
 * bit s set when output q has a neighbour at slot s.  All owned by the map.
 * Any argument may be NULL.  Asking for offsets_host or n_pairs the first
 * time synchronises the stream the map was built on (which must still exist)
 * and may return FVX_ERR_DEVICE_TIMEOUT; the pointers and n_out need no
 * device work. */
fvx_status fvx_kmap_view(fvx_kmap m, const int64_t** offsets_host, const int32_t** in_idx, const int32_t** out_idx,
                         const uint32_t** out_mask, int64_t* n_pairs, int64_t* n_out);

/* Kernel map of the transposed (inverse) convolution
 * [fVDB-ONNX §1.2 ConvTransposeGrid: the transposed conv scatters each input
 * voxel to stride*ijk + d].  For every output voxel q of gout and slot s (d as
 * above), the input voxel p of gin with stride*ijk(p) + d == ijk(q), when
 * ijk(q) - d is divisible by stride.  It pairs exactly what
 * fvx_kernel_map(gout, gin, 3, stride) pairs, with the roles of input and
 * output swapped and the same slot numbers, so
 *   - fvx_sparse_conv over it computes the transposed convolution of gin's
 *     features onto gout (gout usually fvx_refine(gin, 2) for stride 2, or
 *     gin itself for stride 1), and
 *   - fvx_sparse_conv_dgrad over fvx_kernel_map_transposed(gout, gin, ...)
 *     computes the input gradient of a forward conv from gin to gout.
 * Same layout, sizing, synchronisation and errors as fvx_kernel_map; the bf16
 * leaf-densified kernels never run on it. */
fvx_status fvx_kernel_map_transposed(fvx_grid gin, fvx_grid gout, int32_t ksize, int32_t stride, fvx_stream stream,
                                     fvx_kmap* out);

/* ---------------------------------------------------------------------------
 * Sparse convolution (gather - GEMM - scatter)  [fVDB-notes, "Sparse-
 * convolution operators"; effective-TFLOPS definition there]
 *
 *   out[q, co] = sum_s sum_{(p,q) in list s} sum_ci feats[p, ci] * W[s, ci, co]
 *
 * Cross-correlation, no bias; outputs without pairs are 0.
 * feats  device [gin.n_active, cin], row-major (fp32 for FVX_F32, else bf16).
 * W      device [27, cin, cout], row-major (same type as feats).
 * out    device [gout.n_active, cout], row-major, caller-allocated, fully
 *        overwritten; bf16 for FVX_BF16_OUT_BF16, else fp32.
 * FVX_BF16 / FVX_BF16_OUT_BF16: tcgen05 tensor cores, fp32 accumulation in
 *           TMEM.  cin and cout multiples of 8 (cin <= 512, cout <= 256; the
 *           MMA's N is cout rounded up to 16, the extra columns are not
 *           written); feats and out 16-byte aligned.
 * FVX_F32:  fp32 FFMA throughout (no TF32).  cin, cout >= 1.
 * m must have been built for (gin, gout).  Errors: FVX_ERR_INVALID_ARG. */
fvx_status fvx_sparse_conv(fvx_grid gin, fvx_grid gout, fvx_kmap m, fvx_dtype dt, const void* feats, int64_t cin,
                           const void* W, int64_t cout, void* out, fvx_stream stream);

/* Which bf16 kernel fvx_sparse_conv and fvx_sparse_conv_noalloc run
 * [fVDB-notes, "Sparse-convolution operators": several convolution backends,
 * the leaf-densified one for low channel counts on leaves at least 20%
 * occupied, picked per case].
 *   FVX_CONV_AUTO    (default) leaf-densified when the map has stride 1,
 *                    cin is 8 or 16, cout <= 64 and the output grid's leaves
 *                    are at least 20% occupied on average; halo-staged when
 *                    the map has stride 1, cin is 32 (or a larger multiple
 *                    of 32 with fp32 output), cout <= 64 and the output
 *                    leaves hold at least 48 active voxels on average;
 *                    pair-list gather otherwise.
 *   FVX_CONV_GATHER  always the pair-list kernels (128 consecutive outputs
 *                    per tile), direct (below).
 *   FVX_CONV_DIRECT  the pair-list kernel that fetches every pair's input row
 *                    from global memory (TMA gather4 when cin is a multiple
 *                    of 16, else cp.async).
 *   FVX_CONV_UNION   the pair-list kernel that fetches each distinct input
 *                    row of a tile once into shared memory and builds the
 *                    tensor-core operands from there; cin 32 or 64, cout <=
 *                    128, else FVX_ERR_INVALID_ARG.  Same results as the
 *                    direct kernel (bit for bit); slower on the workloads
 *                    measured, so only run when asked for.
 *   FVX_CONV_HALO    always halo-staged (each output leaf's 10^3 input
 *                    window fetched once into shared memory, at the positions
 *                    that hold an input voxel; the operands of the leaf's
 *                    active outputs, 128 per tile, built from there in tensor
 *                    memory; the pair lists are not read, the map's leaf table
 *                    is); one pass per 32 input channels, the passes after
 *                    the first adding to the fp32 output; a call it cannot
 *                    serve (stride 2, a transposed map, cin not a multiple
 *                    of 32, cin > 32 with bf16 output, cout > 64) fails with
 *                    FVX_ERR_INVALID_ARG.
 *   FVX_CONV_LEAF    always leaf-densified (each output leaf's 10^3 input
 *                    window staged densely in shared memory; the pair lists
 *                    are not read; the map's per-leaf table of neighbouring
 *                    input leaves is); a call it cannot serve (stride 2, cin
 *                    other than 8 or 16, cout > 64) fails with
 *                    FVX_ERR_INVALID_ARG.
 * Process-wide; FVX_F32 is unaffected.  Every path meets the same error
 * bound.  Errors: FVX_ERR_INVALID_ARG for an unknown value. */
typedef enum {
  FVX_CONV_AUTO = 0,
  FVX_CONV_GATHER = 1,
  FVX_CONV_LEAF = 2,
  FVX_CONV_DIRECT = 3,
  FVX_CONV_UNION = 4,
  FVX_CONV_HALO = 5
} fvx_conv_algo;
fvx_status fvx_set_conv_algo(fvx_conv_algo algo);
/* The kernel family the last successful bf16 convolution on this host thread
 * launched (FVX_CONV_GATHER for every pair-list kernel, FVX_CONV_LEAF or
 * FVX_CONV_HALO; FVX_CONV_AUTO before any). */
fvx_conv_algo fvx_last_conv_algo(void);
/* Name of the kernel the last convolution on this host thread launched
 * ("conv_halo", "conv_union", "conv_bf16_tma", "conv_bf16_tc", "conv_leaf",
 * "conv_f32";
 * "" before any).  Static storage; not freed. */
const char* fvx_last_conv_kernel(void);

/* Sparse convolution that allocates no device memory.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory while they run — for example an inference
 * runtime whose device memory is planned and reserved once at load time, or a
 * host process whose allocator forbids new device allocations after start-up.
 * Same arguments, result and errors as fvx_sparse_conv (inputs and outputs
 * are still the caller's); its only scratch (the transposed weights and the
 * bounded-wait status word) lives in a fixed array of 2 MiB + 256 bytes in the
 * library's device image, which every GPU that loads the library holds until
 * the process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *   - Limit: 27 * cin * cout16 * 2 bytes <= 2 MiB (cout16 = cout rounded up
 *     to 16; cin * cout16 <= 38836), else FVX_ERR_RANGE; FVX_F32 needs no
 *     scratch and has no such limit.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array and the call clears what must start at
 *     zero: calls that overlap on the GPU (other streams, other threads) race;
 *     order them on one stream.
 *   - A bounded device-side wait that gives up is recorded in that array's
 *     status word, which each call clears when it starts and
 *     fvx_noalloc_status reads (fvx_device_status does not). */
fvx_status fvx_sparse_conv_noalloc(fvx_grid gin, fvx_grid gout, fvx_kmap m, fvx_dtype dt, const void* feats,
                                   int64_t cin, const void* W, int64_t cout, void* out, fvx_stream stream);

/* Status of the last fvx_sparse_conv_noalloc call on the current device,
 * without allocating: synchronises `stream`, reads the status word of the
 * fixed scratch array into a host variable, clears it, and returns FVX_OK,
 * FVX_ERR_DEVICE_TIMEOUT (a bounded wait gave up; the output is incomplete)
 * or FVX_ERR_CHECK.  Call it after each no-alloc call whose result matters:
 * the next call clears the word. */
fvx_status fvx_noalloc_status(fvx_stream stream);

/* ---------------------------------------------------------------------------
 * Backward pass of fvx_sparse_conv  [fVDB-notes, "Limitations and future
 * work": training computes its gradients through the pair-list (IGEMM)
 * backend]
 *
 * Input gradient, for y = conv(x, W) over the map of (gin, gout):
 *   dx[p, ci] = sum_s sum_{(p,q) in list s} sum_co dout[q, co] * W[s, ci, co]
 * mt: fvx_kernel_map_transposed(gout, gin, 3, stride) (FVX_ERR_INVALID_ARG
 *     for any other map).
 * dout device [gout.n_active, cout]; W device [27, cin, cout] as in
 *     fvx_sparse_conv; dx device [gin.n_active, cin], caller-allocated, fully
 *     overwritten (zero where no pair reaches it).
 * Types as fvx_sparse_conv with the roles of cin and cout swapped: bf16
 *     needs cout and cin multiples of 8 (cout <= 512, cin <= 256), dout, W
 *     and dx 16-byte aligned (cin not a multiple of 16: W is first copied
 *     into library scratch with zero rows up to the next multiple); FVX_F32
 *     any sizes >= 1 (it transposes W into library scratch first).
 * Kernels: bf16 stride 1 with cout 8 or 16, cin <= 64 and the grid of dx at
 *     least 20% occupied per leaf (or FVX_CONV_LEAF set) runs the
 *     leaf-densified kernel with the slot-mirrored weights (dx[p] = sum_s
 *     dout[p + d_s] W[26 - s]^T); FVX_CONV_LEAF with any other shape fails
 *     with FVX_ERR_INVALID_ARG; everything else runs the pair-list kernels
 *     over mt.  Same error bound as fvx_sparse_conv. */
fvx_status fvx_sparse_conv_dgrad(fvx_grid gin, fvx_grid gout, fvx_kmap mt, fvx_dtype dt, const void* dout,
                                 int64_t cout, const void* W, int64_t cin, void* dx, fvx_stream stream);

/* Weight gradient over the forward map m of (gin, gout):
 *   dW[s, ci, co] = sum_{(p,q) in list s} feats[p, ci] * dout[q, co]
 * feats device [gin.n_active, cin], dout device [gout.n_active, cout], both
 * fp32 (FVX_F32) or bf16 (FVX_BF16); dW device fp32 [27, cin, cout],
 * caller-allocated, fully overwritten.  Kernels: cin * cout <= 1024 and
 * cin + cout <= 64, fp32 FFMA with the partial in registers; other bf16
 * layers with cin and cout multiples of 8, tcgen05 tensor cores (bf16
 * products, fp32 accumulation in tensor memory; within 2e-3 * sum|x*dy|);
 * the rest, tiled fp32 FFMA (fp32 inputs: within 1e-5 * sum|x*dy|).  Partial
 * sums are added with fp32 atomics, so the summation order is not fixed and
 * results may differ between runs in the last bits.
 * 1 <= cin, cout <= 65536.  Errors: FVX_ERR_INVALID_ARG; FVX_ERR_RANGE past
 * 2^32 tensor-core work units. */
fvx_status fvx_sparse_conv_wgrad(fvx_grid gin, fvx_grid gout, fvx_kmap m, fvx_dtype dt, const void* feats,
                                 int64_t cin, const void* dout, int64_t cout, float* dW, fvx_stream stream);

/* ---------------------------------------------------------------------------
 * Voxels along rays ("fVDB" reading notes, HDDA: one DDA per tree level at
 * 4096^3, 128^3, 8^3 and 1^3 cells; empty nodes are crossed in one step).
 *
 * For each ray, the active voxels it passes through, in order, with the
 * interval of the ray parameter t spent in each.  Definition (exact, fp32):
 *   - voxel (i,j,k) is the cell [i,i+1) x [j,j+1) x [k,k+1) in index space;
 *     the ray is o + t d; inv_a = 1/d_a rounded once; the ray crosses the
 *     plane x_a = n at T_a(n) = ((float)n - o_a) * inv_a (two fp32 roundings);
 *   - [tmin, tmax] is clipped to the batch element's voxels by those plane
 *     times; at time t the ray is in cell c_a = max{n : T_a(n) <= t}
 *     (d_a > 0), min{n : T_a(n) <= t} - 1 (d_a < 0), floor(o_a) (d_a = 0);
 *   - a hit is an active cell occupied for a time interval of positive
 *     length: its voxel index and [t_enter, t_exit) (crossing times clipped
 *     to the segment).  Rays that graze an edge or corner do not hit the
 *     cells they only touch.  d = 0 gives no hits.
 * origins, dirs: device float [n_rays, 3] (finite); ray_batch: device int32
 * [n_rays] batch element of each ray, or NULL (all in element 0).  Voxel
 * coordinates must lie in [-2^24, 2^24) (cell faces exact in fp32).
 * Two passes (count, write) and one host synchronisation (the total sizes
 * the output; nothing is truncated).  The handle owns the result: offsets
 * device int64 [n_rays + 1] (CSR: ray r's hits are [offsets[r],
 * offsets[r+1])), voxel device int32 [n_hits], t device float [n_hits, 2].
 * Errors: FVX_ERR_INVALID_ARG (NULL, negative count, NaN tmin/tmax);
 * FVX_ERR_RANGE (n_rays or n_hits >= 2^31); FVX_ERR_CHECK (a ray_batch value
 * outside [0, B), or voxels outside the coordinate range); FVX_ERR_ALLOC. */
fvx_status fvx_voxels_along_rays(fvx_grid g, const float* origins, const float* dirs, const int32_t* ray_batch,
                                 int64_t n_rays, float tmin, float tmax, fvx_stream stream, fvx_hits* out);
/* Device pointers owned by h (NULL arguments are skipped). */
fvx_status fvx_hits_view(fvx_hits h, const int64_t** offsets, const int32_t** voxel, const float** t,
                         int64_t* n_hits, int64_t* n_rays);
fvx_status fvx_hits_destroy(fvx_hits h);

fvx_status fvx_grid_destroy(fvx_grid g);
fvx_status fvx_kmap_destroy(fvx_kmap m);

/* ---------------------------------------------------------------------------
 * Status, diagnostics, accounting
 */
const char* fvx_status_string(fvx_status st);
/* Message of the last failing call on this host thread ("" if none). */
const char* fvx_last_error(void);

/* Synchronises `stream` and returns the device status word that bounded waits
 * and device-side checks write (FVX_OK, FVX_ERR_DEVICE_TIMEOUT or
 * FVX_ERR_CHECK), then clears it. */
fvx_status fvx_device_status(fvx_stream stream);

/* Number of kernels this library has launched since it was loaded (host
 * counter, all threads). */
uint64_t fvx_launch_count(void);

/* Kernel timing for roofline measurement: while enabled, every launch of a
 * kernel whose name equals `kernel_name` is bracketed with CUDA events on its
 * own stream.  fvx_profile_read synchronises those events and returns the
 * total milliseconds and the number of timed launches since the last enable.
 * Pass NULL to disable. */
fvx_status fvx_profile_enable(const char* kernel_name);
fvx_status fvx_profile_read(double* total_ms, int64_t* launches);
/* The same timed launches one by one, in launch order: writes the duration
 * in milliseconds of the first min(cap, launches) of them to ms_each (host
 * array of cap doubles) and the number of timed launches to *launches.
 * Errors: FVX_ERR_INVALID_ARG for a NULL output or cap < 0. */
fvx_status fvx_profile_read_each(double* ms_each, int64_t cap, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* FVX_H */
