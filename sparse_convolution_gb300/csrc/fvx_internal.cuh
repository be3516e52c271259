// Internal declarations shared by the fvx CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/fvx.h"

namespace fvx {

// ---------------------------------------------------------------- errors
void set_error(const char* fmt, ...);
fvx_status cuda_fail(cudaError_t e, const char* what, const char* file, int line);

#define FVX_TRY(expr)                     \
  do {                                    \
    fvx_status st_ = (expr);              \
    if (st_ != FVX_OK) return st_;        \
  } while (0)

#define FVX_CUDA(expr)                                                       \
  do {                                                                       \
    cudaError_t e_ = (expr);                                                 \
    if (e_ != cudaSuccess) return ::fvx::cuda_fail(e_, #expr, __FILE__, __LINE__); \
  } while (0)

// ---------------------------------------------------------------- memory
// Name of the public call this host thread is in, for messages of helpers
// that do not know it (a failed device allocation names its entry point).
extern thread_local const char* t_entry;
struct EntryScope {
  const char* prev;
  explicit EntryScope(const char* name) : prev(t_entry) { t_entry = name; }
  ~EntryScope() { t_entry = prev; }
};

void* dalloc(size_t bytes, cudaStream_t s);  // NULL on failure (error recorded)
void dfree(void* p, cudaStream_t s);

// Temporary device buffers of one call: carved (256-byte aligned) from a few
// large chunks, freed stream-ordered on scope exit.
struct Scratch {
  cudaStream_t stream;
  std::vector<void*> ptrs;
  char* cur = nullptr;
  size_t left = 0;
  explicit Scratch(cudaStream_t s) : stream(s) {}
  ~Scratch() {
    for (void* p : ptrs) dfree(p, stream);
  }
  template <class T>
  T* get(size_t count) {
    const size_t bytes = (count * sizeof(T) + 16 + 255) & ~(size_t)255;
    if (bytes > left) {
      const size_t chunk = bytes > ((size_t)32 << 20) ? bytes : ((size_t)32 << 20);
      void* p = dalloc(chunk, stream);
      if (!p) return nullptr;
      ptrs.push_back(p);
      cur = (char*)p;
      left = chunk;
    }
    T* r = (T*)cur;
    cur += bytes;
    left -= bytes;
    return r;
  }
};

// Pinned host staging buffer reused by host<->device reads of small values.
void* pinned_staging(size_t bytes);

// ---------------------------------------------------------------- launches
// Counts every kernel launch and, when profiling is enabled for this kernel
// name, brackets it with CUDA events on its stream.
struct LaunchScope {
  const char* name;
  cudaStream_t stream;
  void* ev0;
  LaunchScope(const char* n, cudaStream_t s);
  ~LaunchScope();
};
fvx_status check_launch(const char* name);
// Streaming multiprocessors of the current device (queried once per device).
fvx_status device_sm_count(int* sms);
fvx_status check_staged_status(const char* who, uint32_t staged, cudaStream_t s);
// Kernel map pair lists are allocated for 27 pairs per output (no count
// read-back) up to this many bytes (environment FVX_KMAP_CAP_BYTES, default
// 8 GiB); larger maps read the count first and allocate it exactly.
size_t kmap_capacity_limit();
fvx_status kmap_read_totals(fvx_kmap_s* m, const char* who);

// Device status word written by bounded waits / device-side checks.
uint32_t* device_status_word();  // device pointer (per device, lazily set up)

enum : uint32_t { DEV_OK = 0, DEV_TIMEOUT = 1, DEV_CHECK = 2 };

// Test hooks (fvx_testing_bounded_wait): one bounded wait of each form on
// something nothing completes, giving up after limit_ns.
fvx_status testing_mbar_wait(unsigned long long limit_ns, uint32_t* status, cudaStream_t s);
fvx_status testing_flag_wait(const uint64_t* flag, unsigned long long limit_ns, uint32_t* status, cudaStream_t s);

// ---------------------------------------------------------------- primitives
// Exclusive scan of n uint32 values (in may equal out).  If total != NULL the
// grand total is written to total[0] (device).
fvx_status scan_exclusive_u32(const uint32_t* in, uint32_t* out, int64_t n, uint32_t* total, cudaStream_t s,
                              Scratch& scr);

// Exclusive scan of the popcounts of n uint64 words (bitmap rank offsets);
// total as above.
fvx_status scan_popc64(const uint64_t* words, uint32_t* out, int64_t n, uint32_t* total, cudaStream_t s,
                       Scratch& scr);

// Stable LSD radix sort of (key, value) pairs by key bits [bit_lo, bit_hi)
// with 8-bit digits.  Ping-pongs between (k0,v0) and (k1,v1); returns in
// *result_in_1 whether the sorted data ends in (k1,v1).
fvx_status radix_sort_pairs(uint64_t* k0, uint32_t* v0, uint64_t* k1, uint32_t* v1, int64_t n, int bit_lo,
                            int bit_hi, cudaStream_t s, bool* result_in_1, Scratch& scr);

}  // namespace fvx

// ---------------------------------------------------------------- handles
struct fvx_grid_s {
  int32_t B = 0;
  int64_t n_rows = 0, n_upper = 0, n_lower = 0, n_leaf = 0, n_active = 0;
  void* block = nullptr;  // single allocation holding every array below
  cudaStream_t stream = 0;
  int32_t* ijk = nullptr;
  int32_t* row_to_index = nullptr;
  int64_t* voxel_batch_offsets = nullptr;
  int32_t* leaf_origin = nullptr;
  int32_t* leaf_batch = nullptr;
  uint64_t* leaf_rec = nullptr;  // [n_leaf][10]
  int32_t* lower_origin = nullptr;
  int32_t* lower_batch = nullptr;
  uint64_t* lower_mask = nullptr;
  uint32_t* lower_prefix = nullptr;
  uint32_t* lower_first = nullptr;
  int32_t* upper_origin = nullptr;
  int32_t* upper_batch = nullptr;
  uint64_t* upper_mask = nullptr;
  uint32_t* upper_prefix = nullptr;
  uint32_t* upper_first = nullptr;
  int32_t* upper_tile = nullptr;  // [n_upper][4]: batch, tile i, tile j, tile k (root search keys)
  std::vector<int64_t> host_batch_offsets;  // filled lazily
};

struct fvx_kmap_s {
  int32_t stride = 1;
  bool transposed = false;  // map of the transposed convolution (see fvx_kernel_map_transposed)
  int64_t n_out = 0, n_pairs = 0;
  int64_t offsets_host[28] = {0};
  // the 28 list offsets on the device; copied to offsets_host / n_pairs on
  // the first request (host_ready), so building the map needs no sync
  uint32_t* dtot = nullptr;
  bool host_ready = false;
  int64_t pair_capacity = 0;  // pairs the in_idx / out_idx allocation holds
  void* block = nullptr;   // out_mask + tile_start
  void* block2 = nullptr;  // in_idx + out_idx
  cudaStream_t stream = 0;
  int32_t* in_idx = nullptr;
  int32_t* out_idx = nullptr;
  uint32_t* out_mask = nullptr;
  // conv tiling: for tiles of kTileRows consecutive outputs, tile_start[s*n_tiles + t]
  // is the position in in_idx of the first pair of list s with output >= t*kTileRows.
  uint32_t* tile_start = nullptr;
  int64_t n_tiles = 0;
  // stride 1: for each output leaf, the input leaf at each of the 27 leaf
  // offsets ((ex+1)*9 + (ey+1)*3 + ez+1, -1 if absent); null for stride 2.
  // A forward map keeps it in leaf_nbr, a transposed one in leaf_nbr_t (the
  // forward conv must not take a transposed map for a forward one).
  int32_t* leaf_nbr = nullptr;
  int32_t* leaf_nbr_t = nullptr;
  const fvx_grid_s* gin = nullptr;
  const fvx_grid_s* gout = nullptr;
};

namespace fvx {
constexpr int kTileRows = 128;  // conv output rows per tile (= tcgen05 M)

// Read-only device view of a grid used by lookups.
struct GridDev {
  int64_t n_upper, n_leaf, n_active;
  const int32_t* upper_tile;
  const uint64_t* upper_mask;
  const uint32_t* upper_prefix;
  const uint32_t* upper_first;
  const uint64_t* lower_mask;
  const uint32_t* lower_prefix;
  const uint32_t* lower_first;
  const uint64_t* leaf_rec;
  const int32_t* leaf_origin;
  const int32_t* leaf_batch;
};
inline GridDev grid_dev(const fvx_grid_s* g) {
  return GridDev{g->n_upper,    g->n_leaf,       g->n_active,     g->upper_tile, g->upper_mask,
                 g->upper_prefix, g->upper_first, g->lower_mask,   g->lower_prefix, g->lower_first,
                 g->leaf_rec,   g->leaf_origin,  g->leaf_batch};
}

// Builds a grid from DEVICE coords and DEVICE CSR offsets (used by the public
// build after uploading the offsets, and by coarsen).
fvx_status build_grid_device(const int32_t* coords, int64_t n_rows, const int64_t* batch_offsets_dev, int32_t B,
                             cudaStream_t s, fvx_grid_s** out);
}  // namespace fvx

// ---------------------------------------------------------------- device helpers
#ifdef __CUDACC__
namespace fvx {

// Tree walk from the root to the leaf holding (b, i, j, k); -1 if absent.
__device__ __forceinline__ int find_upper(const GridDev& g, int b, int ti, int tj, int tk) {
  int lo = 0, hi = (int)g.n_upper;  // upper_tile sorted by (b, ti, tj, tk)
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    const int4 t = reinterpret_cast<const int4*>(g.upper_tile)[mid];
    bool less = (t.x != b) ? (t.x < b) : (t.y != ti) ? (t.y < ti) : (t.z != tj) ? (t.z < tj) : (t.w < tk);
    if (less) lo = mid + 1; else hi = mid;
  }
  if (lo < (int)g.n_upper) {
    const int4 t = reinterpret_cast<const int4*>(g.upper_tile)[lo];
    if (t.x == b && t.y == ti && t.z == tj && t.w == tk) return lo;
  }
  return -1;
}

__device__ __forceinline__ int child_index(const uint64_t* mask, const uint32_t* prefix, uint32_t first, int n) {
  const int w = n >> 6, bit = n & 63;
  const uint64_t m = __ldg(reinterpret_cast<const unsigned long long*>(mask) + w);
  if (!((m >> bit) & 1ull)) return -1;
  return (int)(first + __ldg(prefix + w) + (uint32_t)__popcll(m & ((1ull << bit) - 1ull)));
}

// Leaf index of the leaf containing (i, j, k) in batch b, or -1.
__device__ __forceinline__ int find_leaf(const GridDev& g, int b, int i, int j, int k) {
  const int u = find_upper(g, b, i >> 12, j >> 12, k >> 12);
  if (u < 0) return -1;
  const int nu = ((((i >> 7) & 31) << 10) | (((j >> 7) & 31) << 5) | ((k >> 7) & 31));
  const int w = child_index(g.upper_mask + (size_t)u * 512, g.upper_prefix + (size_t)u * 512, __ldg(g.upper_first + u), nu);
  if (w < 0) return -1;
  const int nl = ((((i >> 3) & 15) << 8) | (((j >> 3) & 15) << 4) | ((k >> 3) & 15));
  return child_index(g.lower_mask + (size_t)w * 64, g.lower_prefix + (size_t)w * 64, __ldg(g.lower_first + w), nl);
}

// find_leaf for a leaf origin computed in 64 bits: -1 when it lies outside the
// int32 coordinate range (no grid holds such a leaf).
__device__ __forceinline__ int find_leaf_wide(const GridDev& g, int b, long long i, long long j, long long k) {
  const long long lo = -2147483648ll, hi = 2147483647ll;
  if (i < lo || i > hi || j < lo || j > hi || k < lo || k > hi) return -1;
  return find_leaf(g, b, (int)i, (int)j, (int)k);
}

// Index of voxel n (0..511) inside leaf record rec, or -1: two branches (bit
// inactive; word 0 has no prefix).
__device__ __forceinline__ int leaf_voxel_index(const uint64_t* rec, int n) {
  const int w = n >> 6, bit = n & 63;
  const uint64_t m = __ldg(reinterpret_cast<const unsigned long long*>(rec) + w);
  if (!((m >> bit) & 1ull)) return -1;
  const uint64_t first = __ldg(reinterpret_cast<const unsigned long long*>(rec) + 8);
  const uint64_t pre9 = __ldg(reinterpret_cast<const unsigned long long*>(rec) + 9);
  const uint32_t pre = w ? (uint32_t)((pre9 >> (9 * (w - 1))) & 511ull) : 0u;
  return (int)(first + pre + (uint32_t)__popcll(m & ((1ull << bit) - 1ull)));
}

__device__ __forceinline__ int lookup_index(const GridDev& g, int b, int i, int j, int k) {
  const int l = find_leaf(g, b, i, j, k);
  if (l < 0) return -1;
  return leaf_voxel_index(g.leaf_rec + (size_t)l * 10, ((i & 7) << 6) | ((j & 7) << 3) | (k & 7));
}

__device__ __forceinline__ void report_device_error(uint32_t* status, uint32_t code) {
  if (status) atomicCAS(status, 0u, code);
}

}  // namespace fvx
#endif
