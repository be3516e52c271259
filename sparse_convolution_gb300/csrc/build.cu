// GPU IndexGrid build, lookup and coarsening.
//
// Follows the build of "fVDB: A Deep-Learning Framework for Sparse, Large
// Scale, and High Performance Spatial Intelligence" (reading notes, section
// "GPU-accelerated IndexGrid build"):
//   1  N signed voxel coordinates i, j, k
//   2  a 64-bit key per coordinate from i, j, k shifted right by 12 bits
//      (the root tile), packed side by side
//   3  radix sort of the N keys
//   4  run-length encoding of the sorted keys (one run per root tile)
//   5  a unique 64-bit key per coordinate: run id + the offsets inside the
//      upper, lower and leaf node
//   6  radix sort of those keys
//   7-9  upper / lower / leaf / voxel counts from runs and unique keys
//   10-12  allocation from the counts, then top-down registration of nodes
//      and active-voxel bitmasks (80-byte leaves: "IndexGrid" section).
// Differences from the printed recipe (same result): the tile fields of the
// step-2 key use only as many bits as the data's tile range needs (so the batch
// index fits in the same key), and the step-5 key keeps only the offset bits
// that vary across the input (order-preserving bit compaction), so that the
// sorts run only over significant 8-bit digits.
#include <cuda_runtime.h>
#include <limits.h>
#include <string.h>

#include <algorithm>

#include "block_scan.cuh"
#include "fvx_internal.cuh"

namespace fvx {

namespace {

constexpr int kThreads = 256;

// 36-bit in-tile offset key, x-major inside each level:
//   [35:21] upper child (5+5+5)  [20:9] lower child (4+4+4)  [8:0] voxel (3+3+3)
__device__ __forceinline__ uint64_t offset_key(int i, int j, int k) {
  const uint64_t ui = (i >> 7) & 31, uj = (j >> 7) & 31, uk = (k >> 7) & 31;
  const uint64_t li = (i >> 3) & 15, lj = (j >> 3) & 15, lk = (k >> 3) & 15;
  const uint64_t vi = i & 7, vj = j & 7, vk = k & 7;
  return (ui << 31) | (uj << 26) | (uk << 21) | (li << 17) | (lj << 13) | (lk << 9) | (vi << 6) | (vj << 3) | vk;
}

struct BitRuns {  // contiguous runs of set bits of the varying-offset mask
  int n;
  uint8_t src[36], len[36], dst[36];
};

__device__ __forceinline__ uint64_t compact_bits(uint64_t x, const BitRuns& r) {
  uint64_t y = 0;
  for (int t = 0; t < r.n; ++t) y |= ((x >> r.src[t]) & ((1ull << r.len[t]) - 1ull)) << r.dst[t];
  return y;
}
__device__ __forceinline__ uint64_t expand_bits(uint64_t y, const BitRuns& r) {
  uint64_t x = 0;
  for (int t = 0; t < r.n; ++t) x |= ((y >> r.dst[t]) & ((1ull << r.len[t]) - 1ull)) << r.src[t];
  return x;
}

struct PlanDev {
  int32_t tmin[3];
  int32_t tmax[3];
  unsigned long long off_or, off_and;
};

struct Key1Layout {
  int w[3];  // bits per tile axis
  int32_t tmin[3];
  int tile_bits;  // w0 + w1 + w2
};

__device__ __forceinline__ int batch_of_row(const int64_t* __restrict__ offs, int B, int64_t r) {
  int lo = 0, hi = B;  // largest b with offs[b] <= r
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (__ldg((const long long*)offs + mid) <= r) lo = mid; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- step 2 planning
__global__ void k_plan_init(PlanDev* plan) {
  for (int a = 0; a < 3; ++a) {
    plan->tmin[a] = INT_MAX;
    plan->tmax[a] = INT_MIN;
  }
  plan->off_or = 0ull;
  plan->off_and = ~0ull;
}

__global__ void __launch_bounds__(kThreads) k_plan_reduce(const int32_t* __restrict__ coords, int64_t n,
                                                          PlanDev* __restrict__ plan) {
  int tmin[3] = {INT_MAX, INT_MAX, INT_MAX}, tmax[3] = {INT_MIN, INT_MIN, INT_MIN};
  unsigned long long o_or = 0ull, o_and = ~0ull;
  auto take = [&](int i, int j, int k) {
    const int t[3] = {i >> 12, j >> 12, k >> 12};
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      tmin[a] = min(tmin[a], t[a]);
      tmax[a] = max(tmax[a], t[a]);
    }
    const uint64_t o = offset_key(i, j, k);
    o_or |= o;
    o_and &= o;
  };
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(coords) & 15u) == 0u) {
    // four rows (three 16-byte loads) per thread and step
    const int64_t n4 = n >> 2;
    const int4* c4 = reinterpret_cast<const int4*>(coords);
    for (int64_t g = first; g < n4; g += stride) {
      const int4 a = __ldg(c4 + 3 * g), b = __ldg(c4 + 3 * g + 1), c = __ldg(c4 + 3 * g + 2);
      take(a.x, a.y, a.z);
      take(a.w, b.x, b.y);
      take(b.z, b.w, c.x);
      take(c.y, c.z, c.w);
    }
    for (int64_t r = 4 * n4 + first; r < n; r += stride) take(coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]);
  } else {
    for (int64_t r = first; r < n; r += stride) take(coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      tmin[a] = min(tmin[a], __shfl_xor_sync(0xffffffffu, tmin[a], d));
      tmax[a] = max(tmax[a], __shfl_xor_sync(0xffffffffu, tmax[a], d));
    }
    o_or |= __shfl_xor_sync(0xffffffffu, o_or, d);
    o_and &= __shfl_xor_sync(0xffffffffu, o_and, d);
  }
  // block reduction, then one set of atomics per block
  __shared__ int s_min[3][kThreads / 32], s_max[3][kThreads / 32];
  __shared__ unsigned long long s_or[kThreads / 32], s_and[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      s_min[a][warp] = tmin[a];
      s_max[a][warp] = tmax[a];
    }
    s_or[warp] = o_or;
    s_and[warp] = o_and;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) {
#pragma unroll
      for (int a = 0; a < 3; ++a) {
        tmin[a] = min(tmin[a], s_min[a][w]);
        tmax[a] = max(tmax[a], s_max[a][w]);
      }
      o_or |= s_or[w];
      o_and &= s_and[w];
    }
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      atomicMin(&plan->tmin[a], tmin[a]);
      atomicMax(&plan->tmax[a], tmax[a]);
    }
    atomicOr(&plan->off_or, o_or);
    atomicAnd(&plan->off_and, o_and);
  }
}

// ---------------------------------------------------------------- step 2 key
__global__ void __launch_bounds__(kThreads) k_key1(const int32_t* __restrict__ coords, int64_t n,
                                                   const int64_t* __restrict__ offs, int B, Key1Layout L,
                                                   uint64_t* __restrict__ key, uint32_t* __restrict__ val) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n) return;
  const int b = batch_of_row(offs, B, r);
  const uint64_t ti = (uint64_t)(uint32_t)((coords[3 * r] >> 12) - L.tmin[0]);
  const uint64_t tj = (uint64_t)(uint32_t)((coords[3 * r + 1] >> 12) - L.tmin[1]);
  const uint64_t tk = (uint64_t)(uint32_t)((coords[3 * r + 2] >> 12) - L.tmin[2]);
  key[r] = ((uint64_t)b << L.tile_bits) | (ti << (L.w[1] + L.w[2])) | (tj << L.w[2]) | tk;
  val[r] = (uint32_t)r;
}

// step 5 key when every row lies in one root tile of one batch (no step 2-4)
__global__ void __launch_bounds__(kThreads) k_key2_direct(const int32_t* __restrict__ coords, int64_t n,
                                                          const __grid_constant__ BitRuns runs, int4 tile0,
                                                          uint64_t* __restrict__ key, uint32_t* __restrict__ val,
                                                          int4* __restrict__ run_tile) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r == 0) run_tile[0] = tile0;
  if (r >= n) return;
  key[r] = compact_bits(offset_key(coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]), runs);
  val[r] = (uint32_t)r;
}

// step 5 key when every batch element lies in one root tile (the same one):
// the run of a row is its batch element, so key2 = batch above the compacted
// offsets, without the stage-1 sort and run numbering (run ids may skip
// empty batch elements; they only order keys and index run_tile)
__global__ void __launch_bounds__(kThreads) k_key2_batch(const int32_t* __restrict__ coords, int64_t n,
                                                         const int64_t* __restrict__ offs, int B,
                                                         const __grid_constant__ BitRuns runs, int vbits, int4 tile0,
                                                         uint64_t* __restrict__ key, uint32_t* __restrict__ val,
                                                         int4* __restrict__ run_tile) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r < B) run_tile[r] = make_int4((int)r, tile0.y, tile0.z, tile0.w);
  if (r >= n) return;
  const int b = batch_of_row(offs, B, r);
  key[r] = ((uint64_t)b << vbits) | compact_bits(offset_key(coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]), runs);
  val[r] = (uint32_t)r;
}

// ---------------------------------------------------------------- steps 3-6 by bitmap
// One batch in one root tile whose compacted offset key has at most
// kBitmapMaxBits varying bits: a presence bitmap over the whole key space
// (<= 32 MB, so it stays in L2) replaces the radix sort.  Set one bit per
// row, scan the words' popcounts, and the set bits in word order are the
// unique keys in canonical order; a row's index is the rank of its bit.
constexpr int kBitmapMaxBits = 28;

__global__ void __launch_bounds__(kThreads) k_bitmap_set(const int32_t* __restrict__ coords, int64_t n,
                                                         const __grid_constant__ BitRuns runs, int4 tile0,
                                                         unsigned long long* __restrict__ bm,
                                                         int4* __restrict__ run_tile) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r == 0) run_tile[0] = tile0;
  if (r >= n) return;
  const uint64_t key = compact_bits(offset_key(coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]), runs);
  atomicOr(bm + (key >> 6), 1ull << (key & 63));
}

// One thread per bitmap word; a block gathers the set bits of its 256 words in
// order in shared memory (32-bit keys: the key space has at most 28 bits) and
// writes them out as one contiguous, coalesced run of the key list.
__global__ void __launch_bounds__(kThreads) k_bitmap_emit(const uint64_t* __restrict__ bm,
                                                          const uint32_t* __restrict__ wpre, int64_t nwords,
                                                          uint64_t* __restrict__ keys) {
  extern __shared__ uint32_t skey[];  // kThreads * 64 entries at most
  __shared__ uint32_t tmp[33];
  const int64_t w0 = (int64_t)blockIdx.x * kThreads;
  const int64_t w = w0 + threadIdx.x;
  uint64_t m = (w < nwords) ? bm[w] : 0ull;
  uint32_t total;
  uint32_t pos = block_exclusive_scan<uint32_t>((uint32_t)__popcll(m), tmp, &total);
  while (m) {
    const int b = __ffsll((long long)m) - 1;
    skey[pos++] = ((uint32_t)w << 6) | (uint32_t)b;
    m &= m - 1ull;
  }
  __syncthreads();
  const uint32_t base = wpre[w0];
  for (uint32_t e = threadIdx.x; e < total; e += kThreads) keys[base + e] = skey[e];
}

// Index of every input row: the rank of its key's bit.
__global__ void __launch_bounds__(kThreads) k_bitmap_rank(const int32_t* __restrict__ coords, int64_t n,
                                                          const __grid_constant__ BitRuns runs,
                                                          const uint64_t* __restrict__ bm,
                                                          const uint32_t* __restrict__ wpre,
                                                          int32_t* __restrict__ row_to_index) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n) return;
  const uint64_t key = compact_bits(offset_key(coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]), runs);
  const uint64_t m = bm[key >> 6];
  row_to_index[r] = (int32_t)(wpre[key >> 6] + (uint32_t)__popcll(m & ((1ull << (key & 63)) - 1ull)));
}

// ---------------------------------------------------------------- step 4 RLE + step 5 key
constexpr int kFlagItems = 8;
constexpr int kFlagTile = kThreads * kFlagItems;  // 2048
// Flag passes over sorted keys: each warp takes 256 consecutive keys in 8
// rounds of 32 (coalesced loads, all issued up front); the previous key of
// lane 0 comes from the round before (or memory).
constexpr int kFlagRounds = kFlagTile / kThreads;  // 8 rounds of 32 per warp
static_assert(kFlagRounds * 32 * (kThreads / 32) == kFlagTile, "flag tile = warps x rounds x 32");

// A warp's keys k[r] (item wbase + 32 r + lane; 0 past n) and the key before
// each item (prev; unused for item 0).
__device__ __forceinline__ void warp_keys(const uint64_t* __restrict__ key, int64_t n, int64_t wbase, int lane,
                                          uint64_t (&k)[kFlagRounds], uint64_t (&prev)[kFlagRounds]) {
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    k[r] = (j < n) ? key[j] : 0ull;
  }
  const uint64_t before = (lane == 0 && wbase > 0 && wbase - 1 < n) ? key[wbase - 1] : 0ull;
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const uint64_t up = __shfl_up_sync(0xffffffffu, k[r], 1);
    const uint64_t last = __shfl_sync(0xffffffffu, r ? k[r - 1] : before, 31);
    prev[r] = (lane == 0) ? (r ? last : before) : up;
  }
}

// Block-wide exclusive offset of this warp's count plus the warp counts of
// the block (one value per warp, through shared memory).
__device__ __forceinline__ uint32_t warp_offset(uint32_t warp_total, uint32_t* sh, int warp, int lane,
                                                uint32_t* block_total) {
  if (lane == 0) sh[warp] = warp_total;
  __syncthreads();
  uint32_t off = 0, tot = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const uint32_t c = sh[w];
    off += (w < warp) ? c : 0u;
    tot += c;
  }
  if (block_total) *block_total = tot;
  return off;
}

__global__ void __launch_bounds__(kThreads) k_rle_count(const uint64_t* __restrict__ key, int64_t n,
                                                        uint32_t* __restrict__ partial) {
  __shared__ uint32_t sh[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wbase = (int64_t)blockIdx.x * kFlagTile + (int64_t)warp * (32 * kFlagRounds);
  uint64_t k[kFlagRounds], prev[kFlagRounds];
  warp_keys(key, n, wbase, lane, k, prev);
  uint32_t c = 0;
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    c += __popc(__ballot_sync(0xffffffffu, j < n && (j == 0 || k[r] != prev[r])));
  }
  uint32_t tot;
  warp_offset(c, sh, warp, lane, &tot);
  if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kThreads) k_rle_key2(const uint64_t* __restrict__ key1, int64_t n,
                                                       const uint32_t* __restrict__ val,
                                                       const int32_t* __restrict__ coords,
                                                       const uint32_t* __restrict__ partial, Key1Layout L,
                                                       int vbits, const __grid_constant__ BitRuns runs,
                                                       uint64_t* __restrict__ key2, int4* __restrict__ run_tile) {
  __shared__ uint32_t sh[kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wbase = (int64_t)blockIdx.x * kFlagTile + (int64_t)warp * (32 * kFlagRounds);
  uint64_t k[kFlagRounds], prev[kFlagRounds];
  uint32_t v[kFlagRounds];
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    v[r] = (j < n) ? val[j] : 0u;
  }
  warp_keys(key1, n, wbase, lane, k, prev);
  uint32_t c = 0;
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    c += __popc(__ballot_sync(0xffffffffu, j < n && (j == 0 || k[r] != prev[r])));
  }
  uint32_t run = partial[blockIdx.x] + warp_offset(c, sh, warp, lane, nullptr);  // heads before this warp
  const uint32_t lt = lanemask_lt();
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    const bool head = j < n && (j == 0 || k[r] != prev[r]);
    const uint32_t bal = __ballot_sync(0xffffffffu, head);
    const uint32_t mine = run + __popc(bal & lt) + (head ? 1u : 0u);  // inclusive: run id + 1
    run += __popc(bal);
    if (j >= n) continue;
    const uint32_t rr = v[r];
    const uint64_t o = offset_key(coords[3 * (int64_t)rr], coords[3 * (int64_t)rr + 1], coords[3 * (int64_t)rr + 2]);
    key2[j] = ((uint64_t)(mine - 1) << vbits) | compact_bits(o, runs);
    if (head) {
      const uint64_t k1 = k[r];
      const int w12 = L.w[1] + L.w[2];
      int4 t;
      t.x = (int)(k1 >> L.tile_bits);
      t.y = (int)((k1 >> w12) & ((1ull << L.w[0]) - 1ull)) + L.tmin[0];
      t.z = (int)((k1 >> L.w[2]) & ((1ull << L.w[1]) - 1ull)) + L.tmin[1];
      t.w = (int)(k1 & ((1ull << L.w[2]) - 1ull)) + L.tmin[2];
      run_tile[mine - 1] = t;
    }
  }
}

// ---------------------------------------------------------------- steps 7-9 counts
struct Shifts {
  int leaf, lower, upper;  // key2 >> shift identifies leaf / lower / upper node
};

// Head flags of the sorted key2 per item: bit 0 new voxel, bit 1 new leaf,
// bit 2 new lower node, bit 3 new upper node.

__device__ __forceinline__ uint32_t flags_of(uint64_t a, uint64_t b, bool first, Shifts sh) {
  if (first) return 0xFu;
  return (a != b ? 1u : 0u) | (((a >> sh.leaf) != (b >> sh.leaf)) ? 2u : 0u) |
         (((a >> sh.lower) != (b >> sh.lower)) ? 4u : 0u) | (((a >> sh.upper) != (b >> sh.upper)) ? 8u : 0u);
}

// A warp's 256 keys and their head flags; items past n get flags 0.
__device__ __forceinline__ void warp_flags(const uint64_t* __restrict__ key, int64_t n, int64_t wbase, Shifts sh,
                                           int lane, uint64_t (&k)[kFlagRounds], uint32_t (&fl)[kFlagRounds]) {
  uint64_t prev[kFlagRounds];
  warp_keys(key, n, wbase, lane, k, prev);
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    fl[r] = (j < n) ? flags_of(k[r], prev[r], j == 0, sh) : 0u;
  }
}

// n_live (device, may be NULL): the key list is only that long (<= n).
__global__ void __launch_bounds__(kThreads) k_count_tiles(const uint64_t* __restrict__ key, int64_t n,
                                                          const uint32_t* __restrict__ n_live, Shifts sh,
                                                          uint32_t* __restrict__ partial, int64_t ntiles) {
  __shared__ uint32_t wt[kThreads / 32][4];
  if (n_live) n = min(n, (int64_t)*n_live);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wbase = (int64_t)blockIdx.x * kFlagTile + (int64_t)warp * (32 * kFlagRounds);
  uint64_t k[kFlagRounds];
  uint32_t fl[kFlagRounds];
  warp_flags(key, n, wbase, sh, lane, k, fl);
  uint32_t tot[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r)
#pragma unroll
    for (int f = 0; f < 4; ++f) tot[f] += __popc(__ballot_sync(0xffffffffu, (fl[r] >> f) & 1u));
  if (lane < 4) wt[warp][lane] = tot[0] * (lane == 0) + tot[1] * (lane == 1) + tot[2] * (lane == 2) + tot[3] * (lane == 3);
  __syncthreads();
  if (threadIdx.x < 4) {
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) c += wt[w][threadIdx.x];
    partial[threadIdx.x * ntiles + blockIdx.x] = c;
  }
}

__global__ void k_gather_counts(const uint32_t* __restrict__ scanned, int64_t ntiles, const uint32_t* total,
                                uint32_t* __restrict__ out) {
  // out[f] = count of head flag f = (row f+1 base) - (row f base); last row to the total
  if (threadIdx.x < 4) {
    const uint32_t lo = scanned[threadIdx.x * ntiles];
    const uint32_t hi = threadIdx.x < 3 ? scanned[(threadIdx.x + 1) * ntiles] : *total;
    out[threadIdx.x] = hi - lo;
  }
}

struct DecodeInfo {
  int vbits;
  uint64_t const_bits;  // offset bits that do not vary (their common value)
};

struct BuildOut {
  int32_t* ijk;
  int32_t* row_to_index;
  uint32_t* leaf_first_voxel;
  int32_t* leaf_origin;
  int32_t* leaf_batch;
  uint32_t* lower_first;
  int32_t* lower_origin;
  int32_t* lower_batch;
  uint32_t* upper_first;
  uint32_t* upper_first_voxel;
  int32_t* upper_origin;
  int32_t* upper_batch;
  int4* upper_tile;
  uint64_t* lower_mask;
  uint64_t* upper_mask;
};

// val (row id of each key) may be NULL: row_to_index is then written
// elsewhere (bitmap path, where the keys are already unique).
__global__ void __launch_bounds__(kThreads, 3) k_count_down(const uint64_t* __restrict__ key,
                                                         const uint32_t* __restrict__ val, int64_t n,
                                                         const uint32_t* __restrict__ n_live, Shifts sh,
                                                         const uint32_t* __restrict__ scanned, int64_t ntiles,
                                                         const __grid_constant__ BitRuns runs, DecodeInfo dec,
                                                         const int4* __restrict__ run_tile, BuildOut o) {
  __shared__ uint32_t wt[kThreads / 32][4];
  if (n_live) n = min(n, (int64_t)*n_live);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wbase = (int64_t)blockIdx.x * kFlagTile + (int64_t)warp * (32 * kFlagRounds);
  uint64_t k[kFlagRounds];
  uint32_t fl[kFlagRounds];
  uint32_t v[kFlagRounds];
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    v[r] = (j < n && val) ? val[j] : 0u;
  }
  warp_flags(key, n, wbase, sh, lane, k, fl);
  // warp totals of each flag to shared memory
  uint32_t tot[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r)
#pragma unroll
    for (int f = 0; f < 4; ++f) tot[f] += __popc(__ballot_sync(0xffffffffu, (fl[r] >> f) & 1u));
  if (lane < 4) wt[warp][lane] = tot[0] * (lane == 0) + tot[1] * (lane == 1) + tot[2] * (lane == 2) + tot[3] * (lane == 3);
  __syncthreads();
  // running (exclusive) count of each flag before this warp's first item
  uint32_t cnt[4];
#pragma unroll
  for (int f = 0; f < 4; ++f) {
    uint32_t c = scanned[f * ntiles + blockIdx.x] - scanned[f * ntiles];
    for (int w = 0; w < warp; ++w) c += wt[w][f];
    cnt[f] = c;
  }
  const uint32_t lt = lanemask_lt();
#pragma unroll
  for (int r = 0; r < kFlagRounds; ++r) {
    const int64_t j = wbase + 32 * r + lane;
    const uint32_t f = fl[r];
    uint32_t bal[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) bal[q] = __ballot_sync(0xffffffffu, (f >> q) & 1u);
    // inclusive count of each flag up to this item, minus one = its node index
    const uint32_t vox = cnt[0] + __popc(bal[0] & lt) + (f & 1u) - 1u;
    const uint32_t leaf = cnt[1] + __popc(bal[1] & lt) + ((f >> 1) & 1u) - 1u;
    const uint32_t lower = cnt[2] + __popc(bal[2] & lt) + ((f >> 2) & 1u) - 1u;
    const uint32_t upper = cnt[3] + __popc(bal[3] & lt) + ((f >> 3) & 1u) - 1u;
#pragma unroll
    for (int q = 0; q < 4; ++q) cnt[q] += __popc(bal[q]);
    if (j >= n) continue;
    if (val) o.row_to_index[v[r]] = (int32_t)vox;
    if (!(f & 1u)) continue;
    const uint64_t k2 = k[r];
    const uint64_t off = expand_bits(k2 & ((1ull << dec.vbits) - 1ull), runs) | dec.const_bits;
    const int4 t = run_tile[(uint32_t)(k2 >> dec.vbits)];
    const int ci = t.y * 4096 + (int)(((off >> 31) & 31) << 7 | ((off >> 17) & 15) << 3 | ((off >> 6) & 7));
    const int cj = t.z * 4096 + (int)(((off >> 26) & 31) << 7 | ((off >> 13) & 15) << 3 | ((off >> 3) & 7));
    const int ck = t.w * 4096 + (int)(((off >> 21) & 31) << 7 | ((off >> 9) & 15) << 3 | (off & 7));
    o.ijk[3 * (int64_t)vox] = ci;
    o.ijk[3 * (int64_t)vox + 1] = cj;
    o.ijk[3 * (int64_t)vox + 2] = ck;
    if (f & 2u) {
      o.leaf_first_voxel[leaf] = vox;
      o.leaf_origin[3 * (int64_t)leaf] = ci & ~7;
      o.leaf_origin[3 * (int64_t)leaf + 1] = cj & ~7;
      o.leaf_origin[3 * (int64_t)leaf + 2] = ck & ~7;
      o.leaf_batch[leaf] = t.x;
      // the new leaf is a child of its lower node (masks zeroed before)
      const int nb = (((ci >> 3) & 15) << 8) | (((cj >> 3) & 15) << 4) | ((ck >> 3) & 15);
      atomicOr(reinterpret_cast<unsigned long long*>(o.lower_mask) + (int64_t)lower * 64 + (nb >> 6), 1ull << (nb & 63));
    }
    if (f & 4u) {
      o.lower_first[lower] = leaf;
      o.lower_origin[3 * (int64_t)lower] = ci & ~127;
      o.lower_origin[3 * (int64_t)lower + 1] = cj & ~127;
      o.lower_origin[3 * (int64_t)lower + 2] = ck & ~127;
      o.lower_batch[lower] = t.x;
      const int nb = (((ci >> 7) & 31) << 10) | (((cj >> 7) & 31) << 5) | ((ck >> 7) & 31);
      atomicOr(reinterpret_cast<unsigned long long*>(o.upper_mask) + (int64_t)upper * 512 + (nb >> 6), 1ull << (nb & 63));
    }
    if (f & 8u) {
      o.upper_first[upper] = lower;
      o.upper_first_voxel[upper] = vox;
      o.upper_origin[3 * (int64_t)upper] = t.y * 4096;
      o.upper_origin[3 * (int64_t)upper + 1] = t.z * 4096;
      o.upper_origin[3 * (int64_t)upper + 2] = t.w * 4096;
      o.upper_batch[upper] = t.x;
      o.upper_tile[upper] = t;
    }
  }
}

// ---------------------------------------------------------------- steps 10-12 registration
// One warp per leaf: 8 mask words from its voxels, first index, packed prefix.
__global__ void __launch_bounds__(kThreads) k_leaf_register(const int32_t* __restrict__ ijk,
                                                            const uint32_t* __restrict__ leaf_first_voxel,
                                                            int64_t n_leaf, int64_t n_active,
                                                            uint64_t* __restrict__ rec) {
  const int64_t l = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (l >= n_leaf) return;
  const uint32_t first = leaf_first_voxel[l];
  const uint32_t end = (l + 1 < n_leaf) ? leaf_first_voxel[l + 1] : (uint32_t)n_active;
  uint64_t m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (uint32_t t = first + lane; t < end; t += 32) {
    const int i = ijk[3 * (int64_t)t], j = ijk[3 * (int64_t)t + 1], k = ijk[3 * (int64_t)t + 2];
    const int w = i & 7;
    const uint64_t bit = 1ull << (((j & 7) << 3) | (k & 7));
#pragma unroll
    for (int q = 0; q < 8; ++q) m[q] |= (q == w) ? bit : 0ull;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m[q] |= __shfl_xor_sync(0xffffffffu, m[q], d);
  }
  uint64_t packed = 0, acc = 0;
#pragma unroll
  for (int w = 1; w < 8; ++w) {
    acc += (uint64_t)__popcll(m[w - 1]);
    packed |= acc << (9 * (w - 1));
  }
  uint64_t v = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) v = (lane == q) ? m[q] : v;
  if (lane == 8) v = first;
  if (lane == 9) v = packed;
  if (lane < 10) rec[l * 10 + lane] = v;
}

// Per-word exclusive popcount prefix of the lower-node child masks (one warp
// per node, 64 words); the masks themselves are set in k_count_down.
__global__ void __launch_bounds__(kThreads) k_lower_prefix(const uint64_t* __restrict__ mask, int64_t n_lower,
                                                           uint32_t* __restrict__ prefix) {
  const int lane = threadIdx.x & 31;
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (w >= n_lower) return;
  const unsigned long long* m = reinterpret_cast<const unsigned long long*>(mask) + w * 64;
  const uint32_t pa = __popcll(m[2 * lane]), pb = __popcll(m[2 * lane + 1]);
  const uint32_t ex = warp_inclusive_scan<uint32_t>(pa + pb) - (pa + pb);
  prefix[w * 64 + 2 * lane] = ex;
  prefix[w * 64 + 2 * lane + 1] = ex + pa;
}

// Same for the upper-node masks (one block per node, 512 words).
__global__ void __launch_bounds__(kThreads) k_upper_prefix(const uint64_t* __restrict__ mask,
                                                           uint32_t* __restrict__ prefix) {
  __shared__ uint32_t tmp[33];
  const int64_t u = blockIdx.x;
  const unsigned long long* m = reinterpret_cast<const unsigned long long*>(mask) + u * 512;
  const uint32_t pa = __popcll(m[2 * threadIdx.x]), pb = __popcll(m[2 * threadIdx.x + 1]);
  const uint32_t ex = block_exclusive_scan<uint32_t>(pa + pb, tmp, (uint32_t*)nullptr);
  prefix[u * 512 + 2 * threadIdx.x] = ex;
  prefix[u * 512 + 2 * threadIdx.x + 1] = ex + pa;
}

__global__ void k_batch_offsets(const int4* __restrict__ upper_tile, const uint32_t* __restrict__ upper_first_voxel,
                                int64_t n_upper, int64_t n_active, int B, int64_t* __restrict__ vbo) {
  for (int b = threadIdx.x; b <= B; b += blockDim.x) {
    int lo = 0, hi = (int)n_upper;  // first upper node with batch >= b
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (upper_tile[mid].x < b) lo = mid + 1; else hi = mid;
    }
    vbo[b] = (lo < n_upper) ? (int64_t)upper_first_voxel[lo] : n_active;
  }
}

__global__ void k_lookup(GridDev g, const int32_t* __restrict__ coords, const int32_t* __restrict__ batch, int64_t n,
                         int32_t* __restrict__ out) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n) return;
  const int b = batch ? batch[r] : 0;
  out[r] = lookup_index(g, b, coords[3 * r], coords[3 * r + 1], coords[3 * r + 2]);
}

__global__ void k_coarsen_coords(const int32_t* __restrict__ ijk, int64_t n, int stride, int shift,
                                 int32_t* __restrict__ out) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= 3 * n) return;
  const int c = ijk[t];
  if (shift >= 0) {
    out[t] = c >> shift;  // floor division by a power of two
  } else {
    int q = c / stride;
    if ((c % stride) != 0 && c < 0) q -= 1;
    out[t] = q;
  }
}

// Children of every voxel for the refined grid: row t*f^3 + c holds
// factor * ijk[t] + (c / f^2, (c / f) % f, c % f).  A coordinate that does not
// fit int32 is recorded in the status word (the build reports it).
__global__ void k_refine_coords(const int32_t* __restrict__ ijk, int64_t n, int factor, int32_t* __restrict__ out,
                                uint32_t* status) {
  const int64_t f3 = (int64_t)factor * factor * factor;
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n * f3) return;
  const int64_t t = r / f3;
  const int c = (int)(r - t * f3);
  const int ch[3] = {c / (factor * factor), (c / factor) % factor, c % factor};
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    const int64_t v = (int64_t)factor * ijk[3 * t + a] + ch[a];
    if (v < INT32_MIN || v > INT32_MAX) report_device_error(status, DEV_CHECK);
    out[3 * r + a] = (int32_t)v;
  }
}

__global__ void k_scale_offsets(const int64_t* __restrict__ in, int n, int64_t f, int64_t* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = in[i] * f;
}

int bits_for(uint64_t maxval) {  // bits needed to represent 0..maxval
  int b = 0;
  while (b < 64 && (maxval >> b) != 0) ++b;
  return b;
}

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

unsigned grid_for(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

fvx_status build_grid_device(const int32_t* coords, int64_t n, const int64_t* offs_dev, int32_t B, cudaStream_t s,
                             fvx_grid_s** out) {
  Scratch scr(s);
  fvx_grid_s* g = new fvx_grid_s();
  g->B = B;
  g->n_rows = n;
  g->stream = s;
  struct Guard {
    fvx_grid_s** g;
    ~Guard() {
      if (*g) fvx_grid_destroy(*g);
    }
  } guard{&g};

  int64_t counts[4] = {0, 0, 0, 0};  // voxels, leaves, lower, upper
  uint64_t* ka = nullptr;
  uint32_t* va = nullptr;
  Shifts sh{0, 0, 0};
  BitRuns runs{};
  DecodeInfo dec{0, 0};
  int4* run_tile = nullptr;
  uint32_t* scanned = nullptr;
  int64_t ntiles = 0;
  bool use_bitmap = false;
  uint64_t* bm = nullptr;       // bitmap path: presence bitmap of the key space
  uint32_t* bm_pre = nullptr;   // exclusive popcount prefix of its words (+ total)
  uint32_t* n_live = nullptr;   // device: unique keys (the sorted list's length)
  int64_t bm_words = 0;

  if (n > 0) {
    // ---- step 2 planning: tile range per axis and the varying offset bits
    PlanDev* plan = scr.get<PlanDev>(1);
    if (!plan) return FVX_ERR_ALLOC;
    PlanDev* hp = (PlanDev*)pinned_staging(sizeof(PlanDev));
    if (!hp) {
      set_error("fvx_build_grid: pinned staging allocation failed");
      return FVX_ERR_ALLOC;
    }
    {
      LaunchScope ls("build_plan_init", s);
      k_plan_init<<<1, 1, 0, s>>>(plan);
    }
    FVX_TRY(check_launch("build_plan_init"));
    {
      LaunchScope ls("build_plan_reduce", s);
      int sms = 0;
      FVX_TRY(device_sm_count(&sms));
      unsigned nb = std::min<unsigned>(grid_for((n + 3) / 4, kThreads), (unsigned)sms * 8u);
      k_plan_reduce<<<nb, kThreads, 0, s>>>(coords, n, plan);
    }
    FVX_TRY(check_launch("build_plan_reduce"));
    FVX_CUDA(cudaMemcpyAsync(hp, plan, sizeof(PlanDev), cudaMemcpyDeviceToHost, s));
    FVX_CUDA(cudaStreamSynchronize(s));
    const PlanDev P = *hp;

    Key1Layout L{};
    for (int a = 0; a < 3; ++a) {
      L.tmin[a] = P.tmin[a];
      L.w[a] = bits_for((uint64_t)((int64_t)P.tmax[a] - (int64_t)P.tmin[a]));
    }
    L.tile_bits = L.w[0] + L.w[1] + L.w[2];
    const int width1 = L.tile_bits + bits_for((uint64_t)(B - 1));
    if (width1 > 64) {
      set_error("fvx_build_grid: batch size %d with tile range needs a %d-bit key (max 64)", B, width1);
      return FVX_ERR_RANGE;
    }
    const uint64_t vm = P.off_or & ~P.off_and;
    runs.n = 0;
    int dst = 0;
    for (int b = 0; b < 36;) {
      if (!((vm >> b) & 1ull)) {
        ++b;
        continue;
      }
      int e = b;
      while (e < 36 && ((vm >> e) & 1ull)) ++e;
      runs.src[runs.n] = (uint8_t)b;
      runs.len[runs.n] = (uint8_t)(e - b);
      runs.dst[runs.n] = (uint8_t)dst;
      ++runs.n;
      dst += e - b;
      b = e;
    }
    const int vbits = dst;
    dec.vbits = vbits;
    dec.const_bits = P.off_and & ~vm;
    sh.leaf = __builtin_popcountll(vm & 0x1FFull);
    sh.lower = __builtin_popcountll(vm & 0x1FFFFFull);
    sh.upper = vbits;
    // runs: (batch, tile) pairs present, or with a single tile the batch
    // elements themselves (run id = batch index)
    const uint64_t max_runs = (width1 > 0 && L.tile_bits == 0) ? (uint64_t)B
                              : (width1 >= 63)                 ? (uint64_t)n
                                                               : std::min<uint64_t>((uint64_t)n, 1ull << width1);
    const int runbits = bits_for(max_runs - 1);
    if (runbits + vbits > 64) {
      set_error("fvx_build_grid: %d rows spread over too many root tiles for a 64-bit key", (int)n);
      return FVX_ERR_RANGE;
    }

    use_bitmap = (width1 == 0) && vbits <= kBitmapMaxBits;
    ka = scr.get<uint64_t>((size_t)n);
    va = scr.get<uint32_t>((size_t)n);
    uint64_t* kb = scr.get<uint64_t>((size_t)n);
    uint32_t* vb = scr.get<uint32_t>((size_t)n);
    run_tile = scr.get<int4>((size_t)max_runs);
    if (!ka || !va || !kb || !vb || !run_tile) return FVX_ERR_ALLOC;

    if (use_bitmap) {
      // one batch, one root tile, a key space that fits L2: bitmap instead of sort
      const int4 tile0 = make_int4(0, P.tmin[0], P.tmin[1], P.tmin[2]);
      bm_words = ((int64_t)1 << vbits) > 64 ? ((int64_t)1 << vbits) / 64 : 1;
      bm = scr.get<uint64_t>((size_t)bm_words);
      bm_pre = scr.get<uint32_t>((size_t)bm_words + 1);
      if (!bm || !bm_pre) return FVX_ERR_ALLOC;
      n_live = bm_pre + bm_words;  // the scan's total: number of unique keys
      FVX_CUDA(cudaMemsetAsync(bm, 0, 8 * (size_t)bm_words, s));
      {
        LaunchScope ls("build_bitmap_set", s);
        k_bitmap_set<<<grid_for(n, kThreads), kThreads, 0, s>>>(coords, n, runs, tile0,
                                                                (unsigned long long*)bm, run_tile);
      }
      FVX_TRY(check_launch("build_bitmap_set"));
      FVX_TRY(scan_popc64(bm, bm_pre, bm_words, n_live, s, scr));
      {
        LaunchScope ls("build_bitmap_emit", s);
        FVX_CUDA(cudaFuncSetAttribute(k_bitmap_emit, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kThreads * 64 * 4));
        k_bitmap_emit<<<grid_for(bm_words, kThreads), kThreads, kThreads * 64 * 4, s>>>(bm, bm_pre, bm_words, ka);
      }
      FVX_TRY(check_launch("build_bitmap_emit"));
    } else if (width1 == 0) {
      // one batch, one root tile: steps 2-4 are empty; run 0 is that tile
      const int4 tile0 = make_int4(0, P.tmin[0], P.tmin[1], P.tmin[2]);
      {
        LaunchScope ls("build_key2_direct", s);
        k_key2_direct<<<grid_for(n, kThreads), kThreads, 0, s>>>(coords, n, runs, tile0, ka, va, run_tile);
      }
      FVX_TRY(check_launch("build_key2_direct"));
    } else if (L.tile_bits == 0) {
      // several batch elements, all in the one root tile: run = batch
      const int4 tile0 = make_int4(0, P.tmin[0], P.tmin[1], P.tmin[2]);
      {
        LaunchScope ls("build_key2_batch", s);
        k_key2_batch<<<grid_for(std::max<int64_t>(n, B), kThreads), kThreads, 0, s>>>(coords, n, offs_dev, B, runs,
                                                                                        vbits, tile0, ka, va, run_tile);
      }
      FVX_TRY(check_launch("build_key2_batch"));
    } else {
      {
        LaunchScope ls("build_key1", s);
        k_key1<<<grid_for(n, kThreads), kThreads, 0, s>>>(coords, n, offs_dev, B, L, ka, va);
      }
      FVX_TRY(check_launch("build_key1"));
      bool in1 = false;
      FVX_TRY(radix_sort_pairs(ka, va, kb, vb, n, 0, width1, s, &in1, scr));
      uint64_t* k1 = in1 ? kb : ka;
      uint32_t* v1 = in1 ? vb : va;
      uint64_t* k2 = in1 ? ka : kb;  // the other key buffer receives key2
      const int64_t nt = (n + kFlagTile - 1) / kFlagTile;
      uint32_t* partial = scr.get<uint32_t>((size_t)nt);
      if (!partial) return FVX_ERR_ALLOC;
      {
        LaunchScope ls("build_rle_count", s);
        k_rle_count<<<(unsigned)nt, kThreads, 0, s>>>(k1, n, partial);
      }
      FVX_TRY(check_launch("build_rle_count"));
      FVX_TRY(scan_exclusive_u32(partial, partial, nt, nullptr, s, scr));
      {
        LaunchScope ls("build_rle_key2", s);
        k_rle_key2<<<(unsigned)nt, kThreads, 0, s>>>(k1, n, v1, coords, partial, L, vbits, runs, k2, run_tile);
      }
      FVX_TRY(check_launch("build_rle_key2"));
      // arrange so that (ka, va) hold key2 and the row ids
      if (in1) {
        // key2 in ka, rows in vb
        std::swap(va, vb);
      } else {
        // key2 in kb, rows in va
        std::swap(ka, kb);
      }
    }
    // ---- step 6: sort by key2 (run id above the compacted offsets)
    if (!use_bitmap) {
      bool in1 = false;
      FVX_TRY(radix_sort_pairs(ka, va, kb, vb, n, 0, runbits + vbits, s, &in1, scr));
      if (in1) {
        ka = kb;
        va = vb;
      }
    }
    // ---- steps 7-9: node counts
    ntiles = (n + kFlagTile - 1) / kFlagTile;
    scanned = scr.get<uint32_t>((size_t)(4 * ntiles));
    uint32_t* dcounts = scr.get<uint32_t>(8);
    if (!scanned || !dcounts) return FVX_ERR_ALLOC;
    {
      LaunchScope ls("build_count_tiles", s);
      k_count_tiles<<<(unsigned)ntiles, kThreads, 0, s>>>(ka, n, n_live, sh, scanned, ntiles);
    }
    FVX_TRY(check_launch("build_count_tiles"));
    FVX_TRY(scan_exclusive_u32(scanned, scanned, 4 * ntiles, dcounts + 4, s, scr));
    {
      LaunchScope ls("build_gather_counts", s);
      k_gather_counts<<<1, 32, 0, s>>>(scanned, ntiles, dcounts + 4, dcounts);
    }
    FVX_TRY(check_launch("build_gather_counts"));
    uint32_t* hc = (uint32_t*)pinned_staging(20);
    uint32_t* dstat = device_status_word();
    if (!hc || !dstat) {
      set_error("fvx_build_grid: staging buffer or device status word unavailable");
      return FVX_ERR_ALLOC;
    }
    FVX_CUDA(cudaMemcpyAsync(hc, dcounts, 16, cudaMemcpyDeviceToHost, s));
    FVX_CUDA(cudaMemcpyAsync(hc + 4, dstat, 4, cudaMemcpyDeviceToHost, s));
    FVX_CUDA(cudaStreamSynchronize(s));
    FVX_TRY(check_staged_status("fvx_build_grid", hc[4], s));
    for (int f = 0; f < 4; ++f) counts[f] = hc[f];
  }

  // ---- step 10: allocate the topology from the counts
  g->n_active = counts[0];
  g->n_leaf = counts[1];
  g->n_lower = counts[2];
  g->n_upper = counts[3];
  const int64_t U = g->n_active, Lf = g->n_leaf, NL = g->n_lower, NU = g->n_upper;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += align_up(bytes);
    return o;
  };
  const size_t o_ijk = take(12 * U), o_r2i = take(4 * n), o_vbo = take(8 * (B + 1));
  const size_t o_lfo = take(12 * Lf), o_lfb = take(4 * Lf), o_lfr = take(80 * Lf);
  const size_t o_lwo = take(12 * NL), o_lwb = take(4 * NL), o_lwm = take(512 * NL), o_lwp = take(256 * NL),
               o_lwf = take(4 * NL);
  const size_t o_upo = take(12 * NU), o_upb = take(4 * NU), o_upm = take(4096 * NU), o_upp = take(2048 * NU),
               o_upf = take(4 * NU), o_upt = take(16 * NU);
  g->block = dalloc(off, s);
  if (!g->block) return FVX_ERR_ALLOC;
  char* base = (char*)g->block;
  g->ijk = (int32_t*)(base + o_ijk);
  g->row_to_index = (int32_t*)(base + o_r2i);
  g->voxel_batch_offsets = (int64_t*)(base + o_vbo);
  g->leaf_origin = (int32_t*)(base + o_lfo);
  g->leaf_batch = (int32_t*)(base + o_lfb);
  g->leaf_rec = (uint64_t*)(base + o_lfr);
  g->lower_origin = (int32_t*)(base + o_lwo);
  g->lower_batch = (int32_t*)(base + o_lwb);
  g->lower_mask = (uint64_t*)(base + o_lwm);
  g->lower_prefix = (uint32_t*)(base + o_lwp);
  g->lower_first = (uint32_t*)(base + o_lwf);
  g->upper_origin = (int32_t*)(base + o_upo);
  g->upper_batch = (int32_t*)(base + o_upb);
  g->upper_mask = (uint64_t*)(base + o_upm);
  g->upper_prefix = (uint32_t*)(base + o_upp);
  g->upper_first = (uint32_t*)(base + o_upf);
  g->upper_tile = (int32_t*)(base + o_upt);

  if (n == 0) {
    FVX_CUDA(cudaMemsetAsync(g->voxel_batch_offsets, 0, 8 * (B + 1), s));
  } else {
    uint32_t* leaf_first_voxel = scr.get<uint32_t>((size_t)Lf);
    uint32_t* upper_first_voxel = scr.get<uint32_t>((size_t)NU);
    if (!leaf_first_voxel || !upper_first_voxel) return FVX_ERR_ALLOC;
    BuildOut o{g->ijk,          g->row_to_index, leaf_first_voxel, g->leaf_origin,  g->leaf_batch,
               g->lower_first,  g->lower_origin, g->lower_batch,   g->upper_first,  upper_first_voxel,
               g->upper_origin, g->upper_batch,  (int4*)g->upper_tile, g->lower_mask, g->upper_mask};
    FVX_CUDA(cudaMemsetAsync(g->lower_mask, 0, 512 * (size_t)NL, s));
    FVX_CUDA(cudaMemsetAsync(g->upper_mask, 0, 4096 * (size_t)NU, s));
    {
      LaunchScope ls("build_count_down", s);
      k_count_down<<<(unsigned)ntiles, kThreads, 0, s>>>(ka, use_bitmap ? nullptr : va, n, n_live, sh, scanned,
                                                         ntiles, runs, dec, run_tile, o);
    }
    FVX_TRY(check_launch("build_count_down"));
    if (use_bitmap) {
      LaunchScope ls("build_bitmap_rank", s);
      k_bitmap_rank<<<grid_for(n, kThreads), kThreads, 0, s>>>(coords, n, runs, bm, bm_pre, g->row_to_index);
    }
    FVX_TRY(check_launch("build_bitmap_rank"));
    // ---- steps 11-12: leaf masks and prefix counts at every level
    {
      LaunchScope ls("build_leaf_register", s);
      k_leaf_register<<<grid_for(Lf * 32, kThreads), kThreads, 0, s>>>(g->ijk, leaf_first_voxel, Lf, U, g->leaf_rec);
    }
    FVX_TRY(check_launch("build_leaf_register"));
    {
      LaunchScope ls("build_lower_prefix", s);
      k_lower_prefix<<<grid_for(NL * 32, kThreads), kThreads, 0, s>>>(g->lower_mask, NL, g->lower_prefix);
    }
    FVX_TRY(check_launch("build_lower_prefix"));
    {
      LaunchScope ls("build_upper_prefix", s);
      k_upper_prefix<<<(unsigned)NU, kThreads, 0, s>>>(g->upper_mask, g->upper_prefix);
    }
    FVX_TRY(check_launch("build_upper_prefix"));
    {
      LaunchScope ls("build_batch_offsets", s);
      k_batch_offsets<<<1, 256, 0, s>>>((const int4*)g->upper_tile, upper_first_voxel, NU, U, B,
                                        g->voxel_batch_offsets);
    }
    FVX_TRY(check_launch("build_batch_offsets"));
  }
  *out = g;
  g = nullptr;  // release the guard
  return FVX_OK;
}

}  // namespace fvx

using namespace fvx;

extern "C" {

fvx_status fvx_build_grid(const int32_t* coords, int64_t n_rows, const int64_t* batch_offsets, int32_t B,
                          fvx_stream stream, fvx_grid* out) {
  EntryScope entry_("fvx_build_grid");
  if (!out || !batch_offsets || (n_rows > 0 && !coords)) {
    set_error("fvx_build_grid: NULL argument");
    return FVX_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (B < 1 || n_rows < 0 || n_rows > (int64_t)INT32_MAX - 1) {
    set_error("fvx_build_grid: need B >= 1 and 0 <= n_rows < 2^31 - 1 (got B=%d, n_rows=%lld)", B,
              (long long)n_rows);
    return FVX_ERR_INVALID_ARG;
  }
  if (batch_offsets[0] != 0 || batch_offsets[B] != n_rows) {
    set_error("fvx_build_grid: batch_offsets must start at 0 and end at n_rows (%lld, %lld vs %lld)",
              (long long)batch_offsets[0], (long long)batch_offsets[B], (long long)n_rows);
    return FVX_ERR_INVALID_ARG;
  }
  for (int32_t b = 0; b < B; ++b) {
    if (batch_offsets[b + 1] < batch_offsets[b]) {
      set_error("fvx_build_grid: batch_offsets not monotone at batch %d", b);
      return FVX_ERR_INVALID_ARG;
    }
  }
  cudaStream_t s = (cudaStream_t)stream;
  Scratch scr(s);
  int64_t* offs = scr.get<int64_t>((size_t)B + 1);
  if (!offs) return FVX_ERR_ALLOC;
  int64_t* ho = (int64_t*)pinned_staging(sizeof(int64_t) * (B + 1));
  if (!ho) return FVX_ERR_ALLOC;
  memcpy(ho, batch_offsets, sizeof(int64_t) * (B + 1));
  FVX_CUDA(cudaMemcpyAsync(offs, ho, sizeof(int64_t) * (B + 1), cudaMemcpyHostToDevice, s));
  fvx_grid_s* g = nullptr;
  FVX_TRY(build_grid_device(coords, n_rows, offs, B, s, &g));
  *out = g;
  return FVX_OK;
}

fvx_status fvx_lookup(fvx_grid g, const int32_t* coords, const int32_t* batch_idx, int64_t n, int32_t* out_idx,
                      fvx_stream stream) {
  EntryScope entry_("fvx_lookup");
  if (!g || n < 0 || (n > 0 && (!coords || !out_idx))) {
    set_error("fvx_lookup: bad argument");
    return FVX_ERR_INVALID_ARG;
  }
  if (n == 0) return FVX_OK;
  cudaStream_t s = (cudaStream_t)stream;
  {
    LaunchScope ls("lookup", s);
    k_lookup<<<grid_for(n, kThreads), kThreads, 0, s>>>(grid_dev(g), coords, batch_idx, n, out_idx);
  }
  return check_launch("lookup");
}

fvx_status fvx_coarsen(fvx_grid g, int32_t stride, fvx_stream stream, fvx_grid* out) {
  EntryScope entry_("fvx_coarsen");
  if (!g || !out || stride < 1) {
    set_error("fvx_coarsen: bad argument (stride must be >= 1)");
    return FVX_ERR_INVALID_ARG;
  }
  *out = nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  Scratch scr(s);
  const int64_t U = g->n_active;
  int32_t* c = scr.get<int32_t>((size_t)(3 * U + 3));
  if (!c) return FVX_ERR_ALLOC;
  int shift = -1;
  for (int b = 0; b < 31; ++b)
    if ((1 << b) == stride) shift = b;
  if (U > 0) {
    {
      LaunchScope ls("coarsen_coords", s);
      k_coarsen_coords<<<grid_for(3 * U, kThreads), kThreads, 0, s>>>(g->ijk, U, stride, shift, c);
    }
    FVX_TRY(check_launch("coarsen_coords"));
  }
  fvx_grid_s* r = nullptr;
  FVX_TRY(build_grid_device(c, U, g->voxel_batch_offsets, g->B, s, &r));
  *out = r;
  return FVX_OK;
}

fvx_status fvx_refine(fvx_grid g, int32_t factor, fvx_stream stream, fvx_grid* out) {
  EntryScope entry_("fvx_refine");
  if (!g || !out || factor < 1) {
    set_error("fvx_refine: bad argument (factor must be >= 1)");
    return FVX_ERR_INVALID_ARG;
  }
  *out = nullptr;
  const int64_t U = g->n_active, f3 = (int64_t)factor * factor * factor;
  if (factor > 1024 || U * f3 > (int64_t)INT32_MAX - 1) {
    set_error("fvx_refine: %lld voxels x %lld children exceed the row limit", (long long)U, (long long)f3);
    return FVX_ERR_RANGE;
  }
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* status = device_status_word();
  if (!status) {
    set_error("fvx_refine: device status word unavailable");
    return FVX_ERR_CUDA;
  }
  Scratch scr(s);
  int32_t* c = scr.get<int32_t>((size_t)(3 * U * f3 + 3));
  int64_t* offs = scr.get<int64_t>((size_t)g->B + 1);
  if (!c || !offs) return FVX_ERR_ALLOC;
  if (U > 0) {
    {
      LaunchScope ls("refine_coords", s);
      k_refine_coords<<<grid_for(U * f3, kThreads), kThreads, 0, s>>>(g->ijk, U, factor, c, status);
    }
    FVX_TRY(check_launch("refine_coords"));
  }
  {
    LaunchScope ls("refine_offsets", s);
    k_scale_offsets<<<grid_for(g->B + 1, kThreads), kThreads, 0, s>>>(g->voxel_batch_offsets, g->B + 1, f3, offs);
  }
  FVX_TRY(check_launch("refine_offsets"));
  fvx_grid_s* r = nullptr;
  FVX_TRY(build_grid_device(c, U * f3, offs, g->B, s, &r));
  *out = r;
  return FVX_OK;
}

}  // extern "C"
