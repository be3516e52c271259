// Device-wide primitives for the IndexGrid build and the kernel map:
//   * exclusive scan of uint32 (reduce, scan of tile sums, down-sweep);
//   * stable LSD radix sort of (uint64 key, uint32 value) pairs, 8-bit digits,
//     one histogram pass and one scatter pass per digit, with the per-(digit,
//     tile) offsets produced by the scan above.
// The pages run steps 3-9 of the build on library sort/RLE/scan primitives
// ["fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High
// Performance Spatial Intelligence" notes, "GPU-accelerated IndexGrid build"];
// these are written here for sm_103a with no device-side spin waits.
#include <cuda_runtime.h>

#include "block_scan.cuh"
#include "fvx_internal.cuh"

namespace fvx {

// ============================================================== scan
constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;  // 2048

__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(const uint32_t* __restrict__ in, int64_t n,
                                                              uint32_t* __restrict__ partial) {
  __shared__ uint32_t tmp[33];
  const int64_t base = (int64_t)blockIdx.x * kScanTile;
  uint32_t s = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    int64_t i = base + k * kScanThreads + threadIdx.x;
    if (i < n) s += in[i];
  }
  uint32_t tot;
  block_exclusive_scan<uint32_t>(s, tmp, &tot);
  if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

// Single block: exclusive scan of the tile sums in place; grand total to *total.
__global__ void __launch_bounds__(1024) k_scan_partials(uint32_t* __restrict__ partial, int64_t np,
                                                        uint32_t* __restrict__ total) {
  __shared__ uint32_t tmp[33];
  uint32_t carry = 0;
  for (int64_t base = 0; base < np; base += 1024) {
    int64_t i = base + threadIdx.x;
    uint32_t v = (i < np) ? partial[i] : 0u;
    uint32_t tot;
    uint32_t ex = block_exclusive_scan<uint32_t>(v, tmp, &tot);
    if (i < np) partial[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0 && total) *total = carry;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_down(const uint32_t* in, uint32_t* out, int64_t n,
                                                            const uint32_t* __restrict__ partial) {
  __shared__ uint32_t tmp[33];
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
  uint32_t v[kScanItems];
  uint32_t s = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    v[k] = (base + k < n) ? in[base + k] : 0u;
    s += v[k];
  }
  uint32_t ex = block_exclusive_scan<uint32_t>(s, tmp, (uint32_t*)nullptr) + partial[blockIdx.x];
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    if (base + k < n) out[base + k] = ex;
    ex += v[k];
  }
}

fvx_status scan_exclusive_u32(const uint32_t* in, uint32_t* out, int64_t n, uint32_t* total, cudaStream_t s,
                              Scratch& scr) {
  if (n <= 0) {
    if (total) FVX_CUDA(cudaMemsetAsync(total, 0, 4, s));
    return FVX_OK;
  }
  const int64_t nt = (n + kScanTile - 1) / kScanTile;
  uint32_t* partial = scr.get<uint32_t>((size_t)nt);
  if (!partial) return FVX_ERR_ALLOC;
  {
    LaunchScope ls("scan_reduce", s);
    k_scan_reduce<<<(unsigned)nt, kScanThreads, 0, s>>>(in, n, partial);
  }
  FVX_TRY(check_launch("scan_reduce"));
  {
    LaunchScope ls("scan_partials", s);
    k_scan_partials<<<1, 1024, 0, s>>>(partial, nt, total);
  }
  FVX_TRY(check_launch("scan_partials"));
  {
    LaunchScope ls("scan_down", s);
    k_scan_down<<<(unsigned)nt, kScanThreads, 0, s>>>(in, out, n, partial);
  }
  return check_launch("scan_down");
}

// ============================================================== radix sort
constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kRsItems = 16;                       // per thread
constexpr int kRsTile = kRsThreads * kRsItems;     // 4096 keys per tile
constexpr int kRsWarpItems = kRsTile / kRsWarps;   // 512 consecutive keys per warp
constexpr int kRsRounds = kRsWarpItems / 32;       // 16

__global__ void __launch_bounds__(kRsThreads) k_radix_hist(const uint64_t* __restrict__ keys, int64_t n, int shift,
                                                           uint32_t dmask, uint32_t* __restrict__ counts,
                                                           int64_t ntiles) {
  __shared__ uint32_t h[256];
  h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kRsTile;
#pragma unroll 4
  for (int k = 0; k < kRsItems; ++k) {
    int64_t i = base + k * kRsThreads + threadIdx.x;
    if (i < n) atomicAdd(&h[(uint32_t)(keys[i] >> shift) & dmask], 1u);
  }
  __syncthreads();
  counts[(int64_t)threadIdx.x * ntiles + blockIdx.x] = h[threadIdx.x];
}

struct RsSmem {
  uint64_t keys[kRsTile];
  uint32_t vals[kRsTile];
  uint32_t whist[kRsWarps][256];
  uint32_t dexcl[256];
  uint32_t goff[256];
  uint32_t tmp[33];
};

__global__ void __launch_bounds__(kRsThreads) k_radix_scatter(const uint64_t* __restrict__ kin,
                                                              const uint32_t* __restrict__ vin,
                                                              uint64_t* __restrict__ kout, uint32_t* __restrict__ vout,
                                                              int64_t n, int shift, uint32_t dmask,
                                                              const uint32_t* __restrict__ offs, int64_t ntiles) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RsSmem& sm = *reinterpret_cast<RsSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int d = lane; d < 256; d += 32) sm.whist[warp][d] = 0;
  sm.goff[tid] = offs[(int64_t)tid * ntiles + blockIdx.x];
  __syncwarp();

  const int64_t base = (int64_t)blockIdx.x * kRsTile + (int64_t)warp * kRsWarpItems;
  uint64_t key[kRsRounds];
  uint32_t val[kRsRounds];
  uint32_t rank[kRsRounds];
  const uint32_t lt = lanemask_lt();
#pragma unroll
  for (int r = 0; r < kRsRounds; ++r) {
    const int64_t i = base + r * 32 + lane;
    const bool valid = i < n;
    key[r] = valid ? kin[i] : 0ull;
    val[r] = valid ? vin[i] : 0u;
    const uint32_t d = valid ? ((uint32_t)(key[r] >> shift) & dmask) : (256u + lane);
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const uint32_t old = valid ? sm.whist[warp][d] : 0u;
    __syncwarp();
    if (valid && (peers & lt) == 0) sm.whist[warp][d] = old + __popc(peers);
    __syncwarp();
    rank[r] = old + __popc(peers & lt);
  }
  __syncthreads();
  {  // per digit: exclusive over warps, then exclusive over digits of the tile totals
    const int d = tid;
    uint32_t run = 0;
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) {
      uint32_t c = sm.whist[w][d];
      sm.whist[w][d] = run;
      run += c;
    }
    uint32_t ex = block_exclusive_scan<uint32_t>(run, sm.tmp, (uint32_t*)nullptr);
    sm.dexcl[d] = ex;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRsRounds; ++r) {
    const int64_t i = base + r * 32 + lane;
    if (i < n) {
      const uint32_t d = (uint32_t)(key[r] >> shift) & dmask;
      const uint32_t lpos = sm.dexcl[d] + sm.whist[warp][d] + rank[r];
      sm.keys[lpos] = key[r];
      sm.vals[lpos] = val[r];
    }
  }
  __syncthreads();
  const int64_t tbase = (int64_t)blockIdx.x * kRsTile;
  const int tile_n = (int)((n - tbase) < kRsTile ? (n - tbase) : kRsTile);
  for (int i = tid; i < tile_n; i += kRsThreads) {
    const uint64_t k = sm.keys[i];
    const uint32_t d = (uint32_t)(k >> shift) & dmask;
    const uint32_t g = sm.goff[d] + (uint32_t)i - sm.dexcl[d];
    kout[g] = k;
    vout[g] = sm.vals[i];
  }
}

fvx_status radix_sort_pairs(uint64_t* k0, uint32_t* v0, uint64_t* k1, uint32_t* v1, int64_t n, int bit_lo,
                            int bit_hi, cudaStream_t s, bool* result_in_1, Scratch& scr) {
  *result_in_1 = false;
  if (n <= 1 || bit_hi <= bit_lo) return FVX_OK;
  FVX_CUDA(cudaFuncSetAttribute(k_radix_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(RsSmem)));
  const int64_t ntiles = (n + kRsTile - 1) / kRsTile;
  uint32_t* counts = scr.get<uint32_t>((size_t)(256 * ntiles));
  if (!counts) return FVX_ERR_ALLOC;
  uint64_t* ks = k0;
  uint32_t* vs = v0;
  uint64_t* kd = k1;
  uint32_t* vd = v1;
  bool in1 = false;
  for (int lo = bit_lo; lo < bit_hi; lo += 8) {
    const int nb = (bit_hi - lo) < 8 ? (bit_hi - lo) : 8;
    const uint32_t dmask = (1u << nb) - 1u;
    {
      LaunchScope ls("radix_hist", s);
      k_radix_hist<<<(unsigned)ntiles, kRsThreads, 0, s>>>(ks, n, lo, dmask, counts, ntiles);
    }
    FVX_TRY(check_launch("radix_hist"));
    FVX_TRY(scan_exclusive_u32(counts, counts, 256 * ntiles, nullptr, s, scr));
    {
      LaunchScope ls("radix_scatter", s);
      k_radix_scatter<<<(unsigned)ntiles, kRsThreads, sizeof(RsSmem), s>>>(ks, vs, kd, vd, n, lo, dmask, counts,
                                                                           ntiles);
    }
    FVX_TRY(check_launch("radix_scatter"));
    uint64_t* tk = ks; ks = kd; kd = tk;
    uint32_t* tv = vs; vs = vd; vd = tv;
    in1 = !in1;
  }
  *result_in_1 = in1;
  return FVX_OK;
}

}  // namespace fvx
