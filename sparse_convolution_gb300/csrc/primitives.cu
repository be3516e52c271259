// Device-wide primitives for the IndexGrid build and the kernel map:
//   * exclusive scan of uint32 in a single pass: each 2048-element tile
//     publishes its sum, then its inclusive prefix, and every later tile adds
//     up what its predecessors published (decoupled look-back);
//   * stable LSD radix sort of (uint64 key, uint32 value) pairs, digits of up
//     to 9 bits (the key's bits spread evenly over as few passes as that
//     allows: 33 bits take four passes, not five of 8 bits):
//     one kernel counts the digits of every pass in a single read of the keys,
//     then one kernel per pass ranks each 4096-key tile in shared memory and
//     takes the tile's output offset for each digit from the digit counts its
//     predecessors published.
// Tiles take their position from an atomic ticket, so a tile only ever waits
// for tiles that started before it.  Every wait is bounded (2 s); one that
// gives up records DEV_TIMEOUT in the device status word.
// The pages run steps 3-9 of the build on library sort/RLE/scan primitives
// ["fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High
// Performance Spatial Intelligence" notes, "GPU-accelerated IndexGrid build"];
// these are written here for sm_103a.
#include <cuda_runtime.h>

#include "block_scan.cuh"
#include "fvx_internal.cuh"

namespace fvx {

// ============================================================== look-back helpers
// Published words: bits 32-33 kind (1 = the tile's own total, 2 = inclusive
// prefix through the tile), bits 40-47 a pass tag (radix sort), bits 0-31 the
// value.  Zero = nothing published yet.
constexpr uint64_t kLbAgg = 1ull << 32;
constexpr uint64_t kLbInc = 2ull << 32;
constexpr unsigned long long kLbWaitNs = 2000000000ull;
constexpr int kLbWindow = 8;   // radix sort: predecessors read per round trip

// A published word carries its own value and nothing else is read on the
// strength of it, so relaxed device-scope accesses suffice (and several loads
// can be in flight at once).
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long lb_clock() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// True once a look-back wait that started at t0 has run past limit_ns.
__device__ __forceinline__ bool lb_expired(unsigned long long t0, unsigned long long limit_ns) {
  return lb_clock() - t0 > limit_ns;
}

// ============================================================== scan
constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;  // 2048

// Input of the scan: the uint32 values themselves, or the popcounts of uint64
// words (bitmap ranks).
struct ScanU32 {
  const uint32_t* p;
  __device__ __forceinline__ uint32_t operator()(int64_t i) const { return p[i]; }
};
struct ScanPopc64 {
  const uint64_t* p;
  __device__ __forceinline__ uint32_t operator()(int64_t i) const { return (uint32_t)__popcll(p[i]); }
};

template <class In>
__global__ void __launch_bounds__(kScanThreads) k_scan_1p(In in, uint32_t* out, int64_t n,
                                                          uint32_t* __restrict__ total, uint64_t* flags,
                                                          uint32_t* ticket, int64_t nt, uint32_t* status) {
  __shared__ uint32_t tmp[33];
  __shared__ uint32_t s_tile, s_prefix;
  if (threadIdx.x == 0) s_tile = atomicAdd(ticket, 1u);
  __syncthreads();
  const int64_t t = s_tile;
  const int64_t base = t * kScanTile + (int64_t)threadIdx.x * kScanItems;
  uint32_t v[kScanItems];
  uint32_t sum = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    v[k] = (base + k < n) ? in(base + k) : 0u;
    sum += v[k];
  }
  uint32_t tot;
  uint32_t ex = block_exclusive_scan<uint32_t>(sum, tmp, &tot);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    if (lane == 0) st_relaxed_u64(flags + t, (t == 0 ? kLbInc : kLbAgg) | tot);
    uint32_t prefix = 0;
    if (t > 0) {
      // lane i looks at tile j - i; the window moves back 32 tiles at a time
      int64_t j = t - 1;
      const unsigned long long t0 = lb_clock();
      for (uint32_t it = 1;; ++it) {
        const int64_t jj = j - lane;
        const uint64_t f = (jj >= 0) ? ld_relaxed_u64(flags + jj) : kLbInc;  // before tile 0: prefix 0
        if (!__all_sync(0xffffffffu, ((f >> 32) & 3u) != 0u)) {
          int give_up = 0;
          if (lane == 0 && (it & 255u) == 0u && lb_expired(t0, kLbWaitNs)) give_up = 1;
          if (__shfl_sync(0xffffffffu, give_up, 0)) {
            if (lane == 0) report_device_error(status, DEV_TIMEOUT);
            break;
          }
          continue;
        }
        const uint32_t incl = __ballot_sync(0xffffffffu, ((f >> 32) & 3u) == 2u);
        const int first = incl ? __ffs(incl) - 1 : 32;  // nearest tile with an inclusive prefix
        prefix += warp_reduce_sum<uint32_t>(lane <= first ? (uint32_t)f : 0u);
        if (incl) break;
        j -= 32;
      }
      if (lane == 0) st_relaxed_u64(flags + t, kLbInc | (uint32_t)(prefix + tot));
    }
    if (lane == 0) s_prefix = prefix;
  }
  __syncthreads();
  ex += s_prefix;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    if (base + k < n) out[base + k] = ex;
    ex += v[k];
  }
  if (t == nt - 1 && threadIdx.x == 0 && total) *total = s_prefix + tot;
}

template <class In>
fvx_status scan_1p(In in, uint32_t* out, int64_t n, uint32_t* total, cudaStream_t s, Scratch& scr) {
  if (n <= 0) {
    if (total) FVX_CUDA(cudaMemsetAsync(total, 0, 4, s));
    return FVX_OK;
  }
  uint32_t* status = device_status_word();
  if (!status) {
    set_error("scan: device status word unavailable");
    return FVX_ERR_CUDA;
  }
  const int64_t nt = (n + kScanTile - 1) / kScanTile;
  uint64_t* flags = scr.get<uint64_t>((size_t)nt + 1);  // tile words, then the ticket
  if (!flags) return FVX_ERR_ALLOC;
  FVX_CUDA(cudaMemsetAsync(flags, 0, 8 * ((size_t)nt + 1), s));
  {
    LaunchScope ls("scan_1p", s);
    k_scan_1p<In><<<(unsigned)nt, kScanThreads, 0, s>>>(in, out, n, total, flags, (uint32_t*)(flags + nt), nt,
                                                        status);
  }
  return check_launch("scan_1p");
}

fvx_status scan_exclusive_u32(const uint32_t* in, uint32_t* out, int64_t n, uint32_t* total, cudaStream_t s,
                              Scratch& scr) {
  return scan_1p(ScanU32{in}, out, n, total, s, scr);
}

fvx_status scan_popc64(const uint64_t* words, uint32_t* out, int64_t n, uint32_t* total, cudaStream_t s,
                       Scratch& scr) {
  return scan_1p(ScanPopc64{words}, out, n, total, s, scr);
}

// ============================================================== radix sort
constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kRsItems = 16;                       // per thread
constexpr int kRsTile = kRsThreads * kRsItems;     // 4096 keys per tile
constexpr int kRsWarpItems = kRsTile / kRsWarps;   // 512 consecutive keys per warp
constexpr int kRsRounds = kRsWarpItems / 32;       // 16

constexpr int kRsMaxPasses = 8;                    // 64-bit keys
constexpr int kRsMaxBins = 512;                    // digits of up to 9 bits
constexpr int kRsHistTile = 4096;                  // keys per block of the counting kernel

// The passes of one sort: pass p sorts bits [lo[p], lo[p] + nb[p]).
struct RsPasses {
  int n;
  int lo[kRsMaxPasses], nb[kRsMaxPasses];
};

// Digit counts of every pass in one read of the keys: ghist[p][d] += number of
// keys whose pass-p digit is d (block counts in shared memory, then one global
// add per nonzero count); pass p's counts start at p * kRsMaxBins.
__global__ void __launch_bounds__(kRsThreads) k_radix_hist_all(const uint64_t* __restrict__ keys, int64_t n,
                                                               RsPasses ps, uint32_t* __restrict__ ghist) {
  __shared__ uint32_t h[kRsMaxPasses * kRsMaxBins];
  const int passes = ps.n;
  for (int i = threadIdx.x; i < passes * kRsMaxBins; i += kRsThreads) h[i] = 0u;
  __syncthreads();
  const int64_t b0 = (int64_t)blockIdx.x * kRsHistTile;
#pragma unroll 4
  for (int k = 0; k < kRsHistTile / kRsThreads; ++k) {
    const int64_t i = b0 + k * kRsThreads + threadIdx.x;
    if (i < n) {
      const uint64_t key = keys[i];
      for (int p = 0; p < passes; ++p)
        atomicAdd(&h[p * kRsMaxBins + ((uint32_t)(key >> ps.lo[p]) & ((1u << ps.nb[p]) - 1u))], 1u);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < passes * kRsMaxBins; i += kRsThreads)
    if (h[i]) atomicAdd(&ghist[i], h[i]);
}

template <int BINS>
struct RsSmem {
  uint64_t keys[kRsTile];
  uint32_t vals[kRsTile];
  uint32_t whist[kRsWarps][BINS];
  uint32_t dexcl[BINS];
  uint32_t goff[BINS];
  uint32_t tmp[33];
};

// One pass: tile t (by ticket) ranks its 4096 keys by digit in shared
// memory, publishes its count of each digit, adds up the counts its
// predecessors published (thread j follows digits j * DPT .. j * DPT + DPT-1)
// publishes the inclusive count and writes each key to digit_start[d] +
// predecessors' count + rank.  BINS = 256 (digits of up to 8 bits) or 512.
template <int BINS>
__global__ void __launch_bounds__(kRsThreads, 3) k_radix_onesweep(const uint64_t* __restrict__ kin,
                                                               const uint32_t* __restrict__ vin,
                                                               uint64_t* __restrict__ kout,
                                                               uint32_t* __restrict__ vout, int64_t n, int shift,
                                                               uint32_t dmask, const uint32_t* __restrict__ ghist,
                                                               uint64_t* state, uint32_t* ticket, uint32_t tag,
                                                               uint32_t* status) {
  constexpr int DPT = BINS / kRsThreads;  // digits per thread in the per-digit steps
  extern __shared__ __align__(16) unsigned char smem_raw[];
  RsSmem<BINS>& sm = *reinterpret_cast<RsSmem<BINS>*>(smem_raw);
  __shared__ uint32_t s_tile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_tile = atomicAdd(ticket, 1u);
  for (int d = lane; d < BINS; d += 32) sm.whist[warp][d] = 0;
  // where each digit starts in the output: exclusive scan of the pass's counts
  uint32_t gcnt[DPT], gsum = 0;
#pragma unroll
  for (int j = 0; j < DPT; ++j) {
    gcnt[j] = ghist[tid * DPT + j];
    gsum += gcnt[j];
  }
  const uint32_t gstart0 = block_exclusive_scan<uint32_t>(gsum, sm.tmp, (uint32_t*)nullptr);
  const int64_t t = s_tile;  // visible after the scan's barriers

  const int64_t base = t * kRsTile + (int64_t)warp * kRsWarpItems;
  uint64_t key[kRsRounds];
  uint32_t rank[kRsRounds];  // values are read again when scattered (registers for a third block per SM)
  const uint32_t lt = lanemask_lt();
#pragma unroll
  for (int r = 0; r < kRsRounds; ++r) {
    const int64_t i = base + r * 32 + lane;
    const bool valid = i < n;
    key[r] = valid ? kin[i] : 0ull;
    const uint32_t d = valid ? ((uint32_t)(key[r] >> shift) & dmask) : ((uint32_t)BINS + lane);
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const uint32_t old = valid ? sm.whist[warp][d] : 0u;
    __syncwarp();
    if (valid && (peers & lt) == 0) sm.whist[warp][d] = old + __popc(peers);
    __syncwarp();
    rank[r] = old + __popc(peers & lt);
  }
  __syncthreads();
  {  // per digit: exclusive over warps, the tile's count, then the look-back
    uint32_t run[DPT], prefix[DPT], rsum = 0;
#pragma unroll
    for (int j = 0; j < DPT; ++j) {
      const int d = tid * DPT + j;
      uint32_t acc = 0;
#pragma unroll
      for (int w = 0; w < kRsWarps; ++w) {
        uint32_t c = sm.whist[w][d];
        sm.whist[w][d] = acc;
        acc += c;
      }
      run[j] = acc;
      rsum += acc;
      prefix[j] = 0;
    }
    const uint64_t tagbits = (uint64_t)tag << 40;
#pragma unroll
    for (int j = 0; j < DPT; ++j)
      st_relaxed_u64(state + t * BINS + tid * DPT + j, tagbits | (t == 0 ? kLbInc : kLbAgg) | run[j]);
    if (t > 0) {
      // kLbWindow predecessors per round trip, nearest first; the walk stops
      // at the first inclusive word and resumes at the first unpublished one
      const unsigned long long t0 = lb_clock();
#pragma unroll
      for (int jd = 0; jd < DPT; ++jd) {
        const int d = tid * DPT + jd;
        int64_t j = t - 1;
        bool done = false;
        for (uint32_t it = 1; !done; ++it) {
          uint64_t f[kLbWindow];
#pragma unroll
          for (int q = 0; q < kLbWindow; ++q)
            f[q] = (j - q >= 0) ? ld_relaxed_u64(state + (j - q) * BINS + d) : (tagbits | kLbInc);  // before tile 0
          int q = 0;
#pragma unroll
          for (int r = 0; r < kLbWindow; ++r) {
            if (q != r || done) continue;
            const bool ready = (uint32_t)(f[r] >> 40) == tag && ((f[r] >> 32) & 3u) != 0u;
            if (!ready) continue;
            prefix[jd] += (uint32_t)f[r];
            done = ((f[r] >> 32) & 3u) == 2u;
            q = r + 1;
          }
          j -= q;
          if (!done && q < kLbWindow && (it & 63u) == 0u && lb_expired(t0, kLbWaitNs)) {
            report_device_error(status, DEV_TIMEOUT);
            break;
          }
        }
        st_relaxed_u64(state + t * BINS + d, tagbits | kLbInc | (uint32_t)(prefix[jd] + run[jd]));
      }
    }
    uint32_t gs = gstart0;
#pragma unroll
    for (int j = 0; j < DPT; ++j) {
      sm.goff[tid * DPT + j] = gs + prefix[j];
      gs += gcnt[j];
    }
    uint32_t de = block_exclusive_scan<uint32_t>(rsum, sm.tmp, (uint32_t*)nullptr);
#pragma unroll
    for (int j = 0; j < DPT; ++j) {
      sm.dexcl[tid * DPT + j] = de;
      de += run[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRsRounds; ++r) {
    const int64_t i = base + r * 32 + lane;
    if (i < n) {
      const uint32_t d = (uint32_t)(key[r] >> shift) & dmask;
      const uint32_t lpos = sm.dexcl[d] + sm.whist[warp][d] + rank[r];
      sm.keys[lpos] = key[r];
      sm.vals[lpos] = vin[i];
    }
  }
  __syncthreads();
  const int64_t tbase = t * kRsTile;
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
  uint32_t* status = device_status_word();
  if (!status) {
    set_error("radix sort: device status word unavailable");
    return FVX_ERR_CUDA;
  }
  for (auto kern : {k_radix_onesweep<256>, k_radix_onesweep<512>}) {
    const int bytes = kern == k_radix_onesweep<256> ? (int)sizeof(RsSmem<256>) : (int)sizeof(RsSmem<512>);
    FVX_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
    // three blocks per SM: shared memory for three tiles, registers for three (launch bounds)
    FVX_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared));
  }
  // as few passes as digits of up to 9 bits allow, 8-bit digits when that
  // takes no more passes; the bits spread evenly (first passes one wider)
  const int bits = bit_hi - bit_lo;
  int passes = (bits + 7) / 8;
  if ((bits + 8) / 9 < passes) passes = (bits + 8) / 9;
  RsPasses ps;
  ps.n = passes;
  for (int p = 0, lo = bit_lo; p < passes; ++p) {
    ps.nb[p] = bits / passes + (p < bits % passes ? 1 : 0);
    ps.lo[p] = lo;
    lo += ps.nb[p];
  }
  const int64_t ntiles = (n + kRsTile - 1) / kRsTile;
  // one zeroed region: digit counts [passes][kRsMaxBins], tickets [8], then
  // the published words [ntiles][kRsMaxBins] shared by all passes (told apart
  // by tag)
  const size_t words32 = (size_t)passes * kRsMaxBins + kRsMaxPasses;
  uint64_t* region = scr.get<uint64_t>(words32 / 2 + (size_t)ntiles * kRsMaxBins);
  if (!region) return FVX_ERR_ALLOC;
  uint32_t* ghist = reinterpret_cast<uint32_t*>(region);
  uint32_t* tickets = ghist + (size_t)passes * kRsMaxBins;
  uint64_t* state = region + words32 / 2;
  FVX_CUDA(cudaMemsetAsync(region, 0, 8 * (words32 / 2 + (size_t)ntiles * kRsMaxBins), s));
  {
    LaunchScope ls("radix_hist_all", s);
    const int64_t nb = (n + kRsHistTile - 1) / kRsHistTile;
    k_radix_hist_all<<<(unsigned)nb, kRsThreads, 0, s>>>(k0, n, ps, ghist);
  }
  FVX_TRY(check_launch("radix_hist_all"));
  uint64_t* ks = k0;
  uint32_t* vs = v0;
  uint64_t* kd = k1;
  uint32_t* vd = v1;
  bool in1 = false;
  for (int p = 0; p < passes; ++p) {
    const uint32_t dmask = (1u << ps.nb[p]) - 1u;
    {
      LaunchScope ls("radix_onesweep", s);
      if (ps.nb[p] > 8)
        k_radix_onesweep<512><<<(unsigned)ntiles, kRsThreads, sizeof(RsSmem<512>), s>>>(
            ks, vs, kd, vd, n, ps.lo[p], dmask, ghist + (size_t)p * kRsMaxBins, state, tickets + p,
            (uint32_t)(p + 1), status);
      else
        k_radix_onesweep<256><<<(unsigned)ntiles, kRsThreads, sizeof(RsSmem<256>), s>>>(
            ks, vs, kd, vd, n, ps.lo[p], dmask, ghist + (size_t)p * kRsMaxBins, state, tickets + p,
            (uint32_t)(p + 1), status);
    }
    FVX_TRY(check_launch("radix_onesweep"));
    uint64_t* tk = ks; ks = kd; kd = tk;
    uint32_t* tv = vs; vs = vd; vd = tv;
    in1 = !in1;
  }
  *result_in_1 = in1;
  return FVX_OK;
}

// ============================================================== test hook
// One warp polls a published word that nothing sets, the way the scan's
// look-back polls its predecessors, and gives up after limit_ns the same way:
// the bounded wait and its status report, without a real wait running out.
__global__ void k_testing_flag_wait(const uint64_t* flag, unsigned long long limit_ns, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const unsigned long long t0 = lb_clock();
  for (uint32_t it = 1;; ++it) {
    const uint64_t f = ld_relaxed_u64(flag);
    if (__all_sync(0xffffffffu, ((f >> 32) & 3u) != 0u)) return;
    int give_up = 0;
    if (lane == 0 && (it & 255u) == 0u && lb_expired(t0, limit_ns)) give_up = 1;
    if (__shfl_sync(0xffffffffu, give_up, 0)) {
      if (lane == 0) report_device_error(status, DEV_TIMEOUT);
      return;
    }
  }
}

fvx_status testing_flag_wait(const uint64_t* flag, unsigned long long limit_ns, uint32_t* status, cudaStream_t s) {
  {
    LaunchScope ls("testing_flag_wait", s);
    k_testing_flag_wait<<<1, 32, 0, s>>>(flag, limit_ns, status);
  }
  return check_launch("testing_flag_wait");
}

}  // namespace fvx
