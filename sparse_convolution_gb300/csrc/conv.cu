// Sparse 3x3x3 convolution over a kernel map: gather - GEMM - scatter.
//
//   out[q, co] = sum_s sum_{(p,q) in list s} sum_ci x[p, ci] * W[s, ci, co]
//
// ["fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High
// Performance Spatial Intelligence" notes, "Sparse-convolution operators":
// gather-GEMM-scatter on tiles of consecutive output indices, pairs padded for
// the tensor-core GEMM, a shared-memory accumulator instead of a global
// scatter.]  Here the accumulator is TMEM and the tile is 128 consecutive
// outputs (the tcgen05 M); the K dimension of the tile's GEMM is the
// concatenation, over the offsets that occur in the tile, of Cin channels each,
// so empty offsets cost nothing and small Cin (8, 16) still fills K = 64 per
// pipeline stage.  For output row m and offset s the gathered A row is x[p]
// where (p, q0+m) is a pair of list s, or zeros; the pair is found from the
// 27-bit output mask ["DriveRT", "Kernels selected per GPU"] by the rank of m
// among the tile's rows with bit s, added to the tile's start in list s.
//
// Two kernels, one per dtype (no dispatch between backends):
//   * bf16: cp.async gathers into 128B-swizzled K-major shared tiles,
//     tcgen05.mma kind::f16 (bf16 x bf16 -> fp32 in TMEM) issued by one
//     thread, tcgen05.ld epilogue, bf16 round-to-nearest-even output.
//   * fp32: exact FFMA on CUDA cores (no TF32).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <string.h>

#include "block_scan.cuh"
#include "fvx_internal.cuh"

namespace fvx {
namespace {

constexpr int kRows = kTileRows;  // 128

// ============================================================== shared prologue
// Per tile: for each offset s, the ballot of the tile's rows having bit s, per
// warp (4 warps x 32 rows).  rank of row m in list s = popcount of the bits
// before it.
struct TileMasks {
  uint32_t wb[27][4];
};

__device__ __forceinline__ void tile_ballots(TileMasks& tm, uint32_t mk) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 1
  for (int s = 0; s < 27; ++s) {
    const uint32_t b = __ballot_sync(0xffffffffu, (mk >> s) & 1u);
    if (lane == 0) tm.wb[s][warp] = b;
  }
}

__device__ __forceinline__ uint32_t tile_rank(const TileMasks& tm, int s, int warp, uint32_t lt) {
  uint32_t r = __popc(tm.wb[s][warp] & lt);
  for (int w = 0; w < warp; ++w) r += __popc(tm.wb[s][w]);
  return r;
}

__device__ __forceinline__ uint32_t tile_or(const TileMasks& tm) {
  uint32_t o = 0;
  for (int s = 0; s < 27; ++s)
    if (tm.wb[s][0] | tm.wb[s][1] | tm.wb[s][2] | tm.wb[s][3]) o |= 1u << s;
  return o;
}

// ============================================================== fp32 FFMA
constexpr int kF32Cols = 16;

__global__ void __launch_bounds__(kRows) k_conv_f32(const float* __restrict__ x, const float* __restrict__ W,
                                                    const uint32_t* __restrict__ mask,
                                                    const int32_t* __restrict__ in_idx,
                                                    const uint32_t* __restrict__ tile_start, int64_t ntiles,
                                                    int64_t n_out, int cin, int cout, float* __restrict__ y) {
  __shared__ TileMasks tm;
  const int m = threadIdx.x, warp = m >> 5;
  const int64_t t = blockIdx.x;
  const int64_t q = t * kRows + m;
  const uint32_t mk = (q < n_out) ? mask[q] : 0u;
  tile_ballots(tm, mk);
  __syncthreads();
  const uint32_t lt = lanemask_lt();
  const uint32_t tor = tile_or(tm);
  for (int c0 = 0; c0 < cout; c0 += kF32Cols) {
    float acc[kF32Cols];
#pragma unroll
    for (int c = 0; c < kF32Cols; ++c) acc[c] = 0.f;
    for (int s = 0; s < 27; ++s) {
      if (!((tor >> s) & 1u)) continue;
      if (!((mk >> s) & 1u)) continue;
      const int p = in_idx[tile_start[(int64_t)s * ntiles + t] + tile_rank(tm, s, warp, lt)];
      const float* xp = x + (int64_t)p * cin;
      const float* ws = W + (int64_t)s * cin * cout + c0;
      if (c0 + kF32Cols <= cout) {
        for (int ci = 0; ci < cin; ++ci) {
          const float xv = __ldg(xp + ci);
          const float* wr = ws + (int64_t)ci * cout;
#pragma unroll
          for (int c = 0; c < kF32Cols; ++c) acc[c] = fmaf(xv, __ldg(wr + c), acc[c]);
        }
      } else {
        for (int ci = 0; ci < cin; ++ci) {
          const float xv = __ldg(xp + ci);
          const float* wr = ws + (int64_t)ci * cout;
#pragma unroll
          for (int c = 0; c < kF32Cols; ++c)
            if (c0 + c < cout) acc[c] = fmaf(xv, __ldg(wr + c), acc[c]);
        }
      }
    }
    if (q < n_out) {
      float* yq = y + q * cout + c0;
#pragma unroll
      for (int c = 0; c < kF32Cols; ++c)
        if (c0 + c < cout) yq[c] = acc[c];
    }
  }
}

// ============================================================== bf16 tcgen05
constexpr int kProducerWarps = 4;
constexpr int kConvThreads = (kProducerWarps + 1) * 32;  // + one MMA-issue warp
constexpr int kLag = 2;                                   // cp.async groups kept in flight per producer
constexpr int kATileBytes = kRows * 128;                  // 128 rows x 64 bf16 (one 128B swizzle atom wide)
constexpr unsigned long long kWaitNs = 2000000000ull;     // bounded mbarrier waits: 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Waits for the phase with the given parity to complete; gives up after
// kWaitNs (or when another CTA has already reported a failure), recording
// DEV_TIMEOUT in the status word.  Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
  uint32_t ok = 0;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  if (ok) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (globaltimer() - t0 > kWaitNs || *(volatile uint32_t*)status != 0u) {
      report_device_error(status, DEV_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), leading offset unused for this layout.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

struct ConvSmemHead {
  TileMasks tm;
  int32_t rowp[27][kRows];  // gathered input row for (offset slot, tile row), -1 = zeros
  int32_t slot_s[27];       // offset of each slot (only offsets present in the tile)
  unsigned long long full[8], empty[8], done;
  uint32_t tmem_base;
  int nslots;
};

struct ConvArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* wt;  // [27][cout][cin], K-major per offset
  const uint32_t* mask;
  const int32_t* in_idx;
  const uint32_t* tile_start;
  __nv_bfloat16* y;
  uint32_t* status;
  int64_t ntiles, n_out;
  int cin, cout, stages, stage_bytes, b_bytes, tmem_cols;
};

__global__ void __launch_bounds__(kConvThreads, 1) k_conv_bf16_tc(const __grid_constant__ ConvArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // stage buffers first (1024-aligned), head after them
  unsigned char* sbase = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  ConvSmemHead& h = *reinterpret_cast<ConvSmemHead*>(sbase + (size_t)a.stages * a.stage_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t t = blockIdx.x;
  const int S = a.stages;

  // ---- setup: barriers (thread 0), TMEM allocation (MMA warp)
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&h.full[i]), kProducerWarps * 32);
      mbar_init(smem_u32(&h.empty[i]), 1);
    }
    mbar_init(smem_u32(&h.done), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kProducerWarps) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&h.tmem_base)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // ---- tile prologue (producer warps): masks, ranks, gathered row per slot
  uint32_t mk = 0;
  if (warp < kProducerWarps) {
    const int64_t q = t * kRows + tid;
    mk = (q < a.n_out) ? a.mask[q] : 0u;
    tile_ballots(h.tm, mk);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tor = tile_or(h.tm);
  const int nslots = __popc(tor);
  if (warp < kProducerWarps) {
    const uint32_t lt = lanemask_lt();
    int slot = 0;
    for (int s = 0; s < 27; ++s) {
      if (!((tor >> s) & 1u)) continue;
      int p = -1;
      if ((mk >> s) & 1u) p = a.in_idx[a.tile_start[(int64_t)s * a.ntiles + t] + tile_rank(h.tm, s, warp, lt)];
      h.rowp[slot][tid] = p;
      if (tid == 0) h.slot_s[slot] = s;
      ++slot;
    }
  }
  __syncthreads();
  const uint32_t tmem = h.tmem_base;
  const int ppo = a.cin >> 3;  // 16-byte pieces per (row, offset)
  const int total = nslots * ppo;
  const int nst = (total + 7) >> 3;  // pipeline stages of 8 pieces (K = 64)

  if (warp < kProducerWarps) {
    // ---------------- producers: gather A rows and B (weights) rows
    const int m = tid;
    int signaled = 0;
    for (int k = 0; k < nst; ++k) {
      const int sb = k % S;
      if (k >= S) mbar_wait(smem_u32(&h.empty[sb]), (uint32_t)((k / S - 1) & 1), a.status);
      const uint32_t sA = smem_u32(sbase + (size_t)sb * a.stage_bytes);
      const uint32_t sB = sA + kATileBytes;
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        const int g = 8 * k + pc;
        const void* src = a.x;
        uint32_t bytes = 0;
        if (g < total) {
          const int slot = g / ppo, cb = g - slot * ppo;
          const int p = h.rowp[slot][m];
          if (p >= 0) {
            src = a.x + (int64_t)p * a.cin + cb * 8;
            bytes = 16;
          }
        }
        cp_async16(sA + (m >> 3) * 1024 + (m & 7) * 128 + ((pc ^ (m & 7)) << 4), src, bytes);
      }
      for (int n = m; n < a.cout; n += kProducerWarps * 32) {
#pragma unroll
        for (int pc = 0; pc < 8; ++pc) {
          const int g = 8 * k + pc;
          const void* src = a.wt;
          uint32_t bytes = 0;
          if (g < total) {
            const int slot = g / ppo, cb = g - slot * ppo;
            src = a.wt + ((int64_t)h.slot_s[slot] * a.cout + n) * a.cin + cb * 8;
            bytes = 16;
          }
          cp_async16(sB + (n >> 3) * 1024 + (n & 7) * 128 + ((pc ^ (n & 7)) << 4), src, bytes);
        }
      }
      cp_async_commit();
      if (k - signaled >= kLag) {
        cp_async_wait<kLag>();
        fence_proxy_async();
        mbar_arrive(smem_u32(&h.full[signaled % S]));
        ++signaled;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    while (signaled < nst) {
      mbar_arrive(smem_u32(&h.full[signaled % S]));
      ++signaled;
    }
  } else if (lane == 0) {
    // ---------------- MMA issue (one thread)
    const uint32_t idesc = idesc_bf16(kRows, a.cout);
    for (int k = 0; k < nst; ++k) {
      const int sb = k % S;
      mbar_wait(smem_u32(&h.full[sb]), (uint32_t)((k / S) & 1), a.status);
      tc_fence_after();
      const uint32_t sA = smem_u32(sbase + (size_t)sb * a.stage_bytes);
      const uint32_t sB = sA + kATileBytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(tmem, sdesc_sw128(sA + kk * 32), sdesc_sw128(sB + kk * 32), idesc, (k | kk) ? 1u : 0u);
      umma_commit(smem_u32(&h.empty[sb]));
    }
    if (nst > 0) umma_commit(smem_u32(&h.done));
  }
  if (warp == kProducerWarps) __syncwarp();

  // ---------------- epilogue: TMEM -> registers -> bf16 -> global
  if (warp < kProducerWarps) {
    const int64_t q = t * kRows + tid;
    if (nst > 0) {
      mbar_wait(smem_u32(&h.done), 0u, a.status);
      tc_fence_after();
    }
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c = 0; c < a.cout; c += 16) {
      uint32_t r[16];
      if (nst > 0) {
        tmem_ld16(trow + (uint32_t)c, r);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = 0u;
      }
      if (q < a.n_out) {
        uint4 v0, v1;
        v0.x = pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1]));
        v0.y = pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3]));
        v0.z = pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5]));
        v0.w = pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7]));
        v1.x = pack_bf16x2(__uint_as_float(r[8]), __uint_as_float(r[9]));
        v1.y = pack_bf16x2(__uint_as_float(r[10]), __uint_as_float(r[11]));
        v1.z = pack_bf16x2(__uint_as_float(r[12]), __uint_as_float(r[13]));
        v1.w = pack_bf16x2(__uint_as_float(r[14]), __uint_as_float(r[15]));
        uint4* dst = reinterpret_cast<uint4*>(a.y + q * a.cout + c);
        dst[0] = v0;
        dst[1] = v1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kProducerWarps) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
  }
}

// W [27][cin][cout] -> Wt [27][cout][cin] (bf16), the K-major B operand.
__global__ void k_transpose_w(const __nv_bfloat16* __restrict__ W, int cin, int cout,
                              __nv_bfloat16* __restrict__ wt) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t per = (int64_t)cin * cout;
  if (e >= 27 * per) return;
  const int64_t s = e / per, r = e - s * per;
  const int co = (int)(r / cin), ci = (int)(r - (int64_t)co * cin);
  wt[e] = W[s * per + (int64_t)ci * cout + co];
}

}  // namespace
}  // namespace fvx

using namespace fvx;

extern "C" fvx_status fvx_sparse_conv(fvx_grid gin, fvx_grid gout, fvx_kmap m, fvx_dtype dt, const void* feats,
                                      int64_t cin, const void* W, int64_t cout, void* out, fvx_stream stream) {
  if (!gin || !gout || !m || !W || !out || (gin->n_active > 0 && !feats)) {
    set_error("fvx_sparse_conv: NULL argument");
    return FVX_ERR_INVALID_ARG;
  }
  if (m->gin != gin || m->gout != gout) {
    set_error("fvx_sparse_conv: kernel map was built for other grids");
    return FVX_ERR_INVALID_ARG;
  }
  if (cin < 1 || cout < 1) {
    set_error("fvx_sparse_conv: cin and cout must be >= 1");
    return FVX_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t nt = m->n_tiles;
  if (gout->n_active == 0) return FVX_OK;
  if (dt == FVX_F32) {
    {
      LaunchScope ls("conv_f32", s);
      k_conv_f32<<<(unsigned)nt, kRows, 0, s>>>((const float*)feats, (const float*)W, m->out_mask, m->in_idx,
                                                m->tile_start, nt, m->n_out, (int)cin, (int)cout, (float*)out);
    }
    return check_launch("conv_f32");
  }
  if (dt != FVX_BF16) {
    set_error("fvx_sparse_conv: unknown dtype %d", (int)dt);
    return FVX_ERR_INVALID_ARG;
  }
  if (cin % 8 != 0 || cout % 16 != 0 || cin > 512 || cout > 256) {
    set_error("fvx_sparse_conv: bf16 needs cin %% 8 == 0 (<= 512) and cout %% 16 == 0 (<= 256); got %lld, %lld",
              (long long)cin, (long long)cout);
    return FVX_ERR_INVALID_ARG;
  }
  if (((uintptr_t)feats | (uintptr_t)out) & 15u) {
    set_error("fvx_sparse_conv: feats and out must be 16-byte aligned");
    return FVX_ERR_INVALID_ARG;
  }
  uint32_t* status = device_status_word();
  if (!status) {
    set_error("fvx_sparse_conv: device status word unavailable");
    return FVX_ERR_CUDA;
  }
  Scratch scr(s);
  __nv_bfloat16* wt = scr.get<__nv_bfloat16>((size_t)(27 * cin * cout));
  if (!wt) return FVX_ERR_ALLOC;
  {
    LaunchScope ls("conv_transpose_w", s);
    const int64_t n = 27 * cin * cout;
    k_transpose_w<<<(unsigned)((n + 255) / 256), 256, 0, s>>>((const __nv_bfloat16*)W, (int)cin, (int)cout, wt);
  }
  FVX_TRY(check_launch("conv_transpose_w"));

  ConvArgs a;
  a.x = (const __nv_bfloat16*)feats;
  a.wt = wt;
  a.mask = m->out_mask;
  a.in_idx = m->in_idx;
  a.tile_start = m->tile_start;
  a.y = (__nv_bfloat16*)out;
  a.status = status;
  a.ntiles = nt;
  a.n_out = m->n_out;
  a.cin = (int)cin;
  a.cout = (int)cout;
  a.b_bytes = (int)cout * 128;
  a.stage_bytes = kATileBytes + a.b_bytes;  // multiple of 1024 since cout % 8 == 0
  const int budget = 200 * 1024 - (int)sizeof(ConvSmemHead);
  a.stages = budget / a.stage_bytes;
  if (a.stages > 8) a.stages = 8;
  if (a.stages < kLag + 1) {
    set_error("fvx_sparse_conv: cout %lld leaves too few pipeline stages", (long long)cout);
    return FVX_ERR_INVALID_ARG;
  }
  int cols = 32;
  while (cols < cout) cols <<= 1;
  a.tmem_cols = cols;
  const size_t smem = 1024 + (size_t)a.stages * a.stage_bytes + sizeof(ConvSmemHead);
  FVX_CUDA(cudaFuncSetAttribute(k_conv_bf16_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  {
    LaunchScope ls("conv_bf16_tc", s);
    k_conv_bf16_tc<<<(unsigned)nt, kConvThreads, smem, s>>>(a);
  }
  return check_launch("conv_bf16_tc");
}
