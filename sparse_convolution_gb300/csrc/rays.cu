// Voxels along rays: hierarchical DDA over the IndexGrid.
//
// ["fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High
// Performance Spatial Intelligence" notes, "HDDA"]: a ray is rasterised by one
// DDA per tree level, at 4096^3, 128^3, 8^3 and 1^3 cells; the coarse levels
// cross empty space in one step and only the finest walks voxel by voxel.
// What it yields is the list of active voxels each ray passes through.
//
// Exact definition (the CPU oracle follows the same written rules with its own
// code; the two share nothing):
//   * voxel (i,j,k) is the cell [i,i+1) x [j,j+1) x [k,k+1) in index space;
//     the ray is o + t d with fp32 o, d; inv_a = 1 / d_a, rounded once.
//   * the ray crosses the plane x_a = n at T_a(n) = ((float)n - o_a) * inv_a,
//     two fp32 operations rounded to nearest (no fused multiply-add).
//   * [tmin, tmax] is clipped to a box holding the batch element's active
//     voxels by the same plane times (slab method); a direction component of 0
//     keeps the ray only if lo_a <= o_a < hi_a + 1; d = 0 gives no hits.
//   * at time t the ray is in cell c_a = max{n : T_a(n) <= t} (d_a > 0),
//     min{n : T_a(n) <= t} - 1 (d_a < 0), floor(o_a) (d_a = 0).
//   * a hit is an active cell occupied for a time interval of positive length
//     inside the clipped segment: its index and [t_enter, t_exit), the times
//     of the crossings that enter and leave it, clipped to the segment (a
//     zero is written as +0).  Hits are in order of t_enter.
// The walk keeps exactly that state (current cell, next crossing time per
// axis).  When the upper node, lower node or leaf that would hold the current
// cell is absent, it leaves that 4096^3, 128^3 or 8^3 box in one step: the
// exit time is the earliest far-face crossing, and the cell at that time is
// found from the definition (estimate, then bounded corrections), so the walk
// visits the same cells, with the same times, as a cell-by-cell walk would.
// The clip box here is the batch element's box of leaves (a superset of the
// voxels' box): cells outside hold no voxel and a hit's entry crossing is
// never before the box's, so the hits are the same.
#include <cuda_runtime.h>
#include <limits.h>
#include <string.h>

#include "fvx_internal.cuh"

struct fvx_hits_s {
  int64_t n_rays = 0, n_hits = 0;
  void* block = nullptr;  // offsets int64 [n_rays + 1], voxel int32 [n_hits], t float [n_hits][2]
  cudaStream_t stream = 0;
  int64_t* offsets = nullptr;
  int32_t* voxel = nullptr;
  float* t = nullptr;
};

namespace fvx {
namespace {

constexpr int kRayThreads = 128;
constexpr int kMaxSteps = 1 << 24;  // per ray; a walk inside the clip box takes far fewer
constexpr int kMaxCoord = 1 << 24;  // voxel coordinates must lie in [-2^24, 2^24): every cell face exact in fp32

struct RayArgs {
  GridDev g;
  const float* o;
  const float* d;
  const int32_t* batch;  // NULL: all rays in batch element 0
  int64_t n;
  float tmin, tmax;
  const int32_t* bbox;  // [B][6]: lo x y z, hi x y z (inclusive); lo > hi: no voxels
  int32_t B;
  uint32_t* count;             // counting pass: hits per ray
  unsigned long long* total;   // counting pass: sum of the counts
  const uint32_t* off;         // writing pass: exclusive scan of the counts
  int32_t* voxel;              // writing pass
  float* t;
  uint32_t* status;
};

__device__ __forceinline__ float plane_time(int n, float o, float inv) {
  return __fmul_rn(__fsub_rn(__int2float_rn(n), o), inv);
}

// Cell coordinate along one axis at time t (the definition above): an
// estimate, then corrections against the plane times themselves.
__device__ __forceinline__ int cell_at(float o, float d, float inv, float t) {
  if (d > 0.0f) {
    int n = (int)floorf(__fadd_rn(o, __fmul_rn(t, d)));
    for (int it = 0; it < 64 && plane_time(n + 1, o, inv) <= t; ++it) ++n;
    for (int it = 0; it < 64 && plane_time(n, o, inv) > t; ++it) --n;
    return n;
  }
  if (d < 0.0f) {
    int m = (int)floorf(__fadd_rn(o, __fmul_rn(t, d))) + 1;
    for (int it = 0; it < 64 && plane_time(m - 1, o, inv) <= t; ++it) --m;
    for (int it = 0; it < 64 && plane_time(m, o, inv) > t; ++it) ++m;
    return m - 1;
  }
  return (int)floorf(o);
}

__device__ __forceinline__ float next_crossing(int c, float o, float d, float inv) {
  return d > 0.0f ? plane_time(c + 1, o, inv) : d < 0.0f ? plane_time(c, o, inv) : __int_as_float(0x7f800000);
}

// One ray: the counting pass counts its hits, the writing pass stores them
// from position pos.  Returns the number of hits.
template <bool kWrite>
__device__ uint32_t march(const RayArgs& a, int64_t r, uint32_t pos) {
  const int b = a.batch ? __ldg(a.batch + r) : 0;
  if (b < 0 || b >= a.B) {
    report_device_error(a.status, DEV_CHECK);
    return 0;
  }
  float o[3], d[3], inv[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    o[k] = __ldg(a.o + 3 * r + k);
    d[k] = __ldg(a.d + 3 * r + k);
  }
  if (d[0] == 0.0f && d[1] == 0.0f && d[2] == 0.0f) return 0;
  int lo[3], hi[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    lo[k] = __ldg(a.bbox + 6 * b + k);
    hi[k] = __ldg(a.bbox + 6 * b + 3 + k);
  }
  if (lo[0] > hi[0]) return 0;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    if (lo[k] < -kMaxCoord || hi[k] >= kMaxCoord) {  // cell faces no longer exact in fp32
      report_device_error(a.status, DEV_CHECK);
      return 0;
    }
  }
  float t0 = a.tmin, t1 = a.tmax;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    if (d[k] == 0.0f) {
      inv[k] = 0.0f;
      if (o[k] < __int2float_rn(lo[k]) || o[k] >= __int2float_rn(hi[k] + 1)) return 0;
      continue;
    }
    inv[k] = __fdiv_rn(1.0f, d[k]);
    float ta = plane_time(lo[k], o[k], inv[k]), tb = plane_time(hi[k] + 1, o[k], inv[k]);
    if (ta > tb) {
      const float x = ta;
      ta = tb;
      tb = x;
    }
    t0 = fmaxf(t0, ta);
    t1 = fminf(t1, tb);
  }
  if (!(t0 < t1)) return 0;
  int c[3];
  float nx[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    c[k] = cell_at(o[k], d[k], inv[k], t0);
    nx[k] = next_crossing(c[k], o[k], d[k], inv[k]);
  }
  float enter = t0;
  uint32_t nh = 0;
  const uint32_t cap = kWrite ? __ldg(a.count + r) : 0u;
  // nodes holding the current cell, cached with their origins
  int upper = -1, lower = -1, leaf = -1;
  int up_o[3] = {0, 0, 0}, lw_o[3] = {0, 0, 0}, lf_o[3] = {0, 0, 0};
  uint64_t lm[8];
  uint64_t lfirst = 0, lpre9 = 0;
  const GridDev& g = a.g;
  for (int step = 0;; ++step) {
    if (step == kMaxSteps) {
      report_device_error(a.status, DEV_CHECK);
      break;
    }
    int skip = 0;  // side of the empty box to leave in one step; 0: inside a leaf
    if (leaf < 0 || (c[0] & ~7) != lf_o[0] || (c[1] & ~7) != lf_o[1] || (c[2] & ~7) != lf_o[2]) {
      leaf = -1;
      if (lower < 0 || (c[0] & ~127) != lw_o[0] || (c[1] & ~127) != lw_o[1] || (c[2] & ~127) != lw_o[2]) {
        lower = -1;
        if (upper < 0 || (c[0] & ~4095) != up_o[0] || (c[1] & ~4095) != up_o[1] || (c[2] & ~4095) != up_o[2]) {
          upper = find_upper(g, b, c[0] >> 12, c[1] >> 12, c[2] >> 12);
#pragma unroll
          for (int k = 0; k < 3; ++k) up_o[k] = c[k] & ~4095;
        }
        if (upper < 0) {
          skip = 4096;
        } else {
          const int nu = (((c[0] >> 7) & 31) << 10) | (((c[1] >> 7) & 31) << 5) | ((c[2] >> 7) & 31);
          lower = child_index(g.upper_mask + (size_t)upper * 512, g.upper_prefix + (size_t)upper * 512,
                              __ldg(g.upper_first + upper), nu);
          if (lower < 0) skip = 128;
#pragma unroll
          for (int k = 0; k < 3; ++k) lw_o[k] = c[k] & ~127;
        }
      }
      if (!skip) {
        const int nl = (((c[0] >> 3) & 15) << 8) | (((c[1] >> 3) & 15) << 4) | ((c[2] >> 3) & 15);
        leaf = child_index(g.lower_mask + (size_t)lower * 64, g.lower_prefix + (size_t)lower * 64,
                           __ldg(g.lower_first + lower), nl);
        if (leaf < 0) {
          skip = 8;
        } else {
          const unsigned long long* rec = reinterpret_cast<const unsigned long long*>(g.leaf_rec) + (size_t)leaf * 10;
#pragma unroll
          for (int w = 0; w < 8; ++w) lm[w] = __ldg(rec + w);
          lfirst = __ldg(rec + 8);
          lpre9 = __ldg(rec + 9);
#pragma unroll
          for (int k = 0; k < 3; ++k) lf_o[k] = c[k] & ~7;
        }
      }
    }
    if (skip) {
      // leave the empty box [c & ~(skip-1), + skip) through its far faces
      float tx = __int_as_float(0x7f800000);
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        if (d[k] == 0.0f) continue;
        const int base = c[k] & ~(skip - 1);
        tx = fminf(tx, plane_time(d[k] > 0.0f ? base + skip : base, o[k], inv[k]));
      }
      if (tx >= t1) break;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        c[k] = cell_at(o[k], d[k], inv[k], tx);
        nx[k] = next_crossing(c[k], o[k], d[k], inv[k]);
      }
      enter = tx;
      continue;
    }
    // one voxel of the current leaf
    const float T = fminf(nx[0], fminf(nx[1], nx[2]));
    const float ex = fminf(T, t1);
    const int n = ((c[0] & 7) << 6) | ((c[1] & 7) << 3) | (c[2] & 7);
    const uint64_t word = lm[n >> 6];
    if (ex > enter && ((word >> (n & 63)) & 1ull)) {
      if (kWrite && nh < cap) {  // never past this ray's range (the passes agree; this only guards it)
        const int w = n >> 6;
        const uint32_t pre = w ? (uint32_t)((lpre9 >> (9 * (w - 1))) & 511ull) : 0u;
        const uint64_t below = word & ((1ull << (n & 63)) - 1ull);
        a.voxel[pos + nh] = (int32_t)(lfirst + pre + (uint32_t)__popcll(below));
        a.t[2 * (size_t)(pos + nh)] = __fadd_rn(enter, 0.0f);
        a.t[2 * (size_t)(pos + nh) + 1] = __fadd_rn(ex, 0.0f);
      }
      ++nh;
    }
    if (T >= t1) break;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      if (nx[k] != T) continue;
      c[k] += d[k] > 0.0f ? 1 : -1;
      nx[k] = next_crossing(c[k], o[k], d[k], inv[k]);
    }
    enter = T;
  }
  return nh;
}

__global__ void __launch_bounds__(kRayThreads) k_rays_count(const RayArgs a) {
  const int64_t r = (int64_t)blockIdx.x * kRayThreads + threadIdx.x;
  uint32_t nh = 0;
  if (r < a.n) {
    nh = march<false>(a, r, 0u);
    a.count[r] = nh;
  }
  // one 64-bit atomic per warp for the total (overflow check on the host)
  unsigned long long s = nh;
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) s += __shfl_down_sync(0xffffffffu, s, sh);
  if ((threadIdx.x & 31) == 0 && s) atomicAdd(a.total, s);
}

__global__ void __launch_bounds__(kRayThreads) k_rays_write(const RayArgs a) {
  const int64_t r = (int64_t)blockIdx.x * kRayThreads + threadIdx.x;
  if (r < a.n) march<true>(a, r, __ldg(a.off + r));
}

__global__ void k_ray_bbox_init(int32_t* bbox, int32_t B) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 6 * B) bbox[i] = (i % 6) < 3 ? INT_MAX : INT_MIN;
}

// Box of each batch element's leaves: min origin and max origin + 7.
__global__ void k_ray_bbox(const int32_t* __restrict__ origin, const int32_t* __restrict__ batch, int64_t n_leaf,
                           int32_t* bbox) {
  const int64_t l = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (l >= n_leaf) return;
  const int b = __ldg(batch + l);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int v = __ldg(origin + 3 * l + k);
    atomicMin(bbox + 6 * b + k, v);
    atomicMax(bbox + 6 * b + 3 + k, v + 7);
  }
}

__global__ void k_offsets64(const uint32_t* __restrict__ scan, int64_t n, uint64_t total, int64_t* out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (int64_t)__ldg(scan + i);
  if (i == n) out[n] = (int64_t)total;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace fvx

using namespace fvx;

extern "C" fvx_status fvx_voxels_along_rays(fvx_grid g, const float* origins, const float* dirs,
                                            const int32_t* ray_batch, int64_t n_rays, float tmin, float tmax,
                                            fvx_stream stream, fvx_hits* out) {
  EntryScope entry_("fvx_voxels_along_rays");
  if (!g || !out || n_rays < 0 || (n_rays > 0 && (!origins || !dirs))) {
    set_error("fvx_voxels_along_rays: NULL argument or negative ray count");
    return FVX_ERR_INVALID_ARG;
  }
  if (tmin != tmin || tmax != tmax) {
    set_error("fvx_voxels_along_rays: tmin and tmax must not be NaN");
    return FVX_ERR_INVALID_ARG;
  }
  if (n_rays >= ((int64_t)1 << 31)) {
    set_error("fvx_voxels_along_rays: %lld rays exceed 2^31 - 1", (long long)n_rays);
    return FVX_ERR_RANGE;
  }
  *out = nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  fvx_hits_s* h = new fvx_hits_s();
  struct Guard {
    fvx_hits_s** h;
    ~Guard() {
      if (*h) fvx_hits_destroy(*h);
    }
  } guard{&h};
  h->n_rays = n_rays;
  h->stream = s;
  const bool empty = n_rays == 0 || g->n_active == 0;
  Scratch scr(s);
  uint32_t* scan = nullptr;
  uint64_t total = 0;
  RayArgs a;
  memset(&a, 0, sizeof(a));
  if (!empty) {
    uint32_t* status = device_status_word();
    if (!status) {
      set_error("fvx_voxels_along_rays: device status word unavailable");
      return FVX_ERR_CUDA;
    }
    int32_t* bbox = scr.get<int32_t>((size_t)6 * g->B);
    uint32_t* counts = scr.get<uint32_t>((size_t)n_rays);
    scan = scr.get<uint32_t>((size_t)n_rays);
    unsigned long long* dtot = scr.get<unsigned long long>(1);
    if (!bbox || !counts || !scan || !dtot) return FVX_ERR_ALLOC;
    FVX_CUDA(cudaMemsetAsync(dtot, 0, 8, s));
    {
      LaunchScope ls("ray_bbox_init", s);
      k_ray_bbox_init<<<(unsigned)((6 * g->B + 255) / 256), 256, 0, s>>>(bbox, g->B);
    }
    FVX_TRY(check_launch("ray_bbox_init"));
    {
      LaunchScope ls("ray_bbox", s);
      k_ray_bbox<<<(unsigned)((g->n_leaf + 255) / 256), 256, 0, s>>>(g->leaf_origin, g->leaf_batch, g->n_leaf, bbox);
    }
    FVX_TRY(check_launch("ray_bbox"));
    a.g = grid_dev(g);
    a.o = origins;
    a.d = dirs;
    a.batch = ray_batch;
    a.n = n_rays;
    a.tmin = tmin;
    a.tmax = tmax;
    a.bbox = bbox;
    a.B = g->B;
    a.count = counts;
    a.total = dtot;
    a.status = status;
    const unsigned grid = (unsigned)((n_rays + kRayThreads - 1) / kRayThreads);
    {
      LaunchScope ls("rays_count", s);
      k_rays_count<<<grid, kRayThreads, 0, s>>>(a);
    }
    FVX_TRY(check_launch("rays_count"));
    FVX_TRY(scan_exclusive_u32(counts, scan, n_rays, nullptr, s, scr));
    // one synchronisation: the total sizes the output (never truncated)
    uint32_t* hst = (uint32_t*)pinned_staging(16);
    if (!hst) {
      set_error("fvx_voxels_along_rays: pinned staging buffer unavailable");
      return FVX_ERR_ALLOC;
    }
    FVX_CUDA(cudaMemcpyAsync(hst, dtot, 8, cudaMemcpyDeviceToHost, s));
    FVX_CUDA(cudaMemcpyAsync(hst + 2, status, 4, cudaMemcpyDeviceToHost, s));
    FVX_CUDA(cudaStreamSynchronize(s));
    memcpy(&total, hst, 8);
    if (hst[2] != 0u) {
      FVX_CUDA(cudaMemsetAsync(status, 0, 4, s));
      set_error("fvx_voxels_along_rays: %s",
                hst[2] == DEV_CHECK ? "a ray's batch index lies outside [0, B), or the grid has voxels outside "
                                      "[-2^24, 2^24) where cell faces are not exact in fp32"
                                    : "a bounded device-side wait gave up in an earlier unchecked call");
      return hst[2] == DEV_CHECK ? FVX_ERR_CHECK : FVX_ERR_DEVICE_TIMEOUT;
    }
    if (total >= ((uint64_t)1 << 31)) {
      set_error("fvx_voxels_along_rays: %llu hits exceed 2^31 - 1", (unsigned long long)total);
      return FVX_ERR_RANGE;
    }
  }
  const size_t off_b = align256(8 * ((size_t)n_rays + 1));
  const size_t vox_b = align256(4 * (size_t)total);
  h->block = dalloc(off_b + vox_b + align256(8 * (size_t)total), s);
  if (!h->block) return FVX_ERR_ALLOC;
  h->offsets = (int64_t*)h->block;
  h->voxel = (int32_t*)((char*)h->block + off_b);
  h->t = (float*)((char*)h->block + off_b + vox_b);
  h->n_hits = (int64_t)total;
  if (empty) {
    FVX_CUDA(cudaMemsetAsync(h->offsets, 0, 8 * ((size_t)n_rays + 1), s));
  } else {
    {
      LaunchScope ls("ray_offsets", s);
      k_offsets64<<<(unsigned)((n_rays + 1 + 255) / 256), 256, 0, s>>>(scan, n_rays, total, h->offsets);
    }
    FVX_TRY(check_launch("ray_offsets"));
    a.off = scan;
    a.voxel = h->voxel;
    a.t = h->t;
    {
      LaunchScope ls("rays_write", s);
      k_rays_write<<<(unsigned)((n_rays + kRayThreads - 1) / kRayThreads), kRayThreads, 0, s>>>(a);
    }
    FVX_TRY(check_launch("rays_write"));
  }
  *out = h;
  h = nullptr;
  return FVX_OK;
}

extern "C" fvx_status fvx_hits_view(fvx_hits h, const int64_t** offsets, const int32_t** voxel, const float** t,
                                    int64_t* n_hits, int64_t* n_rays) {
  if (!h) {
    set_error("fvx_hits_view: NULL handle");
    return FVX_ERR_INVALID_ARG;
  }
  if (offsets) *offsets = h->offsets;
  if (voxel) *voxel = h->voxel;
  if (t) *t = h->t;
  if (n_hits) *n_hits = h->n_hits;
  if (n_rays) *n_rays = h->n_rays;
  return FVX_OK;
}

extern "C" fvx_status fvx_hits_destroy(fvx_hits h) {
  if (!h) return FVX_OK;
  dfree(h->block, h->stream);
  delete h;
  return FVX_OK;
}
