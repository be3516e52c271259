// 3x3x3 kernel map (neighbour pair lists) over two IndexGrids.
//
// [DriveRT, "Shared neighbour maps"]: a map is identified by the coordinate
// domain (the grids), the kernel geometry (3x3x3, stride) and the row order
// (the grids' index order); building it can cost more than the convolution.
// [DriveRT, "Kernels selected per GPU"]: the 27 neighbours of a voxel form a
// bit mask, kept here per output voxel.
// [fVDB notes, "IndexGrid"]: coordinate -> index through the leaf bitmask and
// its prefix popcounts.
//
// One CTA per OUTPUT leaf.  The 27 input leaves that can hold a neighbour of
// the leaf's voxels (stride 1: origin-8 .. origin+8; stride 2: 2*origin-8 ..
// 2*origin+8, per axis) are found once by tree walks and staged in shared
// memory; every voxel-offset lookup is then a shared-memory mask test plus a
// popcount.  Pass A counts pairs per (offset, output leaf) and writes the
// 27-bit masks; a device-wide exclusive scan over the offset-major counts gives
// every (offset, leaf) its position; pass B writes the pairs, ordered by output
// inside each offset list, without atomics (deterministic).
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include "block_scan.cuh"
#include "fvx_internal.cuh"

namespace fvx {
namespace {

constexpr int kKmThreads = 256;
constexpr int kKmWarps = kKmThreads / 32;

struct KmSmem {
  unsigned long long mask[27][8];
  unsigned long long pre9[27];
  uint32_t first[27];
  int nleaf[27];
  uint16_t vox[512];
  uint32_t omask[512];
  int nvox;
  uint32_t qfirst;
  int toff[3];  // transposed map: origin / stride minus the input leaf base (0 or 4)
};

// Loads the output leaf's voxels and the 27 input leaves around a base point:
// the input point of the output leaf's origin (stride * origin), or, for the
// transposed map, the origin of the input leaf holding origin / stride.  Leaf
// origins are computed in 64 bits so that none wraps at the int32 edges.
__device__ __forceinline__ void km_prologue(KmSmem& sm, const GridDev& gin, const int32_t* __restrict__ out_origin,
                                            const int32_t* __restrict__ out_batch,
                                            const uint64_t* __restrict__ out_rec, int stride, int transposed,
                                            int lo) {
  const int tid = threadIdx.x;
  if (tid < 3) {
    const int o = out_origin[3 * lo + tid];
    const int q = stride == 2 ? (o >> 1) : o;
    sm.toff[tid] = transposed ? q - (q & ~7) : 0;
  }
  if (tid < 27) {
    const int a = tid / 9, b = (tid / 3) % 3, c = tid % 3;
    const int bt = out_batch[lo];
    long long bs[3];
#pragma unroll
    for (int e = 0; e < 3; ++e) {
      const int o = out_origin[3 * lo + e];
      bs[e] = transposed ? (long long)((stride == 2 ? (o >> 1) : o) & ~7) : (long long)stride * o;
    }
    const int l = find_leaf_wide(gin, bt, bs[0] - 8 + 8 * a, bs[1] - 8 + 8 * b, bs[2] - 8 + 8 * c);
    sm.nleaf[tid] = l;
    if (l >= 0) {
      const unsigned long long* r = reinterpret_cast<const unsigned long long*>(gin.leaf_rec) + (size_t)l * 10;
#pragma unroll
      for (int w = 0; w < 8; ++w) sm.mask[tid][w] = __ldg(r + w);
      sm.first[tid] = (uint32_t)__ldg(r + 8);
      sm.pre9[tid] = __ldg(r + 9);
    }
  }
  // active voxels of the output leaf, ascending bit number = ascending index
  const unsigned long long* orec = reinterpret_cast<const unsigned long long*>(out_rec) + (size_t)lo * 10;
  const unsigned long long pre9 = __ldg(orec + 9);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int n = tid + h * 256;
    const int w = n >> 6, bit = n & 63;
    const unsigned long long m = __ldg(orec + w);
    if ((m >> bit) & 1ull) {
      const uint32_t pre = w ? (uint32_t)((pre9 >> (9 * (w - 1))) & 511ull) : 0u;
      const uint32_t rank = pre + (uint32_t)__popcll(m & ((1ull << bit) - 1ull));
      sm.vox[rank] = (uint16_t)n;
      sm.omask[rank] = 0u;
    }
  }
  if (tid == 0) {
    sm.nvox = (int)(((pre9 >> 54) & 511ull) + (unsigned long long)__popcll(__ldg(orec + 7)));
    sm.qfirst = (uint32_t)__ldg(orec + 8);
  }
  __syncthreads();
}

// input index of the neighbour of output voxel n at offset (di, dj, dk), or -1
__device__ __forceinline__ int km_neighbour(const KmSmem& sm, int n, int stride, int di, int dj, int dk) {
  const int ri = stride * (n >> 6) + 8 + di;
  const int rj = stride * ((n >> 3) & 7) + 8 + dj;
  const int rk = stride * (n & 7) + 8 + dk;
  const int slot = (ri >> 3) * 9 + (rj >> 3) * 3 + (rk >> 3);
  if (sm.nleaf[slot] < 0) return -1;
  const int nn = ((ri & 7) << 6) | ((rj & 7) << 3) | (rk & 7);
  const int w = nn >> 6, bit = nn & 63;
  const unsigned long long m = sm.mask[slot][w];
  if (!((m >> bit) & 1ull)) return -1;
  const uint32_t pre = w ? (uint32_t)((sm.pre9[slot] >> (9 * (w - 1))) & 511ull) : 0u;
  return (int)(sm.first[slot] + pre + (uint32_t)__popcll(m & ((1ull << bit) - 1ull)));
}

// Transposed map: input index of the voxel q with stride * ijk(q) + d = ijk of
// output voxel n, or -1 (also when the division is not exact).  Works on the
// local coordinate (n's position in its leaf minus d, in [-1, 8]); the leaf
// origin is a multiple of 8, so exactness and the quotient follow from it.
__device__ __forceinline__ int km_neighbour_t(const KmSmem& sm, int n, int stride, int di, int dj, int dk) {
  const int li = (n >> 6) - di, lj = ((n >> 3) & 7) - dj, lk = (n & 7) - dk;
  const int sh = stride == 2 ? 1 : 0;
  if (sh && ((li | lj | lk) & 1)) return -1;
  // stride 1: r in [7, 16]; stride 2: li >> 1 in [0, 4], toff in {0, 4}, r in [8, 16]
  const int ri = sm.toff[0] + (li >> sh) + 8, rj = sm.toff[1] + (lj >> sh) + 8, rk = sm.toff[2] + (lk >> sh) + 8;
  const int slot = (ri >> 3) * 9 + (rj >> 3) * 3 + (rk >> 3);
  if (sm.nleaf[slot] < 0) return -1;
  const int nn = ((ri & 7) << 6) | ((rj & 7) << 3) | (rk & 7);
  const int w = nn >> 6, bit = nn & 63;
  const unsigned long long m = sm.mask[slot][w];
  if (!((m >> bit) & 1ull)) return -1;
  const uint32_t pre = w ? (uint32_t)((sm.pre9[slot] >> (9 * (w - 1))) & 511ull) : 0u;
  return (int)(sm.first[slot] + pre + (uint32_t)__popcll(m & ((1ull << bit) - 1ull)));
}

__global__ void __launch_bounds__(kKmThreads) k_kmap_count(GridDev gin, const int32_t* __restrict__ out_origin,
                                                           const int32_t* __restrict__ out_batch,
                                                           const uint64_t* __restrict__ out_rec, int64_t n_out_leaf,
                                                           int stride, int transposed, uint32_t* __restrict__ counts,
                                                           uint32_t* __restrict__ out_mask) {
  __shared__ KmSmem sm;
  const int lo = blockIdx.x;
  km_prologue(sm, gin, out_origin, out_batch, out_rec, stride, transposed, lo);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int s = warp; s < 27; s += kKmWarps) {
    const int di = s / 9 - 1, dj = (s / 3) % 3 - 1, dk = s % 3 - 1;
    uint32_t cnt = 0;
    for (int c0 = 0; c0 < sm.nvox; c0 += 32) {
      const int idx = c0 + lane;
      const int p = (idx < sm.nvox) ? (transposed ? km_neighbour_t(sm, sm.vox[idx], stride, di, dj, dk)
                                                  : km_neighbour(sm, sm.vox[idx], stride, di, dj, dk))
                                    : -1;
      cnt += __popc(__ballot_sync(0xffffffffu, p >= 0));
      if (p >= 0) atomicOr(&sm.omask[idx], 1u << s);
    }
    if (lane == 0) counts[(int64_t)s * n_out_leaf + lo] = cnt;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < sm.nvox; idx += kKmThreads) out_mask[sm.qfirst + idx] = sm.omask[idx];
}

__global__ void __launch_bounds__(kKmThreads) k_kmap_write(GridDev gin, const int32_t* __restrict__ out_origin,
                                                           const int32_t* __restrict__ out_batch,
                                                           const uint64_t* __restrict__ out_rec, int64_t n_out_leaf,
                                                           int stride, int transposed,
                                                           const uint32_t* __restrict__ starts,
                                                           int32_t* __restrict__ in_idx,
                                                           int32_t* __restrict__ out_idx) {
  __shared__ KmSmem sm;
  const int lo = blockIdx.x;
  km_prologue(sm, gin, out_origin, out_batch, out_rec, stride, transposed, lo);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t lt = lanemask_lt();
  for (int s = warp; s < 27; s += kKmWarps) {
    const int di = s / 9 - 1, dj = (s / 3) % 3 - 1, dk = s % 3 - 1;
    uint32_t pos = starts[(int64_t)s * n_out_leaf + lo];
    for (int c0 = 0; c0 < sm.nvox; c0 += 32) {
      const int idx = c0 + lane;
      const int p = (idx < sm.nvox) ? (transposed ? km_neighbour_t(sm, sm.vox[idx], stride, di, dj, dk)
                                                  : km_neighbour(sm, sm.vox[idx], stride, di, dj, dk))
                                    : -1;
      const uint32_t bal = __ballot_sync(0xffffffffu, p >= 0);
      if (p >= 0) {
        const uint32_t e = pos + __popc(bal & lt);
        in_idx[e] = p;
        out_idx[e] = (int32_t)(sm.qfirst + idx);
      }
      pos += __popc(bal);
    }
  }
}

// ------------------------------------------------------------------ stride 1,
// bit-parallel.  A leaf mask is 8 words (word x = one x slice, bit y*8+z).
// For offset d the output voxels of leaf O that have an input neighbour at
// O + (x,y,z) + d are  out_word[x] & shifted_in_word(x, d): the input word of
// slice x+dx, shifted by dy rows and dz bits, with the rows / bits that cross
// the leaf border taken from the y / z / yz neighbour leaves.
struct Km1Smem {
  unsigned long long im[27][8];  // input leaf masks of the 27 slots (0 if absent)
  unsigned long long pre9[27];
  uint32_t first[27];
  unsigned long long R[27][8];   // per offset: output voxels with a neighbour there
  unsigned long long om[8];
  unsigned long long opre9;
  uint32_t qf;
  int nvox;
  uint16_t vox[512];
};

__device__ __forceinline__ unsigned long long shift_rows(unsigned long long c, unsigned long long nb, int dj) {
  return dj == 0 ? c : (dj > 0 ? (c >> 8) | (nb << 56) : (c << 8) | (nb >> 56));
}
__device__ __forceinline__ unsigned long long shift_bits(unsigned long long v, unsigned long long vz, int dk) {
  return dk == 0 ? v
                 : (dk > 0 ? ((v >> 1) & 0x7F7F7F7F7F7F7F7Full) | ((vz & 0x0101010101010101ull) << 7)
                           : ((v << 1) & 0xFEFEFEFEFEFEFEFEull) | ((vz & 0x8080808080808080ull) >> 7));
}

__device__ __forceinline__ unsigned long long km1_word(const Km1Smem& sm, int s, int x) {
  const int di = s / 9 - 1, dj = (s / 3) % 3 - 1, dk = s % 3 - 1;
  const int xs = x + di;
  const int a = (xs + 8) >> 3, xw = xs & 7;
  const unsigned long long A = sm.im[a * 9 + 4][xw];
  const unsigned long long Y = dj ? sm.im[a * 9 + (1 + dj) * 3 + 1][xw] : 0ull;
  const unsigned long long Z = dk ? sm.im[a * 9 + 3 + (1 + dk)][xw] : 0ull;
  const unsigned long long YZ = (dj && dk) ? sm.im[a * 9 + (1 + dj) * 3 + (1 + dk)][xw] : 0ull;
  return sm.om[x] & shift_bits(shift_rows(A, Y, dj), shift_rows(Z, YZ, dj), dk);
}

// Loads the output leaf and its 27 input-leaf slots (tree walks, or the slot
// table written by k_kmap1_nbr).
__device__ __forceinline__ void km1_load(Km1Smem& sm, const GridDev& gin, const int32_t* __restrict__ out_origin,
                                         const int32_t* __restrict__ out_batch,
                                         const uint64_t* __restrict__ out_rec, int lo,
                                         const int32_t* __restrict__ nbr_in, int32_t* __restrict__ nbr_out) {
  const int tid = threadIdx.x;
  if (tid < 27) {
    int l;
    if (nbr_in) {
      l = nbr_in[(int64_t)lo * 27 + tid];
    } else {
      const int a = tid / 9, b = (tid / 3) % 3, c = tid % 3;
      l = find_leaf_wide(gin, out_batch[lo], (long long)out_origin[3 * lo] - 8 + 8 * a,
                         (long long)out_origin[3 * lo + 1] - 8 + 8 * b, (long long)out_origin[3 * lo + 2] - 8 + 8 * c);
      if (nbr_out) nbr_out[(int64_t)lo * 27 + tid] = l;
    }
    const unsigned long long* r = reinterpret_cast<const unsigned long long*>(gin.leaf_rec) + (size_t)(l < 0 ? 0 : l) * 10;
#pragma unroll
    for (int w = 0; w < 8; ++w) sm.im[tid][w] = l >= 0 ? __ldg(r + w) : 0ull;
    sm.first[tid] = l >= 0 ? (uint32_t)__ldg(r + 8) : 0u;
    sm.pre9[tid] = l >= 0 ? __ldg(r + 9) : 0ull;
  } else if (tid >= 32 && tid < 42) {
    const unsigned long long v = __ldg(reinterpret_cast<const unsigned long long*>(out_rec) + (size_t)lo * 10 + (tid - 32));
    if (tid < 40) sm.om[tid - 32] = v;
    else if (tid == 40) sm.qf = (uint32_t)v;
    else sm.opre9 = v;
  }
  __syncthreads();
}

// The 27 input leaves around every output leaf (slot (a,b,c): the leaf at
// origin - 8 + 8 * (a,b,c)), one tree walk per thread: the walks' dependent
// loads overlap across many threads instead of 27 per block.
__global__ void __launch_bounds__(256) k_kmap1_nbr(GridDev gin, const int32_t* __restrict__ out_origin,
                                                   const int32_t* __restrict__ out_batch, int64_t n_out_leaf,
                                                   int32_t* __restrict__ nbr) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= 27 * n_out_leaf) return;
  const int64_t lo = e / 27;
  const int t = (int)(e - lo * 27);
  const int a = t / 9, b = (t / 3) % 3, c = t % 3;
  nbr[e] = find_leaf_wide(gin, out_batch[lo], (long long)out_origin[3 * lo] - 8 + 8 * a,
                          (long long)out_origin[3 * lo + 1] - 8 + 8 * b, (long long)out_origin[3 * lo + 2] - 8 + 8 * c);
}

__global__ void __launch_bounds__(kKmThreads) k_kmap1_count(GridDev gin, const int32_t* __restrict__ out_origin,
                                                            const int32_t* __restrict__ out_batch,
                                                            const uint64_t* __restrict__ out_rec, int64_t n_out_leaf,
                                                            uint32_t* __restrict__ counts,
                                                            uint32_t* __restrict__ out_mask,
                                                            const int32_t* __restrict__ nbr_in, int mirror) {
  __shared__ Km1Smem sm;
  const int lo = blockIdx.x, tid = threadIdx.x;
  km1_load(sm, gin, out_origin, out_batch, out_rec, lo, nbr_in, nullptr);
  const int s = tid >> 3, x = tid & 7;
  const unsigned long long R = (s < 27) ? km1_word(sm, s, x) : 0ull;
  if (s < 27) sm.R[s][x] = R;
  uint32_t c = (uint32_t)__popcll(R);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 4);
  if (s < 27 && x == 0) counts[(int64_t)(mirror ? 26 - s : s) * n_out_leaf + lo] = c;
  // active output voxels in index order
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int n = tid + h * 256;
    const int w = n >> 6, bit = n & 63;
    const unsigned long long m = sm.om[w];
    if ((m >> bit) & 1ull) {
      const uint32_t pre = w ? (uint32_t)((sm.opre9 >> (9 * (w - 1))) & 511ull) : 0u;
      sm.vox[pre + (uint32_t)__popcll(m & ((1ull << bit) - 1ull))] = (uint16_t)n;
    }
  }
  if (tid == 0) sm.nvox = (int)(((sm.opre9 >> 54) & 511ull) + (unsigned long long)__popcll(sm.om[7]));
  __syncthreads();
  for (int idx = tid; idx < sm.nvox; idx += kKmThreads) {
    const int n = sm.vox[idx], w = n >> 6, bit = n & 63;
    uint32_t mk = 0;
#pragma unroll
    for (int t = 0; t < 27; ++t) mk |= (uint32_t)((sm.R[t][w] >> bit) & 1ull) << (mirror ? 26 - t : t);
    out_mask[sm.qf + idx] = mk;
  }
}

// Input index of every position of the output leaf's one-voxel halo
// (10^3 positions, -1 where no input voxel is active), from the 27 slots, and
// where each (offset, slice) run of the leaf's pairs starts in its list.
struct Km1WriteSmem {
  Km1Smem k;
  int32_t hidx[1000];   // (hx+1)*100 + (hy+1)*10 + (hz+1), h in -1..8
  uint32_t pos0[27][8]; // list position of the first pair of (offset s, slice x)
};

// One thread per active output voxel (index order), looping over the 27
// offsets in step: a voxel with a neighbour at offset s writes its pair at
// its rank among the leaf's voxels with that neighbour, so the lanes of a
// warp write consecutive entries of one list at a time.  Work scales with the
// leaf's active voxels, not with its 512 positions.
// kKm1WriteThreads: 128 for sparse leaves (a narrow band's leaf holds about
// 113 voxels, so a 256-thread block would idle half its warps in the voxel
// loop), 256 for leaves with more than 200 voxels on average.
template <int kKm1WriteThreads>
__global__ void __launch_bounds__(kKm1WriteThreads) k_kmap1_write(GridDev gin, const int32_t* __restrict__ out_origin,
                                                            const int32_t* __restrict__ out_batch,
                                                            const uint64_t* __restrict__ out_rec, int64_t n_out_leaf,
                                                            const uint32_t* __restrict__ starts,
                                                            const int32_t* __restrict__ nbr_in,
                                                            int32_t* __restrict__ in_idx,
                                                            int32_t* __restrict__ out_idx, int mirror) {
  static_assert(512 % kKm1WriteThreads == 0 && kKm1WriteThreads % 32 == 0 && kKm1WriteThreads >= 64,
                "the writer's loops over 512 positions and 256 (offset, slice) entries");
  __shared__ Km1WriteSmem sw;
  Km1Smem& sm = sw.k;
  const int lo = blockIdx.x, tid = threadIdx.x;
  km1_load(sm, gin, out_origin, out_batch, out_rec, lo, nbr_in, nullptr);
  for (int h = tid; h < 1000; h += kKm1WriteThreads) {
    const int hx = h / 100 - 1, hy = (h / 10) % 10 - 1, hz = h % 10 - 1;
    const int slot = ((hx + 8) >> 3) * 9 + ((hy + 8) >> 3) * 3 + ((hz + 8) >> 3);
    const int w = hx & 7, bit = ((hy & 7) << 3) | (hz & 7);
    const unsigned long long m = sm.im[slot][w];
    int32_t v = -1;
    if ((m >> bit) & 1ull) {
      const uint32_t pre = w ? (uint32_t)((sm.pre9[slot] >> (9 * (w - 1))) & 511ull) : 0u;
      v = (int32_t)(sm.first[slot] + pre + (uint32_t)__popcll(m & ((1ull << bit) - 1ull)));
    }
    sw.hidx[h] = v;
  }
  // the neighbour words of every (offset, slice), as the count pass had
  // them; entry e = s * 8 + x, so the eight slices of an offset are eight
  // consecutive lanes and their running pair counts one segmented scan
#pragma unroll
  for (int e0 = 0; e0 < 256; e0 += kKm1WriteThreads) {
    const int s = (e0 + tid) >> 3, x = tid & 7;
    const unsigned long long R = (s < 27) ? km1_word(sm, s, x) : 0ull;
    const uint32_t c = (uint32_t)__popcll(R);
    uint32_t incl = c;
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, d, 8);
      if (x >= d) incl += v;
    }
    if (s < 27) {
      sm.R[s][x] = R;
      sw.pos0[s][x] = starts[(int64_t)(mirror ? 26 - s : s) * n_out_leaf + lo] + incl - c;
    }
  }
  // active output voxels in index order
#pragma unroll
  for (int h = 0; h < 512 / kKm1WriteThreads; ++h) {
    const int n = tid + h * kKm1WriteThreads;
    const int w = n >> 6, bit = n & 63;
    const unsigned long long m = sm.om[w];
    if ((m >> bit) & 1ull) {
      const uint32_t pre = w ? (uint32_t)((sm.opre9 >> (9 * (w - 1))) & 511ull) : 0u;
      sm.vox[pre + (uint32_t)__popcll(m & ((1ull << bit) - 1ull))] = (uint16_t)n;
    }
  }
  const int nvox = (int)(((sm.opre9 >> 54) & 511ull) + (unsigned long long)__popcll(sm.om[7]));
  __syncthreads();
  for (int idx = tid; idx < nvox; idx += kKm1WriteThreads) {
    const int n = sm.vox[idx], x = n >> 6, b = n & 63;
    const unsigned long long below = (1ull << b) - 1ull;
    const int h0 = (x + 1) * 100 + ((b >> 3) + 1) * 10 + (b & 7) + 1;  // the voxel's own halo position
    const int32_t q = (int32_t)(sm.qf + (uint32_t)idx);
#pragma unroll
    for (int s = 0; s < 27; ++s) {
      const unsigned long long R = sm.R[s][x];
      if ((R >> b) & 1ull) {
        const uint32_t pos = sw.pos0[s][x] + (uint32_t)__popcll(R & below);
        in_idx[pos] = sw.hidx[h0 + (s / 9 - 1) * 100 + ((s / 3) % 3 - 1) * 10 + (s % 3 - 1)];
        out_idx[pos] = q;
      }
    }
  }
}

__global__ void k_list_offsets(const uint32_t* __restrict__ starts, int64_t n_out_leaf, const uint32_t* total,
                               uint32_t* __restrict__ out) {
  const int s = threadIdx.x;
  if (s < 27) out[s] = (n_out_leaf > 0) ? starts[(int64_t)s * n_out_leaf] : 0u;
  if (s == 27) out[27] = *total;
}

// per conv tile of kTileRows outputs: number of outputs with mask bit s
// (one warp per tile: lane r holds the masks of rows r, r+32, r+64, r+96)
__global__ void __launch_bounds__(256) k_tile_counts(const uint32_t* __restrict__ mask, int64_t n_out,
                                                     int64_t ntiles, uint32_t* __restrict__ cnt) {
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= ntiles) return;
  uint32_t m[kTileRows / 32];
#pragma unroll
  for (int h = 0; h < kTileRows / 32; ++h) {
    const int64_t q = t * kTileRows + h * 32 + lane;
    m[h] = (q < n_out) ? mask[q] : 0u;
  }
  uint32_t mine = 0;  // lane s keeps the count of offset s
#pragma unroll
  for (int s = 0; s < 27; ++s) {
    uint32_t c = 0;
#pragma unroll
    for (int h = 0; h < kTileRows / 32; ++h) c += __popc(__ballot_sync(0xffffffffu, (m[h] >> s) & 1u));
    if (lane == s) mine = c;
  }
  if (lane < 27) cnt[(int64_t)lane * ntiles + t] = mine;
}

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace fvx

using namespace fvx;

size_t fvx::kmap_capacity_limit() {
  static size_t limit = [] {
    const char* e = getenv("FVX_KMAP_CAP_BYTES");
    return e ? (size_t)strtoull(e, nullptr, 10) : ((size_t)8 << 30);
  }();
  return limit;
}

// Copies the map's 28 list offsets to the host (synchronising its stream) and
// checks the device status word for a wait that gave up meanwhile.
fvx_status fvx::kmap_read_totals(fvx_kmap_s* m, const char* who) {
  if (m->host_ready) return FVX_OK;
  uint32_t* h = (uint32_t*)pinned_staging(29 * 4);
  uint32_t* dstat = device_status_word();
  if (!h || !dstat) {
    set_error("%s: staging buffer or device status word unavailable", who);
    return FVX_ERR_ALLOC;
  }
  FVX_CUDA(cudaMemcpyAsync(h, m->dtot, 28 * 4, cudaMemcpyDeviceToHost, m->stream));
  FVX_CUDA(cudaMemcpyAsync(h + 28, dstat, 4, cudaMemcpyDeviceToHost, m->stream));
  FVX_CUDA(cudaStreamSynchronize(m->stream));
  FVX_TRY(check_staged_status(who, h[28], m->stream));
  for (int t = 0; t < 28; ++t) m->offsets_host[t] = h[t];
  m->n_pairs = m->offsets_host[27];
  m->host_ready = true;
  return FVX_OK;
}

namespace {
fvx_status kernel_map_impl(const char* who, fvx_grid gin, fvx_grid gout, int32_t ksize, int32_t stride,
                           bool transposed, fvx_stream stream, fvx_kmap* out) {
  if (!gin || !gout || !out) {
    set_error("%s: NULL argument", who);
    return FVX_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (ksize != 3 || (stride != 1 && stride != 2)) {
    set_error("%s: need ksize == 3 and stride 1 or 2 (got %d, %d)", who, ksize, stride);
    return FVX_ERR_INVALID_ARG;
  }
  if (gin->B != gout->B) {
    set_error("%s: batch sizes differ (%d vs %d)", who, gin->B, gout->B);
    return FVX_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  Scratch scr(s);
  fvx_kmap_s* m = new fvx_kmap_s();
  struct Guard {
    fvx_kmap_s** m;
    ~Guard() {
      if (*m) fvx_kmap_destroy(*m);
    }
  } guard{&m};
  m->stride = stride;
  m->transposed = transposed;
  m->n_out = gout->n_active;
  m->stream = s;
  m->gin = gin;
  m->gout = gout;
  const int64_t Lo = gout->n_leaf, Nout = gout->n_active;
  m->n_tiles = (Nout + kTileRows - 1) / kTileRows;

  uint32_t* counts = scr.get<uint32_t>((size_t)(27 * Lo + 1));
  if (!counts) return FVX_ERR_ALLOC;
  // mask, list totals and conv tiling live in the first block, pairs in the
  // second (and, for stride 1, the input-leaf slot table k_kmap1_nbr
  // writes, which the leaf-densified convolution reads too)
  const size_t o_mask = 0, o_tot = align_up(4 * (size_t)Nout), o_tile = o_tot + align_up(4 * 32);
  const size_t o_nbr = o_tile + align_up(4 * (size_t)(27 * m->n_tiles + 1));
  // Stride 1 runs the bit-parallel kernels.  Its transposed map pairs output
  // p with the input at p - d, which the forward map lists under the mirrored
  // offset -d (slot 26 - s): the same kernels write each list to slot 26 - s.
  const bool bitpar = stride == 1;
  const size_t bytes1 = o_nbr + (bitpar ? align_up(4 * (size_t)(27 * Lo + 1)) : 0);
  m->block = dalloc(bytes1, s);
  if (!m->block) return FVX_ERR_ALLOC;
  m->out_mask = (uint32_t*)((char*)m->block + o_mask);
  m->dtot = (uint32_t*)((char*)m->block + o_tot);
  m->tile_start = (uint32_t*)((char*)m->block + o_tile);
  uint32_t* const dtot = m->dtot;
  // Pair lists sized for every output having all 27 neighbours, so the map
  // is built without reading the pair count back; past kMapCapBytes (or the
  // int32 pair index range) the count is read first and the lists are exact.
  const int64_t cap = 27 * Nout;
  const bool by_capacity = cap < (int64_t)INT32_MAX && (size_t)cap * 8 <= kmap_capacity_limit();
  if (by_capacity) {
    m->pair_capacity = cap;
    m->block2 = dalloc(2 * align_up(4 * (size_t)cap), s);
    if (!m->block2) return FVX_ERR_ALLOC;
    m->in_idx = (int32_t*)m->block2;
    m->out_idx = (int32_t*)((char*)m->block2 + align_up(4 * (size_t)cap));
  }

  const GridDev gd = grid_dev(gin);
  int32_t* nbr = nullptr;  // stride 1: input-leaf slot table (k_kmap1_nbr)
  if (bitpar) {
    nbr = (int32_t*)((char*)m->block + o_nbr);
    (transposed ? m->leaf_nbr_t : m->leaf_nbr) = nbr;  // the forward conv's leaf path takes forward maps only
  }
  if (Lo > 0 && bitpar) {
    LaunchScope ls("kmap_nbr", s);
    k_kmap1_nbr<<<(unsigned)((27 * Lo + 255) / 256), 256, 0, s>>>(gd, gout->leaf_origin, gout->leaf_batch, Lo, nbr);
  }
  FVX_TRY(check_launch("kmap_nbr"));
  if (Lo > 0) {
    LaunchScope ls("kmap_count", s);
    if (bitpar)
      k_kmap1_count<<<(unsigned)Lo, kKmThreads, 0, s>>>(gd, gout->leaf_origin, gout->leaf_batch, gout->leaf_rec, Lo,
                                                        counts, m->out_mask, nbr, transposed ? 1 : 0);
    else
      k_kmap_count<<<(unsigned)Lo, kKmThreads, 0, s>>>(gd, gout->leaf_origin, gout->leaf_batch, gout->leaf_rec, Lo,
                                                       stride, transposed ? 1 : 0, counts, m->out_mask);
  }
  FVX_TRY(check_launch("kmap_count"));
  FVX_TRY(scan_exclusive_u32(counts, counts, 27 * Lo, dtot + 28, s, scr));
  {
    LaunchScope ls("kmap_list_offsets", s);
    k_list_offsets<<<1, 32, 0, s>>>(counts, Lo, dtot + 28, dtot);
  }
  FVX_TRY(check_launch("kmap_list_offsets"));
  if (!by_capacity) {
    FVX_TRY(kmap_read_totals(m, who));
    const int64_t P = m->n_pairs;
    if (P >= (int64_t)INT32_MAX) {
      set_error("%s: %lld pairs exceed the int32 pair index range", who, (long long)P);
      return FVX_ERR_RANGE;
    }
    m->pair_capacity = P;
    m->block2 = dalloc(2 * align_up(4 * (size_t)P), s);
    if (!m->block2) return FVX_ERR_ALLOC;
    m->in_idx = (int32_t*)m->block2;
    m->out_idx = (int32_t*)((char*)m->block2 + align_up(4 * (size_t)P));
  }
  if (Lo > 0 && m->pair_capacity > 0) {
    LaunchScope ls("kmap_write", s);
    if (bitpar) {
      if ((double)Nout > 200.0 * (double)Lo)
        k_kmap1_write<256><<<(unsigned)Lo, 256, 0, s>>>(gd, gout->leaf_origin, gout->leaf_batch, gout->leaf_rec, Lo,
                                                        counts, nbr, m->in_idx, m->out_idx, transposed ? 1 : 0);
      else
        k_kmap1_write<128><<<(unsigned)Lo, 128, 0, s>>>(gd, gout->leaf_origin, gout->leaf_batch, gout->leaf_rec, Lo,
                                                        counts, nbr, m->in_idx, m->out_idx, transposed ? 1 : 0);
    } else {
      k_kmap_write<<<(unsigned)Lo, kKmThreads, 0, s>>>(gd, gout->leaf_origin, gout->leaf_batch, gout->leaf_rec, Lo,
                                                       stride, transposed ? 1 : 0, counts, m->in_idx, m->out_idx);
    }
  }
  FVX_TRY(check_launch("kmap_write"));
  // conv tiling: where each tile's pairs start in every list
  if (m->n_tiles > 0) {
    {
      LaunchScope ls("kmap_tile_counts", s);
      k_tile_counts<<<(unsigned)((m->n_tiles * 32 + 255) / 256), 256, 0, s>>>(m->out_mask, Nout, m->n_tiles,
                                                                             m->tile_start);
    }
    FVX_TRY(check_launch("kmap_tile_counts"));
  }
  FVX_TRY(scan_exclusive_u32(m->tile_start, m->tile_start, 27 * m->n_tiles, m->tile_start + 27 * m->n_tiles, s, scr));
  *out = m;
  m = nullptr;
  return FVX_OK;
}
}  // namespace

extern "C" fvx_status fvx_kernel_map(fvx_grid gin, fvx_grid gout, int32_t ksize, int32_t stride, fvx_stream stream,
                                     fvx_kmap* out) {
  EntryScope entry_("fvx_kernel_map");
  return kernel_map_impl("fvx_kernel_map", gin, gout, ksize, stride, false, stream, out);
}

extern "C" fvx_status fvx_kernel_map_transposed(fvx_grid gin, fvx_grid gout, int32_t ksize, int32_t stride,
                                                fvx_stream stream, fvx_kmap* out) {
  EntryScope entry_("fvx_kernel_map_transposed");
  return kernel_map_impl("fvx_kernel_map_transposed", gin, gout, ksize, stride, true, stream, out);
}
