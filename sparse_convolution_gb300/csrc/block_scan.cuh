// Warp- and block-level scan helpers (device only).
#pragma once
#include <stdint.h>

namespace fvx {

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

template <class T>
__device__ __forceinline__ T warp_inclusive_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

template <class T>
__device__ __forceinline__ T warp_reduce_sum(T v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// Exclusive scan across the whole block (blockDim.x a multiple of 32, at most
// 1024).  `tmp` is shared scratch of >= 33 elements.  Returns the exclusive
// prefix of v; *total receives the block total.  Contains __syncthreads().
template <class T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* tmp, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  T inc = warp_inclusive_scan(v);
  if (lane == 31) tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T w = (lane < nwarps) ? tmp[lane] : T(0);
    T wi = warp_inclusive_scan(w);
    if (lane < nwarps) tmp[lane] = wi - w;
    if (lane == nwarps - 1) tmp[32] = wi;
  }
  __syncthreads();
  T res = tmp[warp] + inc - v;
  if (total) *total = tmp[32];
  __syncthreads();
  return res;
}

}  // namespace fvx
