// CTA-wide helpers shared by the index kernels: exclusive prefix sums and the
// order-preserving float -> uint32 key used by radix selection.
#pragma once
#include <cstdint>

namespace msa {

// Maps a float to a uint32 whose unsigned order equals the float order
// (-0.0 is folded onto +0.0 first, so the two compare equal).
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive prefix sum of `x` over the CTA in thread order; returns the
// prefix and writes the CTA total to *total.  `warp_sums` needs one int per
// warp.  Must be reached by every thread of the CTA.
template <int kThreads>
__device__ __forceinline__ int block_exclusive_scan(int x, int* warp_sums, int* total) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += y;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_sums[lane] : 0;
    int winc = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, winc, d);
      if (lane >= d) winc += y;
    }
    if (lane < kWarps) warp_sums[lane] = winc - w;  // exclusive warp offsets
    if (lane == kWarps - 1) warp_sums[kWarps] = winc;
  }
  __syncthreads();
  const int res = warp_sums[warp] + inc - x;
  *total = warp_sums[kWarps];
  __syncthreads();  // warp_sums may be reused right after
  return res;
}

}  // namespace msa
