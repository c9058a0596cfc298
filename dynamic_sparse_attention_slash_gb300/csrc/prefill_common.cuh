// Helpers shared by the two sparse prefill kernels (prefill.cu: two query
// tiles per CTA; prefill_tile.cu: one query tile per CTA).
#pragma once
#include "msa_internal.h"
#include "sm103_ptx.cuh"

namespace msa {
namespace prefill {

constexpr int kTileBytes = 128 * 128 * 2;  // one 128 x 128 16-bit tile (two 64-column halves)
constexpr int kHalfBytes = kTileBytes / 2;

__device__ __forceinline__ int unit_batch(const PrefillParams& P, int unit) {
  return unit / P.units.n_heads;
}
__device__ __forceinline__ int unit_head(const PrefillParams& P, int unit) {
  return P.units.heads[unit % P.units.n_heads];
}

__device__ __forceinline__ bool dist_bit(const uint32_t* dist, int t) {
  return t >= 0 && ((dist[t >> 5] >> (t & 31)) & 1u);
}

// dist_bit with the bit index checked against the bitset's dist_words words.
__device__ __forceinline__ bool dist_bit_checked(const PrefillParams& P, const uint32_t* dist, int t) {
  return t >= 0 && dist_bit(dist, MSA_IDX(t, 0, 32 * P.dist_words, P.status));
}

// Number of pair distances <= pB (the vertical-slash pair list is ascending).
__device__ __forceinline__ int vs_tiles_upto(const PrefillParams& P, int unit, int pB) {
  const int32_t* qd = P.qdelta + static_cast<int64_t>(unit) * (P.g.NQ + 1);  // (D << 5) | bits
  int lo = 0, hi = MSA_COUNT(P.qdelta_count[unit], P.g.NQ + 1, P.status);
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if ((qd[mid] >> 5) <= pB) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Quadrant mask of key tile q for query tile p (bit a*2 + b), streaming head.
__device__ __forceinline__ uint32_t quad_mask_st(const PrefillParams& P, int p, int q) {
  uint32_t mask = 0;
#pragma unroll
  for (int a = 0; a < 2; ++a) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int m = 2 * p + a, n = 2 * q + b;
      if (m < P.g.NB && n <= m && (n < P.init_num || n >= m - P.local_num + 1))
        mask |= 1u << (a * 2 + b);
    }
  }
  return mask;
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  int never = 0;
  return mbar_wait(bar, parity, &never);
}

}  // namespace prefill
}  // namespace msa
