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

// Admission of a vertical-slash column chunk's keys for the 32 rows of one
// warp, which all lie in row block mblk: keys kbase .. kbase + 32 W - 1 of the
// unit's ascending vertical list V (those at or past kv do not exist).  A key
// j is admitted for row i iff j <= i and its 64x64 tile is not active for the
// row block (tile distance mblk - j/64 not in the bitset).  Every row of the
// warp admits the keys of earlier blocks alike, so lane l loads keys
// kbase + l + 32 q and four (or W) ballots give the warp the bits: adm (a key of
// an earlier block whose tile is inactive) and own (a key of block mblk
// itself, admitted iff j <= i: only those need the row; the caller fetches
// their j by shuffle from jv).
template <int W>
__device__ __forceinline__ void column_bits(const PrefillParams& P, const int32_t* V, int kbase,
                                            const uint32_t* dist, int mblk, uint32_t (&adm)[W],
                                            uint32_t (&own)[W], int (&jv)[W]) {
  const int lane = threadIdx.x & 31;
  const bool own_tile = dist_bit_checked(P, dist, 0);  // block mblk's own tile is active
#pragma unroll
  for (int q = 0; q < W; ++q) {
    const int s = kbase + 32 * q + lane;
    bool a = false, o = false;
    int j = 0x7fffffff;
    if (s < P.kv) {
      j = MSA_IDX(V[s], 0, P.g.N, P.status);
      const int nb = j >> 6;
      a = nb < mblk && !dist_bit_checked(P, dist, mblk - nb);
      o = nb == mblk && !own_tile;
    }
    jv[q] = j;
    adm[q] = __ballot_sync(0xffffffffu, a);
    own[q] = __ballot_sync(0xffffffffu, o);
  }
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
