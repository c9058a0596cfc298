// Sparse prefill attention (MInference 1.0 overview, section 2.2: "block-sparse
// computation of the attention weights and output" over the sparse index, shared
// by the vertical-slash, block-sparse and streaming heads), with the one-pass
// online softmax of FlashAttention-2 (the Novita vLLM article, "Attention
// modification", Fig. 7: keep a running row max and row sum, rescale the output,
// divide by the row sum at the end).
//
// One CTA computes 128 query rows (row blocks 2p and 2p+1) of one (batch, head)
// unit over a list of work items, each 128 keys wide:
//   * a key tile q: keys [128q, 128q+128) of the KV head, with a 4-bit quadrant
//     mask (bit a*2+b: row half a may see key half b) and the causal cut on the
//     diagonal tile;
//   * a column chunk c (vertical-slash only): gathered K/V rows of chosen keys
//     [128c, 128c+128) of the unit's ascending vertical list, each admitted for
//     a row iff the key is <= the row and outside the row block's active tiles.
//
// Warp roles (256 threads):
//   warp 0   TMA producer for Q and K (one thread)
//   warp 1   TMEM allocator and tcgen05.mma issuer (one thread)
//   warp 2   TMA producer for V (one thread)
//   warp 3   idle
//   warps 4-7 softmax: thread r owns query row r (TMEM lane r): reads S from
//            TMEM, masks, online softmax in fp32 (exp2 with log2(e) folded into
//            the scale), writes P as bf16 back over S, rescales O in TMEM when
//            the row max grows by more than 2^8, and writes the output row.
//
// TMEM (512 columns): S/P double buffer at columns [0,128) and [128,256), the
// output accumulator O at [256,384).  S = Q K^T reads Q and K from 128B-swizzled
// shared memory (K-major); O += P V reads P from TMEM and V from shared memory
// (MN-major).  Every mbarrier wait is bounded (see sm103_ptx.cuh); a timeout
// sets the status word and the CTA drains its copies and MMAs and exits.
#include "msa_internal.h"
#include "sm103_ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;
constexpr int kStagesK = 3;
constexpr int kStagesV = 2;
constexpr int kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile (two 64-column halves)
constexpr int kHalfBytes = kTileBytes / 2;
constexpr int kMaxDistWords = 1040;         // tile-distance bitset capacity (N up to 2M)
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows by > 2^8
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;

struct __align__(1024) Smem {
  uint8_t q[kTileBytes];
  uint8_t k[kStagesK][kTileBytes];
  uint8_t v[kStagesV][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full[2], p_full[2];
  uint64_t o_bar, final_bar;
  uint32_t tmem_base;
  int abort;
  uint32_t dist[kMaxDistWords];
};

struct Item {
  bool cols;      // column chunk (true) or key tile (false)
  int idx;        // key tile q or chunk c
  uint32_t qmask; // quadrant mask of a key tile
};

__device__ __forceinline__ int unit_batch(const PrefillParams& P, int unit) {
  return unit / P.units.n_heads;
}
__device__ __forceinline__ int unit_head(const PrefillParams& P, int unit) {
  return P.units.heads[unit % P.units.n_heads];
}

// Number of active 128-tile distances <= p (qdelta is ascending).
__device__ __forceinline__ int vs_tiles_upto(const PrefillParams& P, int unit, int p) {
  const int32_t* qd = P.qdelta + static_cast<int64_t>(unit) * P.g.NQ;
  int lo = 0, hi = P.qdelta_count[unit];
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (qd[mid] <= p) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ const uint32_t* vs_chunk_words(const PrefillParams& P, int unit, int p) {
  return P.col_chunks + (static_cast<int64_t>(unit) * P.g.NQ + p) * P.chunk_words;
}

__device__ __forceinline__ int vs_n_chunks(const PrefillParams& P, int unit, int p) {
  const uint32_t* w = vs_chunk_words(P, unit, p);
  int n = 0;
  for (int i = 0; i < P.chunk_words; ++i) n += __popc(w[i]);
  return n;
}

// Streaming: key tiles [0, sink_hi) and [loc_lo, p] (merged when they overlap).
__device__ __forceinline__ void st_ranges(const PrefillParams& P, int p, int& sink_hi, int& loc_lo) {
  sink_hi = min((P.init_num + 1) >> 1, p + 1);
  loc_lo = max(0, 2 * p - P.local_num + 1) >> 1;
  if (sink_hi >= loc_lo) {
    sink_hi = 0;
    loc_lo = 0;
  }
}

__device__ __forceinline__ int n_items(const PrefillParams& P, int unit, int p) {
  if (P.kind == kPrefillVS) return vs_n_chunks(P, unit, p) + vs_tiles_upto(P, unit, p);
  if (P.kind == kPrefillBS) return P.bs_tile_count[static_cast<int64_t>(unit) * P.g.NQ + p];
  int sink_hi, loc_lo;
  st_ranges(P, p, sink_hi, loc_lo);
  return sink_hi + (p - loc_lo + 1);
}

__device__ __forceinline__ bool dist_bit(const uint32_t* dist, int t) {
  return t >= 0 && ((dist[t >> 5] >> (t & 31)) & 1u);
}

// Quadrant mask of key tile q for query tile p (bit a*2 + b).
__device__ __forceinline__ uint32_t quad_mask_vs(const PrefillParams& P, const uint32_t* dist, int p, int q) {
  uint32_t mask = 0;
#pragma unroll
  for (int a = 0; a < 2; ++a) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int m = 2 * p + a, n = 2 * q + b;
      if (m < P.g.NB && n <= m && dist_bit(dist, m - n)) mask |= 1u << (a * 2 + b);
    }
  }
  return mask;
}
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

// Item i of query tile p.  Vertical-slash: column chunks first (ascending),
// then key tiles ascending (largest distance first).  `dist` may be null when
// the caller does not need the quadrant mask.
__device__ __forceinline__ Item get_item(const PrefillParams& P, int unit, int p, int i,
                                         const uint32_t* dist, int n_chunks, int n_tiles) {
  Item it;
  it.cols = false;
  it.qmask = 0xFu;
  if (P.kind == kPrefillVS) {
    if (i < n_chunks) {
      const uint32_t* w = vs_chunk_words(P, unit, p);
      int seen = 0;
      for (int x = 0;; ++x) {
        const int c = __popc(w[x]);
        if (seen + c > i) {
          uint32_t word = w[x];
          for (int skip = i - seen; skip > 0; --skip) word &= word - 1;
          it.cols = true;
          it.idx = 32 * x + (__ffs(word) - 1);
          return it;
        }
        seen += c;
      }
    }
    const int t = i - n_chunks;
    const int32_t* qd = P.qdelta + static_cast<int64_t>(unit) * P.g.NQ;
    it.idx = p - qd[n_tiles - 1 - t];
    if (dist) it.qmask = quad_mask_vs(P, dist, p, it.idx);
    return it;
  }
  if (P.kind == kPrefillBS) {
    const int32_t e = P.bs_tiles[(static_cast<int64_t>(unit) * P.g.NQ + p) * P.bs_tile_cap + i];
    it.idx = e >> 4;
    it.qmask = static_cast<uint32_t>(e & 15);
    return it;
  }
  int sink_hi, loc_lo;
  st_ranges(P, p, sink_hi, loc_lo);
  it.idx = i < sink_hi ? i : loc_lo + (i - sink_hi);
  it.qmask = quad_mask_st(P, p, it.idx);
  return it;
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  int never = 0;
  return mbar_wait(bar, parity, &never);
}

__global__ void __launch_bounds__(kThreads, 1)
sparse_prefill_kernel(const __grid_constant__ PrefillParams P, const __grid_constant__ CUtensorMap mq,
                      const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                      const __grid_constant__ CUtensorMap mkc,
                      const __grid_constant__ CUtensorMap mvc) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = blockIdx.y;
  const int p = P.g.NQ - 1 - static_cast<int>(blockIdx.x);  // heavy (late) tiles first
  const int b = unit_batch(P, unit), h = unit_head(P, unit), hkv = h / P.g.G;
  volatile int* abort = &sm.abort;

  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kStagesK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < kStagesV; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.p_full[s], 4);  // one arrival per softmax warp
    }
    mbar_init(&sm.o_bar, 1);
    mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  if (P.kind == kPrefillVS && warp >= 4) {
    const uint32_t* d = P.tile_dist + static_cast<int64_t>(unit) * P.dist_words;
    for (int w = tid - 128; w < P.dist_words; w += 128) sm.dist[w] = d[w];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  int n_chunks = 0, n_tiles = 0;
  if (P.kind == kPrefillVS) {
    n_chunks = vs_n_chunks(P, unit, p);
    n_tiles = vs_tiles_upto(P, unit, p);
  }
  const int n = n_items(P, unit, p);

  if (warp == 0) {
    // ------------------------------------------------------------ Q + K producer
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
      tma_load_4d(sm.q, &mq, &sm.q_full, 0, 128 * p, h, b);
      tma_load_4d(sm.q + kHalfBytes, &mq, &sm.q_full, 64, 128 * p, h, b);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % kStagesK;
        if (!mbar_wait(&sm.k_empty[s], ((i / kStagesK) & 1) ^ 1, abort)) break;
        const Item it = get_item(P, unit, p, i, nullptr, n_chunks, n_tiles);
        mbar_arrive_expect_tx(&sm.k_full[s], kTileBytes);
        if (it.cols) {
          const int row = unit * P.kv_pad + 128 * it.idx;
          tma_load_2d(sm.k[s], &mkc, &sm.k_full[s], 0, row);
          tma_load_2d(sm.k[s] + kHalfBytes, &mkc, &sm.k_full[s], 64, row);
        } else {
          tma_load_4d(sm.k[s], &mk, &sm.k_full[s], 0, 128 * it.idx, hkv, b);
          tma_load_4d(sm.k[s] + kHalfBytes, &mk, &sm.k_full[s], 64, 128 * it.idx, hkv, b);
        }
        issued = i + 1;
      }
      // drain: the latest load of every stage, and Q, must land before exit
      wait_drain(&sm.q_full, 0);
      for (int i = max(0, issued - kStagesK); i < issued; ++i)
        wait_drain(&sm.k_full[i % kStagesK], (i / kStagesK) & 1);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      tma_prefetch_desc(&mv);
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % kStagesV;
        if (!mbar_wait(&sm.v_empty[s], ((i / kStagesV) & 1) ^ 1, abort)) break;
        const Item it = get_item(P, unit, p, i, nullptr, n_chunks, n_tiles);
        mbar_arrive_expect_tx(&sm.v_full[s], kTileBytes);
        if (it.cols) {
          const int row = unit * P.kv_pad + 128 * it.idx;
          tma_load_2d(sm.v[s], &mvc, &sm.v_full[s], 0, row);
          tma_load_2d(sm.v[s] + kHalfBytes, &mvc, &sm.v_full[s], 64, row);
        } else {
          tma_load_4d(sm.v[s], &mv, &sm.v_full[s], 0, 128 * it.idx, hkv, b);
          tma_load_4d(sm.v[s] + kHalfBytes, &mv, &sm.v_full[s], 64, 128 * it.idx, hkv, b);
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - kStagesV); i < issued; ++i)
        wait_drain(&sm.v_full[i % kStagesV], (i / kStagesV) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_f32acc(128, 128, /*bf16=*/false, false, true);  // f16 P, f16 V
      const uint32_t q_addr = smem_u32(sm.q);
      bool ok = n == 0 || mbar_wait(&sm.q_full, 0, abort);
      tc_fence_after();
      auto issue_pv = [&](int j) -> bool {
        const int buf = j & 1, sv = j % kStagesV;
        if (!mbar_wait(&sm.p_full[buf], (j >> 1) & 1, abort)) return false;
        if (!mbar_wait(&sm.v_full[sv], (j / kStagesV) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sm.v[sv]);
        const uint32_t p_col = tmem + (buf ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = sdesc_sw128(v_addr + kk * 2048, kHalfBytes, 1024);
          mma_ts(tmem + kColO, p_col + kk * 8, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&sm.v_empty[sv]);
        mma_commit(&sm.o_bar);
        return true;
      };
      for (int i = 0; ok && i < n; ++i) {
        const int sk = i % kStagesK, buf = i & 1;
        if (!mbar_wait(&sm.k_full[sk], (i / kStagesK) & 1, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sm.k[sk]);
        const uint32_t s_col = tmem + (buf ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_ss(s_col, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                 idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&sm.s_full[buf]);
        mma_commit(&sm.k_empty[sk]);
        if (i >= 1 && !issue_pv(i - 1)) { ok = false; break; }
      }
      if (ok && n > 0) issue_pv(n - 1);
      // every MMA issued above must complete before TMEM is released
      mma_commit(&sm.final_bar);
      wait_drain(&sm.final_bar, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int r = tid - 128;                 // query row within the tile == TMEM lane
    const int half = r >> 6;                 // row block 2p + half
    const int row = 128 * p + r;             // query index i
    const int mblk = 2 * p + half;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    named_bar_sync(1, 128);                  // dist bitset copy complete
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const Item it = get_item(P, unit, p, i, sm.dist, n_chunks, n_tiles);
      const int buf = i & 1;
      const uint32_t s_col = lane_base + (buf ? kColS1 : kColS0);
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[buf], (i >> 1) & 1, abort))) { ok = false; break; }
      tc_fence_after();
      // raw logits (unscaled) of this row; scale * log2(e) is folded in below
      float x[128];
      {
        uint32_t raw[128];
        tmem_ld128(s_col, raw);
#pragma unroll
        for (int e = 0; e < 128; ++e) x[e] = __uint_as_float(raw[e]);
      }
      // ---- mask
      if (it.cols) {
        const int32_t* V = P.vertical + static_cast<int64_t>(unit) * P.kv + 128 * it.idx;
        const int valid = min(128, P.kv - 128 * it.idx);
#pragma unroll
        for (int e = 0; e < 128; ++e) {
          bool keep = false;
          if (e < valid) {
            const int j = V[e];
            keep = j <= row && !dist_bit(sm.dist, mblk - (j >> 6));
          }
          if (!keep) x[e] = -INFINITY;
        }
      } else {
        const bool lo_ok = (it.qmask >> (half * 2)) & 1u;
        const bool hi_ok = (it.qmask >> (half * 2 + 1)) & 1u;
        const bool diag = it.idx == p;
        if (!lo_ok || !hi_ok || diag) {
#pragma unroll
          for (int e = 0; e < 128; ++e) {
            const bool in_q = e < 64 ? lo_ok : hi_ok;
            if (!in_q || (diag && e > r)) x[e] = -INFINITY;
          }
        }
      }
      // ---- online softmax (8 independent partial maxima / sums per row)
      float mx8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        float m = fmax3(x[a], x[8 + a], x[16 + a]);
#pragma unroll
        for (int e = 24; e < 120; e += 16) m = fmax3(m, x[e + a], x[e + 8 + a]);
        mx8[a] = fmaxf(m, x[120 + a]);
      }
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      const float m_new = fmaxf(m_run, mx * P.scale_log2);
      const bool grow = m_new > m_run + kRescaleThreshold;  // false when both are -inf
      const float m_use = grow ? m_new : m_run;
      const float neg_base = m_use == -INFINITY ? 0.f : -m_use;
      const float2 scale2 = make_float2(P.scale_log2, P.scale_log2);
      const float2 nb2 = make_float2(neg_base, neg_base);
      float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
      uint32_t pk[64];
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        const float2 a = ffma2(make_float2(x[2 * e], x[2 * e + 1]), scale2, nb2);
        const float2 pe = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        rs2[e & 3] = fadd2(rs2[e & 3], pe);
        pk[e] = pack_f16x2(pe.x, pe.y);
      }
      const float2 rsa = fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3]));
      const float rs = rsa.x + rsa.y;
      const bool correct = grow && m_run != -INFINITY;  // O holds earlier rows' weight
      const float alpha = correct ? ex2_approx(m_run - m_new) : 1.f;
      l_run = (m_run == -INFINITY ? 0.f : l_run * alpha) + rs;
      m_run = m_use;
      // PV of the previous item must be complete before O is touched
      if (i >= 1 && !__all_sync(0xffffffffu, mbar_wait(&sm.o_bar, (i - 1) & 1, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, correct)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + 32 * c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(lane_base + kColO + 32 * c, o);
        }
      }
      {
        uint32_t lo[32], hi[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          lo[e] = pk[e];
          hi[e] = pk[32 + e];
        }
        tmem_st32(s_col, lo);
        tmem_st32(s_col + 32, hi);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[buf]);
    }
    // ---- epilogue
    uint4 outv[16];
    bool have = ok && n > 0 && l_run > 0.f;
    if (ok && n > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_bar, (n - 1) & 1, abort))) ok = false;
      tc_fence_after();
    }
    const bool warp_ok = ok;
    if (warp_ok && n > 0) {
      const float inv = have ? 1.f / l_run : 0.f;
      uint32_t o[128];
      tmem_ld128(lane_base + kColO, o);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
        w.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
        w.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
        w.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
        outv[e] = w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) outv[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (row < P.g.N && ok) {
      uint4* dst = reinterpret_cast<uint4*>(P.out + b * P.out_sb + h * P.out_sh +
                                            static_cast<int64_t>(row) * P.out_sn);
#pragma unroll
      for (int e = 0; e < 16; ++e) dst[e] = outv[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (tid == 0 && sm.abort && P.status) atomicOr(P.status, kStatusTimeout);
}


// v (bf16, any strides, [B][Hkv][N][128]) -> dst (f16, contiguous, same shape).
// The P.V product runs in f16 (P rounded to f16 keeps 3 more mantissa bits than
// bf16); every bf16 value of magnitude <= 65504 is exactly representable in
// f16 (tiny values become f16 subnormals, error < 3e-8).  Larger magnitudes
// set the range bit of the status word.
__global__ void v_to_f16_kernel(const __nv_bfloat16* __restrict__ v, int64_t sb, int64_t sh,
                                int64_t sn, int Hkv, int N, int64_t rows, __half* __restrict__ dst,
                                uint32_t* status) {
  const int64_t n16 = rows * 16;
  bool bad = false;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n16;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = idx >> 4;
    const int c = static_cast<int>(idx & 15);
    const int64_t bh = row / N;
    const int n = static_cast<int>(row % N);
    const int b = static_cast<int>(bh / Hkv), h = static_cast<int>(bh % Hkv);
    const uint4 raw = *reinterpret_cast<const uint4*>(v + b * sb + h * sh + n * sn + c * 8);
    const __nv_bfloat162* in = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __low2float(in[e]), hi = __high2float(in[e]);
      bad |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
      ow[e] = pack_f16x2(lo, hi);
    }
    *reinterpret_cast<uint4*>(dst + row * kHeadDim + c * 8) = o;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && status)
    atomicOr(status, kStatusRange);
}

}  // namespace

cudaError_t launch_v_to_f16(TensorView v, int B, int Hkv, int N, __half* dst, uint32_t* status,
                            cudaStream_t st, int* n_launch) {
  const int64_t rows = static_cast<int64_t>(B) * Hkv * N;
  int64_t blocks = (rows * 16 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  v_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(v.data, v.sb, v.sh, v.sn, Hkv, N,
                                                                 rows, dst, status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const CUtensorMap& mkc, const CUtensorMap& mvc,
                           cudaStream_t st, int* n_launch) {
  const int smem = static_cast<int>(sizeof(Smem)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(sparse_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (p.g.n_units == 0 || p.g.NQ == 0) return cudaSuccess;
  sparse_prefill_kernel<<<dim3(p.g.NQ, p.g.n_units), kThreads, smem, st>>>(p, mq, mk, mv, mkc, mvc);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
