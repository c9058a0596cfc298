// Sparse prefill attention (MInference 1.0 overview, section 2.2: "block-sparse
// computation of the attention weights and output" over the sparse index, shared
// by the vertical-slash, block-sparse and streaming heads), with the one-pass
// online softmax of FlashAttention-2 (the Novita vLLM article, "Attention
// modification", Fig. 7: keep a running row max and row sum, rescale the output,
// divide by the row sum at the end).
//
// One CTA computes 256 query rows of one (batch, head) unit: two adjacent
// 128-row query tiles pA = 2c and pB = 2c + 1 (row blocks 4c .. 4c+3), which
// share every K/V tile they load.  Work items are 128 keys wide:
//   * a key tile q: keys [128q, 128q+128) of the KV head, with a 4-bit quadrant
//     mask per query tile (bit a*2+b: row half a may see key half b) and the
//     causal cut on each tile's diagonal;
//   * a column chunk c (vertical-slash only): gathered K/V rows of chosen keys
//     [128c, 128c+128) of the unit's ascending vertical list, each admitted for
//     a row iff the key is <= the row and outside the row block's active tiles.
// The item list is the union of the two query tiles' lists; a tile that does
// not use an item sees it fully masked.  (Skipping such items per tile was
// measured slower on GB300: it lengthens the single MMA thread's issue path,
// which the tensor core waits on.)  Block-sparse heads, whose per-tile lists
// are short and sparse, run the one-tile kernel of prefill_tile.cu instead.
//
// Warp roles (384 threads; the control warpgroup gives registers to the two
// softmax warpgroups with setmaxnreg):
//   warp 0    TMA producer for Q and K (one thread)
//   warp 1    TMEM allocator and tcgen05.mma issuer (one thread)
//   warp 2    TMA producer for V (one thread)
//   warp 3    idle
//   warps 4-7 softmax of query tile A, warps 8-11 of query tile B: thread r owns
//            query row r of its tile (TMEM lane r): reads S from TMEM, masks,
//            runs the online softmax in fp32 (exp2 with log2(e) folded into the
//            scale) against the row's running max, takes the row max (and
//            rescales O in TMEM) only when the item's row sum would let a P
//            value leave the f16 range, writes P as f16 back over S, and writes
//            the output row.
//
// TMEM (512 columns): S/P of tile A at [0,128), of tile B at [128,256); the
// output accumulators O_A at [256,384) and O_B at [384,512).  S = Q K^T reads Q
// and K from 128B-swizzled shared memory (K-major); O += P V reads P from TMEM
// and V from shared memory (MN-major).  The MMA issue order per item i is
// PV_A(i-1), S_A(i), PV_B(i-1), S_B(i): since tcgen05 operations of one thread
// complete in order, the completion of S_t(i) also certifies that PV_t(i-1) is
// done, so the softmax may rescale O_t without another wait, while the tensor
// core works on the other tile.  Every mbarrier wait is bounded (see
// sm103_ptx.cuh); a timeout sets the status word and the CTA drains its copies
// and MMAs and exits.
#include "prefill_common.cuh"

namespace msa {
namespace {

using namespace prefill;

constexpr int kThreads = 384;
constexpr int kStagesK = 3;
constexpr int kStagesV = 2;
// A row sum of at most 2^15 bounds every p of the item by it: P fits f16.
constexpr float kSumLimit = 32768.f;
// TMEM columns: S/P of tile t at kColS + 128 t, O of tile t at kColO + 128 t
constexpr uint32_t kColS = 0, kColO = 256;
// Register split: the control warpgroup drops to kCtrlRegs, the two softmax
// warpgroups rise to kSoftRegs.  128 * 64 + 256 * 208 = 61440 registers, within
// the 384 * 160 = 61440 the launch is checked to provide.
constexpr int kCtrlRegs = 64;
constexpr int kSoftRegs = 208;
constexpr int kMinLaunchRegs = 160;

struct __align__(1024) Smem {
  uint8_t q[2][kTileBytes];
  uint8_t k[kStagesK][kTileBytes];
  uint8_t v[kStagesV][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t final_bar;
  uint32_t tmem_base;
  int abort;
};

struct Item {
  bool cols;          // column chunk (true) or key tile (false)
  int idx;            // key tile q or chunk c
  uint32_t qmask[2];  // quadrant masks of a key tile for query tiles A and B
};

__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
}
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
}

// Column-chunk word x of the pair: chunks needed by query tile pA or pB.
__device__ __forceinline__ uint32_t vs_chunk_word(const PrefillParams& P, int unit, int pA, int x) {
  const uint32_t* w = P.col_chunks + (static_cast<int64_t>(unit) * P.g.NQ + pA) * P.chunk_words;
  uint32_t word = w[x];
  if (pA + 1 < P.g.NQ) word |= w[P.chunk_words + x];
  return word;
}

__device__ __forceinline__ int vs_n_chunks(const PrefillParams& P, int unit, int pA) {
  int n = 0;
  for (int x = 0; x < P.chunk_words; ++x) n += __popc(vs_chunk_word(P, unit, pA, x));
  return n;
}

// Last key tile a pair may touch: pB, or NQ - 1 when pB is past the sequence
// (an odd number of query tiles leaves the last pair with one real tile).
__device__ __forceinline__ int pair_qmax(const PrefillParams& P, int pA) {
  return min(pA + 1, P.g.NQ - 1);
}

// Streaming: key tiles [0, sink_hi) and [loc_lo, qmax] (merged when they overlap).
__device__ __forceinline__ void st_ranges(const PrefillParams& P, int pA, int& sink_hi, int& loc_lo) {
  sink_hi = min((P.init_num + 1) >> 1, pair_qmax(P, pA) + 1);
  loc_lo = max(0, 2 * pA - P.local_num + 1) >> 1;
  if (sink_hi >= loc_lo) {
    sink_hi = 0;
    loc_lo = 0;
  }
}

// Key tiles of a vertical-slash pair: n_hi distances <= pB in the ascending
// list; the smallest (distance 0, key tile pB) is dropped when pB is past the
// sequence.  Item t maps to distance list[n_hi - 1 - t].
__device__ __forceinline__ int vs_n_tiles(const PrefillParams& P, int unit, int pA, int n_hi) {
  const int32_t* qd = P.qdelta + static_cast<int64_t>(unit) * (P.g.NQ + 1);  // n_hi <= NQ + 1
  const bool drop = pA + 1 > P.g.NQ - 1 && n_hi > 0 && (qd[0] >> 5) == 0;
  return n_hi - (drop ? 1 : 0);
}

__device__ __forceinline__ int n_items(const PrefillParams& P, int unit, int c, int n_chunks,
                                       int n_tiles) {
  const int pA = 2 * c;
  if (P.kind == kPrefillVS) return n_chunks + n_tiles;
  int sink_hi, loc_lo;
  st_ranges(P, pA, sink_hi, loc_lo);
  return sink_hi + (pair_qmax(P, pA) - loc_lo + 1);
}

// Item i of pair c.  Vertical-slash: column chunks first (ascending), then key
// tiles ascending (largest distance first; n_hi from vs_tiles_upto).
// Streaming: the sink tiles, then the local window's tiles, ascending.
__device__ __forceinline__ Item get_item(const PrefillParams& P, int unit, int c, int i,
                                         int n_chunks, int n_hi) {
  const int pA = 2 * c, pB = pA + 1;
  Item it;
  it.cols = false;
  it.qmask[0] = it.qmask[1] = 0xFu;
  if (P.kind == kPrefillVS) {
    if (i < n_chunks) {
      int seen = 0;
      for (int x = 0;; ++x) {
#ifdef MSA_CHECKED
        if (x >= P.chunk_words) {  // fewer chunks than items: report, take chunk 0
          MSA_IDX(x, 0, P.chunk_words, P.status);
          it.cols = true;
          it.idx = 0;
          return it;
        }
#endif
        uint32_t word = vs_chunk_word(P, unit, pA, x);
        const int cnt = __popc(word);
        if (seen + cnt > i) {
          for (int skip = i - seen; skip > 0; --skip) word &= word - 1;
          it.cols = true;
          it.idx = MSA_IDX(32 * x + (__ffs(word) - 1), 0, (P.kv + 127) / 128, P.status);
          return it;
        }
        seen += cnt;
      }
    }
    const int t = i - n_chunks;
    const int32_t e = P.qdelta[static_cast<int64_t>(unit) * (P.g.NQ + 1) +
                               MSA_IDX(n_hi - 1 - t, 0, P.g.NQ + 1, P.status)];
    it.idx = MSA_IDX(pB - (e >> 5), 0, P.g.NQ, P.status);
    // quadrant (a, b) of tile pB sits at distance 2D + a - b (bit a - b + 3 of
    // the packed window), of tile pA at 2D - 2 + a - b (bit a - b + 1)
    uint32_t ma = 0, mb = 0;
#pragma unroll
    for (int a = 0; a < 2; ++a) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        if (2 * pA + a < P.g.NB) ma |= ((e >> (a - b + 1)) & 1u) << (a * 2 + b);
        if (2 * pB + a < P.g.NB) mb |= ((e >> (a - b + 3)) & 1u) << (a * 2 + b);
      }
    }
    it.qmask[0] = ma;
    it.qmask[1] = mb;
    return it;
  }
  // streaming
  int sink_hi, loc_lo;
  st_ranges(P, pA, sink_hi, loc_lo);
  it.idx = MSA_IDX(i < sink_hi ? i : loc_lo + (i - sink_hi), 0, P.g.NQ, P.status);
  it.qmask[0] = quad_mask_st(P, pA, it.idx);
  it.qmask[1] = quad_mask_st(P, pB, it.idx);
  return it;
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
  const int unit = P.units_fast ? blockIdx.x : blockIdx.y;
  const int c = P.npair - 1 - static_cast<int>(P.units_fast ? blockIdx.y : blockIdx.x);  // heavy first
  const int pA = 2 * c;
  const int b = unit_batch(P, unit), h = unit_head(P, unit), hkv = h / P.g.G;
  volatile int* abort = &sm.abort;
  const uint32_t* dist = P.kind == kPrefillVS
                             ? P.tile_dist + static_cast<int64_t>(unit) * P.dist_words
                             : nullptr;

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
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], 4);  // one arrival per softmax warp of the tile
      mbar_init(&sm.o_full[t], 1);
    }
    mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  int n_chunks = 0, n_hi = 0, n_tiles = 0;
  if (P.kind == kPrefillVS) {
    n_chunks = vs_n_chunks(P, unit, pA);
    n_hi = vs_tiles_upto(P, unit, pA + 1);
    n_tiles = vs_n_tiles(P, unit, pA, n_hi);
  }
  const int n = n_items(P, unit, c, n_chunks, n_tiles);

  if (warp < 4) {
  // ============================================================== control warpgroup
  setmaxnreg_dec();
  if (warp == 0) {
    // ------------------------------------------------------------ Q + K producer
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk);
      mbar_arrive_expect_tx(&sm.q_full, 2 * kTileBytes);
      for (int t = 0; t < 2; ++t) {  // a tile past the sequence reloads the last one (never stored)
        const int qrow = 128 * min(pA + t, P.g.NQ - 1);
        tma_load_4d(sm.q[t], &mq, &sm.q_full, 0, qrow, h, b);
        tma_load_4d(sm.q[t] + kHalfBytes, &mq, &sm.q_full, 64, qrow, h, b);
      }
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i % kStagesK;
        if (!mbar_wait(&sm.k_empty[s], ((i / kStagesK) & 1) ^ 1, abort)) break;
        const Item it = get_item(P, unit, c, i, n_chunks, n_hi);
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
        const Item it = get_item(P, unit, c, i, n_chunks, n_hi);
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
      bool ok = n == 0 || mbar_wait(&sm.q_full, 0, abort);
      tc_fence_after();
      // Operand descriptors are built once; a K-step only adds a constant to the
      // start-address field (16-byte units), which cannot carry out of it.
      const uint64_t q_desc0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t q_desc1 = sdesc_sw128(smem_u32(sm.q[1]), 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(smem_u32(sm.v[0]), kHalfBytes, 1024);
      constexpr uint64_t kStageStep = kTileBytes >> 4;
      // O_t += P_t(j) V(j); the second tile's product releases the V stage
      auto issue_pv = [&](int t, int j) -> bool {
        const int sv = j % kStagesV;
        if (!mbar_wait(&sm.p_full[t], j & 1, abort)) return false;
        if (t == 0 && !mbar_wait(&sm.v_full[sv], (j / kStagesV) & 1, abort)) return false;
        tc_fence_after();
        const uint64_t vd = v_desc0 + sv * kStageStep;
        const uint32_t o_tm = tmem + kColO + 128 * t, p_tm = tmem + kColS + 128 * t;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(o_tm, p_tm + kk * 8, vd + ((kk * 2048) >> 4), idO, (j > 0 || kk > 0) ? 1u : 0u);
        if (t == 1) mma_commit(&sm.v_empty[sv]);
        return true;
      };
      // S_t(i) = Q_t K(i)^T
      auto issue_s = [&](int t, int i) {
        const uint64_t qd = t ? q_desc1 : q_desc0;
        const uint64_t kd = k_desc0 + (i % kStagesK) * kStageStep;
        const uint32_t s_tm = tmem + kColS + 128 * t;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          mma_ss(s_tm, qd + off, kd + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&sm.s_full[t]);
      };
      for (int i = 0; ok && i < n; ++i) {
        // K(i) is normally resident long before; waiting for it next to P_A's
        // wait keeps a wait out of the middle of the MMA stream (a wait there
        // stalls behind the queued P.V MMAs and lets the tensor pipe drain)
        if (!mbar_wait(&sm.k_full[i % kStagesK], (i / kStagesK) & 1, abort)) { ok = false; break; }
        if (i >= 1 && !issue_pv(0, i - 1)) { ok = false; break; }
        tc_fence_after();
        issue_s(0, i);
        if (i >= 1 && !issue_pv(1, i - 1)) { ok = false; break; }
        issue_s(1, i);
        mma_commit(&sm.k_empty[i % kStagesK]);
      }
      if (ok && n > 0) {
        if (issue_pv(0, n - 1)) {
          mma_commit(&sm.o_full[0]);
          if (issue_pv(1, n - 1)) mma_commit(&sm.o_full[1]);
        }
      }
      // every MMA issued above must complete before TMEM is released
      mma_commit(&sm.final_bar);
      wait_drain(&sm.final_bar, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (tid == 0 && sm.abort && P.status) atomicOr(P.status, kStatusTimeout);
  } else {
  // ============================================================== softmax warpgroups
  setmaxnreg_inc();
  {
    const int t = (warp - 4) >> 2;           // query tile of this warpgroup
    const int p = pA + t;
    const int r = (tid - 128) & 127;         // query row within the tile == TMEM lane
    const int half = r >> 6;                 // row block 2p + half
    const int row = 128 * p + r;             // query index i
    const int mblk = 2 * p + half;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + (kColS + 128 * t);
    const uint32_t o_col = lane_base + (kColO + 128 * t);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int k = 0;  // items processed so far
    for (int i = 0; i < n; ++i) {
      const Item it = get_item(P, unit, c, i, n_chunks, n_hi);
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[t], k & 1, abort))) { ok = false; break; }
      tc_fence_after();
      // raw logits (unscaled) of this row, masked; scale * log2(e) is folded in
      // below.  S stays in TMEM until P is written over it, so this may run twice.
      auto logits = [&](float (&x)[128]) {
        {
          uint32_t raw[128];
          tmem_ld128(s_col, raw);
#pragma unroll
          for (int e = 0; e < 128; ++e) x[e] = __uint_as_float(raw[e]);
        }
        if (it.cols) {
          // the warp's admission bits for the chunk's 128 keys (column_bits);
          // a key of the row's own block also needs j <= row
          uint32_t adm[4], own[4];
          int jv[4];
          column_bits<4>(P, P.vertical + static_cast<int64_t>(unit) * P.kv, 128 * it.idx, dist,
                         mblk, adm, own, jv);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t keep = adm[q];
            for (uint32_t ob = own[q]; ob; ob &= ob - 1) {  // warp-uniform: own[q] is a ballot
              const int bit = __ffs(static_cast<int>(ob)) - 1;
              if (__shfl_sync(0xffffffffu, jv[q], bit) <= row) keep |= 1u << bit;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((keep >> e) & 1u)) x[32 * q + e] = -INFINITY;
          }
        } else {
          const uint32_t qm = t ? it.qmask[1] : it.qmask[0];
          const bool lo_ok = (qm >> (half * 2)) & 1u;
          const bool hi_ok = (qm >> (half * 2 + 1)) & 1u;
          const bool diag = it.idx == p;
          if (!lo_ok || !hi_ok || diag) {
#pragma unroll
            for (int e = 0; e < 128; ++e) {
              const bool in_q = e < 64 ? lo_ok : hi_ok;
              if (!in_q || (diag && e > r)) x[e] = -INFINITY;
            }
          }
        }
      };
      // p = 2^(z log2(e) - m) as f16 pairs (paired exponent arguments and sums);
      // returns the row sum
      auto exps = [&](const float (&x)[128], float m, uint32_t (&pk)[64]) -> float {
        const float2 scale2 = make_float2(P.scale_log2, P.scale_log2);
        const float nb = m == -INFINITY ? 0.f : -m;
        const float2 nb2 = make_float2(nb, nb);
        float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float2 a = ffma2(make_float2(x[2 * e], x[2 * e + 1]), scale2, nb2);
          const float2 pe = make_float2(ex2_approx(a.x), ex2_approx(a.y));
          rs2[e & 3] = fadd2(rs2[e & 3], pe);
          pk[e] = pack_f16x2(pe.x, pe.y);
        }
        const float2 rsa = fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3]));
        return rsa.x + rsa.y;
      };
      // ---- online softmax.  The exponentials use the running max m_run as
      // they are: while the row sum stays <= kSumLimit, no p exceeds it, so P
      // fits f16 and the row max is not needed.  A row's first item with keys
      // (m_run = -inf), or a sum above the limit (some logit more than
      // log2(kSumLimit / 128) above m_run), takes the row max: S is loaded again,
      // m_run moves to the max, O and l are rescaled, and the warp recomputes its
      // exponentials (rows that did not move get the same values again).
      uint32_t pk[64];
      float rs;
      {
        float x[128];
        logits(x);
        rs = exps(x, m_run, pk);
      }
      const bool redo = m_run == -INFINITY || !(rs <= kSumLimit);
      bool correct = false;
      float alpha = 1.f;
      if (__any_sync(0xffffffffu, redo)) {
        float x[128];
        logits(x);
        float mx8[8];  // 8 independent chains of 3-input max
#pragma unroll
        for (int a = 0; a < 8; ++a) {
          float m = fmax3(x[a], x[8 + a], x[16 + a]);
#pragma unroll
          for (int e = 24; e < 120; e += 16) m = fmax3(m, x[e + a], x[e + 8 + a]);
          mx8[a] = fmaxf(m, x[120 + a]);
        }
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        if (redo) {
          const float m_new = fmaxf(m_run, mx * P.scale_log2);
          correct = m_run != -INFINITY && m_new > m_run;  // O holds earlier items' weight
          alpha = correct ? ex2_approx(m_run - m_new) : 1.f;
          l_run *= alpha;
          m_run = m_new;
        }
        rs = exps(x, m_run, pk);
      }
      l_run += rs;
      // PV_t(i-1) completed before S_t(i) did (in-order tcgen05), so O_t is ready
      if (__any_sync(0xffffffffu, correct)) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t o[32];
          tmem_ld32(o_col + 32 * q4, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(o_col + 32 * q4, o);
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
      if (lane == 0) mbar_arrive(&sm.p_full[t]);
      ++k;
    }
    // ---- epilogue
    uint4 outv[16];
    const bool have = ok && k > 0 && l_run > 0.f;
    if (ok && k > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_full[t], 0, abort))) ok = false;
      tc_fence_after();
    }
    if (ok && k > 0) {
      // 1 / l, times 2^e for a KV head whose f16 copy of v was scaled by 2^-e
      float inv = have ? 1.f / l_run : 0.f;
      if (P.vmax)
        inv = ldexpf(inv, v_scale_exp(__uint_as_float(P.vmax[b * P.g.Hkv + hkv])));
      uint32_t o[128];
      tmem_ld128(o_col, o);
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
      if (P.lse) {
        // ln sum_j exp(z_ij) = (m + log2 l) ln 2: m is the (lazily updated) row
        // max in log2 units, l the row sum relative to it
        const float lse = have ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
        P.lse[(static_cast<int64_t>(b) * P.g.Hq + h) * P.g.N + row] = lse;
      }
    }
  }
  tc_fence_before();
  __syncthreads();  // pairs with the control warpgroup's; TMEM is released after it
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const CUtensorMap& mkc, const CUtensorMap& mvc,
                           cudaStream_t st, int* n_launch) {
  // Block-sparse heads run the one-tile kernel (prefill_tile.cu, launched by
  // the block-sparse entry point): their short, sparse per-tile lists favour
  // items of two kept blocks per query tile; this kernel keeps the tensor core
  // busier on the long lists of vertical-slash and streaming heads.
  if (p.kind == kPrefillBS) return cudaErrorInvalidValue;
  // The register split above needs the launch to provide kMinLaunchRegs per
  // thread; refuse to launch (rather than wait forever) if the build differs.
  static int launch_regs = -1;
  if (launch_regs < 0) {
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, sparse_prefill_kernel);
    if (e != cudaSuccess) return e;
    launch_regs = attr.numRegs;
  }
  if (launch_regs < kMinLaunchRegs) return cudaErrorInvalidConfiguration;
  const int smem = static_cast<int>(sizeof(Smem)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(sparse_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (p.g.n_units == 0 || p.npair == 0) return cudaSuccess;
  const dim3 grid = p.units_fast ? dim3(p.g.n_units, p.npair) : dim3(p.npair, p.g.n_units);
  sparse_prefill_kernel<<<grid, kThreads, smem, st>>>(p, mq, mk, mv, mkc, mvc);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
