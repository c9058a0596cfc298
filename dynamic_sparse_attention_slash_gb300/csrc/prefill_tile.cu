// Sparse prefill attention (MInference 1.0 overview, section 2.2: "block-sparse
// computation of the attention weights and output" over the sparse index, shared
// by the vertical-slash, block-sparse and streaming heads), with the one-pass
// online softmax of FlashAttention-2 (the Novita vLLM article, "Attention
// modification", Fig. 7: keep a running row max and row sum, rescale the output,
// divide by the row sum at the end).
//
// This kernel serves the block-sparse and hierarchical heads, and
// vertical-slash heads whose tiles are sparse (few slash lines for the
// length): one CTA computes one 128-row query tile p of one (batch, head)
// unit (row blocks 2p and 2p + 1).  It walks the tile's items: for
// block-sparse plans the list bs_index.cu builds (the blocks kept by either
// row block, ascending, two 64-key blocks to an item); for vertical-slash
// plans the tile's column chunks, then the blocks either row block admits,
// derived from one per-unit list of active distances (see Tile).  The two blocks of an item
// need not be adjacent, so an item wastes at most the quadrants of a block that
// only one row block kept (on synthetic top-100 heads at 128K: 56 % of the
// computed 64 x 64 quadrants are kept blocks, against 32 % with items of
// aligned 128-key tiles).  An item carries a 4-bit quadrant mask (bit a*2+b:
// row half a may see key half b) and the causal cut where a block reaches
// past a row.
//
// Warp roles (384 threads):
//   warp 0     TMA producer for Q and K (one thread)
//   warp 1     TMEM allocator and tcgen05.mma issuer (one thread)
//   warp 2     TMA producer for V (one thread)
//   warp 3     idle
//   warps 4-11 softmax: warps 4 + w and 8 + w own query rows 32w .. 32w + 31
//              (TMEM lanes) and split each row's 128 keys into two halves.
//              They run the online softmax in fp32 (exp2 with log2(e) folded
//              into the scale) against the row's running max, decide together
//              once per item (one named barrier) whether a row needs its max
//              and only then exchange half-row maxima through shared memory,
//              write P as f16 into the item's P buffer, rescale their half of
//              O in TMEM when the running max moves, and write their half of
//              the output row.  Before P(i) is released, warp 4 waits for V(i)
//              and warp 5 for K(i + 2) to land, so the MMA thread waits on P
//              alone (a wait on that thread stalls its MMA stream).
//
// TMEM (512 columns allocated): two S buffers at [0,128) and [128,256) for even
// and odd items, the output accumulator O at [256,384), two P buffers (f16
// pairs) at [384,448) and [448,512).  S = Q K^T reads Q and K from
// 128B-swizzled shared memory (K-major); O += P V reads P from TMEM and V from
// shared memory (MN-major).  The MMA issue order is S(0), S(1), then per item
// i, once P(i) is complete: S(i + 2) into S(i)'s buffer, then PV(i).  The
// softmax of item i + 1 runs on S(i + 1) while the tensor core computes S(i + 2)
// and PV(i); P(i + 2) is written once PV(i) has read its buffer.  Every
// mbarrier wait is bounded (see sm103_ptx.cuh); a timeout sets the status word
// and the CTA drains its copies and MMAs and exits.  The named barriers
// between the two warps of a row group are reached by both on every path
// (every wait before them is bounded and both leave together).
#include "prefill_common.cuh"

namespace msa {
namespace {

using namespace prefill;

constexpr int kThreads = 384;
constexpr int kStagesK = 3;
constexpr int kStagesV = 2;
constexpr int kRing = 8;  // decoded-item slots (more than kStagesK + 2)
// A sum of at most 2^15 over a half row bounds each of its p: P fits f16.
constexpr float kSumLimit = 32768.f;
// TMEM columns: S of item i at kColS + 128 (i & 1), O at kColO, P (f16 pairs)
// of item i at kColP + 64 (i & 1)
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;

struct __align__(1024) TileSmem {
  uint8_t q[kTileBytes];
  uint8_t k[kStagesK][kTileBytes];
  uint8_t v[kStagesV][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full[2], p_full[2];
  uint64_t final_bar;
  int4 ring[kRing];       // decoded items, K producer -> softmax
  float xmax[2][2][128];  // half-row maxima [item parity][column half][row]
  float xsum[2][128];     // half-row sums at the end
  uint32_t tmem_base;
  int abort;
};

struct Item {
  bool cols;    // vertical-slash column chunk (gathered keys) instead of key blocks
  int idx;      // the column chunk
  int blk[2];   // 64-key block of key half 0 and 1
  uint32_t qm;  // quadrant mask (bit a*2 + b: row half a sees key half b)
};

// The query tile p of a CTA and its items.
//  * block-sparse: the tile's item list; entry i is two int32 slots, one per
//    key half, each blk | flags << 16 (flag bit a: row block 2p + a kept it).
//  * vertical-slash (low tile density): the tile's column chunks (bit c of its
//    col_chunks words: positions [128c, 128c + 128) of the vertical list),
//    then the 64-key blocks of the unit's distance list e2, two to an item.
//    An entry (d + 1) << 2 | flags stands for block n = 2p - d, with flag bit
//    0 set iff tile distance d is active (row block 2p admits n) and bit 1 iff
//    d + 1 is (row block 2p + 1 admits n); the entries with
//    max(-1, 2p - NB + 1) <= d <= 2p belong to tile p, taken in descending d
//    (ascending n).  Flags and the causal cut are those of block-sparse items.
struct Tile {
  int n;  // items
  const int32_t* list;        // block-sparse
  int n_chunks;               // vertical-slash
  const uint32_t* chunks;
  const int32_t* e2;
  int j_hi, j_lo;             // e2 entries [j_lo, j_hi) belong to the tile
};

template <int kKind>
__device__ __forceinline__ Tile make_tile(const PrefillParams& P, int unit, int p) {
  const int64_t t = static_cast<int64_t>(unit) * P.g.NQ + p;
  Tile T;
  if (kKind == kPrefillBS) {
    T.n = MSA_COUNT(P.bs_tile_count[t], P.bs_tile_cap, P.status);
    T.list = P.bs_tiles + t * P.bs_tile_cap * 2;
    return T;
  }
  T.chunks = P.col_chunks + t * P.chunk_words;
  T.n_chunks = 0;
  for (int x = 0; x < P.chunk_words; ++x) T.n_chunks += __popc(T.chunks[x]);
  T.e2 = P.vs_e2 + static_cast<int64_t>(unit) * P.e2_stride;
  const int cnt = MSA_COUNT(P.vs_e2_count[unit], P.e2_stride, P.status);
  // entries ascending by d: first with d >= d_lo, first with d > 2p
  const int d_lo = max(-1, 2 * p - P.g.NB + 1);
  auto first_above = [&](int d) {  // first entry with distance > d
    int lo = 0, hi = cnt;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((T.e2[mid] >> 2) - 1 <= d) lo = mid + 1; else hi = mid;
    }
    return lo;
  };
  T.j_lo = first_above(d_lo - 1);
  T.j_hi = first_above(2 * p);
  T.n = T.n_chunks + (T.j_hi - T.j_lo + 1) / 2;
  return T;
}

template <int kKind>
__device__ __forceinline__ Item get_item(const PrefillParams& P, const Tile& T, int i, int p) {
  Item it;
  it.cols = false;
  it.idx = 0;
  if (kKind == kPrefillBS) {
    const int32_t s0 = T.list[2 * i], s1 = T.list[2 * i + 1];
    const uint32_t f0 = static_cast<uint32_t>(s0 >> 16) & 3u, f1 = static_cast<uint32_t>(s1 >> 16) & 3u;
    it.blk[0] = MSA_IDX(s0 & 0xffff, 0, P.g.NB, P.status);
    it.blk[1] = MSA_IDX(s1 & 0xffff, 0, P.g.NB, P.status);
    it.qm = (f0 & 1u) | ((f1 & 1u) << 1) | ((f0 >> 1) << 2) | ((f1 >> 1) << 3);
    return it;
  }
  if (i < T.n_chunks) {  // the (i+1)-th set chunk bit, ascending
    int seen = 0;
    for (int x = 0; x < P.chunk_words; ++x) {
      uint32_t word = T.chunks[x];
      const int cnt = __popc(word);
      if (seen + cnt > i) {
        for (int skip = i - seen; skip > 0; --skip) word &= word - 1;
        it.cols = true;
        it.idx = MSA_IDX(32 * x + (__ffs(word) - 1), 0, (P.kv + 127) / 128, P.status);
        break;
      }
      seen += cnt;
    }
    it.blk[0] = it.blk[1] = 0;
    it.qm = 0xFu;
    return it;
  }
  const int t = i - T.n_chunks;
  const int j0 = T.j_hi - 1 - 2 * t, j1 = j0 - 1;
  const int32_t e0 = T.e2[MSA_IDX(j0, 0, P.e2_stride, P.status)];
  const int32_t e1 = j1 >= T.j_lo ? T.e2[j1] : e0;
  const bool second_row_block = 2 * p + 1 < P.g.NB;
  uint32_t f0 = static_cast<uint32_t>(e0) & 3u, f1 = j1 >= T.j_lo ? static_cast<uint32_t>(e1) & 3u : 0u;
  if (!second_row_block) {
    f0 &= 1u;
    f1 &= 1u;
  }
  it.blk[0] = MSA_IDX(2 * p - ((e0 >> 2) - 1), 0, P.g.NB, P.status);
  it.blk[1] = MSA_IDX(2 * p - ((e1 >> 2) - 1), 0, P.g.NB, P.status);
  it.qm = (f0 & 1u) | ((f1 & 1u) << 1) | ((f0 >> 1) << 2) | ((f1 >> 1) << 3);
  return it;
}

// Decoded items pass from the K producer to the softmax warps through a ring
// in shared memory (an L2 read of the list entry per item sat on the softmax's
// per-item path): slot i % kRing holds item i as {i, blk0 | blk1 << 16,
// qm | cols << 4, idx}, its tag written last.  The producer writes item i
// before loading K(i) and may only reach item i + kRing once P(i + kRing - 5)
// is complete (K stage reuse), long after every softmax warp has read slot i.
__device__ __forceinline__ void post_item(int4* ring, int i, const Item& it) {
  volatile int* s = reinterpret_cast<volatile int*>(ring + (i % kRing));
  s[1] = it.blk[0] | (it.blk[1] << 16);
  s[2] = static_cast<int>(it.qm) | (it.cols ? 16 : 0);
  s[3] = it.idx;
  __threadfence_block();
  s[0] = i;
}
// Item i from the ring; false (and a fully masked item) if its tag does not
// appear within the wait limit or the CTA has aborted.
__device__ __forceinline__ bool take_item(int4* ring, int i, volatile int* abort, Item& it) {
  volatile int* s = reinterpret_cast<volatile int*>(ring + (i % kRing));
  bool got = true;
  if (s[0] != i) {
    const uint64_t t0 = global_timer_ns();
    while (s[0] != i) {
      if (*abort || global_timer_ns() - t0 > MSA_WAIT_LIMIT_NS) {
        *abort = 1;
        got = false;
        break;
      }
    }
  }
  got = __all_sync(0xffffffffu, got);
  __threadfence_block();
  const int y = s[1], z = s[2];
  it.blk[0] = got ? (y & 0xffff) : 0;
  it.blk[1] = got ? ((y >> 16) & 0xffff) : 0;
  it.qm = got ? static_cast<uint32_t>(z) & 0xFu : 0u;
  it.cols = got && (z & 16);
  it.idx = got ? s[3] : 0;
  return got;
}

// TMA of the item's K (or V) rows into dst, completion on bar: keys of key
// half h are rows [64h, 64h + 64) of the 128-row tile (both 64-column
// halves): block blk[h] of the KV head, or for a column chunk c the gathered
// rows [128c + 64h, +64) of the unit.
__device__ __forceinline__ void load_item(const Item& it, uint8_t* dst, const CUtensorMap* map64,
                                          const CUtensorMap* mapc64, uint64_t* bar, int hkv,
                                          int b, int crow0) {
  mbar_arrive_expect_tx(bar, kTileBytes);
#pragma unroll
  for (int hd = 0; hd < 2; ++hd)
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      uint8_t* d = dst + hd * kHalfBytes + kh * (kHalfBytes / 2);
      if (it.cols)
        tma_load_2d(d, mapc64, bar, 64 * hd, crow0 + 128 * it.idx + 64 * kh);
      else
        tma_load_4d(d, map64, bar, 64 * hd, 64 * it.blk[kh], hkv, b);
    }
}

template <int kKind>
__global__ void __launch_bounds__(kThreads, 1)
sparse_prefill_tile_kernel(const __grid_constant__ PrefillParams P, const __grid_constant__ CUtensorMap mq,
                           const __grid_constant__ CUtensorMap mk64,
                           const __grid_constant__ CUtensorMap mv64,
                           const __grid_constant__ CUtensorMap mkc64,
                           const __grid_constant__ CUtensorMap mvc64) {
  extern __shared__ uint8_t smem_raw[];
  TileSmem& sm = *reinterpret_cast<TileSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int unit = P.units_fast ? blockIdx.x : blockIdx.y;
  const int p = P.g.NQ - 1 - static_cast<int>(P.units_fast ? blockIdx.y : blockIdx.x);  // heavy first
  const Tile T = make_tile<kKind>(P, unit, p);
  const int b = unit_batch(P, unit), h = unit_head(P, unit), hkv = h / P.g.G;
  const int crow0 = unit * P.kv_pad;  // the unit's gathered column rows (vertical-slash)
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
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], 8);  // one arrival per softmax warp
    }
    mbar_init(&sm.final_bar, 1);
    for (int s = 0; s < kRing; ++s) sm.ring[s].x = -1;
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

  if (warp == 0) {
    // ------------------------------------------------------------ Q + K producer
    if (lane == 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mk64);
      if (kKind == kPrefillVS) tma_prefetch_desc(&mkc64);
      mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
      tma_load_4d(sm.q, &mq, &sm.q_full, 0, 128 * p, h, b);
      tma_load_4d(sm.q + kHalfBytes, &mq, &sm.q_full, 64, 128 * p, h, b);
      int issued = 0;
      for (int i = 0; i < T.n; ++i) {
        const int st = i % kStagesK;
        if (!mbar_wait(&sm.k_empty[st], ((i / kStagesK) & 1) ^ 1, abort)) break;
        const Item it = get_item<kKind>(P, T, i, p);
        post_item(sm.ring, i, it);
        load_item(it, sm.k[st], &mk64, &mkc64, &sm.k_full[st], hkv, b, crow0);
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
      tma_prefetch_desc(&mv64);
      if (kKind == kPrefillVS) tma_prefetch_desc(&mvc64);
      int issued = 0;
      for (int i = 0; i < T.n; ++i) {
        const int st = i % kStagesV;
        if (!mbar_wait(&sm.v_empty[st], ((i / kStagesV) & 1) ^ 1, abort)) break;
        load_item(get_item<kKind>(P, T, i, p), sm.v[st], &mv64, &mvc64, &sm.v_full[st], hkv, b,
                  crow0);
        issued = i + 1;
      }
      for (int i = max(0, issued - kStagesV); i < issued; ++i)
        wait_drain(&sm.v_full[i % kStagesV], (i / kStagesV) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const int n = T.n;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_f32acc(128, 128, /*bf16=*/false, false, true);  // f16 P, f16 V
      bool ok = n == 0 || mbar_wait(&sm.q_full, 0, abort);
      tc_fence_after();
      // Operand descriptors are built once; a K-step only adds a constant to the
      // start-address field (16-byte units), which cannot carry out of it.
      const uint64_t q_desc = sdesc_sw128(smem_u32(sm.q), 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(smem_u32(sm.v[0]), kHalfBytes, 1024);
      constexpr uint64_t kStageStep = kTileBytes >> 4;
      // S(i) = Q K(i)^T into S buffer i & 1; its completion releases the K stage.
      // K(0) and K(1) are waited for here; K(i) for i >= 2 has landed once P(i - 2)
      // is complete (a softmax warp waits for it before that arrival), so the
      // MMA thread waits only on P (a wait on this thread stalls its MMA stream).
      auto issue_s = [&](int i) -> bool {
        const int sk = i % kStagesK;
        if (i < 2 && !mbar_wait(&sm.k_full[sk], (i / kStagesK) & 1, abort)) return false;
        tc_fence_after();
        const uint64_t kd = k_desc0 + sk * kStageStep;
        const uint32_t s_tm = tmem + kColS + 128 * (i & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          mma_ss(s_tm, q_desc + off, kd + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&sm.s_full[i & 1]);
        mma_commit(&sm.k_empty[sk]);
        return true;
      };
      // O += P(i) V(i); its completion releases the V stage (and tells the
      // softmax that O holds items 0..i and that P buffer i & 1 is free)
      auto issue_pv = [&](int i) {
        const int sv = i % kStagesV;
        const uint64_t vd = v_desc0 + sv * kStageStep;
        const uint32_t p_tm = tmem + kColP + 64 * (i & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + kColO, p_tm + kk * 8, vd + ((kk * 2048) >> 4), idO,
                 (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&sm.v_empty[sv]);
      };
      // P(i) complete means the softmax is done with S(i) and V(i) has
      // landed: S(i + 2) goes into S(i)'s buffer ahead of P(i) V(i), so the
      // softmax of item i + 1 (on S(i + 1), issued a step earlier) overlaps
      // both products and S(i + 2) is ready before P(i) V(i) runs
      if (ok && n > 0) ok = issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int i = 0; ok && i < n; ++i) {
        if (!mbar_wait(&sm.p_full[i & 1], (i >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (i + 2 < n && !issue_s(i + 2)) {
          ok = false;
          break;
        }
        issue_pv(i);
      }
      // every MMA issued above must complete before TMEM is released
      mma_commit(&sm.final_bar);
      wait_drain(&sm.final_bar, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    // Warps 4 + w and 8 + w share TMEM lanes 32w .. 32w + 31 (query rows) and
    // split the columns: warpgroup g takes keys [64g, 64g + 64) of each item and
    // output dimensions [64g, 64g + 64).  Both halves of a row keep the same
    // running max (they move it together, exchanging half-row maxima through
    // shared memory); their row sums are added at the end.
    const int g = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;        // query row within the tile == TMEM lane
    const uint32_t pair_bar = 1 + quarter;    // named barrier of the two warps of these rows
    const int half = r >> 6;                  // row block 2p + half
    const int row = 128 * p + r;              // query index i
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t o_col = lane_base + kColO + 64 * g;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true, loads_ok = true;
    int k = 0;  // items processed so far
    // Block-sparse items come from the ring one item ahead: the producer posts
    // item k + 1 as soon as K(k + 1)'s stage is free, which the completion of
    // S(k - 2) (before this warp starts item k) guarantees.  Vertical-slash
    // items are taken in place (holding the next one costs that
    // instantiation's registers more than the read saves).
    Item nxt;
    bool nxt_got = true;
    if constexpr (kKind == kPrefillBS)
      if (T.n > 0) nxt_got = take_item(sm.ring, 0, abort, nxt);
    for (; k < T.n;) {
      Item it;
      bool got;
      if constexpr (kKind == kPrefillBS) {
        it = nxt;
        got = nxt_got;
        if (k + 1 < T.n) nxt_got = take_item(sm.ring, k + 1, abort, nxt);
      } else {
        got = take_item(sm.ring, k, abort, it);
      }
      const uint32_t s_col = lane_base + kColS + 128 * (k & 1);
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      const bool waited =
          __all_sync(0xffffffffu, mbar_wait(&sm.s_full[k & 1], (k >> 1) & 1, abort)) && loads_ok &&
          got;
      tc_fence_after();
      // A key tile whose quadrant (row half, key half g) is not admitted leaves
      // this warp nothing to do: its half of P is zero, its maximum -inf.
      const bool idle = !((it.qm >> (half * 2 + g)) & 1u);
      // raw logits (unscaled) of this row's half with the causal cut (key
      // 64 blk + e is admitted iff it is <= the row); scale * log2(e) is
      // folded in below
      const int lim = row - 64 * (g ? it.blk[1] : it.blk[0]);
      auto logits = [&](float (&x)[64]) {
        {
          uint32_t raw[64];
          tmem_ld64(s_col + 64 * g, raw);
#pragma unroll
          for (int e = 0; e < 64; ++e) x[e] = __uint_as_float(raw[e]);
        }
        if (kKind == kPrefillVS && it.cols) {
          // chosen key j of the gathered chunk's half g: admitted iff j <= row
          // and its 64x64 tile is not active for this row block; the warp's
          // bits from column_bits, the own block's keys checked per row
          uint32_t adm[2], own[2];
          int jv[2];
          column_bits<2>(P, P.vertical + static_cast<int64_t>(unit) * P.kv,
                         128 * it.idx + 64 * g,
                         P.tile_dist + static_cast<int64_t>(unit) * P.dist_words, 2 * p + half,
                         adm, own, jv);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t keep = adm[q];
            for (uint32_t ob = own[q]; ob; ob &= ob - 1) {  // warp-uniform: own[q] is a ballot
              const int bit = __ffs(static_cast<int>(ob)) - 1;
              if (__shfl_sync(0xffffffffu, jv[q], bit) <= row) keep |= 1u << bit;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((keep >> e) & 1u)) x[32 * q + e] = -INFINITY;
          }
        } else if (lim < 63) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e > lim) x[e] = -INFINITY;
        }
      };
      // p = 2^(z log2(e) - m) as f16 pairs; returns this half's row sum
      auto exps = [&](const float (&x)[64], float m, uint32_t (&pk)[32]) -> float {
        const float2 scale2 = make_float2(P.scale_log2, P.scale_log2);
        const float nb = m == -INFINITY ? 0.f : -m;
        const float2 nb2 = make_float2(nb, nb);
        float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 a = ffma2(make_float2(x[2 * e], x[2 * e + 1]), scale2, nb2);
          const float2 pe = make_float2(ex2_approx(a.x), ex2_approx(a.y));
          rs2[e & 3] = fadd2(rs2[e & 3], pe);
          pk[e] = pack_f16x2(pe.x, pe.y);
        }
        const float2 rsa = fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3]));
        return rsa.x + rsa.y;
      };
      // ---- online softmax.  Both halves of a row exponentiate against the
      // row's running max m_run as it stands: while each half's sum stays <=
      // kSumLimit no p exceeds it, so P fits f16 and no row max is needed.  The
      // two warps of the rows decide together, in the one barrier every item
      // passes, whether a row needs its max (its first item with keys, or a sum
      // above the limit) or a wait failed; only then do they load S again,
      // exchange half-row maxima and move m_run.
      uint32_t pk[32];
      float rs = 0.f;
      bool want = false;
      if (idle) {
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = 0u;
      } else {
        float x[64];
        logits(x);
        rs = exps(x, m_run, pk);
        want = m_run == -INFINITY || !(rs <= kSumLimit);
      }
      // both warps pass this barrier on every item (every wait above is bounded)
      bool correct = false;
      float alpha = 1.f;
      if (bar_red_or(pair_bar, 64, want || !waited)) {
        if (!bar_red_and(pair_bar, 64, waited)) {  // both leave when either wait failed
          ok = false;
          break;
        }
        float x[64];
        float mxh = -INFINITY;
        if (!idle) {
          logits(x);
          float mx8[8];  // 8 independent chains of 3-input max
#pragma unroll
          for (int a = 0; a < 8; ++a) {
            float m = fmax3(x[a], x[8 + a], x[16 + a]);
#pragma unroll
            for (int e = 24; e < 56; e += 16) m = fmax3(m, x[e + a], x[e + 8 + a]);
            mx8[a] = fmaxf(m, x[56 + a]);
          }
          mxh = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                      fmaxf(mx8[6], mx8[7]));
        }
        sm.xmax[k & 1][g][r] = mxh;
        named_bar_sync(pair_bar, 64);
        const float mx = fmaxf(mxh, sm.xmax[k & 1][g ^ 1][r]);
        const float m_new = fmaxf(m_run, mx * P.scale_log2);
        correct = m_run != -INFINITY && m_new > m_run;  // O holds earlier items' weight
        alpha = correct ? ex2_approx(m_run - m_new) : 1.f;
        l_run *= alpha;
        m_run = m_new;
        if (!idle) rs = exps(x, m_run, pk);
      }
      l_run += rs;
      // P buffer k & 1 was last read by P(k - 2) V(k - 2): its completion
      // released V stage (k - 2) % kStagesV
      if (k >= 2) {
        const int j = k - 2;
        loads_ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_empty[j % kStagesV],
                                                     (j / kStagesV) & 1, abort)) && loads_ok;
        tc_fence_after();
      }
      tmem_st32(lane_base + kColP + 64 * (k & 1) + 32 * g, pk);  // f16 pairs of keys [64g, 64g + 64)
      // both warps of these rows take this branch together (same maxima)
      if (__any_sync(0xffffffffu, correct)) {
        // O must hold P(k-1) V(k-1) before it is rescaled: that product's
        // completion released its V stage
        const int j = k - 1;
        const bool got = __all_sync(
            0xffffffffu, mbar_wait(&sm.v_empty[j % kStagesV], (j / kStagesV) & 1, abort));
        if (!bar_red_and(pair_bar, 64, got)) {
          tmem_st_wait();
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          uint32_t o[32];
          tmem_ld32(o_col + 32 * q2, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(o_col + 32 * q2, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      // for the MMA thread: V(k) (warp 4) and K(k + 2) (warp 5) have landed
      // before P(k) is released; a failed wait ends both warps of these rows
      // at the next item's barrier
      if (warp == 4)
        loads_ok = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[k % kStagesV],
                                                     (k / kStagesV) & 1, abort)) && loads_ok;
      else if (warp == 5 && k + 2 < T.n)
        loads_ok = __all_sync(0xffffffffu, mbar_wait(&sm.k_full[(k + 2) % kStagesK],
                                                     ((k + 2) / kStagesK) & 1, abort)) && loads_ok;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[k & 1]);
      ++k;
    }
    // ---- epilogue: add the two halves' row sums (both warps arrive here)
    sm.xsum[g][r] = l_run;
    ok = bar_red_and(pair_bar, 64, ok && loads_ok);
    const float l_row = l_run + sm.xsum[g ^ 1][r];
    uint4 outv[8];
    const bool have = ok && k > 0 && l_row > 0.f;
    if (ok && k > 0) {
      const int j = k - 1;  // the last product's completion released its V stage
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.v_empty[j % kStagesV], (j / kStagesV) & 1, abort)))
        ok = false;
      tc_fence_after();
    }
    if (ok && k > 0) {
      // 1 / l, times 2^e for a KV head whose f16 copy of v was scaled by 2^-e
      float inv = have ? 1.f / l_row : 0.f;
      if (P.vmax)
        inv = ldexpf(inv, v_scale_exp(__uint_as_float(P.vmax[b * P.g.Hkv + hkv])));
      uint32_t o[64];
      tmem_ld64(o_col, o);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
        w.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
        w.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
        w.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
        outv[e] = w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) outv[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (row < P.g.N && ok) {
      uint4* dst = reinterpret_cast<uint4*>(P.out + b * P.out_sb + h * P.out_sh +
                                            static_cast<int64_t>(row) * P.out_sn + 64 * g);
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = outv[e];
      if (P.lse && g == 0) {
        // ln sum_j exp(z_ij) = (m + log2 l) ln 2: m is the (lazily updated) row
        // max in log2 units, l the row sum relative to it
        const float lse = have ? (m_run + log2f(l_row)) * 0.69314718055994531f : -INFINITY;
        P.lse[(static_cast<int64_t>(b) * P.g.Hq + h) * P.g.N + row] = lse;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (tid == 0 && sm.abort && P.status) atomicOr(P.status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_prefill_tile(const PrefillParams& p, const CUtensorMap& mq,
                                const CUtensorMap& mk64, const CUtensorMap& mv64,
                                const CUtensorMap& mkc64, const CUtensorMap& mvc64,
                                cudaStream_t st, int* n_launch) {
  const int smem = static_cast<int>(sizeof(TileSmem)) + 1024;
  if (p.kind != kPrefillBS && p.kind != kPrefillVS) return cudaErrorInvalidValue;
  auto kernel = p.kind == kPrefillBS ? sparse_prefill_tile_kernel<kPrefillBS>
                                     : sparse_prefill_tile_kernel<kPrefillVS>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (p.g.n_units == 0 || p.g.NQ == 0) return cudaSuccess;
  const dim3 grid = p.units_fast ? dim3(p.g.n_units, p.g.NQ) : dim3(p.g.NQ, p.g.n_units);
  kernel<<<grid, kThreads, smem, st>>>(p, mq, mk64, mv64, mkc64, mvc64);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
