// Hierarchical multi-stage pruning head (InfiniteHiP summary page, section on
// the modular hierarchical token pruning algorithm): the key sequence is cut
// into fixed-length chunks, each chunk is represented by its token with the
// highest attention score, and only the best chunks pass on to the next
// pruning stage; stacked stages narrow the candidate keys of each query block
// down to the block-sparse mask the attention kernel runs on.
//
// Scores.  A key token's score for query block m is scale * Qhat_m . k_j, Qhat_m
// the block's mean-pooled query (the block-sparse head's pooling), over the
// candidates j <= 64m + 63.  Every chunk is a group of whole 64-token blocks,
// so every stage reads only the block maxima r[m][n] = max over the keys of
// block n of the token scores: hip_block_max_kernel computes them for the
// causal blocks n <= m only, on the tensor cores.  The pooled queries (f32)
// are split into three bf16 parts whose sum holds ~24 significant bits
// (hip_split_kernel); each 128 x 128 score tile is the f32-accumulated sum of
// the three parts' products with a TMA-staged bf16 key tile (tcgen05.mma into
// TMEM, two TMEM buffers so the next tile's products overlap the maxima of
// this one), which matches an f32 dot product to within a few f32 roundings.
// Four warps read the tile from TMEM, one query block per thread, and keep
// the maximum of each 64-key half.
//
// Selection.  hip_select_warp_kernel (below) runs the stages for one query
// block per warp over short candidate lists; hip_select_kernel, for stage
// lists whose candidates would not fit, runs them for one query block per CTA:
// a stage's chunk score is the maximum of r over the chunk's surviving
// blocks; the own chunk (the one holding block m) is always kept; the best
// keep - 1 others are found by an 8-bit radix select on an order-preserving
// key with an ascending compaction (ties to the lower chunk), as the
// block-sparse selection does.  Survivors are a bitmap of blocks in shared
// memory.  The last stage's chunks are single blocks: the surviving blocks,
// ascending, are the kept list, in the block-sparse head's format, so the
// one-tile prefill kernel and its item lists serve this head unchanged.
//
// Long sequences are processed in slabs of query blocks (the block maxima of
// one slab at a time), so the workspace grows with N, not N^2, beyond a bound.
#include "block_scan.cuh"
#include "msa_internal.h"
#include "sm103_ptx.cuh"

namespace msa {
namespace {

constexpr int kTileBytes = 128 * 128 * 2;  // 128 rows x 128 dims of 16-bit values
constexpr int kHalfBytes = kTileBytes / 2;   // one 64-dim half (128-byte swizzled rows)
constexpr int kRT = 128;                     // pooled query rows (query blocks) per score CTA
constexpr int kKT = 128;                     // keys per key tile (two key blocks)
constexpr int kChunkTiles = 32;              // key tiles per score CTA
constexpr int kScoreThreads = 256;
constexpr int kSplitThreads = 256;
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

// Pooled queries as three bf16 parts hi + mid + lo (hi = bf16(x), mid =
// bf16(x - hi), lo = bf16(x - hi - mid); each difference is exact in f32), so
// the sum carries ~24 significant bits: three bf16 products with an exact f32
// product and f32 accumulation give the score to about f32 accuracy.
// qsplit is [3][units * NB][128].
__global__ void __launch_bounds__(kSplitThreads) hip_split_kernel(const float* __restrict__ qpool,
                                                                  int64_t n, __nv_bfloat16* qsplit) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kSplitThreads + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * kSplitThreads) {
    const float x = qpool[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    qsplit[i] = hi;
    qsplit[n + i] = mid;
    qsplit[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

struct HipScoreArgs {
  UnitMap u;
  int N, NB, G, n_units;
  int m0, rows;        // the slab: query blocks [m0, m0 + rows)
  int slab_stride;     // rows of rmax per unit
  float scale;
  float* rmax;         // [units][slab_stride][NB]; entry (m - m0, n) for n <= m
  uint32_t* status;
};

struct __align__(1024) ScoreSmem {
  uint8_t q[3][kTileBytes];  // hi, mid, lo parts of 128 pooled rows
  uint8_t k[2][kTileBytes];  // key tiles, two stages
  uint64_t q_full, k_full[2], k_empty[2], s_full[2], s_empty[2], final_bar;
  uint32_t tmem_base;
  int abort;
};

// grid (key chunk, row tile, unit): block maxima of query blocks
// [m0 + 128 rt, +128) against the key tiles [32 chunk, +32) they reach.
// Warp 0 loads (TMA), warp 1 issues tcgen05.mma (S = hi K^T + mid K^T + lo K^T
// into one of two TMEM buffers), warps 4-7 read S from TMEM (thread r: query
// block m0 + 128 rt + r) and write the maxima of its two 64-key halves.
__global__ void __launch_bounds__(kScoreThreads, 1)
hip_block_max_kernel(const __grid_constant__ HipScoreArgs a, const __grid_constant__ CUtensorMap mqs,
                     const __grid_constant__ CUtensorMap mk) {
  extern __shared__ uint8_t smem_raw[];
  ScoreSmem& sm = *reinterpret_cast<ScoreSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
  const int unit = blockIdx.z, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int M0 = a.m0 + blockIdx.y * kRT;                    // first query block of the tile
  const int m_last = min(M0 + kRT, a.m0 + a.rows) - 1;
  const int kt_end = min((a.N + kKT - 1) / kKT, m_last / 2 + 1);  // tiles holding candidates
  const int kt0 = blockIdx.x * kChunkTiles;
  const int n = min(kt_end - kt0, kChunkTiles);
  if (n <= 0) return;  // uniform for the CTA, before any barrier
  const int b = unit / a.u.n_heads, hkv = a.u.heads[unit % a.u.n_heads] / a.G;
  volatile int* abort = &sm.abort;
  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.s_full[s], 1);
      mbar_init(&sm.s_empty[s], 4);  // one arrival per reading warp
    }
    mbar_init(&sm.final_bar, 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&mqs);
      tma_prefetch_desc(&mk);
      const int rows_total = a.n_units * a.NB;
      mbar_arrive_expect_tx(&sm.q_full, 3 * kTileBytes);
      for (int part = 0; part < 3; ++part) {
        const int row = part * rows_total + unit * a.NB + M0;
        tma_load_2d(sm.q[part], &mqs, &sm.q_full, 0, row);
        tma_load_2d(sm.q[part] + kHalfBytes, &mqs, &sm.q_full, 64, row);
      }
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int s = i & 1;
        if (!mbar_wait(&sm.k_empty[s], ((i >> 1) & 1) ^ 1, abort)) break;
        mbar_arrive_expect_tx(&sm.k_full[s], kTileBytes);
        tma_load_4d(sm.k[s], &mk, &sm.k_full[s], 0, kKT * (kt0 + i), hkv, b);
        tma_load_4d(sm.k[s] + kHalfBytes, &mk, &sm.k_full[s], 64, kKT * (kt0 + i), hkv, b);
        issued = i + 1;
      }
      // drain: the latest load of every stage, and Q, must land before exit
      int never = 0;
      mbar_wait(&sm.q_full, 0, &never);
      for (int i = max(0, issued - 2); i < issued; ++i) mbar_wait(&sm.k_full[i & 1], (i >> 1) & 1, &never);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      bool ok = mbar_wait(&sm.q_full, 0, abort);
      tc_fence_after();
      uint64_t qd[3];
      for (int part = 0; part < 3; ++part) qd[part] = sdesc_sw128(smem_u32(sm.q[part]), 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      constexpr uint64_t kStageStep = kTileBytes >> 4;
      for (int i = 0; ok && i < n; ++i) {
        const int s = i & 1;
        if (!mbar_wait(&sm.k_full[s], (i >> 1) & 1, abort) ||
            !mbar_wait(&sm.s_empty[s], ((i >> 1) & 1) ^ 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_tm = tmem + 128 * s;
        const uint64_t kd = kd0 + s * kStageStep;
#pragma unroll
        for (int part = 0; part < 3; ++part) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
            mma_ss(s_tm, qd[part] + off, kd + off, idS, (part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&sm.s_full[s]);
        mma_commit(&sm.k_empty[s]);
      }
      // every MMA issued above must complete before TMEM is released
      mma_commit(&sm.final_bar);
      int never = 0;
      mbar_wait(&sm.final_bar, 0, &never);
    }
  } else if (warp >= 4) {
    const int r = tid - 128;  // TMEM lane == row of the tile
    const int m = M0 + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    for (int i = 0; i < n; ++i) {
      const int s = i & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[s], (i >> 1) & 1, abort))) break;
      tc_fence_after();
      uint32_t raw[128];
      tmem_ld128(lane_base + 128 * s, raw);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_empty[s]);
      const int kt = kt0 + i;
      const int j0 = kKT * kt;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (j0 + 64 * h2 + e < a.N) mx = fmaxf(mx, __uint_as_float(raw[64 * h2 + e]));
        const int nb = 2 * kt + h2;
        if (m <= m_last && nb <= m)
          a.rmax[(static_cast<int64_t>(unit) * a.slab_stride + (m - a.m0)) * a.NB + nb] =
              mx * a.scale;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
  if (tid == 0 && sm.abort && a.status) atomicOr(a.status, kStatusTimeout);
}

struct HipStages {
  int n;
  int c[MSA_HIP_MAX_STAGES];
  int keep[MSA_HIP_MAX_STAGES];
};

struct HipSelArgs {
  int NB, m0, rows, slab_stride;
  int cap, warps;  // warp-level selection: candidate capacity per warp, warps per CTA
  const float* rmax;
  HipStages st;
  int32_t* block_count;  // [units][NB]
  int32_t* block_ids;    // [units][NB][kb]
  int kb;
};

// One CTA per (slab row, unit): the stages for query block m = m0 + blockIdx.x.
__global__ void __launch_bounds__(kSelThreads) hip_select_kernel(const __grid_constant__ HipSelArgs a) {
  extern __shared__ __align__(16) float dyn_sel[];
  float* cs = dyn_sel;                                            // [NB] chunk scores, then keep flags
  uint32_t* alive = reinterpret_cast<uint32_t*>(dyn_sel + a.NB);  // [ceil(NB/32)] surviving blocks
  __shared__ int hist[kSelWarps][256];
  __shared__ int total_hist[256];
  __shared__ int warp_sums[kSelWarps + 1];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need;
  const int m = a.m0 + blockIdx.x, unit = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5;
  const float* row = a.rmax + (static_cast<int64_t>(unit) * a.slab_stride + blockIdx.x) * a.NB;
  const int words = (m >> 5) + 1;
  for (int w = tid; w < words; w += kSelThreads)
    alive[w] = (w < (m >> 5)) ? 0xffffffffu : (0xffffffffu >> (31 - (m & 31)));
  __syncthreads();
  for (int s = 0; s < a.st.n; ++s) {
    const int c = a.st.c[s];
    const int nch = m / c + 1, own = m / c;
    // chunk scores over surviving blocks; the own chunk is kept regardless and
    // takes no part in the ranking
    int elig = 0;
    for (int x = tid; x < nch; x += kSelThreads) {
      float best = -INFINITY;
      if (x != own) {
        const int n_end = min(x * c + c, m + 1);
        for (int nb = x * c; nb < n_end; ++nb)
          if ((alive[nb >> 5] >> (nb & 31)) & 1u) best = fmaxf(best, row[nb]);
      }
      cs[x] = best;
      elig += best != -INFINITY ? 1 : 0;
    }
    int n_elig;
    block_exclusive_scan<kSelThreads>(elig, warp_sums, &n_elig);  // also orders the writes above
    const int need = min(a.st.keep[s] - 1, n_elig);
    if (tid == 0) {
      s_prefix = 0u;
      s_mask = 0u;
      s_need = need;
    }
    __syncthreads();
    if (need > 0) {
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < kSelWarps * 256; i += kSelThreads) (&hist[0][0])[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        for (int x = tid; x < nch; x += kSelThreads) {
          const uint32_t key = ordered_key(cs[x]);
          if ((key & mask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1);
        }
        __syncthreads();
        {
          int cnt = 0;
          for (int w = 0; w < kSelWarps; ++w) cnt += hist[w][tid];
          total_hist[tid] = cnt;
        }
        __syncthreads();
        if (tid == 0) {
          int nd = s_need, above = 0, bucket = 0;
          for (int bb = 255; bb >= 0; --bb) {
            if (above + total_hist[bb] >= nd) {
              bucket = bb;
              break;
            }
            above += total_hist[bb];
          }
          s_need = nd - above;
          s_prefix = prefix | (static_cast<uint32_t>(bucket) << shift);
          s_mask = mask | (255u << shift);
        }
        __syncthreads();
      }
    }
    // keep flags (over the scores, each thread its own chunks): the own chunk,
    // keys above the threshold, and the first keys equal to it (lower chunks first)
    const uint32_t T = s_prefix;
    const int take_equal = s_need;
    int equal_before = 0;
    for (int base = 0; base < nch; base += kSelThreads) {
      const int x = base + tid;
      const uint32_t key = x < nch ? ordered_key(cs[x]) : 0u;
      const bool eq = need > 0 && x < nch && x != own && key == T;
      int eq_total;
      const int eq_rank = equal_before + block_exclusive_scan<kSelThreads>(eq ? 1 : 0, warp_sums, &eq_total);
      const bool keep = x < nch && (x == own || (need > 0 && x != own && cs[x] != -INFINITY &&
                                                 (key > T || (eq && eq_rank < take_equal))));
      if (x < nch) cs[x] = keep ? 1.f : 0.f;
      equal_before += eq_total;
    }
    __syncthreads();
    // blocks of dropped chunks leave the candidates
    for (int w = tid; w < words; w += kSelThreads) {
      uint32_t bits = alive[w];
      uint32_t keep_bits = 0u;
      for (int e = 0; e < 32; ++e) {
        const int nb = 32 * w + e;
        if (nb <= m && cs[nb / c] != 0.f) keep_bits |= 1u << e;
      }
      alive[w] = bits & keep_bits;
    }
    __syncthreads();
  }
  // the survivors of the last stage (single blocks), ascending
  int32_t* ids = a.block_ids + (static_cast<int64_t>(unit) * a.NB + m) * a.kb;
  int placed = 0;
  for (int base = 0; base <= m; base += kSelThreads) {
    const int nb = base + tid;
    const bool on = nb <= m && ((alive[nb >> 5] >> (nb & 31)) & 1u);
    int total;
    const int pos = placed + block_exclusive_scan<kSelThreads>(on ? 1 : 0, warp_sums, &total);
    if (on && pos < a.kb) ids[pos] = nb;
    placed += total;
  }
  if (tid == 0) a.block_count[static_cast<int64_t>(unit) * a.NB + m] = min(placed, a.kb);
}

// Warp-level form of the stages (the usual case): warp w of a CTA runs query
// block m = m0 + 8 blockIdx.x + w alone.  Stage s only looks at the chunks
// that survived stage s - 1: the candidates are the sub-chunks (of size c_s)
// of the kept chunks (of size c_{s-1}), every one of whose blocks <= m is
// still a candidate, because chunk sizes nest.  So a stage is a list of at
// most `cap` candidate chunks, ascending: their scores (the maximum of r over
// the chunk's blocks <= m), an 8-bit radix select of the best keep - 1 others
// on one warp (histograms in shared memory), and an ascending compaction of
// the kept ones (the own chunk always) into the other list.  The same rule as
// hip_select_kernel: scores descending, ties to the lower chunk.
__global__ void __launch_bounds__(kSelThreads) hip_select_warp_kernel(const __grid_constant__ HipSelArgs a) {
  extern __shared__ __align__(16) float dyn_w[];
  __shared__ int hist[kSelWarps][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.y;
  const int r_slab = blockIdx.x * a.warps + warp;  // slab row of this warp
  if (warp >= a.warps || r_slab >= a.rows) return;  // no CTA-wide barrier follows
  const int m = a.m0 + r_slab;
  float* sc = dyn_w + warp * a.cap;                                        // [cap] scores
  int* ids_a = reinterpret_cast<int*>(dyn_w + a.warps * a.cap) + warp * 2 * a.cap;  // [cap]
  int* ids_b = ids_a + a.cap;                                              // [cap]
  int* h = hist[warp];
  const float* row = a.rmax + (static_cast<int64_t>(unit) * a.slab_stride + r_slab) * a.NB;
  const uint32_t lt = (1u << lane) - 1u;
  int* cur = ids_a;  // candidate chunks of this stage (ascending)
  int* nxt = ids_b;  // kept chunks of this stage (ascending)
  int n_c = 0, n_k = 0, c_prev = 1;
  for (int s = 0; s < a.st.n; ++s) {
    const int c = a.st.c[s], own = m / c;
    // candidates: every chunk of [0, m] at the first stage, afterwards the
    // sub-chunks of the previous stage's kept chunks that start at or before m
    if (s == 0) {
      n_c = min(own + 1, a.cap);
      for (int x = lane; x < n_c; x += 32) cur[x] = x;
    } else {
      const int ratio = c_prev / c;
      n_c = 0;
      for (int base = 0; base < n_k * ratio; base += 32) {
        const int i = base + lane;
        int y = 0;
        bool ok = false;
        if (i < n_k * ratio) {
          y = nxt[i / ratio] * ratio + i % ratio;
          ok = y <= own;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, ok);
        const int pos = n_c + __popc(bal & lt);
        if (ok && pos < a.cap) cur[pos] = y;
        n_c += __popc(bal);
      }
      n_c = min(n_c, a.cap);
    }
    __syncwarp();
    // scores; the own chunk takes no part in the ranking (it is kept)
    int own_pos = -1;
    for (int base = 0; base < n_c; base += 32) {
      const int i = base + lane;
      bool is_own = false;
      if (i < n_c) {
        const int x = cur[i];
        float best = -INFINITY;
        if (x != own) {
          const int n_end = min(x * c + c, m + 1);
          for (int nb = x * c; nb < n_end; ++nb) best = fmaxf(best, row[nb]);
        } else {
          is_own = true;
        }
        sc[i] = best;
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, is_own);
      if (bal) own_pos = base + __ffs(static_cast<int>(bal)) - 1;
    }
    __syncwarp();
    const int need = min(a.st.keep[s] - 1, n_c - (own_pos >= 0 ? 1 : 0));
    uint32_t prefix = 0u, mask = 0u;
    int take = need;
    if (need > 0) {
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = lane; i < 256; i += 32) h[i] = 0;
        __syncwarp();
        for (int i = lane; i < n_c; i += 32) {
          const uint32_t key = ordered_key(sc[i]);
          if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1);
        }
        __syncwarp();
        // lane l holds bins 255 - 8l down to 248 - 8l; the bucket is the one
        // in which the count from the top reaches `take`
        int cnt[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = h[255 - 8 * lane - j];
          tot += cnt[j];
        }
        int incl = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        const int excl = incl - tot;
        const bool mine = excl < take && incl >= take;
        const int src = __ffs(static_cast<int>(__ballot_sync(0xffffffffu, mine))) - 1;
        int bucket = 0, above = excl;
        if (mine) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (above + cnt[j] >= take) {
              bucket = 255 - 8 * lane - j;
              break;
            }
            above += cnt[j];
          }
        }
        bucket = __shfl_sync(0xffffffffu, bucket, src);
        above = __shfl_sync(0xffffffffu, above, src);
        take -= above;
        prefix |= static_cast<uint32_t>(bucket) << shift;
        mask |= 255u << shift;
        __syncwarp();  // every lane has read the histogram before it is cleared
      }
    }
    // kept chunks, ascending: the own chunk, keys above the threshold, and the
    // first `take` keys equal to it (lower chunks first)
    n_k = 0;
    int eq_seen = 0;
    for (int base = 0; base < n_c; base += 32) {
      const int i = base + lane;
      bool keep = false, eq = false;
      if (i < n_c) {
        if (i == own_pos) {
          keep = true;
        } else if (need > 0) {
          const uint32_t key = ordered_key(sc[i]);
          eq = key == prefix;
          keep = key > prefix;
        }
      }
      const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
      keep |= eq && eq_seen + __popc(eqb & lt) < take;
      eq_seen += __popc(eqb);
      const uint32_t kb = __ballot_sync(0xffffffffu, keep);
      if (keep) nxt[n_k + __popc(kb & lt)] = cur[i];
      n_k += __popc(kb);
    }
    __syncwarp();
    c_prev = c;
  }
  // the last stage's chunks are single blocks
  int32_t* ids = a.block_ids + (static_cast<int64_t>(unit) * a.NB + m) * a.kb;
  const int cnt = min(n_k, a.kb);
  for (int i = lane; i < cnt; i += 32) ids[i] = nxt[i];
  if (lane == 0) a.block_count[static_cast<int64_t>(unit) * a.NB + m] = cnt;
}

// Candidate chunks a stage can hold at most (the first stage: every chunk of
// [0, NB); later: the previous stage's kept chunks times the size ratio).
int hip_stage_cap(int NB, const int32_t* c, const int32_t* keep, int n) {
  int cap = NB / c[0] + 1;
  for (int s = 1; s < n; ++s) {
    const int64_t v = static_cast<int64_t>(keep[s - 1]) * (c[s - 1] / c[s]);
    cap = static_cast<int>(v > cap ? (v < NB + 1 ? v : NB + 1) : cap);
  }
  return cap;
}

}  // namespace

int hip_slab_rows(int n_units, int NB) {
  // block maxima of one slab: n_units x rows x NB floats, at most 512 MiB
  const int64_t per_row = static_cast<int64_t>(n_units) * NB * 4;
  const int64_t fit = (int64_t{512} << 20) / (per_row > 0 ? per_row : 1);
  if (fit >= NB) return NB;
  const int64_t rows = fit / kRT * kRT;
  return static_cast<int>(rows < kRT ? kRT : rows);
}

cudaError_t launch_hip_index(const Geometry& g, const UnitMap& u, const CUtensorMap& mk,
                             const float* qpool, __nv_bfloat16* qsplit,
                             const CUtensorMap& mqs, const int32_t* stage_c,
                             const int32_t* stage_keep, int n_stages, float* rmax, int slab_rows,
                             int32_t* block_count, int32_t* block_ids, int kb, uint32_t* status,
                             cudaStream_t st, int* n_launch) {
  if (n_stages < 1 || n_stages > MSA_HIP_MAX_STAGES) return cudaErrorInvalidValue;
  const int64_t n_split = static_cast<int64_t>(g.n_units) * g.NB * kHeadDim;
  int64_t split_blocks = (n_split + kSplitThreads - 1) / kSplitThreads;
  if (split_blocks > 152 * 8) split_blocks = 152 * 8;
  hip_split_kernel<<<static_cast<unsigned>(split_blocks), kSplitThreads, 0, st>>>(qpool, n_split,
                                                                                qsplit);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*n_launch;
  HipScoreArgs sa;
  sa.u = u;
  sa.N = g.N;
  sa.NB = g.NB;
  sa.G = g.G;
  sa.n_units = g.n_units;
  sa.slab_stride = slab_rows;
  sa.scale = g.scale;
  sa.rmax = rmax;
  sa.status = status;
  HipSelArgs ta;
  ta.NB = g.NB;
  ta.slab_stride = slab_rows;
  ta.rmax = rmax;
  ta.st.n = n_stages;
  for (int s = 0; s < n_stages; ++s) {
    ta.st.c[s] = stage_c[s];
    ta.st.keep[s] = stage_keep[s];
  }
  ta.block_count = block_count;
  ta.block_ids = block_ids;
  ta.kb = kb;
  const int score_smem = static_cast<int>(sizeof(ScoreSmem)) + 1024;
  // the warp-level selection while eight warps' candidate lists (a score and
  // two ids per candidate) fit in 160 KB of shared memory, else a CTA per
  // query block
  ta.cap = hip_stage_cap(g.NB, stage_c, stage_keep, n_stages);
  ta.warps = kSelWarps;
  const bool warp_sel = static_cast<int64_t>(ta.cap) * 12 * kSelWarps <= 160 * 1024;
  const int sel_smem = warp_sel ? ta.cap * 12 * kSelWarps : (g.NB + (g.NB + 31) / 32) * 4;
  e = cudaFuncSetAttribute(hip_block_max_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           score_smem);
  if (e != cudaSuccess) return e;
  if (sel_smem > 48 * 1024) {
    e = warp_sel ? cudaFuncSetAttribute(hip_select_warp_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, sel_smem)
                 : cudaFuncSetAttribute(hip_select_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, sel_smem);
    if (e != cudaSuccess) return e;
  }
  const int n_kt = (g.N + kKT - 1) / kKT;
  for (int m0 = 0; m0 < g.NB; m0 += slab_rows) {
    const int rows = min(slab_rows, g.NB - m0);
    sa.m0 = m0;
    sa.rows = rows;
    // key tiles past the slab's last query block hold no candidate
    const int kt_end = min(n_kt, (m0 + rows - 1) / 2 + 1);
    const int chunks = (kt_end + kChunkTiles - 1) / kChunkTiles;
    hip_block_max_kernel<<<dim3(chunks, (rows + kRT - 1) / kRT, g.n_units), kScoreThreads,
                           score_smem, st>>>(sa, mqs, mk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++*n_launch;
    ta.m0 = m0;
    ta.rows = rows;
    if (warp_sel)
      hip_select_warp_kernel<<<dim3((rows + kSelWarps - 1) / kSelWarps, g.n_units), kSelThreads,
                               sel_smem, st>>>(ta);
    else
      hip_select_kernel<<<dim3(rows, g.n_units), kSelThreads, sel_smem, st>>>(ta);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++*n_launch;
  }
  return cudaSuccess;
}

}  // namespace msa
