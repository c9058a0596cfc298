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
// block n of the token scores: hip_block_max_kernel computes them, fp32 with
// packed f32x2 FMAs in a fixed order (deterministic), for the causal blocks
// n <= m only.  It is a register-tiled product of 64 pooled queries with 128
// keys per CTA: each thread holds 8 rows x 8 keys, the two operands staged in
// shared memory transposed (dimension-major), so one dimension step is four
// 16-byte shared loads for 32 f32x2 FMAs.
//
// Selection.  hip_select_kernel runs the stages for one query block per CTA:
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

constexpr int kRT = 64;             // pooled query rows (query blocks) per score CTA
constexpr int kKT = 128;            // keys per score CTA (two key blocks)
constexpr int kScoreThreads = 128;  // 8 x 16 threads: 8 rows x 8 keys each
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

struct HipScoreArgs {
  UnitMap u;
  int N, NB, G;
  int m0, rows;        // the slab: query blocks [m0, m0 + rows)
  int slab_stride;     // rows of rmax per unit
  float scale;
  const float* qpool;  // [units][NB][128]
  const __nv_bfloat16* k;
  int64_t k_sb, k_sh, k_sn;
  float* rmax;         // [units][slab_stride][NB]; entry (m - m0, n) for n <= m
};

struct __align__(16) ScoreSmem {
  float q[kHeadDim][kRT];  // q[d][r]: dimension d of pooled row r
  float k[kHeadDim][kKT];  // k[d][j]: dimension d of key j
};

// grid (key tile kt, row tile, unit): block maxima of query blocks
// [m0 + 64 rt, +64) against key blocks 2kt and 2kt + 1.
__global__ void __launch_bounds__(kScoreThreads) hip_block_max_kernel(const __grid_constant__ HipScoreArgs a) {
  extern __shared__ __align__(16) uint8_t dyn[];
  ScoreSmem& sm = *reinterpret_cast<ScoreSmem*>(dyn);
  const int kt = blockIdx.x, unit = blockIdx.z;
  const int r0 = blockIdx.y * kRT;                 // first slab row of the tile
  const int m_first = a.m0 + r0;
  const int m_last = a.m0 + min(r0 + kRT, a.rows) - 1;
  if (2 * kt > m_last) return;  // every key of the tile is after every row's candidates
  const int tid = threadIdx.x;
  const int b = unit / a.u.n_heads;
  const int hkv = a.u.heads[unit % a.u.n_heads] / a.G;
  // stage the pooled queries (rows past the slab read as zero)
  const float* qp = a.qpool + static_cast<int64_t>(unit) * a.NB * kHeadDim;
  for (int i = tid; i < kRT * (kHeadDim / 4); i += kScoreThreads) {
    const int r = i % kRT, d4 = i / kRT;  // consecutive threads: consecutive rows (no bank conflict)
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m_first + r <= m_last)
      v = reinterpret_cast<const float4*>(qp + static_cast<int64_t>(m_first + r) * kHeadDim)[d4];
    sm.q[4 * d4 + 0][r] = v.x;
    sm.q[4 * d4 + 1][r] = v.y;
    sm.q[4 * d4 + 2][r] = v.z;
    sm.q[4 * d4 + 3][r] = v.w;
  }
  // stage the keys as f32 (keys past N read as zero; they are masked below)
  {
    const int j = kKT * kt + tid;
    const __nv_bfloat16* kr = a.k + b * a.k_sb + hkv * a.k_sh + static_cast<int64_t>(j) * a.k_sn;
#pragma unroll 4
    for (int d8 = 0; d8 < kHeadDim / 8; ++d8) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (j < a.N) raw = reinterpret_cast<const uint4*>(kr)[d8];
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sm.k[8 * d8 + 2 * e][tid] = __low2float(h2[e]);
        sm.k[8 * d8 + 2 * e + 1][tid] = __high2float(h2[e]);
      }
    }
  }
  __syncthreads();
  const int ty = tid >> 4, tx = tid & 15;  // rows 8 ty .. + 7, keys 8 tx .. + 7
  float2 acc[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = make_float2(0.f, 0.f);
#pragma unroll 4
  for (int d = 0; d < kHeadDim; ++d) {
    const float4 qa = *reinterpret_cast<const float4*>(&sm.q[d][8 * ty]);
    const float4 qb = *reinterpret_cast<const float4*>(&sm.q[d][8 * ty + 4]);
    const float4 ka = *reinterpret_cast<const float4*>(&sm.k[d][8 * tx]);
    const float4 kb = *reinterpret_cast<const float4*>(&sm.k[d][8 * tx + 4]);
    const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const float2 kv[4] = {make_float2(ka.x, ka.y), make_float2(ka.z, ka.w),
                          make_float2(kb.x, kb.y), make_float2(kb.z, kb.w)};
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float2 q2 = make_float2(qv[r], qv[r]);
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = ffma2(q2, kv[c], acc[r][c]);
    }
  }
  // block maxima: this thread's 8 keys, then the 8 threads of a key block
  // (lanes differing in bits 0..2); keys past N do not count
  const int j0 = kKT * kt + 8 * tx;
  const int n = 2 * kt + (tx >> 3);
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (j0 + 2 * c < a.N) mx = fmaxf(mx, acc[r][c].x);
      if (j0 + 2 * c + 1 < a.N) mx = fmaxf(mx, acc[r][c].y);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    const int m = m_first + 8 * ty + r;
    if ((tx & 7) == 0 && m <= m_last && n <= m)
      a.rmax[(static_cast<int64_t>(unit) * a.slab_stride + (m - a.m0)) * a.NB + n] = mx * a.scale;
  }
}

struct HipStages {
  int n;
  int c[MSA_HIP_MAX_STAGES];
  int keep[MSA_HIP_MAX_STAGES];
};

struct HipSelArgs {
  int NB, m0, slab_stride;
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

}  // namespace

int hip_slab_rows(int n_units, int NB) {
  // block maxima of one slab: n_units x rows x NB floats, at most 512 MiB
  const int64_t per_row = static_cast<int64_t>(n_units) * NB * 4;
  const int64_t fit = (int64_t{512} << 20) / (per_row > 0 ? per_row : 1);
  if (fit >= NB) return NB;
  const int64_t rows = fit / kRT * kRT;
  return static_cast<int>(rows < kRT ? kRT : rows);
}

cudaError_t launch_hip_index(const Geometry& g, const UnitMap& u, TensorView k, const float* qpool,
                             const int32_t* stage_c, const int32_t* stage_keep, int n_stages,
                             float* rmax, int slab_rows, int32_t* block_count, int32_t* block_ids,
                             int kb, cudaStream_t st, int* n_launch) {
  if (n_stages < 1 || n_stages > MSA_HIP_MAX_STAGES) return cudaErrorInvalidValue;
  HipScoreArgs sa;
  sa.u = u;
  sa.N = g.N;
  sa.NB = g.NB;
  sa.G = g.G;
  sa.slab_stride = slab_rows;
  sa.scale = g.scale;
  sa.qpool = qpool;
  sa.k = k.data; sa.k_sb = k.sb; sa.k_sh = k.sh; sa.k_sn = k.sn;
  sa.rmax = rmax;
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
  const int score_smem = static_cast<int>(sizeof(ScoreSmem));
  const int sel_smem = (g.NB + (g.NB + 31) / 32) * 4;
  cudaError_t e = cudaFuncSetAttribute(hip_block_max_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, score_smem);
  if (e != cudaSuccess) return e;
  if (sel_smem > 48 * 1024) {
    e = cudaFuncSetAttribute(hip_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             sel_smem);
    if (e != cudaSuccess) return e;
  }
  const int n_kt = (g.N + kKT - 1) / kKT;
  for (int m0 = 0; m0 < g.NB; m0 += slab_rows) {
    const int rows = min(slab_rows, g.NB - m0);
    sa.m0 = m0;
    sa.rows = rows;
    // key tiles past the slab's last query block hold no candidate
    const int kt_end = min(n_kt, (m0 + rows - 1) / 2 + 1);
    hip_block_max_kernel<<<dim3(kt_end, (rows + kRT - 1) / kRT, g.n_units), kScoreThreads,
                           score_smem, st>>>(sa);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++*n_launch;
    ta.m0 = m0;
    hip_select_kernel<<<dim3(rows, g.n_units), kSelThreads, sel_smem, st>>>(ta);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++*n_launch;
  }
  return cudaSuccess;
}

}  // namespace msa
