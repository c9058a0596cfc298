// Vertical-slash estimate (MInference 1.0 overview, section 2.2, "Vertical-Slash
// Head", first step): the last `last_q` query rows are multiplied with every key,
// soft-maxed causally, and reduced into
//   v_score[j] = sum_i A[i, j]           (vertical line through key j)
//   s_score[o] = sum_i A[i, i - o]       (slash line at offset o = i - j)
// The softmax normaliser comes from a first pass (row max and row sum per key
// range, the two quantities the Novita vLLM article's "Attention modification"
// section exports from FlashAttention); the second pass recomputes the logits
// and forms the probabilities.  Both passes run on the warp-level bf16 tensor
// core instruction; the estimate is under 1% of a prefill.
//
// Determinism: every v_score / s_score entry is summed by exactly one thread in a
// fixed row order; no atomics.
#include "mma16.cuh"

namespace msa {
namespace {

using namespace mma16;
constexpr int kChunk = 256;       // keys (and diagonals) owned by one second-pass CTA
constexpr int kWindow = kChunk + kKeyTile;  // keys a second-pass CTA computes
constexpr int kWinTiles = kWindow / kKeyTile;
constexpr int kAStride = kWindow + 4;       // fp32 row stride of the probability tile
constexpr int kScoreThreads = 256;          // two groups of four warps, alternate key tiles
constexpr float kLog2e = 1.4426950408889634f;

struct EstArgs {
  Geometry g;
  UnitMap u;
  const __nv_bfloat16* q;
  int64_t q_sb, q_sh, q_sn;
  const __nv_bfloat16* k;
  int64_t k_sb, k_sh, k_sn;
  int last_q;
  int n_split;
  float scale_log2;
  float* partial;    // [units][n_split][64][2] (row max in log2 units, row sum)
  float* v_score;    // [units][N]
  float* s_score;    // [units][N]
};

__device__ __forceinline__ void unit_ptrs(const EstArgs& a, int unit, const __nv_bfloat16*& qb,
                                          const __nv_bfloat16*& kb) {
  const int b = unit / a.u.n_heads;
  const int h = a.u.heads[unit % a.u.n_heads];
  qb = a.q + b * a.q_sb + h * a.q_sh;
  kb = a.k + b * a.k_sb + (h / a.g.G) * a.k_sh;
}

// Pass 1: per key range, running row max / row sum of exp over causal keys.
__global__ void __launch_bounds__(kThreads) vs_estimate_stats_kernel(const __grid_constant__ EstArgs a) {
  __shared__ __align__(1024) uint8_t sm_q[64 * 256];
  __shared__ __align__(1024) uint8_t sm_k[2][kKeyTile * 256];
  const int unit = blockIdx.y, split = blockIdx.x;
  const int N = a.g.N;
  const __nv_bfloat16 *qb, *kb;
  unit_ptrs(a, unit, qb, kb);
  const int n_tiles = (N + kKeyTile - 1) / kKeyTile;
  const int t_begin = static_cast<int>((static_cast<int64_t>(n_tiles) * split) / a.n_split);
  const int t_end = static_cast<int>((static_cast<int64_t>(n_tiles) * (split + 1)) / a.n_split);
  const int row0 = N - 64;  // window row r is query i = row0 + r; valid iff r >= 64 - last_q
  const uint32_t q_s = smem_u32(sm_q);
  load_rows(q_s, qb, a.q_sn, row0, 64, N);
  if (t_begin < t_end) load_rows(smem_u32(sm_k[0]), kb, a.k_sn, t_begin * kKeyTile, kKeyTile, N);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();
  uint32_t qa[8][4];
  load_q_frags(q_s, qa);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rA = warp * 16 + (lane >> 2), rB = rA + 8;
  const int iA = row0 + rA, iB = row0 + rB;
  const bool vA = rA >= 64 - a.last_q, vB = rB >= 64 - a.last_q;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  for (int t = t_begin; t < t_end; ++t) {
    const int buf = (t - t_begin) & 1;
    if (t + 1 < t_end)
      load_rows(smem_u32(sm_k[buf ^ 1]), kb, a.k_sn, (t + 1) * kKeyTile, kKeyTile, N);
    cp_async_commit();
    float acc[8][4];
    tile_logits(qa, smem_u32(sm_k[buf]), acc);
    float tmA = -INFINITY, tmB = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = t * kKeyTile + nt * 8 + 2 * (lane & 3) + e;
        const float xA = (vA && j <= iA) ? acc[nt][e] * a.scale_log2 : -INFINITY;
        const float xB = (vB && j <= iB) ? acc[nt][2 + e] * a.scale_log2 : -INFINITY;
        acc[nt][e] = xA;
        acc[nt][2 + e] = xB;
        tmA = fmaxf(tmA, xA);
        tmB = fmaxf(tmB, xB);
      }
    }
    tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 1));
    tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 2));
    tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 1));
    tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 2));
    const float nmA = fmaxf(mA, tmA), nmB = fmaxf(mB, tmB);
    float sA = 0.f, sB = 0.f;
    if (nmA != -INFINITY) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) sA += ex2_approx(acc[nt][0] - nmA) + ex2_approx(acc[nt][1] - nmA);
      lA = lA * ex2_approx(mA - nmA) + sA;
      mA = nmA;
    }
    if (nmB != -INFINITY) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) sB += ex2_approx(acc[nt][2] - nmB) + ex2_approx(acc[nt][3] - nmB);
      lB = lB * ex2_approx(mB - nmB) + sB;
      mB = nmB;
    }
    cp_async_wait_all();
    __syncthreads();
  }
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  if ((lane & 3) == 0) {
    float* p = a.partial + (static_cast<int64_t>(unit) * a.n_split + split) * 128;
    p[2 * rA] = mA;
    p[2 * rA + 1] = lA;
    p[2 * rB] = mB;
    p[2 * rB + 1] = lB;
  }
}

// Pass 2: probabilities for keys [j0, j0 + 320) (the owned keys [j0, j0 + 256)
// and the 64 after them, which the owned diagonals reach), then column sums for
// the owned keys and diagonal sums for the owned offsets.
__global__ void __launch_bounds__(kScoreThreads) vs_estimate_scores_kernel(const __grid_constant__ EstArgs a) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  uint8_t* sm_q = dyn;                          // 16 KB
  uint8_t* sm_k = dyn + 64 * 256;               // 4 x 16 KB: two key tiles per step, two steps
  float* sm_a = reinterpret_cast<float*>(dyn + 64 * 256 + 4 * kKeyTile * 256);  // 64 x kAStride
  __shared__ float s_m[64], s_linv[64];
  const int unit = blockIdx.y, chunk = blockIdx.x;
  const int N = a.g.N;
  const int j0 = chunk * kChunk;
  const __nv_bfloat16 *qb, *kb;
  unit_ptrs(a, unit, qb, kb);
  const int row0 = N - 64;
  const uint32_t q_s = smem_u32(sm_q);
  auto k_buf = [&](int i) { return smem_u32(sm_k + i * kKeyTile * 256); };
  load_rows(q_s, qb, a.q_sn, row0, 64, N);
  load_rows(k_buf(0), kb, a.k_sn, j0, kKeyTile, N);
  load_rows(k_buf(1), kb, a.k_sn, j0 + kKeyTile, kKeyTile, N);
  cp_async_commit();
  // combine the first pass: m = max_s m_s, l = sum_s l_s 2^(m_s - m)
  if (threadIdx.x < 64) {
    const float* p = a.partial + static_cast<int64_t>(unit) * a.n_split * 128 + 2 * threadIdx.x;
    float m = -INFINITY;
    for (int s = 0; s < a.n_split; ++s) m = fmaxf(m, p[s * 128]);
    float l = 0.f;
    if (m != -INFINITY)
      for (int s = 0; s < a.n_split; ++s)
        if (p[s * 128] != -INFINITY) l += p[s * 128 + 1] * ex2_approx(p[s * 128] - m);
    s_m[threadIdx.x] = m;
    s_linv[threadIdx.x] = l > 0.f ? 1.f / l : 0.f;
  }
  cp_async_wait_all();
  __syncthreads();
  // warp w: query rows 16 (w % 4) .. + 15 of key tiles w / 4, w / 4 + 2, ...
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = warp >> 2, wq = warp & 3;
  uint32_t qa[8][4];
  load_q_frags(q_s, qa, wq);
  const int rA = wq * 16 + (lane >> 2), rB = rA + 8;
  const int iA = row0 + rA, iB = row0 + rB;
  const bool vA = rA >= 64 - a.last_q, vB = rB >= 64 - a.last_q;
  const float mA = s_m[rA], mB = s_m[rB], liA = s_linv[rA], liB = s_linv[rB];
  constexpr int kSteps = (kWinTiles + 1) / 2;
  for (int step = 0; step < kSteps; ++step) {
    const int buf = step & 1;
    if (step + 1 < kSteps) {  // the next step's two tiles into the other buffer pair
      for (int g2 = 0; g2 < 2; ++g2) {
        const int tn = 2 * (step + 1) + g2;
        if (tn < kWinTiles)
          load_rows(k_buf((buf ^ 1) * 2 + g2), kb, a.k_sn, j0 + tn * kKeyTile, kKeyTile, N);
      }
    }
    cp_async_commit();
    const int t = 2 * step + grp;
    if (t < kWinTiles) {
      float acc[8][4];
      tile_logits(qa, k_buf(buf * 2 + grp), acc);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = t * kKeyTile + nt * 8 + 2 * (lane & 3) + e;
          const int j = j0 + col;
          const float pA = (vA && j <= iA) ? ex2_approx(acc[nt][e] * a.scale_log2 - mA) * liA : 0.f;
          const float pB = (vB && j <= iB) ? ex2_approx(acc[nt][2 + e] * a.scale_log2 - mB) * liB : 0.f;
          sm_a[rA * kAStride + col] = pA;
          sm_a[rB * kAStride + col] = pB;
        }
      }
    }
    cp_async_wait_all();
    __syncthreads();
  }
  const int t = threadIdx.x;
  float* vs = a.v_score + static_cast<int64_t>(unit) * N;
  float* ss = a.s_score + static_cast<int64_t>(unit) * N;
  // vertical: key j0 + t
  if (j0 + t < N) {
    float s = 0.f;
    for (int r = 0; r < 64; ++r) s += sm_a[r * kAStride + t];
    vs[j0 + t] = s;
  }
  // slash: offset o whose first window key N-64-o equals j0 + t
  {
    const int o = N - 64 - j0 - t;
    if (o >= 0) {
      float s = 0.f;
      for (int r = 0; r < 64; ++r) s += sm_a[r * kAStride + t + r];
      ss[o] = s;
    }
  }
  // offsets o > N-64 start before key 0; chunk 0 owns them
  if (chunk == 0 && t < 63 && N - 63 + t >= 0) {
    const int o = N - 63 + t;  // first key N-64-o = -(t+1); o >= 0 when N < 64 too
    float s = 0.f;
    for (int r = t + 1; r < 64; ++r) s += sm_a[r * kAStride + (r - t - 1)];
    ss[o] = s;
  }
}

}  // namespace

cudaError_t launch_vs_estimate(const Geometry& g, const UnitMap& u, TensorView q, TensorView k,
                               int last_q, float* partial, int n_split, float* row_stats,
                               float* v_score, float* s_score, cudaStream_t st, int* n_launch) {
  (void)row_stats;
  EstArgs a;
  a.g = g;
  a.u = u;
  a.q = q.data; a.q_sb = q.sb; a.q_sh = q.sh; a.q_sn = q.sn;
  a.k = k.data; a.k_sb = k.sb; a.k_sh = k.sh; a.k_sn = k.sn;
  a.last_q = last_q;
  a.n_split = n_split;
  a.scale_log2 = g.scale * kLog2e;
  a.partial = partial;
  a.v_score = v_score;
  a.s_score = s_score;
  vs_estimate_stats_kernel<<<dim3(n_split, g.n_units), kThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*n_launch;
  const int smem = 64 * 256 + 4 * kKeyTile * 256 + 64 * kAStride * 4;
  // per call: the attribute belongs to the current device
  e = cudaFuncSetAttribute(vs_estimate_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_chunks = (g.N + kChunk - 1) / kChunk;
  vs_estimate_scores_kernel<<<dim3(n_chunks, g.n_units), kScoreThreads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
