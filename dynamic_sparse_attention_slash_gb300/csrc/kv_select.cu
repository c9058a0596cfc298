// KV-selection score after the prefill ("How KV sparsity achieves 1.5x
// acceleration for vLLM", Novita AI blog, section "2. Attention modification"):
// the attention pass exports each row's normaliser lse_i = ln sum_{j in J_i}
// exp(z_ij); this second pass runs in key-major order, as the page prescribes,
// so that each key's sum stays with one thread:
//   S_j = sum over window rows i (i in [N - window, N), j <= i, j in J_i)
//         of exp(z_ij - lse_i),       z_ij = scale * q_i . k_j.
// J_i is the key set the call's own attention used for row i (vertical-slash:
// active 64x64 tiles plus vertical columns; block-sparse: the kept blocks;
// streaming: sinks plus the local window), so S sums the probabilities that
// the call actually computed.
//
// One CTA owns 128 keys of one unit and loops over the window's 64-row blocks
// (only those with a row at or after its first key): Q K^T on the warp-level
// bf16 tensor cores, probabilities into shared memory, then thread t adds
// column t over the block's rows in a fixed order.  No atomics: the score is
// deterministic.
#include "mma16.cuh"

namespace msa {
namespace {

using namespace mma16;

constexpr int kChunk = 128;              // keys per CTA (two 64-key tiles)
constexpr int kPStride = kChunk + 4;     // f32 row stride of the probability tile
constexpr float kLog2e = 1.4426950408889634f;

struct KvArgs {
  Geometry g;
  UnitMap u;
  const __nv_bfloat16* q;
  int64_t q_sb, q_sh, q_sn;
  const __nv_bfloat16* k;
  int64_t k_sb, k_sh, k_sn;
  const float* lse;   // [B][Hq][N]
  float* score;       // [B][Hq][N]
  int window;
  float scale_log2;
  KvMask mask;
};

// Is 64-key block n admitted for row block m (before the causal cut)?
__device__ __forceinline__ bool block_admitted(const KvMask& mk, int unit, int m, int n) {
  if (n > m) return false;
  if (mk.kind == kPrefillVS) {
    const uint32_t* dist = mk.tile_dist + static_cast<int64_t>(unit) * mk.dist_words;
    const int t = m - n;
    return (dist[t >> 5] >> (t & 31)) & 1u;
  }
  if (mk.kind == kPrefillBS) {
    const int64_t rb = static_cast<int64_t>(unit) * mk.NB + m;
    const int cnt = mk.block_count[rb];
    const int32_t* ids = mk.block_ids + rb * mk.kb;
    int lo = 0, hi = cnt;  // ids ascending
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (ids[mid] < n) lo = mid + 1; else hi = mid;
    }
    return lo < cnt && ids[lo] == n;
  }
  return n < mk.init_num || n > m - mk.local_num;
}

__global__ void __launch_bounds__(kThreads) kv_score_kernel(const __grid_constant__ KvArgs a) {
  extern __shared__ __align__(1024) uint8_t dyn[];
  uint8_t* sm_q = dyn;                          // 64 rows x 256 B
  uint8_t* sm_k = dyn + 64 * 256;               // 128 keys x 256 B
  float* sm_p = reinterpret_cast<float*>(dyn + 64 * 256 + kChunk * 256);  // 64 x kPStride
  __shared__ float s_lse2[64];                  // lse * log2(e) of the block's rows
  __shared__ uint32_t s_col[kChunk / 32];       // vertical columns among this CTA's keys
  __shared__ int s_adm[2];                      // the two key blocks admitted for row block m?
  const int unit = blockIdx.y, chunk = blockIdx.x;
  const int N = a.g.N;
  const int j0 = chunk * kChunk;
  const int b = unit / a.u.n_heads, h = a.u.heads[unit % a.u.n_heads];
  const __nv_bfloat16* qb = a.q + b * a.q_sb + h * a.q_sh;
  const __nv_bfloat16* kb = a.k + b * a.k_sb + (h / a.g.G) * a.k_sh;
  const int64_t row_base = (static_cast<int64_t>(b) * a.g.Hq + h) * N;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  load_rows(smem_u32(sm_k), kb, a.k_sn, j0, kChunk, N);
  cp_async_commit();
  if (tid < kChunk / 32) s_col[tid] = 0u;
  __syncthreads();
  if (a.mask.kind == kPrefillVS) {
    // the unit's vertical columns are ascending: mark those in [j0, j0 + 128)
    const int32_t* V = a.mask.vertical + static_cast<int64_t>(unit) * a.mask.kv;
    for (int x = tid; x < a.mask.kv; x += kThreads) {
      const int j = V[x];
      if (j >= j0 && j < j0 + kChunk) atomicOr(&s_col[(j - j0) >> 5], 1u << ((j - j0) & 31));
    }
  }
  const int w0 = N - a.window;          // first window row
  const int m_first = w0 >> 6;          // first window row block
  const int m_lo = max(m_first, j0 >> 6);  // earlier row blocks end before key j0
  const int NB = (N + 63) >> 6;          // a partial last block counts
  float acc_s = 0.f;                    // score of key j0 + tid
  for (int m = m_lo; m < NB; ++m) {
    const int r0 = m * 64;
    load_rows(smem_u32(sm_q), qb, a.q_sn, r0, 64, N);
    cp_async_commit();
    if (tid < 64) {
      const int i = r0 + tid;
      const float l = i < N ? a.lse[row_base + i] : -INFINITY;
      // rows before the window, padded rows and rows without keys contribute nothing
      s_lse2[tid] = (i >= w0 && l != -INFINITY) ? l * kLog2e : INFINITY;
    }
    if (tid < 2) s_adm[tid] = block_admitted(a.mask, unit, m, (j0 >> 6) + tid) ? 1 : 0;
    cp_async_wait_all();
    __syncthreads();
    uint32_t qa[8][4];
    load_q_frags(smem_u32(sm_q), qa);
    const int rA = warp * 16 + (lane >> 2), rB = rA + 8;
    const int iA = r0 + rA, iB = r0 + rB;
    const float lA = s_lse2[rA], lB = s_lse2[rB];
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      float acc[8][4];
      tile_logits(qa, smem_u32(sm_k + kt * kKeyTile * 256), acc);
      const bool adm = s_adm[kt] != 0;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = kt * kKeyTile + nt * 8 + 2 * (lane & 3) + e;
          const int j = j0 + col;
          const bool in_j = adm || ((s_col[col >> 5] >> (col & 31)) & 1u);
          // lA / lB is +inf for rows outside the window: ex2(-inf) = 0
          const float pA = (in_j && j <= iA) ? ex2_approx(acc[nt][e] * a.scale_log2 - lA) : 0.f;
          const float pB = (in_j && j <= iB) ? ex2_approx(acc[nt][2 + e] * a.scale_log2 - lB) : 0.f;
          sm_p[rA * kPStride + col] = pA;
          sm_p[rB * kPStride + col] = pB;
        }
      }
    }
    __syncthreads();
    float s = 0.f;
    for (int r = 0; r < 64; ++r) s += sm_p[r * kPStride + tid];
    acc_s += s;
    __syncthreads();
  }
  if (j0 + tid < N) a.score[row_base + j0 + tid] = acc_s;
}

}  // namespace

cudaError_t launch_kv_score(const Geometry& g, const UnitMap& u, TensorView q, TensorView k,
                            const float* lse, float* score, int window, const KvMask& mask,
                            cudaStream_t st, int* n_launch) {
  KvArgs a;
  a.g = g;
  a.u = u;
  a.q = q.data; a.q_sb = q.sb; a.q_sh = q.sh; a.q_sn = q.sn;
  a.k = k.data; a.k_sb = k.sb; a.k_sh = k.sh; a.k_sn = k.sn;
  a.lse = lse;
  a.score = score;
  a.window = window;
  a.scale_log2 = g.scale * kLog2e;
  a.mask = mask;
  const int smem = 64 * 256 + kChunk * 256 + 64 * kPStride * 4;
  // per call: the attribute belongs to the current device
  cudaError_t e =
      cudaFuncSetAttribute(kv_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_chunks = (g.N + kChunk - 1) / kChunk;
  kv_score_kernel<<<dim3(n_chunks, g.n_units), kThreads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
