// Exact top-k selection of line scores (MInference 1.0 overview, section 2.2,
// "Vertical-Slash Head": pick the vertical lines and slash lines).
//
// Order: score descending, ties to the lower index; the chosen indices are
// written in ascending order.  Method: a 4-pass 8-bit radix select on the
// order-preserving uint32 key finds the k-th largest key T and how many of the
// elements equal to T are taken; one more pass in index order keeps every
// element above T and the first such elements equal to T, and compacts the
// kept indices with a CTA-wide prefix sum (so the output is ascending by
// construction).  One 1024-thread CTA per score row; deterministic.
#include "block_scan.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 8;  // consecutive elements per thread in the compaction pass

// Top-k of one row s[0, n) into o[0, min(k, n)).
__device__ __forceinline__ void topk_row(const float* __restrict__ s, int64_t n, int k,
                                         int32_t* __restrict__ o) {
  __shared__ int hist[kWarps][256];
  __shared__ int total_hist[256];
  __shared__ int warp_sums[kWarps + 1];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (k >= n) {
    for (int64_t j = tid; j < n; j += kThreads) o[j] = static_cast<int32_t>(j);
    return;
  }
  if (k <= 0) return;
  if (tid == 0) {
    s_prefix = 0u;
    s_mask = 0u;
    s_need = k;
  }
  __syncthreads();
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < kWarps * 256; i += kThreads) (&hist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int64_t j = tid; j < n; j += kThreads) {
      const uint32_t key = ordered_key(s[j]);
      if ((key & mask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 256) {
      int c = 0;
      for (int w = 0; w < kWarps; ++w) c += hist[w][tid];
      total_hist[tid] = c;
    }
    __syncthreads();
    if (tid == 0) {
      int need = s_need, above = 0, bucket = 0;
      for (int b = 255; b >= 0; --b) {
        if (above + total_hist[b] >= need) {
          bucket = b;
          break;
        }
        above += total_hist[b];
      }
      s_need = need - above;
      s_prefix = prefix | (static_cast<uint32_t>(bucket) << shift);
      s_mask = mask | (255u << shift);
    }
    __syncthreads();
  }
  const uint32_t T = s_prefix;  // key of the k-th largest element
  const int take_equal = s_need; // elements equal to T to keep, lowest indices first
  int kept_before = 0, equal_before = 0;
  for (int64_t base = 0; base < n; base += static_cast<int64_t>(kThreads) * kItems) {
    const int64_t j0 = base + static_cast<int64_t>(tid) * kItems;
    uint32_t keys[kItems];
    int n_eq = 0;
#pragma unroll
    for (int e = 0; e < kItems; ++e) {
      keys[e] = (j0 + e < n) ? ordered_key(s[j0 + e]) : 0u;
      n_eq += (j0 + e < n && keys[e] == T) ? 1 : 0;
    }
    int eq_total;
    int eq_rank = equal_before + block_exclusive_scan<kThreads>(n_eq, warp_sums, &eq_total);
    int n_keep = 0;
    bool keep[kItems];
#pragma unroll
    for (int e = 0; e < kItems; ++e) {
      bool kp = false;
      if (j0 + e < n) {
        if (keys[e] > T) {
          kp = true;
        } else if (keys[e] == T) {
          kp = eq_rank < take_equal;
          ++eq_rank;
        }
      }
      keep[e] = kp;
      n_keep += kp ? 1 : 0;
    }
    int keep_total;
    int pos = kept_before + block_exclusive_scan<kThreads>(n_keep, warp_sums, &keep_total);
#pragma unroll
    for (int e = 0; e < kItems; ++e)
      if (keep[e]) o[pos++] = static_cast<int32_t>(j0 + e);
    kept_before += keep_total;
    equal_before += eq_total;
  }
}

// One CTA per row of one of two row sets (blockIdx.y); row r of set s at
// jobs[s].scores + r * row_stride.
__global__ void __launch_bounds__(kThreads, 1) topk_rows_kernel(int64_t n,
                                                             const __grid_constant__ TopkRows job0,
                                                             const __grid_constant__ TopkRows job1) {
  const bool second = blockIdx.y != 0;
  const float* scores = second ? job1.scores : job0.scores;
  const int64_t row_stride = second ? job1.row_stride : job0.row_stride;
  int32_t* out = second ? job1.out : job0.out;
  const int64_t out_stride = second ? job1.out_stride : job0.out_stride;
  topk_row(scores + static_cast<int64_t>(blockIdx.x) * row_stride, n, second ? job1.k : job0.k,
           out + static_cast<int64_t>(blockIdx.x) * out_stride);
}

// One CTA per selected (batch, head) unit u; its row lives at query-head index
// (u / n_heads) * Hq + heads[u % n_heads] of [B][Hq][n] scores and [B][Hq][k] out.
__global__ void __launch_bounds__(kThreads) topk_units_kernel(const float* __restrict__ scores,
                                                              int64_t n, int k, int Hq,
                                                              const __grid_constant__ UnitMap u,
                                                              int32_t* __restrict__ out) {
  const int unit = blockIdx.x;
  const int64_t row = static_cast<int64_t>(unit / u.n_heads) * Hq + u.heads[unit % u.n_heads];
  const int kk = k < n ? k : static_cast<int>(n);
  topk_row(scores + row * n, n, k, out + row * kk);
}

}  // namespace

cudaError_t launch_topk_units(const float* scores, int64_t n, int k, int Hq, const UnitMap& u,
                              int units, int32_t* out_idx, cudaStream_t st, int* n_launch) {
  if (units <= 0) return cudaSuccess;
  topk_units_kernel<<<units, kThreads, 0, st>>>(scores, n, k, Hq, u, out_idx);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

cudaError_t launch_topk_pair(int64_t n, int rows, const TopkRows& job0, const TopkRows& job1,
                             cudaStream_t st, int* n_launch) {
  if (rows <= 0) return cudaSuccess;
  topk_rows_kernel<<<dim3(rows, 2), kThreads, 0, st>>>(n, job0, job1);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
