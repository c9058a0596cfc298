// Recall of the dense attention that a sparse mask keeps, per head (MInference
// 1.0 overview, section 2.1 "Kernel-Aware Optimal Sparse Pattern Search": the
// search compares candidate patterns by the recall of the attention output).
// For row i the kept mass is sum_{j in J_i} softmax_dense(i)_j
// = exp(lse_M,i - lse_dense,i), with both normalisers exported by the attention
// kernel (msa_kv_select.lse).  One CTA per selected (batch, head) averages it
// over rows [row0, N): each thread sums a fixed strided set of rows in order,
// in double, then a fixed-order tree combines the threads, so the result does
// not depend on scheduling.
#include <cmath>

#include "../../include/msa.h"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) recall_kernel(const float* __restrict__ lse,
                                                          const float* __restrict__ ref, int Hq,
                                                          int N, int row0,
                                                          const __grid_constant__ UnitMap u,
                                                          float* __restrict__ recall) {
  __shared__ double part[kThreads];
  const int unit = blockIdx.x;
  const int64_t row = static_cast<int64_t>(unit / u.n_heads) * Hq + u.heads[unit % u.n_heads];
  const float* a = lse + row * N;
  const float* r = ref + row * N;
  double s = 0.0;
  for (int i = row0 + threadIdx.x; i < N; i += kThreads) {
    const float x = a[i], y = r[i];
    // an empty row keeps nothing; the dense row is never empty (key i <= i)
    if (x != -INFINITY && y != -INFINITY) s += exp(static_cast<double>(x) - static_cast<double>(y));
  }
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = kThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) recall[row] = static_cast<float>(part[0] / (N - row0));
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" int msa_mass_recall(const float* lse, const float* ref_lse, int64_t B, int64_t H,
                               int64_t N, int64_t row0, const int32_t* heads, int32_t n_heads,
                               float* recall, void* stream) {
  if (!lse || !ref_lse || !recall || B <= 0 || H <= 0 || N <= 0 || row0 < 0 || row0 >= N)
    return MSA_ERR_INVALID;
  if (N > (int64_t{1} << 21) || H > MSA_MAX_HEADS) return MSA_ERR_UNSUPPORTED;
  UnitMap u;
  if (heads) {
    if (n_heads <= 0 || n_heads > MSA_MAX_HEADS) return MSA_ERR_INVALID;
    bool seen[MSA_MAX_HEADS] = {};
    for (int i = 0; i < n_heads; ++i) {
      if (heads[i] < 0 || heads[i] >= H || seen[heads[i]]) return MSA_ERR_INVALID;
      seen[heads[i]] = true;
      u.heads[i] = heads[i];
    }
    u.n_heads = n_heads;
  } else {
    for (int i = 0; i < H; ++i) u.heads[i] = i;
    u.n_heads = static_cast<int>(H);
  }
  const int64_t units = B * u.n_heads;
  if (units > kMaxUnits) return MSA_ERR_UNSUPPORTED;
  recall_kernel<<<static_cast<unsigned>(units), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      lse, ref_lse, static_cast<int>(H), static_cast<int>(N), static_cast<int>(row0), u, recall);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  note_launches(1);
  return MSA_OK;
}
