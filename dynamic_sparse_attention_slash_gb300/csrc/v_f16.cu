// The f16 copy of v that the sparse prefill kernels read for the P.V product.
#include "msa_internal.h"
#include "sm103_ptx.cuh"

namespace msa {
namespace {

// v (bf16, any strides, [B][Hkv][N][128]) -> dst (f16, contiguous, same shape),
// for the KV heads in kv only: those a call's query heads read.
// The P.V product runs in f16 (P rounded to f16 keeps 3 more mantissa bits than
// bf16); every bf16 value of magnitude <= 65504 is exactly representable in
// f16 (tiny values become f16 subnormals, error < 3e-8).  Larger magnitudes
// set the range bit of the status word.
__global__ void v_to_f16_kernel(const __nv_bfloat16* __restrict__ v, int64_t sb, int64_t sh,
                                int64_t sn, int Hkv, const __grid_constant__ KvHeads kv, int N,
                                int64_t rows, __half* __restrict__ dst, uint32_t* status) {
  const int64_t n16 = rows * 16;
  bool bad = false;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n16;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = idx >> 4;  // row among the converted heads
    const int cc = static_cast<int>(idx & 15);
    const int64_t bh = r / N;
    const int n = static_cast<int>(r % N);
    const int b = static_cast<int>(bh / kv.n), h = kv.h[bh % kv.n];
    const int64_t row = (static_cast<int64_t>(b) * Hkv + h) * N + n;
    const uint4 raw = *reinterpret_cast<const uint4*>(v + b * sb + h * sh + n * sn + cc * 8);
    const __nv_bfloat162* in = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __low2float(in[e]), hi = __high2float(in[e]);
      bad |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
      ow[e] = pack_f16x2(lo, hi);
    }
    *reinterpret_cast<uint4*>(dst + row * kHeadDim + cc * 8) = o;
  }
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0 && status)
    atomicOr(status, kStatusRange);
}

}  // namespace

cudaError_t launch_v_to_f16(TensorView v, const Geometry& g, const UnitMap& u, __half* dst,
                            uint32_t* status, cudaStream_t st, int* n_launch) {
  const KvHeads kv = kv_heads_of(g.Hkv, g.G, u);
  if (kv.n == 0) return cudaSuccess;
  const int64_t rows = static_cast<int64_t>(g.B) * kv.n * g.N;
  int64_t blocks = (rows * 16 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  v_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      v.data, v.sb, v.sh, v.sn, g.Hkv, kv, g.N, rows, dst, status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
