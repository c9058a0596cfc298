// The f16 copy of v that the sparse prefill kernels read for the P.V product.
//
// The P.V product runs in f16 (P rounded to f16 keeps 3 more mantissa bits than
// bf16).  Every bf16 value of magnitude <= 65504 is exactly representable in
// f16 (tiny values become f16 subnormals, error < 3e-8), so the copy is exact
// for a KV head whose values all fit.  A head with a larger value is copied
// scaled by 2^-e, e the smallest exponent that brings its largest magnitude
// into range (v_scale_exp); the attention kernels multiply that head's output
// by 2^e, which undoes the scaling exactly (powers of two scale every product
// and sum exactly).  The conversion runs optimistically with e = 0 while it
// takes each head's largest magnitude; a second kernel re-converts only the
// heads that need a scale and exits at once for the others.
#include "msa_internal.h"
#include "sm103_ptx.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;

struct ConvArgs {
  const __nv_bfloat16* v;
  int64_t sb, sh, sn;
  int Hkv, N;
  KvHeads kv;        // the KV heads converted (those the call's query heads read)
  int64_t rows_per_cta;
  __half* dst;       // [B][Hkv][N][128]
  uint32_t* vmax;    // [B][Hkv] largest |v| per head, as float bits (zeroed before)
};

__device__ __forceinline__ void head_of(const ConvArgs& a, int y, int& b, int& h) {
  b = y / a.kv.n;
  h = a.kv.h[y % a.kv.n];
}

// Rows [r0, r1) of one head (16 threads per 128-value row), scaled by s.
__device__ __forceinline__ float convert_rows(const ConvArgs& a, int b, int h, int64_t r0,
                                              int64_t r1, float s) {
  float mx = 0.f;
  const int64_t base = (static_cast<int64_t>(b) * a.Hkv + h) * a.N;
  for (int64_t idx = r0 * 16 + threadIdx.x; idx < r1 * 16; idx += kThreads) {
    const int64_t n = idx >> 4;
    const int cc = static_cast<int>(idx & 15);
    const uint4 raw = *reinterpret_cast<const uint4*>(a.v + b * a.sb + h * a.sh + n * a.sn + cc * 8);
    const __nv_bfloat162* in = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __low2float(in[e]), hi = __high2float(in[e]);
      mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
      ow[e] = pack_f16x2(lo * s, hi * s);
    }
    *reinterpret_cast<uint4*>(a.dst + (base + n) * kHeadDim + cc * 8) = o;
  }
  return mx;
}

// grid (slices, converted heads): copy with e = 0 and record the largest |v|.
__global__ void __launch_bounds__(kThreads) v_to_f16_kernel(const __grid_constant__ ConvArgs a) {
  __shared__ float warp_max[kThreads / 32];
  int b, h;
  head_of(a, blockIdx.y, b, h);
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
  const int64_t r1 = min(r0 + a.rows_per_cta, static_cast<int64_t>(a.N));
  float mx = convert_rows(a, b, h, r0, r1, 1.f);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
    // non-negative floats order like their bit patterns
    atomicMax(a.vmax + static_cast<int64_t>(b) * a.Hkv + h, __float_as_uint(m));
  }
}

// grid as above: heads whose largest |v| exceeds the f16 range are converted
// again with the scale 2^-e; every other CTA returns at once.
__global__ void __launch_bounds__(kThreads) v_rescale_kernel(const __grid_constant__ ConvArgs a) {
  int b, h;
  head_of(a, blockIdx.y, b, h);
  const int e = v_scale_exp(__uint_as_float(a.vmax[static_cast<int64_t>(b) * a.Hkv + h]));
  if (e == 0) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
  const int64_t r1 = min(r0 + a.rows_per_cta, static_cast<int64_t>(a.N));
  convert_rows(a, b, h, r0, r1, ldexpf(1.f, -e));
}

}  // namespace

cudaError_t launch_v_to_f16(TensorView v, const Geometry& g, const UnitMap& u, __half* dst,
                            uint32_t* vmax, cudaStream_t st, int* n_launch) {
  ConvArgs a;
  a.kv = kv_heads_of(g.Hkv, g.G, u);
  if (a.kv.n == 0) return cudaSuccess;
  a.v = v.data; a.sb = v.sb; a.sh = v.sh; a.sn = v.sn;
  a.Hkv = g.Hkv;
  a.N = g.N;
  a.dst = dst;
  a.vmax = vmax;
  const int heads = g.B * a.kv.n;
  // about 8 CTAs per SM over all heads, at least 64 rows each
  int64_t slices = (152 * 8 + heads - 1) / heads;
  if (slices > (g.N + 63) / 64) slices = (g.N + 63) / 64;
  if (slices < 1) slices = 1;
  a.rows_per_cta = (g.N + slices - 1) / slices;
  const dim3 grid(static_cast<unsigned>((g.N + a.rows_per_cta - 1) / a.rows_per_cta),
                  static_cast<unsigned>(heads));
  v_to_f16_kernel<<<grid, kThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*n_launch;
  v_rescale_kernel<<<grid, kThreads, 0, st>>>(a);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

}  // namespace msa
