// Warp-level bf16 tensor-core helpers (mma.sync m16n8k16) shared by the
// kernels that multiply a 64-row query block with 64-key tiles: the
// vertical-slash estimate and the KV-selection score.  Tiles are [rows][128]
// bf16 in shared memory with a 128-byte XOR swizzle (16-byte chunk c of row r
// sits at chunk c ^ (r & 7)), loaded with cp.async.
#pragma once
#include "msa_internal.h"
#include "sm103_ptx.cuh"

namespace msa {
namespace mma16 {

constexpr int kThreads = 128;  // 4 warps x 16 query rows
constexpr int kKeyTile = 64;   // keys per MMA tile

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 256 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Loads rows [r0, r0 + rows) of a [n_rows, 128] bf16 matrix into a swizzled
// smem tile; rows outside [0, n_rows) are zero-filled.
__device__ __forceinline__ void load_rows(uint32_t smem, const __nv_bfloat16* base, int64_t sn,
                                          int r0, int rows, int n_rows) {
  for (int idx = threadIdx.x; idx < rows * 16; idx += blockDim.x) {
    const int r = idx >> 4, c = idx & 15;
    const int gr = r0 + r;
    const bool ok = gr >= 0 && gr < n_rows;
    cp_async16(smem + swz(r, c), base + static_cast<int64_t>(ok ? gr : 0) * sn + c * 8, ok);
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Q fragments of this warp's 16 estimate rows, all 8 k-steps.
// A fragments of query rows 16 g .. 16 g + 15 (row group g) for all 128 dims.
__device__ __forceinline__ void load_q_frags(uint32_t q_smem, uint32_t (&qa)[8][4], int g) {
  const int lane = threadIdx.x & 31;
  const int row = g * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    ldsm_x4(q_smem + swz(row, 2 * kk + (lane >> 4)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
}
// Row group = warp index (kThreads = 4 warps x 16 rows).
__device__ __forceinline__ void load_q_frags(uint32_t q_smem, uint32_t (&qa)[8][4]) {
  load_q_frags(q_smem, qa, static_cast<int>(threadIdx.x >> 5));
}

// acc[nt][*] = this warp's 16 rows x 64 keys of Q K^T (raw dot products).
__device__ __forceinline__ void tile_logits(const uint32_t (&qa)[8][4], uint32_t k_smem,
                                            float (&acc)[8][4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(k_smem + swz(key, 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
      mma_bf16(acc[2 * np], qa[kk], b0, b1);
      mma_bf16(acc[2 * np + 1], qa[kk], b2, b3);
    }
  }
}

}  // namespace mma16
}  // namespace msa
