// Vertical-slash sparse format (MInference 1.0 overview, section 2.2,
// "Vertical-Slash Head": convert the chosen vertical and slash lines to a
// sparse format for block-sparse computation).
//
// The format is kept compact instead of listing tiles per row block:
//  * tile_dist: bit t is set iff some chosen offset o has floor(o/64) == t, or
//    floor(o/64) + 1 == t with o % 64 != 0.  For row block m, key tile n <= m is
//    active iff bit m - n is set: the diagonal at offset o = 64a + b (b > 0)
//    through rows [64m, 64m+63] lands on keys [64(m-a) - b, 64(m-a) + 63 - b],
//    which meets tiles m-a and m-a-1 (only m-a when b == 0).  The set is the
//    same for every row block.
//  * qdelta: for the attention CTAs, which each serve two adjacent 128-row
//    query tiles pA and pB = pA + 1, the ascending distances D = pB - q to the
//    128-key tiles q that hold an active 64x64 quadrant for either query tile.
//    A 128x128 tile at query-tile distance E holds quadrant distances 2E-1, 2E
//    and 2E+1; query tile pB sees key tile q at E = D and pA at E = D - 1.
//    Entries are (D << 5) | bits 2D-3 .. 2D+1 of tile_dist, the bits that the
//    quadrant masks of both query tiles read.
//  * e2: for the one-tile kernel (used when the tiles are sparse), the
//    ascending distances d in [-1, NB] with d or d + 1 active: query tile p
//    (row blocks 2p, 2p + 1) sees 64-key block 2p - d at distances d and d + 1.
//  * col_chunks: per 128-row query tile p, bit c is set iff some chosen key in
//    positions [128c, 128c+128) of the ascending vertical list is needed as a
//    column by row block 2p or 2p+1, i.e. lies at or before the block's last
//    row and outside the block's active tiles.
//  * kc / vc: the K rows and the f16 V rows (from the f16 copy of v, so with
//    the head's scale) of the chosen vertical keys, gathered into a
//    contiguous per-unit buffer so column chunks load like ordinary tiles.
#include "block_scan.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kTilesThreads = 512;

__global__ void __launch_bounds__(kTilesThreads) vs_tile_dist_kernel(
    const int32_t* __restrict__ slash, int ks, int N, int NB, int NQ, uint32_t* __restrict__ tile_dist,
    int dist_words, int32_t* __restrict__ qdelta, int32_t* __restrict__ qdelta_count,
    int32_t* __restrict__ e2, int32_t* __restrict__ e2_count, uint32_t* status) {
  extern __shared__ uint32_t bits[];
  __shared__ int warp_sums[kTilesThreads / 32 + 1];
  const int unit = blockIdx.x, tid = threadIdx.x;
  for (int w = tid; w < dist_words; w += kTilesThreads) bits[w] = 0u;
  __syncthreads();
  const int32_t* S = slash + static_cast<int64_t>(unit) * ks;
  for (int s = tid; s < ks; s += kTilesThreads) {
    const int o = MSA_IDX(S[s], 0, N, status);  // t + 1 <= NB < 32 * dist_words
    const int t = o >> 6;
    atomicOr(&bits[t >> 5], 1u << (t & 31));
    if (o & 63) atomicOr(&bits[(t + 1) >> 5], 1u << ((t + 1) & 31));
  }
  __syncthreads();
  uint32_t* dst = tile_dist + static_cast<int64_t>(unit) * dist_words;
  for (int w = tid; w < dist_words; w += kTilesThreads) dst[w] = bits[w];
  auto bit = [&](int t) -> bool { return t >= 0 && t <= NB && ((bits[t >> 5] >> (t & 31)) & 1u); };
  auto tile_active = [&](int e) -> bool { return e >= 0 && (bit(2 * e) || bit(2 * e + 1) || bit(2 * e - 1)); };
  int32_t* qd = qdelta + static_cast<int64_t>(unit) * (NQ + 1);
  int written = 0;
  for (int base = 0; base <= NQ; base += kTilesThreads) {
    const int d = base + tid;
    const bool act = d <= NQ && (tile_active(d) || tile_active(d - 1));
    int total;
    const int pos = block_exclusive_scan<kTilesThreads>(act ? 1 : 0, warp_sums, &total);
    uint32_t near = 0;  // tile-distance bits 2d-3 .. 2d+1: all the quadrant masks need
    for (int k = 0; k < 5; ++k) near |= (bit(2 * d - 3 + k) ? 1u : 0u) << k;
    if (act) qd[MSA_IDX(written + pos, 0, NQ + 1, status)] = (d << 5) | static_cast<int>(near);
    written += total;
  }
  if (tid == 0) qdelta_count[unit] = written;
  // e2: distances d in [-1, NB] for the one-tile kernel's query tiles (row
  // blocks 2p and 2p + 1 see block 2p - d at distances d and d + 1)
  int32_t* ed = e2 + static_cast<int64_t>(unit) * (NB + 2);
  written = 0;
  for (int base = -1; base <= NB; base += kTilesThreads) {
    const int d = base + tid;
    const int flags = d <= NB ? (bit(d) ? 1 : 0) | (bit(d + 1) ? 2 : 0) : 0;
    int total;
    const int pos = block_exclusive_scan<kTilesThreads>(flags ? 1 : 0, warp_sums, &total);
    if (flags) ed[MSA_IDX(written + pos, 0, NB + 2, status)] = ((d + 1) << 2) | flags;
    written += total;
  }
  if (tid == 0) e2_count[unit] = written;
}

// One warp per (unit, query tile p, 32-chunk word).
__global__ void vs_col_chunks_kernel(const int32_t* __restrict__ vertical, int kv, int N, int NB,
                                     int NQ, const uint32_t* __restrict__ tile_dist, int dist_words,
                                     uint32_t* __restrict__ col_chunks, int chunk_words,
                                     int n_units, uint32_t* status) {
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t per_unit = static_cast<int64_t>(NQ) * chunk_words;
  if (gw >= per_unit * n_units) return;
  const int unit = static_cast<int>(gw / per_unit);
  const int rem = static_cast<int>(gw % per_unit);
  const int p = rem / chunk_words, w = rem % chunk_words;
  const int n_chunks = (kv + 127) / 128;
  const int c = 32 * w + lane;
  const int32_t* V = vertical + static_cast<int64_t>(unit) * kv;
  const uint32_t* dist = tile_dist + static_cast<int64_t>(unit) * dist_words;
  bool need = false;
  if (c < n_chunks) {
    const int s_end = min(128 * c + 128, kv);
    const int last_row = min(64 * (2 * p + 1) + 63, 64 * NB - 1);
    for (int s = 128 * c; s < s_end && !need; ++s) {
      const int j = MSA_IDX(V[s], 0, N, status);
      if (j > last_row) break;  // ascending: later keys are after the tile too
      for (int a = 0; a < 2; ++a) {
        const int m = 2 * p + a;
        if (m >= NB || j > 64 * m + 63) continue;
        const int t = m - (j >> 6);
        if (!((dist[t >> 5] >> (t & 31)) & 1u)) need = true;
      }
    }
  }
  const uint32_t word = __ballot_sync(0xffffffffu, need);
  if (lane == 0) col_chunks[(static_cast<int64_t>(unit) * NQ + p) * chunk_words + w] = word;
}

struct GatherArgs {
  UnitMap u;
  int G, Hkv, N, kv, kv_pad;
  const __nv_bfloat16* k;
  int64_t k_sb, k_sh, k_sn;
  const __half* v16;  // [B][Hkv][N][128], the (scaled) f16 copy of v
  const int32_t* vertical;
  __nv_bfloat16* kc;
  __half* vc;
  uint32_t* status;
};

// One warp per gathered row; rows past kv are zero.  K rows stay bf16; V rows
// come from the f16 copy of v that the tiles read, so columns and tiles share
// the head's scale.
__global__ void vs_gather_kernel(const __grid_constant__ GatherArgs a) {
  const int unit = blockIdx.y;
  const int s = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (s >= a.kv_pad) return;
  const int b = unit / a.u.n_heads;
  const int hkv = a.u.heads[unit % a.u.n_heads] / a.G;
  uint2 kx = make_uint2(0u, 0u), vx = make_uint2(0u, 0u);
  if (s < a.kv) {
    const int j = MSA_IDX(a.vertical[static_cast<int64_t>(unit) * a.kv + s], 0, a.N, a.status);
    kx = reinterpret_cast<const uint2*>(a.k + b * a.k_sb + hkv * a.k_sh + j * a.k_sn)[lane];
    const int64_t vrow = (static_cast<int64_t>(b) * a.Hkv + hkv) * a.N + j;
    vx = reinterpret_cast<const uint2*>(a.v16 + vrow * kHeadDim)[lane];
  }
  const int64_t row = static_cast<int64_t>(unit) * a.kv_pad + s;
  reinterpret_cast<uint2*>(a.kc + row * kHeadDim)[lane] = kx;
  reinterpret_cast<uint2*>(a.vc + row * kHeadDim)[lane] = vx;
}

// Export only (the per-row-block column counts of the format): one warp per
// (unit, row block m) counts the chosen keys j <= 64m + 63 whose tile
// distance m - j/64 is not active.  The list is ascending, so the warp stops
// at the first key past the block.
__global__ void vs_col_count_kernel(const int32_t* __restrict__ vertical, int kv, int N, int NB,
                                    const uint32_t* __restrict__ tile_dist, int dist_words,
                                    int32_t* __restrict__ col_count, int n_units,
                                    uint32_t* status) {
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= static_cast<int64_t>(n_units) * NB) return;
  const int unit = static_cast<int>(gw / NB), m = static_cast<int>(gw % NB);
  const int32_t* V = vertical + static_cast<int64_t>(unit) * kv;
  const uint32_t* dist = tile_dist + static_cast<int64_t>(unit) * dist_words;
  const int last_row = 64 * m + 63;
  int cnt = 0;
  for (int s0 = 0; s0 < kv; s0 += 32) {
    const int s = s0 + lane;
    bool col = false, past = false;
    if (s < kv) {
      const int j = MSA_IDX(V[s], 0, N, status);
      if (j > last_row) {
        past = true;
      } else {
        const int t = m - (j >> 6);
        col = !((dist[t >> 5] >> (t & 31)) & 1u);
      }
    }
    cnt += __popc(__ballot_sync(0xffffffffu, col));
    if (__any_sync(0xffffffffu, past)) break;
  }
  if (lane == 0) col_count[gw] = cnt;
}

}  // namespace

cudaError_t launch_vs_col_count(const Geometry& g, const int32_t* vertical, int kv,
                                const uint32_t* tile_dist, int dist_words, int32_t* col_count,
                                uint32_t* status, cudaStream_t st, int* n_launch) {
  const int64_t warps = static_cast<int64_t>(g.n_units) * g.NB;
  if (warps == 0) return cudaSuccess;
  vs_col_count_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(
      vertical, kv, g.N, g.NB, tile_dist, dist_words, col_count, g.n_units, status);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

cudaError_t launch_vs_index(const Geometry& g, const UnitMap& u, TensorView k, const __half* v16,
                            const int32_t* slash, int ks, const int32_t* vertical, int kv,
                            uint32_t* tile_dist, int dist_words, int32_t* qdelta,
                            int32_t* qdelta_count, int32_t* e2, int32_t* e2_count,
                            uint32_t* col_chunks, int chunk_words,
                            __nv_bfloat16* kc, __half* vc, int kv_pad, uint32_t* status,
                            cudaStream_t st, int* n_launch) {
  cudaError_t e;
  const int smem = dist_words * 4;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(vs_tile_dist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  vs_tile_dist_kernel<<<g.n_units, kTilesThreads, smem, st>>>(slash, ks, g.N, g.NB, g.NQ, tile_dist,
                                                             dist_words, qdelta, qdelta_count,
                                                             e2, e2_count, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  const int64_t warps = static_cast<int64_t>(g.n_units) * g.NQ * chunk_words;
  const int64_t blocks = (warps * 32 + 255) / 256;
  vs_col_chunks_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      vertical, kv, g.N, g.NB, g.NQ, tile_dist, dist_words, col_chunks, chunk_words, g.n_units,
      status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  GatherArgs a;
  a.u = u;
  a.G = g.G;
  a.Hkv = g.Hkv;
  a.N = g.N;
  a.kv = kv;
  a.kv_pad = kv_pad;
  a.k = k.data; a.k_sb = k.sb; a.k_sh = k.sh; a.k_sn = k.sn;
  a.v16 = v16;
  a.vertical = vertical;
  a.kc = kc;
  a.vc = vc;
  a.status = status;
  vs_gather_kernel<<<dim3((kv_pad + 7) / 8, g.n_units), 256, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  return cudaSuccess;
}

}  // namespace msa
