// Block-sparse index (MInference 1.0 overview, section 2.2, "Block-Sparse
// Head"): mean-pool Q and K over 64-token blocks, score the pooled blocks, and
// keep per row block its own block plus the best earlier ones.
//
// Scores scale * Qhat_m . Khat_n are ranked directly: the page's block weights
// are a row softmax of these scores, which is monotone per row and so keeps the
// same set.  Ties go to the lower block.  Selection is an 8-bit radix select
// over the row's scores in shared memory followed by an order-preserving
// compaction, so the kept blocks come out ascending.  Everything is fp32 and
// deterministic (fixed reduction trees, no atomics on values).
#include "block_scan.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kPoolWarps = 4;
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

struct PoolArgs {
  UnitMap u;
  int NB, N, G;
  const __nv_bfloat16* x;
  int64_t sb, sh, sn;
  int n_heads_x;     // heads of x per batch entry (pool of every head when u is unused)
  bool use_units;    // true: pool unit heads of q; false: pool every head of k
  float* out;        // [rows of (b, head)][NB][128]
};

// One warp per (head, block): lane c holds dims 4c..4c+3.
__global__ void bs_pool_kernel(const __grid_constant__ PoolArgs a) {
  const int m = blockIdx.x * kPoolWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= a.NB) return;
  const int row = blockIdx.y;
  int b, h;
  if (a.use_units) {
    b = row / a.u.n_heads;
    h = a.u.heads[row % a.u.n_heads];
  } else {
    b = row / a.n_heads_x;
    h = row % a.n_heads_x;
  }
  const __nv_bfloat16* base = a.x + b * a.sb + h * a.sh;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int r_end = min(64 * m + 64, a.N);
  for (int r = 64 * m; r < r_end; ++r) {
    const uint2 raw = reinterpret_cast<const uint2*>(base + static_cast<int64_t>(r) * a.sn)[lane];
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    acc[0] += __low2float(lo);
    acc[1] += __high2float(lo);
    acc[2] += __low2float(hi);
    acc[3] += __high2float(hi);
  }
  const float inv = 1.f / static_cast<float>(r_end - 64 * m);
  float4 o = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
  reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(row) * a.NB + m) * kHeadDim)[lane] = o;
}

struct SelArgs {
  UnitMap u;
  int NB, G, Hkv, topk;
  float scale;
  const float* qpool;  // [units][NB][128]
  const float* kpool;  // [B*Hkv][NB][128]
  int32_t* block_count;  // [units][NB]
  int32_t* block_ids;    // [units][NB][kb]
  int kb;
};

// One CTA per (row block m, unit): scores of blocks n < m, then selection.
__global__ void __launch_bounds__(kSelThreads) bs_select_kernel(const __grid_constant__ SelArgs a) {
  extern __shared__ float sc[];  // [m] scores
  __shared__ int hist[kSelWarps][256];
  __shared__ int total_hist[256];
  __shared__ int warp_sums[kSelWarps + 1];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need;
  const int m = blockIdx.x, unit = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = unit / a.u.n_heads;
  const int hkv = a.u.heads[unit % a.u.n_heads] / a.G;
  int32_t* ids = a.block_ids + (static_cast<int64_t>(unit) * a.NB + m) * a.kb;
  const int k_earlier = min(a.topk - 1, m);  // earlier blocks to keep
  if (tid == 0) a.block_count[static_cast<int64_t>(unit) * a.NB + m] = k_earlier + 1;
  if (k_earlier == m) {  // every earlier block is kept
    for (int n = tid; n <= m; n += kSelThreads) ids[n] = n;
    return;
  }
  const float4 qv =
      reinterpret_cast<const float4*>(a.qpool + (static_cast<int64_t>(unit) * a.NB + m) * kHeadDim)[lane];
  const float* kp = a.kpool + static_cast<int64_t>(b * a.Hkv + hkv) * a.NB * kHeadDim;
  for (int n = warp; n < m; n += kSelWarps) {
    const float4 kv = reinterpret_cast<const float4*>(kp + static_cast<int64_t>(n) * kHeadDim)[lane];
    float d = qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) sc[n] = d * a.scale;
  }
  if (tid == 0) {
    s_prefix = 0u;
    s_mask = 0u;
    s_need = k_earlier;
  }
  __syncthreads();
  if (k_earlier > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < kSelWarps * 256; i += kSelThreads) (&hist[0][0])[i] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix, mask = s_mask;
      for (int n = tid; n < m; n += kSelThreads) {
        const uint32_t key = ordered_key(sc[n]);
        if ((key & mask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1);
      }
      __syncthreads();
      {
        int c = 0;
        for (int w = 0; w < kSelWarps; ++w) c += hist[w][tid];
        total_hist[tid] = c;
      }
      __syncthreads();
      if (tid == 0) {
        int need = s_need, above = 0, bucket = 0;
        for (int bb = 255; bb >= 0; --bb) {
          if (above + total_hist[bb] >= need) {
            bucket = bb;
            break;
          }
          above += total_hist[bb];
        }
        s_need = need - above;
        s_prefix = prefix | (static_cast<uint32_t>(bucket) << shift);
        s_mask = mask | (255u << shift);
      }
      __syncthreads();
    }
  }
  const uint32_t T = s_prefix;
  const int take_equal = s_need;
  int kept_before = 0, equal_before = 0;
  if (k_earlier > 0) {
    for (int base = 0; base < m; base += kSelThreads) {
      const int n = base + tid;
      const uint32_t key = n < m ? ordered_key(sc[n]) : 0u;
      const bool eq = n < m && key == T;
      int eq_total;
      const int eq_rank = equal_before + block_exclusive_scan<kSelThreads>(eq ? 1 : 0, warp_sums, &eq_total);
      const bool keep = n < m && (key > T || (eq && eq_rank < take_equal));
      int keep_total;
      const int pos = kept_before + block_exclusive_scan<kSelThreads>(keep ? 1 : 0, warp_sums, &keep_total);
      if (keep) ids[pos] = n;
      kept_before += keep_total;
      equal_before += eq_total;
    }
  }
  if (tid == 0) ids[k_earlier] = m;  // the diagonal block, largest id
}

struct TileArgs {
  int NB, npair, kb, tile_cap, n_units;
  const int32_t* block_count;
  const int32_t* block_ids;
  int32_t* tiles;       // [units][npair][tile_cap] (q << 8) | maskB << 4 | maskA
  int32_t* tile_count;  // [units][npair]
};

// One thread per (unit, pair c of 128-row query tiles): merge the ascending
// block lists of row blocks 4c .. 4c+3 into 128-key tiles with one 4-bit
// quadrant mask per query tile (bit a*2 + b: row half a sees key half b).
__global__ void bs_tiles_kernel(TileArgs a) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= static_cast<int64_t>(a.n_units) * a.npair) return;
  const int unit = static_cast<int>(gid / a.npair), c = static_cast<int>(gid % a.npair);
  const int32_t* lists[4];
  int cnt[4], pos[4] = {0, 0, 0, 0};
  for (int j = 0; j < 4; ++j) {
    const int m = 4 * c + j;
    lists[j] = a.block_ids + (static_cast<int64_t>(unit) * a.NB + m) * a.kb;
    cnt[j] = m < a.NB ? a.block_count[static_cast<int64_t>(unit) * a.NB + m] : 0;
  }
  int32_t* out = a.tiles + gid * a.tile_cap;
  int n = 0, cur_q = -1, cur_mask = 0;
  for (;;) {
    int best = -1, blk = 0;
    for (int j = 0; j < 4; ++j)
      if (pos[j] < cnt[j] && (best < 0 || lists[j][pos[j]] < blk)) {
        best = j;
        blk = lists[j][pos[j]];
      }
    if (best < 0) break;
    ++pos[best];
    const int q = blk >> 1;
    const int bit = (best >> 1) * 4 + (best & 1) * 2 + (blk & 1);  // tile, row half, key half
    if (q != cur_q) {
      if (cur_q >= 0) out[n++] = (cur_q << 8) | cur_mask;
      cur_q = q;
      cur_mask = 0;
    }
    cur_mask |= 1 << bit;
  }
  if (cur_q >= 0) out[n++] = (cur_q << 8) | cur_mask;
  a.tile_count[gid] = n;
}

}  // namespace

cudaError_t launch_bs_index(const Geometry& g, const UnitMap& u, TensorView q, TensorView k,
                            int topk, float* qpool, float* kpool, int32_t* block_count,
                            int32_t* block_ids, int32_t* tiles, int32_t* tile_count,
                            int tile_cap, cudaStream_t st, int* n_launch) {
  cudaError_t e;
  PoolArgs pa;
  pa.u = u;
  pa.NB = g.NB;
  pa.N = g.N;
  pa.G = g.G;
  pa.x = q.data; pa.sb = q.sb; pa.sh = q.sh; pa.sn = q.sn;
  pa.n_heads_x = g.Hq;
  pa.use_units = true;
  pa.out = qpool;
  bs_pool_kernel<<<dim3((g.NB + kPoolWarps - 1) / kPoolWarps, g.n_units), 32 * kPoolWarps, 0, st>>>(pa);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  pa.x = k.data; pa.sb = k.sb; pa.sh = k.sh; pa.sn = k.sn;
  pa.n_heads_x = g.Hkv;
  pa.use_units = false;
  pa.out = kpool;
  bs_pool_kernel<<<dim3((g.NB + kPoolWarps - 1) / kPoolWarps, g.B * g.Hkv), 32 * kPoolWarps, 0, st>>>(pa);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  SelArgs sa;
  sa.u = u;
  sa.NB = g.NB;
  sa.G = g.G;
  sa.Hkv = g.Hkv;
  sa.topk = topk;
  sa.scale = g.scale;
  sa.qpool = qpool;
  sa.kpool = kpool;
  sa.block_count = block_count;
  sa.block_ids = block_ids;
  sa.kb = min(topk, g.NB);
  const int smem = g.NB * 4;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(bs_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  bs_select_kernel<<<dim3(g.NB, g.n_units), kSelThreads, smem, st>>>(sa);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  TileArgs ta;
  ta.NB = g.NB;
  ta.npair = (g.NQ + 1) / 2;
  ta.kb = sa.kb;
  ta.tile_cap = tile_cap;
  ta.n_units = g.n_units;
  ta.block_count = block_count;
  ta.block_ids = block_ids;
  ta.tiles = tiles;
  ta.tile_count = tile_count;
  const int64_t threads = static_cast<int64_t>(g.n_units) * ta.npair;
  bs_tiles_kernel<<<static_cast<unsigned>((threads + 127) / 128), 128, 0, st>>>(ta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  return cudaSuccess;
}

}  // namespace msa
