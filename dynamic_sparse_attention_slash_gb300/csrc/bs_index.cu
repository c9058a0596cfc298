// Block-sparse index (MInference 1.0 overview, section 2.2, "Block-Sparse
// Head"): mean-pool Q and K over 64-token blocks, score the pooled blocks, and
// keep per row block its own block plus the best earlier ones.
//
// Scores scale * Qhat_m . Khat_n are ranked directly: the page's block weights
// are a row softmax of these scores, which is monotone per row and so keeps the
// same set.  Ties go to the lower block.  Selection is an 8-bit radix select
// over the row's scores in shared memory followed by an order-preserving
// compaction, so the kept blocks come out ascending.  Everything is fp32 and
// deterministic (fixed reduction trees, no atomics on values).  Last, each
// 128-row query tile gets the prefill's item list: the union of the blocks its
// two row blocks kept, ascending, two blocks to an item.
#include "block_scan.cuh"
#include "msa_internal.h"

namespace msa {
namespace {

constexpr int kPoolWarps = 4;
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
// Selection with shared key chunks: kSelWarps row blocks per CTA score against
// pooled key blocks staged kKeyChunk at a time in shared memory (row stride
// kHeadDim + 4 floats: 16-byte rows whose float4 reads by eight consecutive
// lanes cover all 32 banks); warp w takes keys 32 (w % 4) .. + 31 of a chunk
// (one per lane) against row blocks 4 (w / 4) .. + 3, so each float4 of a key
// is read once for four rows.  Used while the CTA's scores fit:
// NB <= kRowsMaxNB.
constexpr int kKeyChunk = 128;
constexpr int kKStride = kHeadDim + 4;
constexpr int kRowsMaxNB = 4096;
constexpr int kTilesWarps = 4;

struct PoolArgs {
  UnitMap u;
  int NB, N, G;
  const __nv_bfloat16* x;
  int64_t sb, sh, sn;
  int n_heads_x;     // heads of x per batch entry
  KvHeads kv;        // without units: the heads of k to pool in every batch entry
  bool use_units;    // true: pool unit heads of q (out row = unit); false: heads kv of k
                     // (out row = b * n_heads_x + h)
  float* out;        // [rows of (b, head)][NB][128]
};

// One warp per (head, block): lane c holds dims 4c..4c+3.
__global__ void bs_pool_kernel(const __grid_constant__ PoolArgs a) {
  const int m = blockIdx.x * kPoolWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= a.NB) return;
  int row = blockIdx.y;
  int b, h;
  if (a.use_units) {
    b = row / a.u.n_heads;
    h = a.u.heads[row % a.u.n_heads];
  } else {
    b = row / a.kv.n;
    h = a.kv.h[row % a.kv.n];
    row = b * a.n_heads_x + h;
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

// One CTA per kSelWarps consecutive row blocks of a unit: the CTA scores its
// rows against every earlier block (pooled keys staged in shared memory, each
// lane one key against four rows), then warp w runs row block m0 + w's radix
// select and ascending compaction alone, as bs_select_kernel does with a CTA.
__global__ void __launch_bounds__(kSelThreads) bs_select_rows_kernel(const __grid_constant__ SelArgs a) {
  extern __shared__ __align__(16) float dyn[];
  float* sc = dyn;                              // [kSelWarps][NB] scores
  float* kc = sc + kSelWarps * a.NB;            // [kKeyChunk][kKStride] pooled keys
  float* qs = kc + kKeyChunk * kKStride;        // [kSelWarps][kHeadDim] pooled queries
  __shared__ int hist[kSelWarps][256];
  const int unit = blockIdx.y, m0 = blockIdx.x * kSelWarps;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = unit / a.u.n_heads;
  const int hkv = a.u.heads[unit % a.u.n_heads] / a.G;
  const int rows = min(kSelWarps, a.NB - m0);
  for (int i = tid; i < kSelWarps * kHeadDim; i += kSelThreads) {
    const int r = i / kHeadDim;
    qs[i] = r < rows
                ? a.qpool[(static_cast<int64_t>(unit) * a.NB + m0 + r) * kHeadDim + i % kHeadDim]
                : 0.f;
  }
  const float* kp = a.kpool + static_cast<int64_t>(b * a.Hkv + hkv) * a.NB * kHeadDim;
  const int n_end = m0 + rows - 1;  // the CTA's last row block scores keys n < n_end
  const int m = m0 + warp;          // the row block this warp selects for
  const int kg = warp & 3, rg = warp >> 2;  // score phase: key group, row group
  for (int n0 = 0; n0 < n_end; n0 += kKeyChunk) {
    __syncthreads();  // the previous chunk is consumed (and qs is written)
    for (int i = tid; i < kKeyChunk * (kHeadDim / 4); i += kSelThreads) {
      const int j = i / (kHeadDim / 4), c4 = i % (kHeadDim / 4);
      const float4 val = n0 + j < n_end
                             ? reinterpret_cast<const float4*>(kp + static_cast<int64_t>(n0 + j) * kHeadDim)[c4]
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(kc + j * kKStride + 4 * c4) = val;
    }
    __syncthreads();
    const int j = 32 * kg + lane, n = n0 + j;
    const float* kr = kc + j * kKStride;
    const float* q0 = qs + 4 * rg * kHeadDim;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int c = 0; c < kHeadDim; c += 4) {
      const float4 kv = *reinterpret_cast<const float4*>(kr + c);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 qv = *reinterpret_cast<const float4*>(q0 + r * kHeadDim + c);
        d[r] = fmaf(qv.x, kv.x, d[r]);
        d[r] = fmaf(qv.y, kv.y, d[r]);
        d[r] = fmaf(qv.z, kv.z, d[r]);
        d[r] = fmaf(qv.w, kv.w, d[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = 4 * rg + r;
      if (row < rows && n < m0 + row) sc[row * a.NB + n] = d[r] * a.scale;
    }
  }
  __syncthreads();  // every row's scores are written (by other warps)
  if (warp >= rows) return;  // no CTA-wide barrier follows
  __syncwarp();
  int32_t* ids = a.block_ids + (static_cast<int64_t>(unit) * a.NB + m) * a.kb;
  const int k_earlier = min(a.topk - 1, m);  // earlier blocks to keep
  if (lane == 0) a.block_count[static_cast<int64_t>(unit) * a.NB + m] = k_earlier + 1;
  if (k_earlier == m) {  // every earlier block is kept
    for (int n = lane; n <= m; n += 32) ids[n] = n;
    return;
  }
  const float* s = sc + warp * a.NB;
  int* h = hist[warp];
  uint32_t prefix = 0u, mask = 0u;
  int need = k_earlier;
  if (k_earlier > 0) {
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = lane; i < 256; i += 32) h[i] = 0;
      __syncwarp();
      for (int n = lane; n < m; n += 32) {
        const uint32_t key = ordered_key(s[n]);
        if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1);
      }
      __syncwarp();
      // lane l holds bins 255 - 8l down to 248 - 8l; the bucket is the one in
      // which the count from the top reaches `need`
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = h[255 - 8 * lane - j];
        tot += cnt[j];
      }
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const int excl = incl - tot;
      const bool mine = excl < need && incl >= need;
      const int src = __ffs(static_cast<int>(__ballot_sync(0xffffffffu, mine))) - 1;
      int bucket = 0, above = excl;
      if (mine) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + cnt[j] >= need) {
            bucket = 255 - 8 * lane - j;
            break;
          }
          above += cnt[j];
        }
      }
      bucket = __shfl_sync(0xffffffffu, bucket, src);
      above = __shfl_sync(0xffffffffu, above, src);
      need -= above;
      prefix |= static_cast<uint32_t>(bucket) << shift;
      mask |= 255u << shift;
      __syncwarp();  // every lane has read the histogram before it is cleared
    }
    // keys above the threshold, and the first `need` keys equal to it (lower
    // blocks first), in ascending block order
    const uint32_t lt = (1u << lane) - 1u;
    int kept = 0, eq_seen = 0;
    for (int base = 0; base < m; base += 32) {
      const int n = base + lane;
      const uint32_t key = n < m ? ordered_key(s[n]) : 0u;
      const bool eq = n < m && key == prefix;
      const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
      const bool keep = n < m && (key > prefix || (eq && eq_seen + __popc(eqb & lt) < need));
      const uint32_t kb = __ballot_sync(0xffffffffu, keep);
      if (keep) ids[kept + __popc(kb & lt)] = n;
      kept += __popc(kb);
      eq_seen += __popc(eqb);
    }
  }
  if (lane == 0) ids[k_earlier] = m;  // the diagonal block, largest id
}

struct TileArgs {
  int NB, NQ, kb, tile_cap, n_units;
  int words_per_warp;   // shared words per warp: two bitmaps of ceil(NB / 32) words
  const int32_t* block_count;
  const int32_t* block_ids;
  int32_t* tiles;       // [units][NQ][tile_cap][2]: key-block slots, blk | flags << 16
  int32_t* tile_count;  // [units][NQ]
  uint32_t* status;
};

// One warp per (unit, 128-row query tile p): the union U of the blocks kept by
// row blocks 2p and 2p + 1, ascending, packed two blocks to an item.  The kept
// blocks set bits of two bitmaps in shared memory (one per row block); a scan
// over the words of their OR gives each block of U its rank r, and the block
// goes to item r >> 1, key half r & 1, as blk | flags << 16 with flag bit a
// set when row block 2p + a kept it.  An odd |U| leaves the last item's second
// half a copy of its first block with no flags (a valid load that the softmax
// masks out).
__global__ void __launch_bounds__(32 * kTilesWarps) bs_tiles_kernel(TileArgs a) {
  extern __shared__ uint32_t tile_bits[];  // [kTilesWarps][2][words_per_warp / 2]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kTilesWarps + warp;
  if (gid >= static_cast<int64_t>(a.n_units) * a.NQ) return;  // no CTA-wide barrier follows
  const int unit = static_cast<int>(gid / a.NQ), p = static_cast<int>(gid % a.NQ);
  const int nblk = min(2 * p + 2, a.NB);  // blocks <= 2p + 1 within the sequence
  const int words = (nblk + 31) >> 5;
  uint32_t* w0 = tile_bits + warp * a.words_per_warp;
  uint32_t* w1 = w0 + (a.words_per_warp >> 1);
  for (int i = lane; i < words; i += 32) w0[i] = w1[i] = 0u;
  __syncwarp();
  for (int t = 0; t < 2 && 2 * p + t < a.NB; ++t) {
    const int64_t rb = static_cast<int64_t>(unit) * a.NB + 2 * p + t;
    const int cnt = MSA_COUNT(a.block_count[rb], a.kb, a.status);
    const int32_t* L = a.block_ids + rb * a.kb;
    uint32_t* w = t ? w1 : w0;
    for (int i = lane; i < cnt; i += 32) {
      const int blk = MSA_IDX(L[i], 0, nblk, a.status);
      atomicOr(&w[blk >> 5], 1u << (blk & 31));
    }
  }
  __syncwarp();
  int32_t* out = a.tiles + gid * a.tile_cap * 2;
  int n = 0, last = 0;  // blocks of U placed so far; the largest of them
  for (int base = 0; base < words; base += 32) {
    const int i = base + lane;
    const uint32_t b0 = i < words ? w0[i] : 0u, b1 = i < words ? w1[i] : 0u;
    uint32_t u = b0 | b1;
    const int cw = __popc(u);
    int incl = cw;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int r = n + incl - cw;
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      const int flags = static_cast<int>(((b0 >> bit) & 1u) | (((b1 >> bit) & 1u) << 1));
      out[MSA_IDX(r, 0, 2 * a.tile_cap, a.status)] = (32 * i + bit) | (flags << 16);
      ++r;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total > 0) {  // the highest lane with a block holds the largest so far
      const uint32_t has = __ballot_sync(0xffffffffu, cw > 0);
      const int src = 31 - __clz(static_cast<int>(has));
      const int top = cw > 0 ? 32 * i + 31 - __clz(static_cast<int>(b0 | b1)) : 0;
      last = __shfl_sync(0xffffffffu, top, src);
    }
    n += total;
  }
  if (lane == 0) {
    if (n & 1) out[MSA_IDX(n, 0, 2 * a.tile_cap, a.status)] = last;  // second half of the last
                                                                    // item: same block, no flags
    a.tile_count[gid] = (n + 1) >> 1;
  }
}

}  // namespace

cudaError_t launch_pool_q(const Geometry& g, const UnitMap& u, TensorView q, float* qpool,
                          cudaStream_t st, int* n_launch) {
  PoolArgs pa;
  pa.u = u;
  pa.NB = g.NB;
  pa.N = g.N;
  pa.G = g.G;
  pa.x = q.data; pa.sb = q.sb; pa.sh = q.sh; pa.sn = q.sn;
  pa.n_heads_x = g.Hq;
  pa.kv.n = 0;
  pa.use_units = true;
  pa.out = qpool;
  bs_pool_kernel<<<dim3((g.NB + kPoolWarps - 1) / kPoolWarps, g.n_units), 32 * kPoolWarps, 0, st>>>(pa);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*n_launch;
  return e;
}

cudaError_t launch_bs_tiles(const Geometry& g, int kb, const int32_t* block_count,
                            const int32_t* block_ids, int32_t* tiles, int32_t* tile_count,
                            int tile_cap, uint32_t* status, cudaStream_t st, int* n_launch) {
  TileArgs ta;
  ta.NB = g.NB;
  ta.NQ = g.NQ;
  ta.kb = kb;
  ta.tile_cap = tile_cap;
  ta.n_units = g.n_units;
  ta.block_count = block_count;
  ta.block_ids = block_ids;
  ta.tiles = tiles;
  ta.tile_count = tile_count;
  ta.status = status;
  ta.words_per_warp = 2 * ((g.NB + 31) >> 5);
  const int tsmem = kTilesWarps * ta.words_per_warp * 4;
  cudaError_t e;
  if (tsmem > 48 * 1024) {
    e = cudaFuncSetAttribute(bs_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tsmem);
    if (e != cudaSuccess) return e;
  }
  const int64_t warps = static_cast<int64_t>(g.n_units) * g.NQ;
  bs_tiles_kernel<<<static_cast<unsigned>((warps + kTilesWarps - 1) / kTilesWarps),
                    32 * kTilesWarps, tsmem, st>>>(ta);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  return cudaSuccess;
}

cudaError_t launch_bs_index(const Geometry& g, const UnitMap& u, TensorView q, TensorView k,
                            int topk, float* qpool, float* kpool, int32_t* block_count,
                            int32_t* block_ids, int32_t* tiles, int32_t* tile_count,
                            int tile_cap, uint32_t* status, cudaStream_t st, int* n_launch) {
  cudaError_t e = launch_pool_q(g, u, q, qpool, st, n_launch);
  if (e != cudaSuccess) return e;
  PoolArgs pa;
  pa.u = u;
  pa.NB = g.NB;
  pa.N = g.N;
  pa.G = g.G;
  pa.x = k.data; pa.sb = k.sb; pa.sh = k.sh; pa.sn = k.sn;
  pa.n_heads_x = g.Hkv;
  pa.kv = kv_heads_of(g.Hkv, g.G, u);  // the KV heads the selected query heads read
  if (pa.kv.n == 0) return cudaErrorInvalidValue;
  pa.use_units = false;
  pa.out = kpool;
  bs_pool_kernel<<<dim3((g.NB + kPoolWarps - 1) / kPoolWarps, g.B * pa.kv.n), 32 * kPoolWarps, 0,
                   st>>>(pa);
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
  if (g.NB <= kRowsMaxNB) {
    const int smem = (kSelWarps * g.NB + kKeyChunk * kKStride + kSelWarps * kHeadDim) * 4;
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(bs_select_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
      if (e != cudaSuccess) return e;
    }
    bs_select_rows_kernel<<<dim3((g.NB + kSelWarps - 1) / kSelWarps, g.n_units), kSelThreads, smem,
                            st>>>(sa);
  } else {
    const int smem = g.NB * 4;
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(bs_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
    }
    bs_select_kernel<<<dim3(g.NB, g.n_units), kSelThreads, smem, st>>>(sa);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n_launch;
  return launch_bs_tiles(g, sa.kb, block_count, block_ids, tiles, tile_count, tile_cap, status,
                         st, n_launch);
}

}  // namespace msa
