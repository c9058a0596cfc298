// Internal interfaces between the host-side C ABI (msa_api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/msa.h"

namespace msa {

constexpr int kHeadDim = 128;
constexpr int kBlock = 64;     // token block of the sparse formats
constexpr int kTileM = 128;    // query rows per attention CTA (two row blocks)
constexpr int kTileN = 128;    // keys per attention tile (two key blocks)
constexpr int kLastQMax = 64;  // estimate rows handled by one estimate CTA
constexpr int kMaxUnits = 65535;

// Device status word bits (first word of every workspace).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBounds = 2u;  // bounds-checking build: an index read was out of range

// Bounds checks of the indices the kernels read from index data (the
// bounds-checking build, compiled with MSA_CHECKED).  An index outside
// [lo, hi) sets kStatusBounds in the status word and is replaced by lo, so the
// access stays inside its buffer (the result is then wrong, and the status
// says so); there is no trap.  A count above cap is reported and cut to cap.
// In the ordinary build both are the plain value.
#ifdef MSA_CHECKED
__device__ __forceinline__ int checked_index(int i, int lo, int hi, uint32_t* status) {
  if (i >= lo && i < hi) return i;
  if (status) atomicOr(status, kStatusBounds);
  return lo;
}
__device__ __forceinline__ int checked_count(int c, int cap, uint32_t* status) {
  if (c >= 0 && c <= cap) return c;
  if (status) atomicOr(status, kStatusBounds);
  return c < 0 ? 0 : cap;
}
#define MSA_IDX(i, lo, hi, status) ::msa::checked_index((i), (lo), (hi), (status))
#define MSA_COUNT(c, cap, status) ::msa::checked_count((c), (cap), (status))
#else
#define MSA_IDX(i, lo, hi, status) (i)
#define MSA_COUNT(c, cap, status) (c)
#endif

// Exponent e >= 0 of the power-of-two scale 2^-e that brings a KV head's
// largest |v| (amax) into the f16 range of the P.V product: 0 when amax <=
// 65504, else the smallest e with amax * 2^-e <= 65504 (ldexpf is exact).
__host__ __device__ inline int v_scale_exp(float amax) {
  int e = 0;
  while (e < 200 && ldexpf(amax, -e) > 65504.f) ++e;
  return e;
}

// A selected (batch, query head) pair and the KV head it reads.
struct UnitMap {
  int n_heads;   // selected query heads per batch entry
  int heads[1024];
};

// The KV heads a call's query heads read (h / G over the selected heads),
// ascending, without repeats.
struct KvHeads {
  int n;
  int h[1024];
};

inline KvHeads kv_heads_of(int Hkv, int G, const UnitMap& u) {
  KvHeads kv;
  kv.n = 0;
  for (int x = 0; x < Hkv; ++x) {
    bool used = false;
    for (int i = 0; i < u.n_heads && !used; ++i) used = u.heads[i] / G == x;
    if (used) kv.h[kv.n++] = x;
  }
  return kv;
}

struct TensorView {
  const __nv_bfloat16* data;
  int64_t sb, sh, sn;
};

// Per-call geometry shared by the kernels.
struct Geometry {
  int B, Hq, Hkv, G, N, NB, NQ;  // NB = N/64 row blocks, NQ = ceil(N/128) query tiles
  int n_units;
  float scale;
};

// ---------------------------------------------------------------- prefill
enum PrefillKind : int { kPrefillVS = 0, kPrefillBS = 1, kPrefillST = 2 };

struct PrefillParams {
  Geometry g;
  int kind;
  int npair;         // ceil(NQ / 2): pairs of 128-row query tiles, one CTA each
  float scale_log2;  // scale * log2(e)
  __nv_bfloat16* out;
  int64_t out_sb, out_sh, out_sn;
  // vertical-slash plan (per unit strides)
  const uint32_t* tile_dist;  // [units][dist_words] bit t: tile distance t active
  int dist_words;
  const int32_t* qdelta;       // [units][NQ+1] ascending tile distances used by a query-tile pair
  const int32_t* qdelta_count; // [units]
  const uint32_t* col_chunks;  // [units][NQ][chunk_words] bit c: column chunk c needed
  int chunk_words;
  const int32_t* vertical;     // [units][kv] ascending chosen key columns
  int kv;                      // number of chosen columns
  // vertical-slash on the one-tile kernel: per unit, the ascending distances
  // d in [-1, NB] with d or d + 1 active, as (d + 1) << 2 | (bit 0: d active,
  // bit 1: d + 1 active), and their count
  const int32_t* vs_e2;        // [units][e2_stride]
  const int32_t* vs_e2_count;  // [units]
  int e2_stride;               // NB + 2
  int kv_pad;                  // rows per unit in the gathered K/V buffers (multiple of 128)
  // block-sparse plan
  const int32_t* bs_tiles;       // [units][NQ][bs_tile_cap][2] 64-key block | flags << 16
  const int32_t* bs_tile_count;  // [units][NQ] items per query tile
  int bs_tile_cap;
  // streaming plan
  int init_num, local_num;
  // row normalisers lse_i (natural log) for KV selection: [B][Hq][N] f32, or null
  float* lse;
  // largest |v| per (batch, KV head) as float bits: the output of a head copied
  // with the scale 2^-e (v_scale_exp) is multiplied by 2^e
  const uint32_t* vmax;
  uint32_t* status;
  UnitMap units;
  // grid order: 0 — x enumerates a unit's query tiles (heavy first), y the
  // units, so the CTAs resident at a time read nearby K/V of one KV head; 1 —
  // x enumerates the units, y the tiles (heavy first over every unit), when
  // the K/V the call reads fit L2 and only the balance of the last waves counts
  int units_fast;
};

// Key set J_i of the call's attention, for the KV-selection score: which 64-key
// blocks row block m admits (then the causal cut j <= i), plus vertical columns.
struct KvMask {
  int kind;                    // PrefillKind
  int NB;
  // vertical-slash: tile-distance bitset and the ascending vertical columns
  const uint32_t* tile_dist;   // [units][dist_words]
  int dist_words;
  const int32_t* vertical;     // [units][kv]
  int kv;
  // block-sparse: kept blocks per row block, ascending
  const int32_t* block_count;  // [units][NB]
  const int32_t* block_ids;    // [units][NB][kb]
  int kb;
  // streaming
  int init_num, local_num;
};

// Adds n to the library's kernel-launch counter (msa_kernel_launches).
void note_launches(int n);

// Every host-side check msa_vertical_slash makes on its arguments before it
// looks at the workspace (shapes, strides, overlaps, options, line counts); on
// MSA_OK, *need holds the workspace bytes that call needs.  Enqueues nothing.
int vertical_slash_need(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                        int64_t vertical_topk, int64_t slash, const msa_tensor* out,
                        const msa_opts* opts, size_t* need);

// ---------------------------------------------------------------- launches
cudaError_t launch_vs_estimate(const Geometry& g, const UnitMap& u, TensorView q, TensorView k,
                               int last_q, float* partial, int n_split, float* row_stats,
                               float* v_score, float* s_score, cudaStream_t st, int* n_launch);
// Top-k of `rows` score rows of length n for two row sets at once (one launch,
// one CTA per row of each set).
struct TopkRows {
  const float* scores;
  int64_t row_stride;
  int k;
  int32_t* out;
  int64_t out_stride;
};
cudaError_t launch_topk_pair(int64_t n, int rows, const TopkRows& job0, const TopkRows& job1,
                             cudaStream_t st, int* n_launch);
// Top-k of the rows of the selected units in [B][Hq][n] scores into [B][Hq][min(k, n)].
cudaError_t launch_topk_units(const float* scores, int64_t n, int k, int Hq, const UnitMap& u,
                              int units, int32_t* out_idx, cudaStream_t st, int* n_launch);
// KV-selection score S of the selected units ([B][Hq][N] lse in, score out).
cudaError_t launch_kv_score(const Geometry& g, const UnitMap& u, TensorView q, TensorView k,
                            const float* lse, float* score, int window, const KvMask& mask,
                            cudaStream_t st, int* n_launch);
// The vertical-slash format; the gathered V rows of the columns are copied
// from the f16 copy of v (v16, [B][Hkv][N][128], already scaled).
cudaError_t launch_vs_index(const Geometry& g, const UnitMap& u, TensorView k, const __half* v16,
                            const int32_t* slash, int ks, const int32_t* vertical, int kv,
                            uint32_t* tile_dist, int dist_words, int32_t* qdelta,
                            int32_t* qdelta_count, int32_t* e2, int32_t* e2_count,
                            uint32_t* col_chunks, int chunk_words,
                            __nv_bfloat16* kc, __half* vc, int kv_pad, uint32_t* status,
                            cudaStream_t st, int* n_launch);
// Export only: columns per row block of the vertical-slash format ([units][NB]).
cudaError_t launch_vs_col_count(const Geometry& g, const int32_t* vertical, int kv,
                                const uint32_t* tile_dist, int dist_words, int32_t* col_count,
                                uint32_t* status, cudaStream_t st, int* n_launch);
cudaError_t launch_bs_index(const Geometry& g, const UnitMap& u, TensorView q, TensorView k,
                            int topk, float* qpool, float* kpool, int32_t* block_count,
                            int32_t* block_ids, int32_t* tiles, int32_t* tile_count,
                            int tile_cap, uint32_t* status, cudaStream_t st, int* n_launch);
// Mean of each 64-row block of q for the selected units ([units][NB][128] f32).
cudaError_t launch_pool_q(const Geometry& g, const UnitMap& u, TensorView q, float* qpool,
                          cudaStream_t st, int* n_launch);
// Per-query-tile item lists of the one-tile prefill from kept blocks per row
// block ([units][NB] counts, [units][NB][kb] ascending ids).
cudaError_t launch_bs_tiles(const Geometry& g, int kb, const int32_t* block_count,
                            const int32_t* block_ids, int32_t* tiles, int32_t* tile_count,
                            int tile_cap, uint32_t* status, cudaStream_t st, int* n_launch);
// Hierarchical pruning head: block maxima of the token scores and the stages,
// slab by slab of slab_rows query blocks; writes kept blocks in the
// block-sparse format.  hip_slab_rows gives the slab height for a call.
int hip_slab_rows(int n_units, int NB);
// mk: TMA map of k in 128-key boxes; qsplit: [3][units * NB][128] bf16 scratch
// for the split pooled queries, mqs its 2-D TMA map (128-row boxes).
cudaError_t launch_hip_index(const Geometry& g, const UnitMap& u, const CUtensorMap& mk,
                             const float* qpool, __nv_bfloat16* qsplit,
                             const CUtensorMap& mqs, const int32_t* stage_c,
                             const int32_t* stage_keep, int n_stages, float* rmax, int slab_rows,
                             int32_t* block_count, int32_t* block_ids, int kb, uint32_t* status,
                             cudaStream_t st, int* n_launch);
// The f16 copy of v for the KV heads the call reads, with each head's largest
// |v| in vmax ([B][Hkv] float bits, zeroed before the call) and heads beyond
// the f16 range scaled by 2^-v_scale_exp(vmax).
cudaError_t launch_v_to_f16(TensorView v, const Geometry& g, const UnitMap& u, __half* dst,
                            uint32_t* vmax, cudaStream_t st, int* n_launch);
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const CUtensorMap& mkc, const CUtensorMap& mvc,
                           cudaStream_t st, int* n_launch);
// One query tile per CTA, for block-sparse plans and vertical-slash plans
// (any other kind returns cudaErrorInvalidValue).  mk64 / mv64 map K and the
// f16 copy of v in 64-key boxes; mkc64 / mvc64 the gathered column rows in
// 64-row boxes (vertical-slash only; unused otherwise).
cudaError_t launch_prefill_tile(const PrefillParams& p, const CUtensorMap& mq,
                                const CUtensorMap& mk64, const CUtensorMap& mv64,
                                const CUtensorMap& mkc64, const CUtensorMap& mvc64,
                                cudaStream_t st, int* n_launch);

}  // namespace msa
