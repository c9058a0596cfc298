// Host side of the C ABI declared in include/msa.h: argument validation,
// workspace layout, TMA descriptor construction and kernel launches.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <utility>

#include <cudaTypedefs.h>

#include "../../include/msa.h"
#include "msa_internal.h"

namespace msa {
namespace {

std::atomic<uint64_t> g_launches{0};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// ------------------------------------------------------------------ validation
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_tensor(const msa_tensor* t) {
  if (!t || !t->data) return MSA_ERR_INVALID;
  if (t->B <= 0 || t->H <= 0 || t->N <= 0 || t->D <= 0) return MSA_ERR_INVALID;
  if (t->D != kHeadDim) return MSA_ERR_UNSUPPORTED;
  if (t->N > (int64_t{1} << 21)) return MSA_ERR_UNSUPPORTED;
  if (!aligned(t->data, 16)) return MSA_ERR_INVALID;
  if (t->sn % 8 || t->sh % 8 || t->sb % 8 || t->sn < 0 || t->sh < 0 || t->sb < 0)
    return MSA_ERR_INVALID;
  // Distinct indices must address distinct elements, in any dimension order
  // ([B, H, N, D] or the [B, N, H, D] storage of a projection, seen as a view):
  // with the dimensions of extent > 1 taken by increasing stride, each stride
  // must pass the largest offset the smaller ones reach.
  int64_t st[4] = {1, t->sn, t->sh, t->sb}, ex[4] = {t->D, t->N, t->H, t->B};
  for (int i = 1; i < 4; ++i)  // insertion sort by stride
    for (int j = i; j > 0 && st[j] < st[j - 1]; --j) {
      std::swap(st[j], st[j - 1]);
      std::swap(ex[j], ex[j - 1]);
    }
  int64_t reach = 0;  // largest element offset of the dimensions taken so far
  for (int i = 0; i < 4; ++i) {
    if (ex[i] == 1) continue;
    if (st[i] <= reach) return MSA_ERR_INVALID;
    reach += st[i] * (ex[i] - 1);
  }
  return MSA_OK;
}

// Byte range [lo, hi) that a tensor view spans (validated views: non-negative
// strides, so the last element is at the sum of the highest indices' offsets).
struct Span {
  uintptr_t lo, hi;
};

Span span(const msa_tensor* t) {
  const int64_t last = (t->B - 1) * t->sb + (t->H - 1) * t->sh + (t->N - 1) * t->sn + t->D;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(t->data);
  return {lo, lo + static_cast<uintptr_t>(last) * 2};
}

bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

struct Call {
  Geometry g;
  UnitMap u;
  cudaStream_t st;
  int last_q;
  float scale;
  const msa_opts* opts;
  Span tensors[4];  // q, k, v, out
};

int prepare(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v, const msa_tensor* out,
            const msa_opts* opts, Call& c) {
  int s;
  if ((s = check_tensor(q)) || (s = check_tensor(k)) || (s = check_tensor(v)) ||
      (s = check_tensor(out)))
    return s;
  if (k->B != q->B || v->B != q->B || out->B != q->B) return MSA_ERR_INVALID;
  if (k->N != q->N || v->N != q->N || out->N != q->N) return MSA_ERR_INVALID;
  if (v->H != k->H || out->H != q->H) return MSA_ERR_INVALID;
  if (q->H % k->H != 0) return MSA_ERR_INVALID;
  // out is written while q, k and v are still read (and q again by KV selection)
  const Span so = span(out);
  if (overlap(so, span(q)) || overlap(so, span(k)) || overlap(so, span(v))) return MSA_ERR_INVALID;
  if (opts && opts->flags != 0) return MSA_ERR_INVALID;
  if (const msa_kv_select* kv = opts ? opts->kv_select : nullptr) {
    if (!kv->lse || !aligned(kv->lse, 4)) return MSA_ERR_INVALID;
    if (kv->keep && !kv->score) return MSA_ERR_INVALID;
    if (kv->score && (!aligned(kv->score, 4) || kv->window < 1 || kv->window > q->N))
      return MSA_ERR_INVALID;
    if (kv->keep && (!aligned(kv->keep, 4) || kv->keep_k < 1)) return MSA_ERR_INVALID;
  }
  c.opts = opts;
  c.tensors[0] = span(q);
  c.tensors[1] = span(k);
  c.tensors[2] = span(v);
  c.tensors[3] = so;
  c.st = opts ? static_cast<cudaStream_t>(opts->stream) : nullptr;
  c.last_q = (opts && opts->last_q) ? static_cast<int>(opts->last_q) : kLastQMax;
  if (opts && (opts->last_q < 0 || opts->last_q > kLastQMax)) return MSA_ERR_INVALID;
  if (c.last_q > q->N) c.last_q = static_cast<int>(q->N);  // a sequence shorter than the window
  c.scale = (opts && opts->scale != 0.f) ? opts->scale : 1.0f / std::sqrt(static_cast<float>(q->D));
  if (!std::isfinite(c.scale) || c.scale <= 0.f) return MSA_ERR_INVALID;
  // head selection
  std::memset(&c.u, 0, sizeof(c.u));
  if (opts && opts->heads) {
    if (opts->n_heads <= 0 || opts->n_heads > MSA_MAX_HEADS) return MSA_ERR_INVALID;
    static_assert(MSA_MAX_HEADS <= static_cast<int>(sizeof(c.u.heads) / sizeof(c.u.heads[0])),
                  "head list capacity");
    bool seen[MSA_MAX_HEADS] = {};
    for (int i = 0; i < opts->n_heads; ++i) {
      const int32_t h = opts->heads[i];
      if (h < 0 || h >= q->H || h >= MSA_MAX_HEADS || seen[h]) return MSA_ERR_INVALID;
      seen[h] = true;
      c.u.heads[i] = h;
    }
    c.u.n_heads = opts->n_heads;
  } else {
    if (q->H > MSA_MAX_HEADS) return MSA_ERR_UNSUPPORTED;
    for (int i = 0; i < q->H; ++i) c.u.heads[i] = i;
    c.u.n_heads = static_cast<int>(q->H);
  }
  const int64_t units = q->B * c.u.n_heads;
  if (units > kMaxUnits) return MSA_ERR_UNSUPPORTED;
  Geometry& g = c.g;
  g.B = static_cast<int>(q->B);
  g.Hq = static_cast<int>(q->H);
  g.Hkv = static_cast<int>(k->H);
  g.G = g.Hq / g.Hkv;
  g.N = static_cast<int>(q->N);
  g.NB = (g.N + kBlock - 1) / kBlock;  // a partial last block counts as a padded block
  g.NQ = (g.N + kTileM - 1) / kTileM;
  g.n_units = static_cast<int>(units);
  g.scale = c.scale;
  return MSA_OK;
}

// ------------------------------------------------------------------ workspace
struct Carver {
  size_t off = 0;
  template <typename T>
  size_t take(size_t count) {
    off = (off + 255) & ~size_t{255};
    const size_t at = off;
    off += count * sizeof(T);
    return at;
  }
};

constexpr size_t kStatusBytes = 256;

struct VSLayout {
  int kv, ks, kv_pad, n_split, dist_words, chunk_words;
  size_t vmax, partial, v_score, s_score, vertical, slash, tile_dist, qdelta, qdelta_count, e2,
      e2_count, col_chunks, kc, vc, v16, total;
};

// Largest |v| per (batch, KV head), right after the status word; both are
// cleared by one memset at the start of every call.
size_t vmax_count(const Geometry& g) { return static_cast<size_t>(g.B) * g.Hkv; }

template <typename L>
size_t cleared_bytes(const L& layout, const Geometry& g) {
  return layout.vmax + vmax_count(g) * sizeof(uint32_t);
}

// f16 copy of v for the P.V product: [B][Hkv][N][128], contiguous.
size_t v16_elems(const Geometry& g) {
  return static_cast<size_t>(g.B) * g.Hkv * g.N * kHeadDim;
}

int vs_split(int units, int NB) {
  int s = (608 + units - 1) / units;
  if (s > 64) s = 64;
  if (s > NB) s = NB;
  return s < 1 ? 1 : s;
}

VSLayout vs_layout(const Geometry& g, int64_t vertical_topk, int64_t slash) {
  VSLayout L;
  L.kv = static_cast<int>(vertical_topk < g.N ? vertical_topk : g.N);
  L.ks = static_cast<int>(slash < g.N ? slash : g.N);
  L.kv_pad = (L.kv + 127) / 128 * 128;
  L.n_split = vs_split(g.n_units, g.NB);
  L.dist_words = (g.NB + 32) / 32;
  L.chunk_words = ((L.kv + 127) / 128 + 31) / 32;
  const size_t U = static_cast<size_t>(g.n_units);
  Carver c;
  c.off = kStatusBytes;
  L.vmax = c.take<uint32_t>(vmax_count(g));
  L.partial = c.take<float>(U * L.n_split * 128);
  L.v_score = c.take<float>(U * g.N);
  L.s_score = c.take<float>(U * g.N);
  L.vertical = c.take<int32_t>(U * L.kv);
  L.slash = c.take<int32_t>(U * L.ks);
  L.tile_dist = c.take<uint32_t>(U * L.dist_words);
  L.qdelta = c.take<int32_t>(U * (g.NQ + 1));
  L.qdelta_count = c.take<int32_t>(U);
  L.e2 = c.take<int32_t>(U * (g.NB + 2));
  L.e2_count = c.take<int32_t>(U);
  L.col_chunks = c.take<uint32_t>(U * g.NQ * L.chunk_words);
  L.kc = c.take<__nv_bfloat16>(U * L.kv_pad * kHeadDim);
  L.vc = c.take<__half>(U * L.kv_pad * kHeadDim);
  L.v16 = c.take<__half>(v16_elems(g));
  L.total = (c.off + 255) & ~size_t{255};
  return L;
}

struct BSLayout {
  int kb, tile_cap;
  size_t vmax, qpool, kpool, block_count, block_ids, tiles, tile_count, v16, total;
};

BSLayout bs_layout(const Geometry& g, int64_t topk) {
  BSLayout L;
  L.kb = static_cast<int>(topk < g.NB ? topk : g.NB);
  L.tile_cap = L.kb;  // a query tile's two row blocks keep at most 2 kb blocks, two per item
  const size_t U = static_cast<size_t>(g.n_units);
  Carver c;
  c.off = kStatusBytes;
  L.vmax = c.take<uint32_t>(vmax_count(g));
  L.qpool = c.take<float>(U * g.NB * kHeadDim);
  L.kpool = c.take<float>(static_cast<size_t>(g.B) * g.Hkv * g.NB * kHeadDim);
  L.block_count = c.take<int32_t>(U * g.NB);
  L.block_ids = c.take<int32_t>(U * g.NB * L.kb);
  L.tiles = c.take<int32_t>(U * g.NQ * L.tile_cap * 2);
  L.tile_count = c.take<int32_t>(U * g.NQ);
  L.v16 = c.take<__half>(v16_elems(g));
  L.total = (c.off + 255) & ~size_t{255};
  return L;
}

// Hierarchical pruning head: pooled queries, the block maxima of one slab of
// query blocks, the kept blocks (block-sparse format) and their item lists.
struct HIPLayout {
  int kb, tile_cap, slab;
  size_t vmax, qpool, qsplit, rmax, block_count, block_ids, tiles, tile_count, v16, total;
};

HIPLayout hip_layout(const Geometry& g, int64_t keep_last) {
  HIPLayout L;
  L.kb = static_cast<int>(keep_last < g.NB ? keep_last : g.NB);
  L.tile_cap = L.kb;
  L.slab = hip_slab_rows(g.n_units, g.NB);
  const size_t U = static_cast<size_t>(g.n_units);
  Carver c;
  c.off = kStatusBytes;
  L.vmax = c.take<uint32_t>(vmax_count(g));
  L.qpool = c.take<float>(U * g.NB * kHeadDim);
  L.qsplit = c.take<__nv_bfloat16>(3 * U * g.NB * kHeadDim);
  L.rmax = c.take<float>(U * L.slab * g.NB);
  L.block_count = c.take<int32_t>(U * g.NB);
  L.block_ids = c.take<int32_t>(U * g.NB * L.kb);
  L.tiles = c.take<int32_t>(U * g.NQ * L.tile_cap * 2);
  L.tile_count = c.take<int32_t>(U * g.NQ);
  L.v16 = c.take<__half>(v16_elems(g));
  L.total = (c.off + 255) & ~size_t{255};
  return L;
}

// Stage list of the hierarchical head (see include/msa.h); fills c[] and keep[]
// (keep clamped to what can matter: one more than the number of blocks).
int check_hip_stages(const msa_hip_stage* stages, int32_t n, int NB, int32_t* c, int32_t* keep) {
  if (!stages || n < 1 || n > MSA_HIP_MAX_STAGES) return MSA_ERR_INVALID;
  for (int s = 0; s < n; ++s) {
    const int64_t cb = stages[s].chunk_blocks, kp = stages[s].keep;
    if (cb < 1 || cb > (int64_t{1} << 21) || kp < 1) return MSA_ERR_INVALID;
    if (s > 0 && (cb >= stages[s - 1].chunk_blocks || stages[s - 1].chunk_blocks % cb != 0))
      return MSA_ERR_INVALID;
    c[s] = static_cast<int32_t>(cb);
    keep[s] = static_cast<int32_t>(kp < NB + 1 ? kp : NB + 1);
  }
  return stages[n - 1].chunk_blocks == 1 ? MSA_OK : MSA_ERR_INVALID;
}

struct STLayout {
  size_t vmax, v16, total;
};

STLayout st_layout(const Geometry& g) {
  STLayout L;
  Carver c;
  c.off = kStatusBytes;
  L.vmax = c.take<uint32_t>(vmax_count(g));
  L.v16 = c.take<__half>(v16_elems(g));
  L.total = (c.off + 255) & ~size_t{255};
  return L;
}

int check_workspace(const Call& c, size_t need) {
  const msa_opts* opts = c.opts;
  if (!opts || !opts->workspace) return MSA_ERR_WORKSPACE;
  if (!aligned(opts->workspace, 256)) return MSA_ERR_WORKSPACE;
  if (opts->workspace_bytes < need) return MSA_ERR_WORKSPACE;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(opts->workspace);
  for (const Span& t : c.tensors)
    if (overlap({lo, lo + need}, t)) return MSA_ERR_WORKSPACE;
  return MSA_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// ------------------------------------------------------------------ TMA maps
int make_map_4d(CUtensorMap* m, const msa_tensor* t,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                cuuint32_t box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return MSA_ERR_CUDA;
  const int64_t sh = t->H > 1 ? t->sh : t->N * t->sn;
  const int64_t sb = t->B > 1 ? t->sb : t->H * sh;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(t->D), static_cast<cuuint64_t>(t->N),
                        static_cast<cuuint64_t>(t->H), static_cast<cuuint64_t>(t->B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(t->sn * 2), static_cast<cuuint64_t>(sh * 2),
                           static_cast<cuuint64_t>(sb * 2)};
  cuuint32_t box[4] = {64, box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(m, dtype, 4, t->data, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MSA_OK : MSA_ERR_INVALID;
}

// Contiguous [B][H][N][128] f16 buffer (the staged copy of v).
int make_map_f16(CUtensorMap* m, void* base, const Geometry& g, cuuint32_t box_rows = 128) {
  msa_tensor t;
  t.data = base;
  t.B = g.B;
  t.H = g.Hkv;
  t.N = g.N;
  t.D = kHeadDim;
  t.sn = kHeadDim;
  t.sh = static_cast<int64_t>(g.N) * kHeadDim;
  t.sb = t.sh * g.Hkv;
  return make_map_4d(m, &t, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, box_rows);
}

int make_map_rows(CUtensorMap* m, void* base, int64_t rows, CUtensorMapDataType dtype,
                  cuuint32_t box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return MSA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, dtype, 2, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MSA_OK : MSA_ERR_INVALID;
}

TensorView view(const msa_tensor* t) {
  return TensorView{static_cast<const __nv_bfloat16*>(t->data), t->sb, t->sh, t->sn};
}

// ------------------------------------------------------------------ stage events
struct StageTimer {
  void* const* ev;
  cudaStream_t st;
  void begin(int s) const {
    if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev[2 * s]), st);
  }
  void end(int s) const {
    if (ev) cudaEventRecord(static_cast<cudaEvent_t>(ev[2 * s + 1]), st);
  }
};

int finish(cudaError_t e, int launches) {
  g_launches.fetch_add(static_cast<uint64_t>(launches));
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

PrefillParams base_prefill(const Call& c, msa_tensor* out, uint32_t* status,
                           const uint32_t* vmax) {
  PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.lse = (c.opts && c.opts->kv_select) ? c.opts->kv_select->lse : nullptr;
  p.g = c.g;
  p.npair = (c.g.NQ + 1) / 2;
  p.scale_log2 = c.scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(out->data);
  p.out_sb = out->sb;
  p.out_sh = out->sh;
  p.out_sn = out->sn;
  p.status = status;
  p.vmax = vmax;
  p.units = c.u;
  // K and the f16 copy of v of the KV heads the call reads, against L2 (128 MiB)
  const int64_t kv_bytes = static_cast<int64_t>(kv_heads_of(c.g.Hkv, c.g.G, c.u).n) * c.g.B *
                           c.g.N * kHeadDim * 4;
  p.units_fast = kv_bytes <= (int64_t{128} << 20) ? 1 : 0;
  return p;
}

// KV selection after the prefill: the window score from the exported row
// normalisers, then the keep set.  Nothing to do without opts->kv_select->score.
cudaError_t run_kv_select(const Call& c, const msa_tensor* q, const msa_tensor* k,
                          const KvMask& mask, const StageTimer& tm, int* launches) {
  const msa_kv_select* kv = c.opts ? c.opts->kv_select : nullptr;
  if (!kv || !kv->score) return cudaSuccess;
  tm.begin(MSA_STAGE_KV_SELECT);
  cudaError_t e = launch_kv_score(c.g, c.u, view(q), view(k), kv->lse, kv->score,
                                  static_cast<int>(kv->window), mask, c.st, launches);
  if (e == cudaSuccess && kv->keep) {
    const int kk = static_cast<int>(kv->keep_k < c.g.N ? kv->keep_k : c.g.N);
    e = launch_topk_units(kv->score, c.g.N, kk, c.g.Hq, c.u, c.g.n_units, kv->keep, c.st,
                          launches);
  }
  tm.end(MSA_STAGE_KV_SELECT);
  return e;
}

// Whether a vertical-slash call runs on the one-tile kernel: when the chosen
// offsets would cover under half of the 64-key bins on average (128 ks < N).
bool vs_one_tile(int ks, int N) { return 128LL * ks < N; }

// Every host-side check of a vertical-slash call that does not involve the
// workspace; on MSA_OK, c and L describe the call.
int vs_check(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v, int64_t vertical_topk,
             int64_t slash, const msa_tensor* out, const msa_opts* opts, Call& c, VSLayout& L) {
  const int s = prepare(q, k, v, out, opts, c);
  if (s) return s;
  if (vertical_topk <= 0 || slash <= 0) return MSA_ERR_INVALID;
  L = vs_layout(c.g, vertical_topk, slash);
  return MSA_OK;
}

KvMask base_mask(const Call& c, int kind) {
  KvMask m;
  std::memset(&m, 0, sizeof(m));
  m.kind = kind;
  m.NB = c.g.NB;
  return m;
}

}  // namespace

void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

int vertical_slash_need(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                        int64_t vertical_topk, int64_t slash, const msa_tensor* out,
                        const msa_opts* opts, size_t* need) {
  Call c;
  VSLayout L;
  const int s = vs_check(q, k, v, vertical_topk, slash, out, opts, c, L);
  if (s == MSA_OK) *need = L.total;
  return s;
}

}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_workspace_bytes(int kind, const msa_tensor* q, const msa_tensor* k, int64_t p0,
                           int64_t p1, int32_t n_heads) {
  if (check_tensor(q) != MSA_OK || check_tensor(k) != MSA_OK) return 0;
  Geometry g;
  g.B = static_cast<int>(q->B);
  g.Hq = static_cast<int>(q->H);
  g.Hkv = static_cast<int>(k->H);
  g.G = g.Hkv > 0 ? g.Hq / g.Hkv : 1;
  g.N = static_cast<int>(q->N);
  g.NB = (g.N + kBlock - 1) / kBlock;  // a partial last block counts as a padded block
  g.NQ = (g.N + kTileM - 1) / kTileM;
  g.n_units = static_cast<int>(q->B * (n_heads > 0 ? n_heads : q->H));
  if (kind == MSA_KIND_VERTICAL_SLASH) {
    if (p0 <= 0 || p1 <= 0) return 0;
    return vs_layout(g, p0, p1).total;
  }
  if (kind == MSA_KIND_BLOCK_SPARSE) {
    if (p0 <= 0) return 0;
    return bs_layout(g, p0).total;
  }
  if (kind == MSA_KIND_STREAMING) return st_layout(g).total;
  if (kind == MSA_KIND_HIERARCHICAL) {
    if (p0 <= 0) return 0;
    return hip_layout(g, p0).total;
  }
  return 0;
}

int msa_vertical_slash(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                       int64_t vertical_topk, int64_t slash, msa_tensor* out,
                       const msa_opts* opts) {
  Call c;
  VSLayout L;
  int s = vs_check(q, k, v, vertical_topk, slash, out, opts, c, L);
  if (s) return s;
  if ((s = check_workspace(c, L.total))) return s;
  void* ws = opts->workspace;
  // Sparse tiles (slash lines cover under half the 64-key bins on average)
  // run on the one-tile kernel, whose items pack 64-key blocks; denser ones
  // on the two-tile kernel, which shares each 128-key tile between two query
  // tiles.
  const bool tile_kernel = vs_one_tile(L.ks, c.g.N);
  CUtensorMap mq, mk, mv, mkc, mvc;
  const int64_t crow = static_cast<int64_t>(c.g.n_units) * L.kv_pad;
  const cuuint32_t box = tile_kernel ? 64 : 128;
  if ((s = make_map_4d(&mq, q)) ||
      (s = make_map_4d(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, box)) ||
      (s = make_map_f16(&mv, at<void>(ws, L.v16), c.g, box)) ||
      (s = make_map_rows(&mkc, at<void>(ws, L.kc), crow, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, box)) ||
      (s = make_map_rows(&mvc, at<void>(ws, L.vc), crow, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, box)))
    return s;
  const StageTimer tm{opts->stage_events, c.st};
  int launches = 0;
  cudaError_t e = cudaMemsetAsync(ws, 0, cleared_bytes(L, c.g), c.st);
  if (e != cudaSuccess) return finish(e, launches);
  tm.begin(MSA_STAGE_ESTIMATE);
  e = launch_vs_estimate(c.g, c.u, view(q), view(k), c.last_q, at<float>(ws, L.partial), L.n_split,
                         nullptr, at<float>(ws, L.v_score), at<float>(ws, L.s_score), c.st,
                         &launches);
  tm.end(MSA_STAGE_ESTIMATE);
  if (e != cudaSuccess) return finish(e, launches);
  tm.begin(MSA_STAGE_TOPK);
  {  // vertical and slash lines in one launch
    const TopkRows vert{at<float>(ws, L.v_score), c.g.N, L.kv, at<int32_t>(ws, L.vertical), L.kv};
    const TopkRows slash{at<float>(ws, L.s_score), c.g.N, L.ks, at<int32_t>(ws, L.slash), L.ks};
    e = launch_topk_pair(c.g.N, c.g.n_units, vert, slash, c.st, &launches);
  }
  tm.end(MSA_STAGE_TOPK);
  if (e != cudaSuccess) return finish(e, launches);
  tm.begin(MSA_STAGE_INDEX);
  // the f16 copy of v first: the format's gathered column rows copy from it
  e = launch_v_to_f16(view(v), c.g, c.u, at<__half>(ws, L.v16), at<uint32_t>(ws, L.vmax), c.st,
                      &launches);
  if (e == cudaSuccess)
    e = launch_vs_index(c.g, c.u, view(k), at<__half>(ws, L.v16), at<int32_t>(ws, L.slash), L.ks,
                        at<int32_t>(ws, L.vertical), L.kv, at<uint32_t>(ws, L.tile_dist),
                        L.dist_words, at<int32_t>(ws, L.qdelta), at<int32_t>(ws, L.qdelta_count),
                        at<int32_t>(ws, L.e2), at<int32_t>(ws, L.e2_count),
                        at<uint32_t>(ws, L.col_chunks), L.chunk_words,
                        at<__nv_bfloat16>(ws, L.kc), at<__half>(ws, L.vc), L.kv_pad,
                        at<uint32_t>(ws, 0), c.st, &launches);
  tm.end(MSA_STAGE_INDEX);
  if (e != cudaSuccess) return finish(e, launches);
  PrefillParams p = base_prefill(c, out, at<uint32_t>(ws, 0), at<uint32_t>(ws, L.vmax));
  p.kind = kPrefillVS;
  p.tile_dist = at<uint32_t>(ws, L.tile_dist);
  p.dist_words = L.dist_words;
  p.qdelta = at<int32_t>(ws, L.qdelta);
  p.qdelta_count = at<int32_t>(ws, L.qdelta_count);
  p.col_chunks = at<uint32_t>(ws, L.col_chunks);
  p.chunk_words = L.chunk_words;
  p.vertical = at<int32_t>(ws, L.vertical);
  p.kv = L.kv;
  p.kv_pad = L.kv_pad;
  p.vs_e2 = at<int32_t>(ws, L.e2);
  p.vs_e2_count = at<int32_t>(ws, L.e2_count);
  p.e2_stride = c.g.NB + 2;
  tm.begin(MSA_STAGE_PREFILL);
  e = tile_kernel ? launch_prefill_tile(p, mq, mk, mv, mkc, mvc, c.st, &launches)
                  : launch_prefill(p, mq, mk, mv, mkc, mvc, c.st, &launches);
  tm.end(MSA_STAGE_PREFILL);
  if (e != cudaSuccess) return finish(e, launches);
  {
    KvMask km = base_mask(c, kPrefillVS);
    km.tile_dist = p.tile_dist;
    km.dist_words = p.dist_words;
    km.vertical = p.vertical;
    km.kv = p.kv;
    e = run_kv_select(c, q, k, km, tm, &launches);
    if (e != cudaSuccess) return finish(e, launches);
  }
  if (const msa_index_export* x = opts->export_idx) {
    const size_t U = static_cast<size_t>(c.g.n_units);
    auto cp = [&](void* dst, size_t off, size_t bytes) {
      if (dst && e == cudaSuccess)
        e = cudaMemcpyAsync(dst, at<void>(ws, off), bytes, cudaMemcpyDeviceToDevice, c.st);
    };
    cp(x->v_score, L.v_score, U * c.g.N * sizeof(float));
    cp(x->s_score, L.s_score, U * c.g.N * sizeof(float));
    cp(x->vertical, L.vertical, U * L.kv * sizeof(int32_t));
    cp(x->slash, L.slash, U * L.ks * sizeof(int32_t));
    cp(x->tile_dist, L.tile_dist, U * L.dist_words * sizeof(uint32_t));
    cp(x->col_chunks, L.col_chunks, U * c.g.NQ * L.chunk_words * sizeof(uint32_t));
    if (x->col_count && e == cudaSuccess)
      e = launch_vs_col_count(c.g, at<int32_t>(ws, L.vertical), L.kv, at<uint32_t>(ws, L.tile_dist),
                              L.dist_words, x->col_count, at<uint32_t>(ws, 0), c.st, &launches);
  }
  return finish(e, launches);
}

int msa_block_sparse(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v, int64_t topk,
                     msa_tensor* out, const msa_opts* opts) {
  Call c;
  int s = prepare(q, k, v, out, opts, c);
  if (s) return s;
  if (topk <= 0) return MSA_ERR_INVALID;
  const BSLayout L = bs_layout(c.g, topk);
  if ((s = check_workspace(c, L.total))) return s;
  void* ws = opts->workspace;
  // K and the f16 copy of v are read as 64-key blocks: an item pairs two kept
  // blocks that need not be adjacent
  CUtensorMap mq, mk64, mv64, mdummy;
  std::memset(&mdummy, 0, sizeof(mdummy));
  if ((s = make_map_4d(&mq, q)) ||
      (s = make_map_4d(&mk64, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64)) ||
      (s = make_map_f16(&mv64, at<void>(ws, L.v16), c.g, 64)))
    return s;
  const StageTimer tm{opts->stage_events, c.st};
  int launches = 0;
  cudaError_t e = cudaMemsetAsync(ws, 0, cleared_bytes(L, c.g), c.st);
  if (e != cudaSuccess) return finish(e, launches);
  tm.begin(MSA_STAGE_INDEX);
  e = launch_v_to_f16(view(v), c.g, c.u, at<__half>(ws, L.v16), at<uint32_t>(ws, L.vmax),
                      c.st, &launches);
  if (e != cudaSuccess) return finish(e, launches);
  e = launch_bs_index(c.g, c.u, view(q), view(k), static_cast<int>(L.kb < topk ? L.kb : topk),
                      at<float>(ws, L.qpool), at<float>(ws, L.kpool), at<int32_t>(ws, L.block_count),
                      at<int32_t>(ws, L.block_ids), at<int32_t>(ws, L.tiles),
                      at<int32_t>(ws, L.tile_count), L.tile_cap, at<uint32_t>(ws, 0), c.st,
                      &launches);
  tm.end(MSA_STAGE_INDEX);
  if (e != cudaSuccess) return finish(e, launches);
  PrefillParams p = base_prefill(c, out, at<uint32_t>(ws, 0), at<uint32_t>(ws, L.vmax));
  p.kind = kPrefillBS;
  p.bs_tiles = at<int32_t>(ws, L.tiles);
  p.bs_tile_count = at<int32_t>(ws, L.tile_count);
  p.bs_tile_cap = L.tile_cap;
  tm.begin(MSA_STAGE_PREFILL);
  e = launch_prefill_tile(p, mq, mk64, mv64, mk64, mv64, c.st, &launches);
  tm.end(MSA_STAGE_PREFILL);
  if (e != cudaSuccess) return finish(e, launches);
  {
    KvMask km = base_mask(c, kPrefillBS);
    km.block_count = at<int32_t>(ws, L.block_count);
    km.block_ids = at<int32_t>(ws, L.block_ids);
    km.kb = L.kb;
    e = run_kv_select(c, q, k, km, tm, &launches);
    if (e != cudaSuccess) return finish(e, launches);
  }
  if (const msa_index_export* x = opts->export_idx) {
    const size_t U = static_cast<size_t>(c.g.n_units);
    if (x->block_count)
      e = cudaMemcpyAsync(x->block_count, at<void>(ws, L.block_count), U * c.g.NB * sizeof(int32_t),
                          cudaMemcpyDeviceToDevice, c.st);
    if (x->block_ids && e == cudaSuccess)
      e = cudaMemcpyAsync(x->block_ids, at<void>(ws, L.block_ids),
                          U * c.g.NB * L.kb * sizeof(int32_t), cudaMemcpyDeviceToDevice, c.st);
  }
  return finish(e, launches);
}

int msa_hierarchical(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                     const msa_hip_stage* stages, int32_t n_stages, msa_tensor* out,
                     const msa_opts* opts) {
  Call c;
  int s = prepare(q, k, v, out, opts, c);
  if (s) return s;
  int32_t sc[MSA_HIP_MAX_STAGES], sk[MSA_HIP_MAX_STAGES];
  if ((s = check_hip_stages(stages, n_stages, c.g.NB, sc, sk))) return s;
  const HIPLayout L = hip_layout(c.g, stages[n_stages - 1].keep);
  if ((s = check_workspace(c, L.total))) return s;
  void* ws = opts->workspace;
  // the kept blocks feed the block-sparse attention kernel: K and the f16 copy
  // of v are read in 64-key boxes
  CUtensorMap mq, mk, mk64, mv64, mqs;
  if ((s = make_map_4d(&mq, q)) || (s = make_map_4d(&mk, k)) ||
      (s = make_map_4d(&mk64, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 64)) ||
      (s = make_map_f16(&mv64, at<void>(ws, L.v16), c.g, 64)) ||
      (s = make_map_rows(&mqs, at<void>(ws, L.qsplit),
                         3 * static_cast<int64_t>(c.g.n_units) * c.g.NB,
                         CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)))
    return s;
  const StageTimer tm{opts->stage_events, c.st};
  int launches = 0;
  cudaError_t e = cudaMemsetAsync(ws, 0, cleared_bytes(L, c.g), c.st);
  if (e != cudaSuccess) return finish(e, launches);
  tm.begin(MSA_STAGE_INDEX);
  e = launch_v_to_f16(view(v), c.g, c.u, at<__half>(ws, L.v16), at<uint32_t>(ws, L.vmax), c.st,
                      &launches);
  if (e == cudaSuccess) e = launch_pool_q(c.g, c.u, view(q), at<float>(ws, L.qpool), c.st, &launches);
  if (e == cudaSuccess)
    e = launch_hip_index(c.g, c.u, mk, at<float>(ws, L.qpool), at<__nv_bfloat16>(ws, L.qsplit), mqs,
                         sc, sk, n_stages, at<float>(ws, L.rmax), L.slab,
                         at<int32_t>(ws, L.block_count), at<int32_t>(ws, L.block_ids), L.kb,
                         at<uint32_t>(ws, 0), c.st, &launches);
  if (e == cudaSuccess)
    e = launch_bs_tiles(c.g, L.kb, at<int32_t>(ws, L.block_count), at<int32_t>(ws, L.block_ids),
                        at<int32_t>(ws, L.tiles), at<int32_t>(ws, L.tile_count), L.tile_cap,
                        at<uint32_t>(ws, 0), c.st, &launches);
  tm.end(MSA_STAGE_INDEX);
  if (e != cudaSuccess) return finish(e, launches);
  PrefillParams p = base_prefill(c, out, at<uint32_t>(ws, 0), at<uint32_t>(ws, L.vmax));
  p.kind = kPrefillBS;  // same per-query-tile item lists as the block-sparse head
  p.bs_tiles = at<int32_t>(ws, L.tiles);
  p.bs_tile_count = at<int32_t>(ws, L.tile_count);
  p.bs_tile_cap = L.tile_cap;
  tm.begin(MSA_STAGE_PREFILL);
  e = launch_prefill_tile(p, mq, mk64, mv64, mk64, mv64, c.st, &launches);
  tm.end(MSA_STAGE_PREFILL);
  if (e != cudaSuccess) return finish(e, launches);
  {
    KvMask km = base_mask(c, kPrefillBS);
    km.block_count = at<int32_t>(ws, L.block_count);
    km.block_ids = at<int32_t>(ws, L.block_ids);
    km.kb = L.kb;
    e = run_kv_select(c, q, k, km, tm, &launches);
    if (e != cudaSuccess) return finish(e, launches);
  }
  if (const msa_index_export* x = opts->export_idx) {
    const size_t U = static_cast<size_t>(c.g.n_units);
    if (x->block_count)
      e = cudaMemcpyAsync(x->block_count, at<void>(ws, L.block_count), U * c.g.NB * sizeof(int32_t),
                          cudaMemcpyDeviceToDevice, c.st);
    if (x->block_ids && e == cudaSuccess)
      e = cudaMemcpyAsync(x->block_ids, at<void>(ws, L.block_ids),
                          U * c.g.NB * L.kb * sizeof(int32_t), cudaMemcpyDeviceToDevice, c.st);
  }
  return finish(e, launches);
}

int msa_streaming(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v, int64_t init_num,
                  int64_t local_window_num, msa_tensor* out, const msa_opts* opts) {
  Call c;
  int s = prepare(q, k, v, out, opts, c);
  if (s) return s;
  if (init_num < 0 || local_window_num < 1) return MSA_ERR_INVALID;
  const STLayout L = st_layout(c.g);
  if ((s = check_workspace(c, L.total))) return s;
  void* ws = opts->workspace;
  CUtensorMap mq, mk, mv, mdummy;
  std::memset(&mdummy, 0, sizeof(mdummy));
  if ((s = make_map_4d(&mq, q)) || (s = make_map_4d(&mk, k)) ||
      (s = make_map_f16(&mv, at<void>(ws, L.v16), c.g)))
    return s;
  const StageTimer tm{opts->stage_events, c.st};
  int launches = 0;
  cudaError_t e = cudaMemsetAsync(ws, 0, cleared_bytes(L, c.g), c.st);
  if (e != cudaSuccess) return finish(e, launches);
  tm.begin(MSA_STAGE_INDEX);
  e = launch_v_to_f16(view(v), c.g, c.u, at<__half>(ws, L.v16), at<uint32_t>(ws, L.vmax),
                      c.st, &launches);
  tm.end(MSA_STAGE_INDEX);
  if (e != cudaSuccess) return finish(e, launches);
  PrefillParams p = base_prefill(c, out, at<uint32_t>(ws, 0), at<uint32_t>(ws, L.vmax));
  p.kind = kPrefillST;
  const int64_t nb = c.g.NB;
  p.init_num = static_cast<int>(init_num < nb ? init_num : nb);
  p.local_num = static_cast<int>(local_window_num < nb ? local_window_num : nb);
  tm.begin(MSA_STAGE_PREFILL);
  e = launch_prefill(p, mq, mk, mv, mdummy, mdummy, c.st, &launches);
  tm.end(MSA_STAGE_PREFILL);
  if (e == cudaSuccess) {
    KvMask km = base_mask(c, kPrefillST);
    km.init_num = p.init_num;
    km.local_num = p.local_num;
    e = run_kv_select(c, q, k, km, tm, &launches);
  }
  return finish(e, launches);
}

int msa_device_status(void* workspace, void* stream) {
  if (!workspace) return MSA_ERR_INVALID;
  uint32_t h = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MSA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st) != cudaSuccess) return MSA_ERR_CUDA;
  if (h & kStatusTimeout) return MSA_ERR_TIMEOUT;
  if (h & kStatusBounds) return MSA_ERR_BOUNDS;
  return MSA_OK;
}

const char* msa_status_string(int status) {
  switch (status) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case MSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_TIMEOUT: return "device-side wait timed out";
    case MSA_ERR_BOUNDS: return "a kernel read an index out of range (bounds-checking build)";
    default: return "unknown status";
  }
}

uint64_t msa_kernel_launches(void) { return g_launches.load(); }

}  // extern "C"
