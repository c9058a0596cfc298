/*
 * msa.h -- C ABI of libmsa: MInference-style dynamic sparse prefill attention
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * The three entry points mirror the kernel-level API listed on the MInference
 * 1.0 overview page (developer.volcengine.com article, "using only the kernel"):
 *
 *   vertical_slash_sparse_attention(q, k, v, vertical_topk, slash)
 *   block_sparse_attention(q, k, v, topk)
 *   streaming_forward(q, k, v, init_num, local_window_num)
 *
 * Each computes, for every selected query head, A(M) = Softmax(Q K^T / sqrt(d)
 * - c (1 - M)) V (same page, section 1 "Problem Formulation") with masked
 * entries excluded exactly (c -> infinity) and a per-head dynamic mask M built
 * as that page's section 2.2 describes.  A row whose mask admits no key is
 * written as zeros.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Tensors   q and out are [B, Hq, N, D]; k and v are [B, Hkv, N, D]; all bf16 in
 *           device memory, innermost dimension contiguous, other strides given
 *           in elements and multiples of 8 (16 bytes), base addresses 16-byte
 *           aligned.  The strides may order the dimensions in any way (a
 *           [B, N, H, D] buffer passes as sb = N H D, sh = D, sn = H D) as
 *           long as distinct indices address distinct elements; anything else
 *           is MSA_ERR_INVALID.  Query head h reads KV head h / (Hq / Hkv).
 * Supported D = 128, 1 <= N <= 2^21, Hq a multiple of Hkv.  Other shapes return
 *           MSA_ERR_UNSUPPORTED before anything is enqueued.  When N is not a
 *           multiple of 64 the block formats treat the last block as a padded
 *           64-token block (causality keeps padded keys out of every real
 *           row; padded rows are never written).
 * Causal    Key j is admitted for query i only if j <= i.
 * Blocks    Block quantities count 64-token blocks.
 * Memory    The caller owns every buffer.  The library allocates no device
 *           memory; every entry point takes its scratch space from
 *           opts->workspace, sized by msa_workspace_bytes().  One workspace
 *           must not be shared by calls that may overlap on the GPU.  The
 *           byte range out spans must not overlap those of q, k and v
 *           (MSA_ERR_INVALID), nor the workspace's first
 *           msa_workspace_bytes() bytes any of the four (MSA_ERR_WORKSPACE);
 *           q, k and v may share memory with one another.
 * Precision S = Q K^T is a bf16 x bf16 product with f32 accumulation; the
 *           softmax runs in f32; P and a staged f16 copy of v form the P.V
 *           product with f32 accumulation; out is written as bf16 (round to
 *           nearest even).  The f16 copy is exact for a KV head whose values
 *           all lie within |v| <= 65504; a head with larger values is copied
 *           scaled by a power of two 2^-e that brings it into range, and its
 *           output is multiplied by 2^e (exact).
 * Streams   Work is enqueued on opts->stream (NULL: the legacy default
 *           stream) and runs asynchronously; a return of MSA_OK means every
 *           launch was enqueued.  Nothing synchronises with the host.
 * Errors    No exception crosses this ABI.  Invalid arguments are rejected on
 *           the host with MSA_ERR_INVALID / MSA_ERR_UNSUPPORTED /
 *           MSA_ERR_WORKSPACE before any work is enqueued; a launch failure
 *           returns MSA_ERR_CUDA.  Every device-side wait is bounded: a wait
 *           that runs out records MSA_ERR_TIMEOUT in the workspace status word,
 *           which msa_device_status() reads back.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define MSA_OK 0
#define MSA_ERR_INVALID 1     /* bad pointer, shape, stride or parameter value */
#define MSA_ERR_UNSUPPORTED 2 /* valid but outside what the library handles (D != 128, N > 2^21) */
#define MSA_ERR_WORKSPACE 3   /* workspace missing, misaligned or too small */
#define MSA_ERR_CUDA 4        /* a CUDA call or kernel launch failed */
#define MSA_ERR_TIMEOUT 5     /* a bounded device-side wait gave up (read by msa_device_status) */
#define MSA_ERR_BOUNDS 6      /* bounds-checking build (libmsa_checked.so): a kernel read an
                                 index out of range and used a valid one instead (read by
                                 msa_device_status; the output of that call is not valid) */

/* Workspace kinds for msa_workspace_bytes(). */
#define MSA_KIND_VERTICAL_SLASH 0
#define MSA_KIND_BLOCK_SPARSE 1
#define MSA_KIND_STREAMING 2
#define MSA_KIND_HIERARCHICAL 3

/* Stage ids for msa_opts.stage_events (CUDA events recorded around each stage). */
#define MSA_STAGE_ESTIMATE 0 /* vertical-slash: last-query estimate (both passes) */
#define MSA_STAGE_TOPK 1     /* vertical-slash: top-k of vertical and slash scores */
#define MSA_STAGE_INDEX 2    /* sparse format / pooling and selection, and the f16 copy of v */
#define MSA_STAGE_PREFILL 3  /* sparse attention itself */
#define MSA_STAGE_KV_SELECT 4 /* KV-selection score and keep set (only with opts->kv_select) */
#define MSA_STAGE_COUNT 5

#define MSA_MAX_HEADS 1024 /* most query heads one call may select */

/* A bf16 tensor [B, H, N, D] in device memory. Strides are in elements. */
typedef struct msa_tensor {
  void* data;
  int64_t B, H, N, D;
  int64_t sb, sh, sn; /* the D dimension is contiguous (stride 1) */
} msa_tensor;

/*
 * Optional copies of intermediate index data, for tests and diagnostics.
 * Every pointer is a caller-owned device buffer or NULL (skipped).  "units"
 * are the selected (batch, head) pairs in order b * n_heads + t, where t is
 * the position of the head in opts->heads.
 *
 * vertical-slash:
 *   v_score   float [units][N]   column sums of the estimated attention
 *   s_score   float [units][N]   diagonal sums, index = offset o = i - j
 *   vertical  int32 [units][min(vertical_topk, N)] chosen key columns, ascending
 *   slash     int32 [units][min(slash, N)]          chosen offsets, ascending
 *   tile_dist uint32 [units][(N/64 + 32) / 32]      bit t set iff 64x64 key tile
 *             m - t is active for row block m (the set is the same for every m)
 *   col_count  int32 [units][N/64]  number of columns of row block m: chosen keys
 *              j <= 64 m + 63 whose key tile m - t (t = m - j/64) is not active
 *   col_chunks uint32 [units][NQ][CW] with NQ = ceil(N/128) query tiles of 128
 *              rows and CW = ceil(ceil(min(vertical_topk, N)/128)/32) words: bit c
 *              of tile p is set iff positions [128c, 128c+128) of the ascending
 *              vertical list hold a column of row block 2p or 2p + 1
 * block-sparse:
 *   block_count int32 [units][N/64]             blocks kept per row block
 *   block_ids   int32 [units][N/64][min(topk, N/64)] kept key blocks, ascending
 *               (entries past block_count are unspecified)
 * (N/64 and N/128 round up when N is not a multiple.)
 */
typedef struct msa_index_export {
  float* v_score;
  float* s_score;
  int32_t* vertical;
  int32_t* slash;
  uint32_t* tile_dist;
  int32_t* block_count;
  int32_t* block_ids;
  int32_t* col_count;
  uint32_t* col_chunks;
} msa_index_export;

/*
 * KV selection after the prefill ("How KV sparsity achieves 1.5x acceleration
 * for vLLM", Novita AI blog, section "2. Attention modification", and the
 * PyramidKV score it quotes): the attention kernel also returns each row's
 * softmax normaliser (row max and running sum, here combined into one number); a
 * second pass in key-major ("kq") order forms the probabilities of the query
 * rows of the instruction window [N - window, N) from it and sums them per key;
 * each head then keeps the keep_k keys with the highest sums.
 *
 * Every buffer is caller-owned device memory, contiguous, indexed by the query
 * head h of q (not by the position in opts->heads); entries of heads that are
 * not selected are left untouched.  J_i below is the key set row i attends to
 * under the call's mask (causal, sparse).
 *   lse     float [B][Hq][N], required: lse_i = ln sum_{j in J_i} exp(z_ij) with
 *           z_ij = scale * q_i . k_j, i.e. rowmax_i + ln(rowsum_i); -inf for a row
 *           with no key.  Written for every row of the selected heads.
 *   score   float [B][Hq][N] or NULL (skip the score and the keep set):
 *           S_j = sum over window rows i with j in J_i of exp(z_ij - lse_i).
 *   keep    int32 [B][Hq][min(keep_k, N)] or NULL: the keys with the highest S
 *           (ties to the lower index), ascending.  Needs score.
 *   window  1 <= window <= N when score is set.
 *   keep_k  >= 1 when keep is set (larger than N is clamped).
 */
typedef struct msa_kv_select {
  float* lse;
  float* score;
  int32_t* keep;
  int64_t window;
  int64_t keep_k;
} msa_kv_select;

typedef struct msa_opts {
  void* stream;          /* cudaStream_t; NULL = legacy default stream */
  int64_t last_q;        /* vertical-slash estimate rows; 0 = 64; 1..64 accepted */
  float scale;           /* logit scale; 0 = 1/sqrt(D) */
  const int32_t* heads;  /* HOST array of query-head ids (ascending not required, no repeats); NULL = all */
  int32_t n_heads;       /* length of heads (ignored when heads is NULL) */
  void* workspace;       /* device scratch, 256-byte aligned */
  size_t workspace_bytes;
  const msa_index_export* export_idx; /* NULL = no export */
  void* const* stage_events; /* NULL, or cudaEvent_t[2 * MSA_STAGE_COUNT]: start/stop per stage
                                (a stage a call does not run records nothing) */
  int32_t flags;             /* reserved, must be 0 */
  const msa_kv_select* kv_select; /* NULL = no row normalisers, no KV selection */
} msa_opts;

/*
 * Vertical-slash head (MInference 1.0 overview, section 2.2, "Vertical-Slash Head").
 *
 * For each selected query head: the last last_q query rows are multiplied with
 * every key and soft-maxed causally (the estimate A-hat); the vertical score of
 * key j is the column sum of A-hat, the slash score of offset o the sum along
 * diagonal i - j = o.  The top min(vertical_topk, N) keys and top min(slash, N)
 * offsets are kept (score descending, ties to the lower index).  Every kept
 * offset is widened to the 64x64 key tiles its diagonal crosses; kept keys that
 * no active tile of a row block covers become extra columns of that block.
 * Attention then runs over active tiles plus columns.
 *
 * vertical_topk >= 1, slash >= 1 (larger than N is clamped).  Needs a workspace
 * of msa_workspace_bytes(MSA_KIND_VERTICAL_SLASH, q, k, vertical_topk, slash).
 */
int msa_vertical_slash(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                       int64_t vertical_topk, int64_t slash, msa_tensor* out,
                       const msa_opts* opts);

/*
 * Block-sparse head (same page, section 2.2, "Block-Sparse Head").
 *
 * Q and K are mean-pooled over 64-token blocks; block scores are
 * scale * Qhat_m . Khat_n for n <= m.  Row block m keeps its own (diagonal)
 * block plus the min(topk, m+1) - 1 best earlier blocks (score descending, ties
 * to the lower block), then attends to the kept blocks.
 *
 * topk >= 1 (larger than N/64 is clamped).  Needs a workspace of
 * msa_workspace_bytes(MSA_KIND_BLOCK_SPARSE, q, k, topk, 0).
 */
int msa_block_sparse(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                     int64_t topk, msa_tensor* out, const msa_opts* opts);

/*
 * Streaming / A-shape head (same page, kernel listing: streaming_forward).
 *
 * Row block m attends to key blocks [0, init_num) and [m - local_window_num + 1, m]
 * (the window counts the query's own block), each cut to [0, m].
 *
 * init_num >= 0, local_window_num >= 1.  Needs a workspace of
 * msa_workspace_bytes(MSA_KIND_STREAMING, q, k, 0, 0).
 */
int msa_streaming(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                  int64_t init_num, int64_t local_window_num, msa_tensor* out,
                  const msa_opts* opts);

/*
 * Hierarchical multi-stage pruning head (InfiniteHiP summary page, section on
 * the modular hierarchical token pruning algorithm: the key sequence is cut
 * into fixed-length chunks, each represented by its token with the highest
 * attention score; only the best chunks pass on, and stacked stages refine the
 * block-sparse mask of the current query block).
 *
 * For query block m (64 rows) a key token's score is scale * Qhat_m . k_j,
 * Qhat_m the mean of the block's query rows, over the candidates j <= 64m + 63.
 * Stage s splits the surviving candidates into chunks of
 * stages[s].chunk_blocks consecutive 64-token blocks (chunk x = blocks
 * [x c, (x + 1) c)); a chunk's score is its best surviving token's score; the
 * chunk holding block m and the stages[s].keep - 1 best other chunks (ties to
 * the lower chunk) survive.  The last stage has chunk_blocks = 1: its
 * surviving blocks, ascending (block m included), are the mask, and attention
 * runs over them as for the block-sparse head.
 *
 * 1 <= n_stages <= MSA_HIP_MAX_STAGES; chunk_blocks >= 1, strictly
 * decreasing, each dividing the one before, the last 1; keep >= 1.  Other
 * stage lists return MSA_ERR_INVALID.  Needs a workspace of
 * msa_workspace_bytes(MSA_KIND_HIERARCHICAL, q, k, stages[n_stages-1].keep, 0,
 * n_heads).  The index export fills block_count / block_ids as for the
 * block-sparse head (min(keep_last, N/64) ids per row block).
 */
#define MSA_HIP_MAX_STAGES 8
typedef struct msa_hip_stage {
  int64_t chunk_blocks; /* chunk size in 64-token blocks */
  int64_t keep;         /* chunks kept, the query block's own chunk included */
} msa_hip_stage;
int msa_hierarchical(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                     const msa_hip_stage* stages, int32_t n_stages, msa_tensor* out,
                     const msa_opts* opts);

/*
 * Vertical-slash attention without a caller-provided workspace.  The MInference
 * pages have no counterpart; this entry point exists for callers that cannot
 * allocate device memory where they run attention: an allocator frozen for the
 * duration of a request in a fixed-pool serving runtime, a plugin host that
 * hands an operator only its inputs and outputs, or code that must avoid the
 * implicit synchronisation an allocation can cause.
 *
 * It computes what msa_vertical_slash computes for all heads of q (last_q = 64,
 * scale = 1/sqrt(D), no index export), taking its scratch space from one
 * file-scope device array of MSA_STATIC_SCRATCH_BYTES that the CUDA runtime
 * reserves on every GPU that loads this library, until the process exits.  It
 * calls no cudaMalloc, cudaFree or allocating library routine.
 *
 *  - A problem whose msa_workspace_bytes(MSA_KIND_VERTICAL_SLASH, ...) exceeds
 *    MSA_STATIC_SCRATCH_BYTES returns MSA_ERR_WORKSPACE before anything is
 *    enqueued (4 query heads over 2 KV heads at N = 32768 with vertical_topk
 *    1000 and slash 6096 fit; 32 heads over 8 KV heads at that N do not);
 *    invalid arguments return MSA_ERR_INVALID.
 *  - The first call in a CUDA context (normally: the first call on a device)
 *    looks up the array's device address (cudaGetSymbolAddress, with that
 *    device current) and caches it under the context's id: make that first
 *    call before any stream capture.  A context created anew (for instance
 *    after cudaDeviceReset) gets a lookup of its own.
 *  - Every call on a device shares the one array, which keeps the last call's
 *    contents (each call clears what must start at zero).  Calls that may
 *    overlap on the GPU (different streams or host threads) race on it; the
 *    caller must serialise them.
 *  - Device-side status (a bounded wait that gave up) lands in the array;
 *    msa_vertical_slash_static_status() reads and clears it.
 * stream is a cudaStream_t (NULL: the legacy default stream).
 */
#define MSA_STATIC_SCRATCH_BYTES (64u << 20)
int msa_vertical_slash_static(const msa_tensor* q, const msa_tensor* k, const msa_tensor* v,
                              int64_t vertical_topk, int64_t slash, msa_tensor* out,
                              void* stream);

/*
 * Device status of msa_vertical_slash_static's array on the current device,
 * as msa_device_status() reports it for a workspace: enqueues a read of the
 * status word on `stream` after the work already enqueued there, synchronises
 * that stream, then clears the word.  Returns MSA_OK, MSA_ERR_TIMEOUT,
 * MSA_ERR_BOUNDS (bounds-checking build only), or MSA_ERR_CUDA if the lookup or
 * the copy failed.  Allocates nothing.
 */
int msa_vertical_slash_static_status(void* stream);

/*
 * Recall of the dense attention that a sparse mask keeps, per head (MInference
 * 1.0 overview, section 2.1 "Kernel-Aware Optimal Sparse Pattern Search": the
 * search compares candidate patterns at similar kernel FLOPs by the recall of
 * the attention output).  For row i the kept mass is
 *   sum_{j in J_i} softmax_dense(i)_j = exp(lse_i - ref_lse_i),
 * lse from a sparse call and ref_lse from a dense call (msa_streaming with
 * init_num 0 and local_window_num N/64), both through msa_kv_select.lse.
 *   lse, ref_lse  float [B][H][N] device buffers (as msa_kv_select.lse)
 *   recall        float [B][H] device buffer: entry (b, h) of every selected
 *                 head receives the mean kept mass over rows [row0, N); other
 *                 entries are left untouched.  Rows with lse = -inf keep 0.
 *   heads         HOST array of n_heads query-head ids (no repeats); NULL = all.
 * 0 <= row0 < N.  Enqueued on `stream` (cudaStream_t; NULL = legacy default);
 * deterministic (fixed-order reduction in double).
 */
int msa_mass_recall(const float* lse, const float* ref_lse, int64_t B, int64_t H, int64_t N,
                    int64_t row0, const int32_t* heads, int32_t n_heads, float* recall,
                    void* stream);

/*
 * Workspace bytes needed by one call.  kind is MSA_KIND_*; p0/p1 are
 * (vertical_topk, slash) for vertical-slash, (topk, unused) for block-sparse,
 * (keep of the last stage, unused) for the hierarchical head.
 * n_heads is the number of selected query heads (<= 0: all of q's heads).
 * Returns 0 for invalid arguments.
 */
size_t msa_workspace_bytes(int kind, const msa_tensor* q, const msa_tensor* k, int64_t p0,
                           int64_t p1, int32_t n_heads);

/*
 * Reads (and clears) the device status word of a workspace after the work of
 * an earlier call has been enqueued on `stream`; synchronises that stream.
 * Returns MSA_OK, MSA_ERR_TIMEOUT, MSA_ERR_BOUNDS (bounds-checking build only),
 * or MSA_ERR_CUDA if the copy itself failed.
 */
int msa_device_status(void* workspace, void* stream);

/*
 * Self-test of the bounded device-side waits behind MSA_ERR_TIMEOUT: enqueues
 * on `stream` one 32-thread CTA that waits, with a limit of `limit_us`
 * microseconds (1 .. 1000000), on an mbarrier nothing arrives at, and on a
 * control mbarrier its own threads complete.  The first wait gives up and sets
 * the timeout bit of the status word at `workspace`, so msa_device_status
 * (workspace, stream) then returns MSA_ERR_TIMEOUT.  It also writes two 32-bit
 * words after the status word: word 1 = 1 if the control wait succeeded, word
 * 2 = microseconds the first wait lasted.  `workspace`: device memory of at
 * least 256 bytes, 256-byte aligned, caller-owned (a call's workspace will do).
 * Nothing faults or hangs: the waits are bounded and no copy or tensor-core
 * work is in flight.  Returns MSA_OK when enqueued, MSA_ERR_INVALID for a bad
 * pointer or limit, MSA_ERR_CUDA if the launch failed.
 */
int msa_selftest_wait_timeout(void* workspace, int64_t limit_us, void* stream);

/* Human-readable name of a status code (static storage). */
const char* msa_status_string(int status);

/* Number of kernel launches this library has enqueued in this process. */
uint64_t msa_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
