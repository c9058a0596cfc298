// Vertical-slash attention for callers that may not allocate device memory.
//
// Some callers cannot call cudaMalloc (or torch's allocator) at the point
// where they run attention: code executing under an allocator that is frozen
// for the duration of a request (fixed-pool serving runtimes), plugin hosts
// that hand an operator only its input and output buffers, or code that must
// not trigger the implicit synchronisation an allocation can cause.  For them
// this file keeps one fixed scratch area in a file-scope __device__ array: the
// CUDA runtime reserves it on every GPU that loads this library, and it stays
// reserved until the process exits.  The caller still provides q, k, v and out.
//
// The array's name, used in host code, is only a host-side stand-in for the
// symbol: handing it to a kernel would fault, or silently use the wrong memory
// where the GPU can reach host memory.  Host code therefore asks the runtime for
// the device address (cudaGetSymbolAddress, with the device current) and passes
// that address on.  The lookup is made once per CUDA context and cached under
// the context's id: a context that is destroyed and created again (after
// cudaDeviceReset, or a driver-API caller's own context) gets an id of its own
// and so a fresh lookup, never a stale address.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/msa.h"
#include "msa_internal.h"

namespace {

// MSA_STATIC_SCRATCH_BYTES bytes on every device that loads this library.
static __device__ __align__(256) unsigned char g_scratch[MSA_STATIC_SCRATCH_BYTES];

constexpr int kMaxContexts = 64;
struct CachedAddress {
  unsigned long long ctx_id;
  void* addr;
};
CachedAddress g_cache[kMaxContexts];
int g_cache_n = 0;     // entries in use
int g_cache_next = 0;  // slot replaced next once the cache is full
std::mutex g_scratch_mutex;

// Driver entry points for the current context and its id (resolved through
// the runtime, so the library needs no link-time dependency on libcuda).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return f;
}

// Id of the current context; false if none is current yet or the driver
// calls are unavailable.
bool current_context_id(unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return false;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return f.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch in the current context, looked up on the first
// call in that context.  Returns MSA_OK or MSA_ERR_CUDA.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long id = 0;
  if (current_context_id(&id)) {
    for (int i = 0; i < g_cache_n; ++i)
      if (g_cache[i].ctx_id == id) {
        *out = g_cache[i].addr;
        return MSA_OK;
      }
  }
  // First use in this context (the lookup also makes the runtime's context
  // current when none was yet).
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MSA_ERR_CUDA;
  if (current_context_id(&id)) {
    const int slot = g_cache_n < kMaxContexts ? g_cache_n++ : (g_cache_next++ % kMaxContexts);
    g_cache[slot] = {id, p};
  }
  *out = p;
  return MSA_OK;
}

}  // namespace

extern "C" int msa_vertical_slash_static(const msa_tensor* q, const msa_tensor* k,
                                         const msa_tensor* v, int64_t vertical_topk,
                                         int64_t slash, msa_tensor* out, void* stream) {
  // Every argument check of msa_vertical_slash first, without touching the
  // device; it also gives the scratch bytes this problem needs.
  msa_opts opts = {};
  opts.stream = stream;
  size_t need = 0;
  const int valid = msa::vertical_slash_need(q, k, v, vertical_topk, slash, out, &opts, &need);
  if (valid != MSA_OK) return valid;
  if (need > MSA_STATIC_SCRATCH_BYTES) return MSA_ERR_WORKSPACE;  // too large for the array
  void* scratch = nullptr;
  const int s = scratch_address(&scratch);
  if (s != MSA_OK) return s;
  // The workspace path clears the status word itself; every other scratch
  // buffer is written before it is read, so leftovers of earlier calls are
  // harmless.
  opts.workspace = scratch;
  opts.workspace_bytes = MSA_STATIC_SCRATCH_BYTES;
  return msa_vertical_slash(q, k, v, vertical_topk, slash, out, &opts);
}

extern "C" int msa_vertical_slash_static_status(void* stream) {
  void* scratch = nullptr;
  const int s = scratch_address(&scratch);
  if (s != MSA_OK) return s;
  return msa_device_status(scratch, stream);
}
