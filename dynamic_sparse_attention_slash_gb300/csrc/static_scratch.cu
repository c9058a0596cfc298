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
// the device address once per device (cudaGetSymbolAddress, with that device
// current) and passes that address on.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/msa.h"

namespace {

// MSA_STATIC_SCRATCH_BYTES bytes on every device that loads this library.
static __device__ __align__(256) unsigned char g_scratch[MSA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of g_scratch on the current device, looked up on the first
// call per device.  Returns MSA_OK or MSA_ERR_CUDA.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MSA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MSA_OK;
}

}  // namespace

extern "C" int msa_vertical_slash_static(const msa_tensor* q, const msa_tensor* k,
                                         const msa_tensor* v, int64_t vertical_topk,
                                         int64_t slash, msa_tensor* out, void* stream) {
  // Full host-side validation first, without touching the device: with no
  // workspace the call checks every argument and then stops at the workspace
  // check, so anything but MSA_ERR_WORKSPACE is the argument error.
  msa_opts check = {};
  check.stream = stream;
  const int valid = msa_vertical_slash(q, k, v, vertical_topk, slash, out, &check);
  if (valid != MSA_ERR_WORKSPACE) return valid;
  const int32_t n_heads = static_cast<int32_t>(q->H);
  const size_t need =
      msa_workspace_bytes(MSA_KIND_VERTICAL_SLASH, q, k, vertical_topk, slash, n_heads);
  if (need == 0) return MSA_ERR_INVALID;
  if (need > MSA_STATIC_SCRATCH_BYTES) return MSA_ERR_WORKSPACE;  // too large for the array
  void* scratch = nullptr;
  const int s = scratch_address(&scratch);
  if (s != MSA_OK) return s;
  // The workspace path clears the status word itself; every other scratch
  // buffer is written before it is read, so leftovers of earlier calls are
  // harmless.
  msa_opts opts = {};
  opts.stream = stream;
  opts.workspace = scratch;
  opts.workspace_bytes = MSA_STATIC_SCRATCH_BYTES;
  return msa_vertical_slash(q, k, v, vertical_topk, slash, out, &opts);
}
