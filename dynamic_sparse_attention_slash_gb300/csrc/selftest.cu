// Self-test of the bounded device-side waits (failure detection without a GPU
// fault).  Every kernel of the library waits on mbarriers through
// mbar_wait_for: a wait that runs past its limit raises the CTA's abort flag,
// the CTA drains and exits, and the status word of the call's workspace gets
// the timeout bit, which msa_device_status reports as MSA_ERR_TIMEOUT.  This
// entry point runs that machinery on a barrier nothing arrives at (the wait
// must give up after the limit) beside a control barrier its own threads
// complete (the wait must succeed), so a test can check the status path and
// that the context stays usable, without making the GPU fault or hang.
#include "../../include/msa.h"
#include "msa_internal.h"
#include "sm103_ptx.cuh"

namespace msa {
namespace {

__global__ void __launch_bounds__(32) selftest_wait_kernel(uint32_t* ws, uint64_t limit_ns) {
  __shared__ uint64_t never_bar, control_bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&never_bar, 1);
    mbar_init(&control_bar, 32);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_arrive(&control_bar);  // 32 arrivals complete the control barrier's phase 0
  int no_abort = 0;
  const bool control = mbar_wait_for(&control_bar, 0, &no_abort, limit_ns);
  const uint64_t t0 = global_timer_ns();
  const bool got = mbar_wait_for(&never_bar, 0, &abort_flag, limit_ns);  // nothing arrives
  const uint64_t waited = global_timer_ns() - t0;
  const bool all_control = __all_sync(0xffffffffu, control);
  if (threadIdx.x == 0) {
    if (!got && abort_flag) atomicOr(ws, kStatusTimeout);
    ws[1] = all_control ? 1u : 0u;
    ws[2] = static_cast<uint32_t>(min(waited / 1000, static_cast<uint64_t>(0xffffffffu)));
  }
}

}  // namespace
}  // namespace msa

using namespace msa;

extern "C" int msa_selftest_wait_timeout(void* workspace, int64_t limit_us, void* stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MSA_ERR_INVALID;
  if (limit_us < 1 || limit_us > 1000000) return MSA_ERR_INVALID;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t*>(workspace), static_cast<uint64_t>(limit_us) * 1000u);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  note_launches(1);
  return MSA_OK;
}
