// Diagnostics: the library's bounded waits, run on a barrier phase that no
// thread ever completes.  Each wait gives up after the wait limit, reports
// MTP_STATUS_TIMEOUT through the status word and returns, so a caller can
// check that a stalled wait ends in a status the host reads and that the CUDA
// context stays usable.  Nothing here faults, traps or spins without a limit.
#include "common.cuh"
#include "internal.h"
#include "mtpspec.h"

namespace mtp {
namespace {

// Warp 0 waits with the spinning form (mbar_wait), warp 1 with the parked form
// (mbar_sleep_wait), both on phase 0 of a barrier that expects one arrival
// which no thread makes.
__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(int *status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x < 32) mbar_wait(&bar, 0u, status);
  else mbar_sleep_wait(&bar, 0u, status);
}

}  // namespace
MTP_TRACE_COLLECTOR(diag)

}  // namespace mtp

extern "C" int mtp_selftest_wait_timeout(int32_t *status, mtp_stream_t stream) {
  if (!status || (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return MTP_ERR_INVALID_ARG;
  mtp::note_launch();
  mtp::wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}
