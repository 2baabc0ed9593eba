// Self-test of the failure detection every attention kernel relies on: a
// wait on an mbarrier that nothing arrives on must run out after the bounded
// budget (the production mbar_wait, about two seconds), raise the CTA's abort
// flag so that the CTA's other waiting warp gives up too, record
// VS_ERR_TIMEOUT in the caller's device error word and return, leaving the
// CUDA context usable.  No fault, trap or endless loop is involved.
#include "vs_internal.h"
#include "vs_kernel_common.cuh"

namespace vs {
namespace {

__global__ void __launch_bounds__(64, 1) selftest_timeout_kernel(int* err, int* done) {
  __shared__ uint64_t never[2];  // barriers nothing arrives on
  __shared__ int abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&never[0], 1);
    mbar_init(&never[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const Abort ab{&abort_flag, err};
  // warp 0 runs its budget out; warp 1 waits as well and leaves on the abort
  // flag (or on its own budget)
  const bool ok = mbar_wait(&never[warp], 0, ab, VS_ERR_TIMEOUT);
  if (lane == 0) atomicAdd(done, ok ? 100 : 1);
}

}  // namespace
}  // namespace vs

extern "C" vs_status vs_selftest_wait_timeout(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws) return VS_ERR_ARG;
  if (ws_bytes < 256) return VS_ERR_WORKSPACE;
  int* words = static_cast<int*>(ws);
  if (cudaMemsetAsync(words + 1, 0, sizeof(int), stream) != cudaSuccess) return VS_ERR_CUDA;
  vs::trace_begin("selftest_timeout", stream);
  vs::selftest_timeout_kernel<<<1, 64, 0, stream>>>(words, words + 1);
  vs::trace_end(stream);
  vs::note_launch();
  return cudaGetLastError() == cudaSuccess ? VS_OK : VS_ERR_CUDA;
}
