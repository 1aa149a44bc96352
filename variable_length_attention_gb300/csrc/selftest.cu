// selftest.cu -- jfa_selftest_wait_timeout: exercises the kernels' failure path
// on the GPU without faulting it.
//
// Every wait of the library's kernels on an mbarrier is bounded: after the wait
// limit the waiting thread raises the CTA's abort flag, records
// JFA_ERR_DEVICE_TIMEOUT in the caller's workspace error word and returns, and
// jfa_device_status() reports it.  This entry point launches one CTA that waits,
// through that same bounded wait, on an mbarrier that nothing ever completes, so
// the limit runs out for certain; the context stays usable afterwards.
#include <cuda_runtime.h>

#include "../../include/jfa.h"
#include "ptx.cuh"

namespace jfa {
namespace {

__global__ void wait_forever_kernel(int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none ever comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Abort ab{&abort_flag, err};
  if (mbar_wait(&bar, 0, ab)) {
    // unreachable: nothing arrives on the barrier
    if (threadIdx.x == 0) atomicCAS(err, 0, -1);
  }
  __syncthreads();
}

}  // namespace

// Launches the never-completing bounded wait with its error word at `err`
// (device memory); used by both self-test entry points.
int launch_wait_forever(int* err, cudaStream_t stream) {
  if (cudaMemsetAsync(err, 0, sizeof(int), stream) != cudaSuccess) return JFA_ERR_CUDA;
  wait_forever_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace jfa

extern "C" int jfa_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream_) {
  if (workspace == nullptr || workspace_bytes < sizeof(int)) return JFA_ERR_INVALID_ARG;
  return jfa::launch_wait_forever(static_cast<int*>(workspace), static_cast<cudaStream_t>(stream_));
}
