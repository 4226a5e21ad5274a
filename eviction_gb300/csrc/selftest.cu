// selftest.cu -- exercises the failure path of the bounded mbarrier wait.
//
// The pipelined kernels (window attention, redundancy score) wait on mbarriers
// with mbar_wait, which gives up after kWaitLimitNs, sets
// KVC_STATUS_WAIT_TIMEOUT and returns false instead of spinning forever.  This
// kernel makes that happen on purpose, with no memory access outside its own
// shared memory and no copy in flight: one thread waits for a phase of a barrier
// that no thread or copy will ever complete.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

__global__ void wait_self_test_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that never comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, &abort_flag, status);
}

}  // namespace

cudaError_t launch_wait_self_test(const kvc_handle* h, cudaStream_t s) {
  wait_self_test_kernel<<<1, 32, 0, s>>>(h->ws.status);
  return cudaGetLastError();
}

}  // namespace kvc
