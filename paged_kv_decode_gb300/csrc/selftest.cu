// selftest.cu -- diagnostic for the bounded device-side waits.
//
// Every wait of the libpkv kernels on an mbarrier (a TMA copy landing, a
// stage being released, an MMA finishing) gives up after a bounded number of
// SM cycles, records PKV_ERR_DEVICE_TIMEOUT in the workspace status word and
// lets the kernel wind down, so a lost copy can never hang the GPU. This
// kernel exercises that path on purpose: it initialises a barrier that
// nothing ever arrives on, waits on it with a short limit through the same
// helper the kernels use, and reports the outcome.
#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {

__global__ void wait_timeout_kernel(int* status, long long limit_cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  fence_barrier_init();
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: no thread arrives and no copy is pending
    if (!mbar_wait_bounded(&bar, 0, limit_cycles)) set_status(status, PKV_ERR_DEVICE_TIMEOUT);
  }
}

int launch_wait_timeout_selftest(void* workspace, long long limit_cycles, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<int*>(workspace), limit_cycles);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
