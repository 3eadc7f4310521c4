// prefill.cu -- chunked-prefill attention (kernel to follow).
#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {

size_t prefill_workspace_bytes(int32_t, int32_t, int) { return PKV_STATUS_BYTES; }

int launch_prefill(const void*, const void*, const void*, const int32_t*, const int32_t*, const int32_t*, int32_t,
                   void*, float, int32_t, int32_t, int32_t, void*, int, cudaStream_t) {
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
