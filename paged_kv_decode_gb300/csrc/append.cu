// append.cu -- KV append: scatter new K/V rows into their page slots.
//
// The KV cache grows by one row per generated token and by a chunk of rows per
// prefill chunk ("FunASR vLLM Inference Engine Guide", section 2, PagedAttention
// with on-demand allocation). The copy is bit-exact: 16-byte vector loads and
// stores, one thread per 16 bytes of a row.
#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {

// Each token carries kKVHeads * kHeadDim bf16 of K and the same of V:
// 2 * 8 * 128 * 2 B = 4 KiB = 256 chunks of 16 B.
constexpr int kChunksPerRow = kRowBytes / 16;                  // 16
constexpr int kChunksPerTokenKV = kKVHeads * kChunksPerRow;     // 128 (K or V)
constexpr int kChunksPerToken = 2 * kChunksPerTokenKV;          // 256

__global__ void __launch_bounds__(256) append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                                     const int* __restrict__ slot_mapping, int n_tokens,
                                                     uint4* __restrict__ k_pages, uint4* __restrict__ v_pages,
                                                     int num_pages, int* status) {
  grid_dependency_wait();
  allow_dependents();
  const long long total = static_cast<long long>(n_tokens) * kChunksPerToken;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(u / kChunksPerToken);
    const int r = static_cast<int>(u % kChunksPerToken);
    const int s = __ldg(slot_mapping + t);
    if (s < 0) continue;
    const int page = s / kPageSize;
    const int slot = s % kPageSize;
    if (page >= num_pages) {
      set_status(status, PKV_ERR_OUT_OF_BOUNDS);
      continue;
    }
    const int is_v = r / kChunksPerTokenKV;
    const int c = r % kChunksPerTokenKV;
    const int head = c / kChunksPerRow;
    const int chunk = c % kChunksPerRow;
    const uint4* src = is_v ? v_new : k_new;
    uint4* dst = is_v ? v_pages : k_pages;
    const long long di = ((static_cast<long long>(page) * kKVHeads + head) * kPageSize + slot) * kChunksPerRow + chunk;
    dst[di] = __ldg(src + static_cast<long long>(t) * kChunksPerTokenKV + c);
  }
}

int launch_append(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t n_tokens, void* k_pages,
                  void* v_pages, int32_t num_pages, int* status, int num_sms, cudaStream_t stream) {
  if (n_tokens == 0) return PKV_OK;
  const long long units = static_cast<long long>(n_tokens) * kChunksPerToken;
  long long blocks = (units + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = launch_pdl(append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                                   static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
                                   n_tokens, static_cast<uint4*>(k_pages), static_cast<uint4*>(v_pages), num_pages,
                                   status);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
