// append.cu -- KV append: scatter new K/V rows into their page slots.
//
// The KV cache grows by one row per generated token and by a chunk of rows per
// prefill chunk ("FunASR vLLM Inference Engine Guide", section 2, PagedAttention
// with on-demand allocation). The copy is bit-exact: 16-byte vector loads and
// stores, one thread per 16 bytes of a row.
#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {

// Each token carries num_kv_heads rows of head_dim bf16 for K and the same for
// V; a row is head_dim / 8 chunks of 16 B (for the Qwen3 decoder 2 * 8 * 16 =
// 256 chunks per token).
__global__ void __launch_bounds__(256) append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                                     const int* __restrict__ slot_mapping, int n_tokens,
                                                     uint4* __restrict__ k_pages, uint4* __restrict__ v_pages,
                                                     int num_pages, int hkv, int row_chunks, int* status) {
  grid_dependency_wait();
  allow_dependents();
  const int token_kv = hkv * row_chunks;  // chunks of K (or V) per token
  const long long total = static_cast<long long>(n_tokens) * 2 * token_kv;
  for (long long u = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(u / (2 * token_kv));
    const int r = static_cast<int>(u % (2 * token_kv));
    const int s = __ldg(slot_mapping + t);
    if (s < 0) continue;
    const int page = s / kPageSize;
    const int slot = s % kPageSize;
    if (page >= num_pages) {
      set_status(status, PKV_ERR_OUT_OF_BOUNDS);
      continue;
    }
    const int is_v = r / token_kv;
    const int c = r % token_kv;
    const int head = c / row_chunks;
    const int chunk = c % row_chunks;
    const uint4* src = is_v ? v_new : k_new;
    uint4* dst = is_v ? v_pages : k_pages;
    const long long di = ((static_cast<long long>(page) * hkv + head) * kPageSize + slot) * row_chunks + chunk;
    dst[di] = __ldg(src + static_cast<long long>(t) * token_kv + c);
  }
}

int launch_append(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t n_tokens, void* k_pages,
                  void* v_pages, int32_t num_pages, int32_t num_kv_heads, int32_t head_dim, int* status, int num_sms,
                  cudaStream_t stream) {
  if (n_tokens == 0) return PKV_OK;
  const int row_chunks = head_dim / 8;
  const long long units = static_cast<long long>(n_tokens) * 2 * num_kv_heads * row_chunks;
  long long blocks = (units + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  const cudaError_t e = launch_pdl(append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                                   static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
                                   n_tokens, static_cast<uint4*>(k_pages), static_cast<uint4*>(v_pages), num_pages,
                                   static_cast<int>(num_kv_heads), row_chunks, status);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
