// decode_noalloc.cu -- pkv_decode_attn_noalloc: decode attention whose split-KV
// scratch lives in a fixed device array owned by the library, so the caller
// never has to allocate device memory for it.
//
// Who needs this: code that is not allowed to call cudaMalloc at the point
// where it runs decode attention -- for example a plug-in loaded into a host
// runtime that owns all device memory through its own pool, or a serving loop
// that reserves its memory once at start-up and must never allocate (or
// implicitly synchronise) afterwards. Such a caller can still pass its inputs
// and outputs, but it cannot hand over a workspace.
//
// The scratch is one file-scope __device__ array of kScratchBytes. Every GPU
// that loads the library holds it until the process exits. Host code must not
// pass the array's name to a kernel (on the host it is only a stand-in, not a
// device address), so the entry point looks the device address up with
// cudaGetSymbolAddress, once per device and context, with that device current.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkv.h"
#include "pkv_kernels.h"

namespace {

constexpr size_t kScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};
int g_scratch_sms[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The driver's cuCtxGetCurrent, found through the runtime (the library links
// only the runtime).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  }
  return fn;
}

// Device address of the scratch array and SM count of the current device.
// The first call on a device does the lookup, and so does the first call in
// any other context on it: each context loads its own copy of the module, and
// with it of the array.
int scratch_of_current_device(void** addr, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (get_ctx == nullptr) return PKV_ERR_CUDA;
  // the context current now (none yet if no runtime call has needed one on this thread)
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (ctx == nullptr || g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ERR_CUDA;
    if (!(major == 10 && minor == 3)) return PKV_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
    // the lookup made the device's context current if none was
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx;
    g_scratch_sms[dev] = sms;
  }
  *addr = g_scratch_addr[dev];
  *num_sms = g_scratch_sms[dev];
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int pkv_decode_attn_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* block_table, const int32_t* seq_lens, void* out, float scale,
                                       pkv_stream_t stream, const pkv_cache_desc* desc, int32_t batch,
                                       int32_t max_pages_per_seq) {
  if (desc == nullptr) return PKV_ERR_NULL_ARG;
  if (desc->num_q_heads <= 0 || desc->num_kv_heads <= 0 || desc->head_dim <= 0 || desc->page_size <= 0 ||
      desc->num_pages <= 0)
    return PKV_ERR_BAD_SHAPE;
  if (desc->num_q_heads != 16 || desc->num_kv_heads != 8 || desc->head_dim != 128 || desc->page_size != 16)
    return PKV_ERR_UNSUPPORTED;
  if (batch < 0 || max_pages_per_seq < 1) return PKV_ERR_BAD_SHAPE;
  if (batch > PKV_NOALLOC_MAX_BATCH) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (static_cast<long long>(batch) * max_pages_per_seq * 8 >= (1LL << 31)) return PKV_ERR_BAD_SHAPE;
  if (batch == 0) return PKV_OK;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out) return PKV_ERR_NULL_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)) return PKV_ERR_MISALIGNED;

  void* scratch = nullptr;
  int sms = 0;
  int rc = scratch_of_current_device(&scratch, &sms);
  if (rc != PKV_OK) return rc;
  if (pkv::decode_workspace_bytes(16, 8, 128, batch, sms) > kScratchBytes) return PKV_ERR_WORKSPACE_TOO_SMALL;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left. The status word and the
  // split records must start at zero; a call that stopped early (a timed-out
  // wait) could have left tagged words behind.
  if (cudaMemsetAsync(scratch, 0, pkv::decode_workspace_bytes(16, 8, 128, batch, sms), s) != cudaSuccess)
    return PKV_ERR_CUDA;
  return pkv::launch_decode(q, nullptr, nullptr, k_pages, v_pages, block_table, seq_lens, nullptr, 0, out, scale, 16, 8,
                            128, batch, max_pages_per_seq, desc->num_pages, scratch, sms, s, 0u);
}
