// pkv_abi.cu -- the extern "C" entry points of libpkv: argument checks on the
// host, launch-configuration choice, and the status word helpers. All device
// work is in append.cu, decode.cu (decode_kernel.cuh) and prefill.cu.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pkv.h"
#include "pkv_kernels.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool known = false;
  bool supported = false;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// SM count of the current device, and whether it is an sm_103 part (the only
// architecture the kernels are compiled for).
int current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.known) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.known = true;
  }
  if (!d.supported) return PKV_ERR_UNSUPPORTED;
  *num_sms = d.num_sms;
  return PKV_OK;
}

// The geometry every call supports: the Qwen3 decoder's 16 query / 8 KV heads
// of dimension 128, page size 16 (decode.cu, prefill.cu, the fused calls).
int check_desc(const pkv_cache_desc* d) {
  if (d == nullptr) return PKV_ERR_NULL_ARG;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->page_size <= 0 || d->num_pages <= 0)
    return PKV_ERR_BAD_SHAPE;
  if (d->num_q_heads != 16 || d->num_kv_heads != 8 || d->head_dim != 128 || d->page_size != 16)
    return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

// Geometries pkv_append and the decode calls serve: page size 16, head_dim 64
// or 128, 1 to 8 query heads per KV head (16 / 8 / 128 on an instantiation
// with the head counts fixed at compile time).
int check_desc_decode(const pkv_cache_desc* d) {
  const int rc = check_desc(d);
  if (rc != PKV_ERR_UNSUPPORTED) return rc;
  return pkv::decode_supported(d->num_q_heads, d->num_kv_heads, d->head_dim, d->page_size) ? PKV_OK
                                                                                          : PKV_ERR_UNSUPPORTED;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest block table the kernels index with 32-bit counts of (request, KV
// head, page) triples (the decode kernel's flattened list: at most rows *
// max_pages * KV heads entries).
bool table_fits(int32_t rows, int32_t max_pages, int32_t kv_heads = 8) {
  const long long h = kv_heads > 8 ? kv_heads : 8;
  return static_cast<long long>(rows) * max_pages * h < (1LL << 31);
}

}  // namespace

extern "C" {

int pkv_workspace_init(void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (workspace == nullptr) return PKV_ERR_NULL_ARG;
  if (workspace_bytes < PKV_STATUS_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
  return cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

int pkv_read_status(const void* workspace, pkv_stream_t stream) {
  if (workspace == nullptr) return PKV_ERR_NULL_ARG;
  int v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  return v;
}

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL_ARG: return "a required pointer is NULL";
    case PKV_ERR_BAD_SHAPE: return "bad or inconsistent size";
    case PKV_ERR_UNSUPPORTED:
      return "unsupported geometry or device (sm_103; decode, the fused calls, append and prefill: page 16, "
             "head_dim 64/128, 1 to 8 query heads per KV head; the no-alloc call: 16/8/128/16)";
    case PKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKV_ERR_CUDA: return "CUDA runtime or launch error";
    case PKV_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
    case PKV_ERR_OUT_OF_BOUNDS: return "page id, slot or length outside the pool or block table";
    case PKV_ERR_MISALIGNED: return "buffer not 16-byte aligned";
    default: return "unknown status";
  }
}

int pkv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t n_tokens, void* k_pages,
               void* v_pages, const pkv_cache_desc* desc, pkv_stream_t stream, void* workspace,
               size_t workspace_bytes) {
  int rc = check_desc_decode(desc);
  if (rc != PKV_OK) return rc;
  if (n_tokens < 0) return PKV_ERR_BAD_SHAPE;
  if (workspace != nullptr && workspace_bytes < PKV_STATUS_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (n_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_pages || !v_pages) return PKV_ERR_NULL_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
    return PKV_ERR_MISALIGNED;
  int sms = 0;
  rc = current_device(&sms);
  if (rc != PKV_OK) return rc;
  return pkv::launch_append(k_new, v_new, slot_mapping, n_tokens, k_pages, v_pages, desc->num_pages,
                            desc->num_kv_heads, desc->head_dim, static_cast<int*>(workspace), sms,
                            reinterpret_cast<cudaStream_t>(stream));
}

// Workspace bytes of a decode call for this geometry.
static size_t decode_ws(const pkv_cache_desc* desc, int32_t batch, int sms) {
  return pkv::decode_workspace_bytes(desc->num_q_heads, desc->num_kv_heads, desc->head_dim, batch, sms);
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq) {
  if (check_desc_decode(desc) != PKV_OK || batch < 0 || max_pages_per_seq < 1) return 0;
  if (batch > pkv::decode_max_batch() || !table_fits(batch, max_pages_per_seq, desc->num_kv_heads)) return 0;
  int sms = 0;
  if (current_device(&sms) != PKV_OK) return 0;
  return decode_ws(desc, batch, sms);
}

int pkv_decode_attn(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                    const int32_t* seq_lens, void* out, float scale, pkv_stream_t stream,
                    const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq, void* workspace,
                    size_t workspace_bytes) {
  int rc = check_desc_decode(desc);
  if (rc != PKV_OK) return rc;
  if (batch < 0 || max_pages_per_seq < 1) return PKV_ERR_BAD_SHAPE;
  if (batch > pkv::decode_max_batch()) return PKV_ERR_UNSUPPORTED;
  if (!table_fits(batch, max_pages_per_seq, desc->num_kv_heads)) return PKV_ERR_BAD_SHAPE;
  if (workspace == nullptr) return PKV_ERR_NULL_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out) return PKV_ERR_NULL_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) || !aligned16(workspace))
    return PKV_ERR_MISALIGNED;
  int sms = 0;
  rc = current_device(&sms);
  if (rc != PKV_OK) return rc;
  if (workspace_bytes < decode_ws(desc, batch, sms)) return PKV_ERR_WORKSPACE_TOO_SMALL;
  return pkv::launch_decode(q, nullptr, nullptr, k_pages, v_pages, block_table, seq_lens, nullptr, 0, out, scale,
                            desc->num_q_heads, desc->num_kv_heads, desc->head_dim, batch, max_pages_per_seq,
                            desc->num_pages, workspace, sms, reinterpret_cast<cudaStream_t>(stream), 0u);
}

static int decode_append(const void* q, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                         const int32_t* block_table, const int32_t* seq_lens, const float* rope_cos_sin,
                         int32_t rope_max_pos, void* out, float scale, pkv_stream_t stream, const pkv_cache_desc* desc,
                         int32_t batch, int32_t max_pages_per_seq, void* workspace, size_t workspace_bytes,
                         uint32_t flags) {
  int rc = check_desc_decode(desc);
  if (rc != PKV_OK) return rc;
  if (batch < 0 || max_pages_per_seq < 1) return PKV_ERR_BAD_SHAPE;
  if (batch > pkv::decode_max_batch()) return PKV_ERR_UNSUPPORTED;
  if (!table_fits(batch, max_pages_per_seq, desc->num_kv_heads)) return PKV_ERR_BAD_SHAPE;
  if (workspace == nullptr) return PKV_ERR_NULL_ARG;
  if (batch == 0) return PKV_OK;
  if (!q || !k_new || !v_new || !k_pages || !v_pages || !block_table || !seq_lens || !out) return PKV_ERR_NULL_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages) ||
      !aligned16(out) || !aligned16(workspace))
    return PKV_ERR_MISALIGNED;
  int sms = 0;
  rc = current_device(&sms);
  if (rc != PKV_OK) return rc;
  if (workspace_bytes < decode_ws(desc, batch, sms)) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if ((flags & ~static_cast<uint32_t>(PKV_DECODE_EARLY_PREFETCH)) != 0) return PKV_ERR_UNSUPPORTED;
  return pkv::launch_decode(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, rope_cos_sin, rope_max_pos, out,
                            scale, desc->num_q_heads, desc->num_kv_heads, desc->head_dim, batch, max_pages_per_seq,
                            desc->num_pages, workspace, sms, reinterpret_cast<cudaStream_t>(stream), flags);
}

int pkv_decode_append_attn(const void* q, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                           const int32_t* block_table, const int32_t* seq_lens, void* out, float scale,
                           pkv_stream_t stream, const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq,
                           void* workspace, size_t workspace_bytes, uint32_t flags) {
  return decode_append(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, nullptr, 0, out, scale, stream, desc,
                       batch, max_pages_per_seq, workspace, workspace_bytes, flags);
}

int pkv_decode_append_rope_attn(const void* q, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                                const int32_t* block_table, const int32_t* seq_lens, const float* rope_cos_sin,
                                int32_t rope_max_pos, void* out, float scale, pkv_stream_t stream,
                                const pkv_cache_desc* desc, int32_t batch, int32_t max_pages_per_seq, void* workspace,
                                size_t workspace_bytes, uint32_t flags) {
  if (batch > 0 && rope_cos_sin == nullptr) return PKV_ERR_NULL_ARG;
  if (rope_max_pos < 1) return PKV_ERR_BAD_SHAPE;
  if (batch > 0 && !aligned16(rope_cos_sin)) return PKV_ERR_MISALIGNED;
  return decode_append(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, rope_cos_sin, rope_max_pos, out,
                       scale, stream, desc, batch, max_pages_per_seq, workspace, workspace_bytes, flags);
}

// Geometries pkv_prefill_chunk_attn serves (prefill.cu): page size 16, head_dim 64 or 128, 1 to 8
// query heads per KV head; 16/8/128 among them.
static int check_desc_prefill(const pkv_cache_desc* d) {
  const int rc = check_desc(d);
  if (rc != PKV_ERR_UNSUPPORTED) return rc;
  return pkv::prefill_supported(d->num_q_heads, d->num_kv_heads, d->head_dim, d->page_size) ? PKV_OK
                                                                                           : PKV_ERR_UNSUPPORTED;
}

size_t pkv_prefill_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs, int32_t max_q_len) {
  if (check_desc_prefill(desc) != PKV_OK || num_seqs < 0 || max_q_len < 0) return 0;
  int sms = 0;
  if (current_device(&sms) != PKV_OK) return 0;
  return pkv::prefill_workspace_bytes(desc->num_q_heads, desc->num_kv_heads, desc->head_dim, num_seqs, max_q_len,
                                      sms);
}

int pkv_prefill_chunk_attn(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                           const int32_t* prefix_lens, const int32_t* cu_q_lens, int32_t num_seqs, int32_t total_q,
                           void* out, float scale, pkv_stream_t stream, const pkv_cache_desc* desc,
                           int32_t max_pages_per_seq, int32_t max_q_len, void* workspace, size_t workspace_bytes) {
  int rc = check_desc_prefill(desc);
  if (rc != PKV_OK) return rc;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_pages_per_seq < 1) return PKV_ERR_BAD_SHAPE;
  if (!table_fits(num_seqs, max_pages_per_seq)) return PKV_ERR_BAD_SHAPE;
  if (static_cast<long long>(desc->num_pages) * desc->num_kv_heads * desc->page_size >= (1LL << 31))
    return PKV_ERR_UNSUPPORTED;
  if (num_seqs > pkv::prefill_max_seqs()) return PKV_ERR_UNSUPPORTED;
  if (workspace == nullptr) return PKV_ERR_NULL_ARG;
  if (workspace_bytes < PKV_STATUS_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (num_seqs == 0 || max_q_len == 0 || total_q == 0) return PKV_OK;
  if (!q || !k_pages || !v_pages || !block_table || !prefix_lens || !cu_q_lens || !out) return PKV_ERR_NULL_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) || !aligned16(workspace))
    return PKV_ERR_MISALIGNED;
  int sms = 0;
  rc = current_device(&sms);
  if (rc != PKV_OK) return rc;
  if (workspace_bytes < pkv::prefill_workspace_bytes(desc->num_q_heads, desc->num_kv_heads, desc->head_dim, num_seqs,
                                                     max_q_len, sms))
    return PKV_ERR_WORKSPACE_TOO_SMALL;
  return pkv::launch_prefill(q, k_pages, v_pages, block_table, prefix_lens, cu_q_lens, num_seqs, total_q, out, scale,
                             desc->num_q_heads, desc->num_kv_heads, desc->head_dim, max_pages_per_seq, max_q_len,
                             desc->num_pages, workspace, reinterpret_cast<cudaStream_t>(stream));
}

size_t pkv_mixed_workspace_bytes(const pkv_cache_desc* desc, int32_t num_seqs, int32_t max_q_len, int32_t dec_batch,
                                 int32_t dec_max_pages_per_seq) {
  if (check_desc(desc) != PKV_OK || num_seqs < 0 || max_q_len < 0 || dec_batch < 0 || dec_max_pages_per_seq < 1)
    return 0;
  if (num_seqs > pkv::prefill_max_seqs() || dec_batch > pkv::decode_max_batch()) return 0;
  int sms = 0;
  if (current_device(&sms) != PKV_OK) return 0;
  const bool chunk = num_seqs > 0 && max_q_len > 0;
  return pkv::mixed_workspace_bytes(chunk ? num_seqs : 0, chunk ? max_q_len : 0, dec_batch, dec_max_pages_per_seq, sms);
}

int pkv_mixed_step_attn(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                        const int32_t* prefix_lens, const int32_t* cu_q_lens, int32_t num_seqs, int32_t total_q,
                        void* out, int32_t max_pages_per_seq, int32_t max_q_len, const void* dec_q,
                        const int32_t* dec_block_table, const int32_t* dec_seq_lens, void* dec_out, int32_t dec_batch,
                        int32_t dec_max_pages_per_seq, float scale, pkv_stream_t stream, const pkv_cache_desc* desc,
                        void* workspace, size_t workspace_bytes) {
  int rc = check_desc(desc);  // the tuned 16/8/128 geometry only
  if (rc != PKV_OK) return rc;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_pages_per_seq < 1) return PKV_ERR_BAD_SHAPE;
  if (dec_batch < 0 || dec_max_pages_per_seq < 1) return PKV_ERR_BAD_SHAPE;
  if (!table_fits(num_seqs, max_pages_per_seq) || !table_fits(dec_batch, dec_max_pages_per_seq))
    return PKV_ERR_BAD_SHAPE;
  if (static_cast<long long>(desc->num_pages) * desc->num_kv_heads * desc->page_size >= (1LL << 31))
    return PKV_ERR_UNSUPPORTED;
  if (num_seqs > pkv::prefill_max_seqs() || dec_batch > pkv::decode_max_batch()) return PKV_ERR_UNSUPPORTED;
  if (workspace == nullptr) return PKV_ERR_NULL_ARG;
  if (workspace_bytes < PKV_STATUS_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
  const bool chunk = num_seqs > 0 && max_q_len > 0 && total_q > 0;
  if (!chunk && dec_batch == 0) return PKV_OK;
  if (!k_pages || !v_pages) return PKV_ERR_NULL_ARG;
  if (chunk && (!q || !block_table || !prefix_lens || !cu_q_lens || !out)) return PKV_ERR_NULL_ARG;
  if (dec_batch > 0 && (!dec_q || !dec_block_table || !dec_seq_lens || !dec_out)) return PKV_ERR_NULL_ARG;
  if (!aligned16(k_pages) || !aligned16(v_pages) || !aligned16(workspace)) return PKV_ERR_MISALIGNED;
  if (chunk && (!aligned16(q) || !aligned16(out))) return PKV_ERR_MISALIGNED;
  if (dec_batch > 0 && (!aligned16(dec_q) || !aligned16(dec_out))) return PKV_ERR_MISALIGNED;
  int sms = 0;
  rc = current_device(&sms);
  if (rc != PKV_OK) return rc;
  const int32_t ns = chunk ? num_seqs : 0, mq = chunk ? max_q_len : 0;
  if (workspace_bytes < pkv::mixed_workspace_bytes(ns, mq, dec_batch, dec_max_pages_per_seq, sms))
    return PKV_ERR_WORKSPACE_TOO_SMALL;
  const pkv::MixedDecode dec = {dec_q, dec_block_table, dec_seq_lens, dec_out, dec_batch, dec_max_pages_per_seq};
  return pkv::launch_prefill(chunk ? q : nullptr, k_pages, v_pages, block_table, prefix_lens, cu_q_lens, ns,
                             chunk ? total_q : 0, out, scale, desc->num_q_heads, desc->num_kv_heads, desc->head_dim,
                             max_pages_per_seq, mq, desc->num_pages, workspace, reinterpret_cast<cudaStream_t>(stream),
                             dec_batch > 0 ? &dec : nullptr);
}

int pkv_rope_table(float* table, int32_t max_pos, int32_t head_dim, double theta, pkv_stream_t stream) {
  if (table == nullptr) return PKV_ERR_NULL_ARG;
  if (max_pos < 1 || head_dim < 2 || head_dim > 1024 || (head_dim % 2) != 0 || !(theta > 0.0))
    return PKV_ERR_BAD_SHAPE;
  if (!aligned16(table)) return PKV_ERR_MISALIGNED;
  int sms = 0;
  const int rc = current_device(&sms);
  if (rc != PKV_OK) return rc;
  return pkv::launch_rope_table(table, max_pos, head_dim, theta, reinterpret_cast<cudaStream_t>(stream));
}

int pkv_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t limit_cycles, pkv_stream_t stream) {
  if (workspace == nullptr) return PKV_ERR_NULL_ARG;
  if (workspace_bytes < PKV_STATUS_BYTES) return PKV_ERR_WORKSPACE_TOO_SMALL;
  if (limit_cycles < 0 || limit_cycles > (1LL << 32)) return PKV_ERR_BAD_SHAPE;
  int sms = 0;
  const int rc = current_device(&sms);
  if (rc != PKV_OK) return rc;
  return pkv::launch_wait_timeout_selftest(workspace, limit_cycles, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
