// pkv_kernels.h -- internal launchers behind the C ABI (host side).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Rows of num_kv_heads x head_dim bf16 (head_dim a multiple of 8), page size 16.
int launch_append(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t n_tokens, void* k_pages,
                  void* v_pages, int32_t num_pages, int32_t num_kv_heads, int32_t head_dim, int* status, int num_sms,
                  cudaStream_t stream);

// Decode (decode.cu, decode_kernel.cuh): page size 16, head_dim 64 or 128, num_q_heads / num_kv_heads
// from 1 to 8. Workspace = [status header | counters (batch * kv heads) | records].
bool decode_supported(int num_q_heads, int num_kv_heads, int head_dim, int page_size);
size_t decode_workspace_bytes(int num_q_heads, int num_kv_heads, int head_dim, int32_t batch, int num_sms);
// k_new / v_new (nullable): fused append of each request's new token at position seq_lens[b] - 1.
// rope (nullable, needs k_new): cos/sin table [rope_max_pos][head_dim]; the new key row and the
// query rows are rotated at that position. flags: 0 or PKV_DECODE_EARLY_PREFETCH.
int launch_decode(const void* q, const void* k_new, const void* v_new, const void* k_pages, const void* v_pages,
                  const int32_t* block_table, const int32_t* seq_lens, const float* rope, int32_t rope_max_pos,
                  void* out, float scale, int num_q_heads, int num_kv_heads, int head_dim, int32_t batch,
                  int32_t max_pages, int32_t num_pages, void* workspace, int num_sms, cudaStream_t stream,
                  uint32_t flags);
int decode_max_batch();


// Rotary-embedding table (rope.cu): fp32 [max_pos][head_dim], row p = cos(p w_i) for i < head_dim / 2,
// then sin(p w_i), w_i = theta^(-2 i / head_dim), angles in double rounded to float once.
int launch_rope_table(float* table, int32_t max_pos, int32_t head_dim, double theta, cudaStream_t stream);

// Chunked prefill (prefill.cu): page size 16, head_dim 64 or 128, 1 to 8 query heads per KV head.
bool prefill_supported(int num_q_heads, int num_kv_heads, int head_dim, int page_size);
size_t prefill_workspace_bytes(int num_q_heads, int num_kv_heads, int head_dim, int32_t num_seqs, int32_t max_q_len,
                               int num_sms);
int prefill_max_seqs();
// The decode half of a mixed step (16/8/128 only): decode requests attended in the prefill launch.
struct MixedDecode {
  const void* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  int32_t batch;
  int32_t max_pages;
};
// Workspace of the mixed step: the prefill workspace, then the decode chunks' counters and records.
size_t mixed_workspace_bytes(int32_t num_seqs, int32_t max_q_len, int32_t dec_batch, int32_t dec_max_pages,
                             int num_sms);
// dec: nullptr for prefill alone; otherwise the launch also attends the decode requests (the mixed step).
int launch_prefill(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                   const int32_t* prefix_lens, const int32_t* cu_q_lens, int32_t num_seqs, int32_t total_q,
                   void* out, float scale, int num_q_heads, int num_kv_heads, int head_dim, int32_t max_pages,
                   int32_t max_q_len, int32_t num_pages, void* workspace, cudaStream_t stream,
                   const MixedDecode* dec = nullptr);

int launch_wait_timeout_selftest(void* workspace, long long limit_cycles, cudaStream_t stream);

}  // namespace pkv
