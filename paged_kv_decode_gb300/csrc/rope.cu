// rope.cu -- the cos/sin table of the rotary position embedding, built on the device.
//
// The decoder is a Qwen3-style causal LM with RoPE theta 1e6 ("Fun-ASR-Nano
// Native Runtime Design", section "Decoder And Prompt"); the pages name the
// embedding and theta only, and the rotate-half form of Qwen3 decoders is
// taken: dims i and i + head_dim/2 form a pair rotated by p * w_i,
// w_i = theta^(-2i / head_dim). Row p of the table holds cos(p w_i) for
// i < head_dim/2, then sin(p w_i), each evaluated in double and rounded to
// float once -- the table the RoPE decode call reads, built here so that a
// caller without a host-side numerics library can make it with one call.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) rope_table_kernel(float* table, int max_pos, int head_dim, double theta) {
  grid_dependency_wait();
  allow_dependents();
  const int half = head_dim / 2;
  const long long n = static_cast<long long>(max_pos) * half;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long p = e / half;
    const int i = static_cast<int>(e - p * half);
    const double w = pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(head_dim));
    const double ang = static_cast<double>(p) * w;
    double sn, cs;
    sincos(ang, &sn, &cs);
    table[p * head_dim + i] = __double2float_rn(cs);
    table[p * head_dim + half + i] = __double2float_rn(sn);
  }
}

}  // namespace

int launch_rope_table(float* table, int32_t max_pos, int32_t head_dim, double theta, cudaStream_t stream) {
  const long long n = static_cast<long long>(max_pos) * (head_dim / 2);
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, table,
                    static_cast<int>(max_pos), static_cast<int>(head_dim), theta) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // namespace pkv
