// pkv_mma.cuh -- warp-level bf16 tensor-core MMA step of a decode page, used by
// the decode kernel (decode_kernel.cuh) and the mixed step's decode CTAs
// (prefill.cu).
//
// A page of one (request, KV head) is 16 token rows of K and of V, each
// head_dim bf16 values, in shared memory as written by 128-byte-swizzled tiled
// TMA boxes (one box of 16 rows x 64 dims per 64 dims, 2 KiB, 1024-byte
// aligned). The step computes the scores of the 16 tokens for up to 8 query
// heads (S^T = K Q^T), updates the online softmax of the lane's two heads, and
// accumulates the values (O^T += V^T P^T), with mma.sync m16n8k16 (bf16
// operands, fp32 accumulators) and ldmatrix / movmatrix moving the operands.
// PTX forms as in the PTX ISA (ldmatrix, movmatrix, mma.sync).
#pragma once

#include <cuda.h>
#include <math_constants.h>
#include <stdint.h>

#include "pkv_device.cuh"

namespace pkv {

// Tensor maps of the two pools for the MMA kernels, over [page * hkv + KV head][16 rows][head_dim] bf16
// viewed as 4-D (64 dims, 16 rows, head_dim / 64 halves, tile), the halves' stride (128 bytes) below the
// rows' (2 * head_dim bytes). One box is a whole tile: coordinates (0, 0, 0, tile) copy it with one
// instruction into head_dim / 64 consecutive 2 KiB blocks of 16 rows x 64 dims, 128-byte swizzled (the
// layout swz() reads). PKV_ERR_UNSUPPORTED past 2^31 tiles.
int encode_page_maps(const void* k_pages, const void* v_pages, int head_dim, int num_pages, int hkv, CUtensorMap* kmap,
                     CUtensorMap* vmap);

// Byte offset of 16-byte chunk c of token row t in a tile written by the
// 128-byte swizzled TMA boxes: box c / 8 (kBox bytes apart, each 1024-byte
// aligned; 2 KiB when a page's boxes are back to back), row t of 128 bytes,
// chunk (c mod 8) XOR (t mod 8).
template <int kBox = 2048>
__device__ __forceinline__ uint32_t swz(int t, int c) {
  return static_cast<uint32_t>((c >> 3) * kBox + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// c += a * b, m16n8k16, bf16 operands, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// This lane's ldmatrix row addresses inside a page tile, per 16-dim step ks:
// K as the A operand of the score product (matrices: tokens 0-7 / 8-15 x the
// two 8-dim halves of the step), V, read transposed, as the A operand of the
// value product (the same four blocks in the order that operand wants). kBox:
// the distance between a page's 64-dim boxes.
template <int KS, int kBox = 2048>
__device__ __forceinline__ void mma_offsets(uint32_t (&koff)[KS], uint32_t (&voff)[KS]) {
  const int lane = threadIdx.x & 31, mi = lane >> 3, mr = lane & 7;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    koff[ks] = swz<kBox>(mr + ((mi & 1) << 3), 2 * ks + (mi >> 1));
    voff[ks] = swz<kBox>(mr + ((mi >> 1) << 3), 2 * ks + (mi & 1));
  }
}

// One page of the tensor-core path: the scores of its 16 tokens for the 8 head
// columns, the online-softmax update of this lane's two heads (2c, 2c + 1), and
// the value product. kt, vt: shared addresses of the page's swizzled K and V
// tiles; nv: its tokens before seq_len.
template <int KS>
__device__ __forceinline__ void mma_page(uint32_t kt, uint32_t vt, const uint32_t (&koff)[KS],
                                         const uint32_t (&voff)[KS], const uint32_t (&qf)[KS][2], int nv,
                                         float qscale, float (&o)[KS][4], float& m0, float& m1, float& l0,
                                         float& l1) {
  const int lane = threadIdx.x & 31, r = lane >> 2, c = lane & 3;
  // ---- scores (two accumulators: the k-steps form two dependent chains)
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t kf[4];
    ldsm4(kt + koff[ks], kf);
    if (ks & 1)
      mma_bf16(sb, kf, qf[ks][0], qf[ks][1]);
    else
      mma_bf16(sa, kf, qf[ks][0], qf[ks][1]);
  }
  const bool v0 = r < nv, v1 = r + 8 < nv;
  const float s00 = v0 ? (sa[0] + sb[0]) * qscale : -CUDART_INF_F;  // token r, head 2c
  const float s01 = v0 ? (sa[1] + sb[1]) * qscale : -CUDART_INF_F;  // token r, head 2c + 1
  const float s10 = v1 ? (sa[2] + sb[2]) * qscale : -CUDART_INF_F;  // token r + 8
  const float s11 = v1 ? (sa[3] + sb[3]) * qscale : -CUDART_INF_F;

  // ---- online softmax of heads 2c, 2c + 1 over the page's 16 tokens
  float x0 = fmaxf(s00, s10), x1 = fmaxf(s01, s11);
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, m));
    x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, m));
  }
  const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
  const uint32_t pk0 = pack_bf16x2(ex2(s00 - n0), ex2(s01 - n1));  // token r
  const uint32_t pk1 = pack_bf16x2(ex2(s10 - n0), ex2(s11 - n1));  // token r + 8
  const float2 q0 = bf2_to_f2(pk0), q1 = bf2_to_f2(pk1);
  if (__any_sync(0xffffffffu, n0 != m0 || n1 != m1)) {
    const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);  // 0 on the first page
    l0 *= al0;
    l1 *= al1;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      o[ks][0] *= al0;
      o[ks][1] *= al1;
      o[ks][2] *= al0;
      o[ks][3] *= al1;
    }
    m0 = n0;
    m1 = n1;
  }
  l0 += q0.x + q1.x;
  l1 += q0.y + q1.y;

  // ---- values: P^T as the B operand (head r, tokens 2c, 2c + 1 and 8 + 2c, 9 + 2c)
  const uint32_t pb0 = movm_t(pk0), pb1 = movm_t(pk1);
  uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;  // value rows past seq_len read as zero
  if (nv < kPageSize) {
    mlo = (2 * c < nv ? 0x0000ffffu : 0u) | (2 * c + 1 < nv ? 0xffff0000u : 0u);
    mhi = (2 * c + 8 < nv ? 0x0000ffffu : 0u) | (2 * c + 9 < nv ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t vf[4];
    ldsm4_t(vt + voff[ks], vf);
    vf[0] &= mlo;
    vf[1] &= mlo;
    vf[2] &= mhi;
    vf[3] &= mhi;
    mma_bf16(o[ks], vf, pb0, pb1);
  }
}

}  // namespace pkv
