// decode_generic.cu -- decode attention for any cache geometry the descriptor
// may give: G = num_q_heads / num_kv_heads query heads per KV head with G from
// 1 to 8, head_dim 64 or 128, any number of KV heads, page size 16 (decode.cu
// keeps its own tuned kernel for the Qwen3 decoder's 16 query / 8 KV heads of
// dimension 128). A group of 3, 5, 6 or 7 heads runs in the kernel for 4 or 8,
// the extra query rows zero and their outputs not written.
//
// The operation is the one of decode.cu (PagedAttention decoding, "FunASR vLLM
// Inference Engine Guide", section 2): for every request and query head, the
// softmax-weighted mean of the value rows over the cached positions, scores
// scale * <q, k_j>. The pages name other backbones for the same decoder slot
// (Llama-style and larger Qwen3 / OLMo / SmolLM decoders) without their head
// counts, so this path serves whatever geometry the cache descriptor gives.
//
// Arithmetic: both products of a page are warp-level bf16 tensor-core MMAs
// (mma.sync m16n8k16, fp32 accumulation), about 100 warp instructions per page
// for any group up to 8 heads, where CUDA-core score and value passes need up
// to 1000 and run out of issue slots long before HBM does:
//  * scores, transposed: S^T[16 tokens][8 heads] = K[16][D] * Q^T[D][8], one MMA
//    per 16 dims (the query rows sit in registers as the B operand, rows past
//    the group zero);
//  * softmax in registers: a lane holds tokens r and r + 8 of heads 2c, 2c + 1
//    (r = lane / 4, c = lane % 4), so a head's page max takes three shuffles;
//    p is rounded to bf16 for the value product, and the running sum adds the
//    rounded p, so the output is an exact convex combination of value rows;
//  * values, transposed: O^T[D][8] += V^T[D][16] * P^T[16][8], one MMA per 16
//    dims; movmatrix turns the score accumulator's (token, head) pairs into
//    the (head, token) pairs the B operand wants, and the rescale factors of
//    the online softmax apply to the lane's own accumulator columns.
// The per-page contraction (16 tokens x at most 8 heads x head_dim) is far below
// the smallest tcgen05 tile (64 rows), and the softmax sits between the two
// products of every page, so the warp-level MMA with S and P in registers is
// the fitting unit here; the prefill kernel, whose tiles are 128 x 128, uses
// tcgen05 and TMEM.
//
// Schedule:
//  * The grid is (splits, KV heads, requests). CTA (s, h, b) takes pages
//    [s * pps, (s + 1) * pps) of request b, KV head h; pps and the number of
//    splits come from the host sizes (one wave of CTAs: every SM holds all of
//    its CTAs from the start), with splits of at least 8 pages. CTAs past a
//    request's last page exit at once.
//  * Each of the 4 warps takes every 4th page of the split and keeps a ring of
//    its own (2 stages for head_dim 128, 3 for 64); lane 0 issues the page's K
//    and V tiles a ring's depth ahead as tiled TMA copies (one 16-row box of
//    128 bytes per 64 dims) with 128-byte swizzle, so the ldmatrix reads of
//    eight token rows at the same dims hit eight different bank groups. Tokens
//    past seq_len are masked in the scores and in the value operand's registers
//    (unused slots may hold NaN).
//  * The warps' states are merged in shared memory. A request whose pages fit
//    one split writes the bf16 output; otherwise each split writes an fp32
//    record (o, m, l per head), counts itself in (fence, atomic), and the CTA
//    completing the count merges the request's records (log-sum-exp) and
//    resets the counter.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_kernels.h"
#include "pkv_mma.cuh"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kGenWarps = 4;
constexpr int kGenThreads = kGenWarps * 32;
constexpr unsigned kGenFull = 0xffffffffu;

// Shared memory of a CTA: the warps' rings | full barriers | flags | page ids of the split.
template <int G, int D>
struct Lay {
  static constexpr int kTile = kPageSize * D * 2;  // one (page, KV head) K or V tile: D / 64 swizzled boxes
  static constexpr int kStage = 2 * kTile;
  static constexpr int kStages = D == 128 ? 2 : 3;  // per warp: 3 (head_dim 128) or 4 (64) CTAs per SM
  static constexpr int kRing = kStages * kStage;   // per warp; a multiple of 1024 bytes
  static constexpr int kKS = D / 16;               // 16-dim steps of both products
  static constexpr int kRec = D + 4;               // floats per head in a state or record: o[D], m, l, 2 pad
  static constexpr int kState = G * kRec;
  static_assert(kState * 4 <= kRing, "a warp's state fits its drained ring");
  static_assert(G <= 8, "one 8-column MMA tile of heads");
  static constexpr int kOffBars = kGenWarps * kRing;
  static constexpr int kOffFlag = kOffBars + kGenWarps * kStages * 8;
  static constexpr int kOffIds = kOffFlag + 16;
  static size_t smem_bytes(int pps) { return 1024 + kOffIds + static_cast<size_t>(pps) * 4; }
};

struct GenArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;  // fused append: [batch][hkv][D], the new token's rows (kernel kFused only)
  const __nv_bfloat16* v_new;
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  const int* block_table;
  const int* seq_lens;
  __nv_bfloat16* out;
  float qscale;  // scale * log2(e)
  int max_pages;
  int num_pages;
  int hkv;
  int gq;      // query heads per KV head (<= G; the rest of the G are padding)
  int pps;     // pages per split
  int splits;  // splits per (request, KV head) in the records
  int* status;
  int* counters;   // [batch][hkv], zero between calls
  float* records;  // [batch][hkv][splits][G][D + 4]
  int early;       // copy pages before the grid dependency (the caller's promise: the predecessor writes
                   // neither the pools nor the block table nor the lengths)
  const float* rope;  // fused append only, optional: cos/sin table [rope_max_pos][D] (rotary embedding)
  int rope_max_pos;
};

// Rotary embedding of 8 dims of the new key row (16-byte chunk ch of D / 8): the rotate-half form,
// dims i and i + D / 2 a pair rotated by the table row's angle for i, in fp32 as
// y1 = fma(x1, c, -(x2 s)) and y2 = fma(x2, c, x1 s) with each product rounded first, then rounded
// to bf16 (ties to even), the operation order the tuned kernel and the header state.
template <int D>
__device__ __forceinline__ uint4 rope_key_chunk(const __nv_bfloat16* krow, int ch, const float* cs) {
  constexpr int kHalfChunks = D / 16;
  const bool first = ch < kHalfChunks;  // this chunk holds x1 of its pairs, else x2
  const int pch = first ? ch + kHalfChunks : ch - kHalfChunks;
  const uint4 own = __ldg(reinterpret_cast<const uint4*>(krow) + ch);
  const uint4 par = __ldg(reinterpret_cast<const uint4*>(krow) + pch);
  const uint32_t ow[4] = {own.x, own.y, own.z, own.w}, pw[4] = {par.x, par.y, par.z, par.w};
  const int i0 = 8 * (first ? ch : pch);  // pair index of the chunk's first dim
  uint32_t res[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 xo = bf2_to_f2(ow[e]), xp = bf2_to_f2(pw[e]);
    const int i = i0 + 2 * e;
    const float c0 = __ldg(cs + i), c1 = __ldg(cs + i + 1);
    const float s0 = __ldg(cs + D / 2 + i), s1 = __ldg(cs + D / 2 + i + 1);
    float y0, y1;
    if (first) {
      y0 = __fmaf_rn(xo.x, c0, -__fmul_rn(xp.x, s0));
      y1 = __fmaf_rn(xo.y, c1, -__fmul_rn(xp.y, s1));
    } else {
      y0 = __fmaf_rn(xo.x, c0, __fmul_rn(xp.x, s0));
      y1 = __fmaf_rn(xo.y, c1, __fmul_rn(xp.y, s1));
    }
    res[e] = pack_bf16x2(y0, y1);
  }
  return make_uint4(res[0], res[1], res[2], res[3]);
}

// Log-sum-exp merge of the nrec records of one (request, KV head) into its bf16
// output rows, by the whole CTA. rec_at(r): record r, rows [G][D + 4] of o[D],
// m, l. Every (m, l) is read at once; one warp per head turns the m into
// weights (kept in `scratch`, 2 * nrec * G + G floats of shared memory); then
// the o rows are summed as float4 with several records in flight.
template <int G, int D, class RecAt>
__device__ __forceinline__ void merge_records(RecAt rec_at, int nrec, int gq, float* scratch, __nv_bfloat16* orow) {
  constexpr int kRec = D + 4;
  const int tid = threadIdx.x;
  float* wgt = scratch;            // [nrec][G]: m, then the weight
  float* lsp = wgt + nrec * G;     // [nrec][G]: l
  float* inv = lsp + nrec * G;     // [G]: 1 / merged l
  for (int e = tid; e < nrec * G; e += kGenThreads) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(rec_at(e / G) + (e % G) * kRec + D));
    wgt[e] = ml.x;
    lsp[e] = ml.y;
  }
  __syncthreads();
  {
    const int warp = tid >> 5, lane = tid & 31;
    for (int g = warp; g < gq; g += kGenWarps) {
      float m = -CUDART_INF_F;
      for (int r = lane; r < nrec; r += 32) m = fmaxf(m, wgt[r * G + g]);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float l = 0.f;
      for (int r = lane; r < nrec; r += 32) {
        const float w = ex2(wgt[r * G + g] - m);  // every record holds at least one token
        wgt[r * G + g] = w;
        l += lsp[r * G + g] * w;
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) inv[g] = 1.f / l;
    }
  }
  __syncthreads();
  for (int e = tid; e < gq * (D / 4); e += kGenThreads) {
    const int g = e / (D / 4), d = (e % (D / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < nrec; ++r) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(rec_at(r) + g * kRec + d));
      const float w = wgt[r * G + g];
      acc.x += v.x * w;
      acc.y += v.y * w;
      acc.z += v.z * w;
      acc.w += v.w * w;
    }
    const float il = inv[g];
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * il, acc.y * il);
    packed.y = pack_bf16x2(acc.z * il, acc.w * il);
    *reinterpret_cast<uint2*>(orow + g * D + d) = packed;
  }
}

// The end of a split, once each warp has left its (o, m, l) of the G heads at
// the start of its drained ring (ring w at rings + w * kRingBytes, layout
// [G][D + 4]): merge the warps' states; a request whose pages fit one split
// writes its bf16 output, otherwise the split writes its fp32 record, counts
// itself in (fence, atomic), and the CTA completing the count merges the
// request's records (log-sum-exp, in split order) and resets the counter.
template <int G, int D, int kRingBytes>
__device__ __forceinline__ void finish_split(const GenArgs& a, const unsigned char* rings, int* flag, int b, int h,
                                             int s, int nsplit, __nv_bfloat16* orow) {
  constexpr int kRec = D + 4, kState = G * kRec;  // rows o[D], m, l, 2 pad: 16-byte aligned
  const int tid = threadIdx.x;
  __syncthreads();
  if (flag[0] != 0) return;  // a wait failed: copies may still land, write nothing
  const bool whole = nsplit == 1;
  float* rec = a.records + ((static_cast<size_t>(b) * a.hkv + h) * a.splits + s) * kState;
  for (int e = tid; e < G * (D + 1); e += kGenThreads) {
    const int g = e / (D + 1), d = e % (D + 1);  // d == D: this head's m and l
    float m = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kGenWarps; ++w)
      m = fmaxf(m, reinterpret_cast<const float*>(rings + w * kRingBytes)[g * kRec + D]);
    float l = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kGenWarps; ++w) {
      const float* r = reinterpret_cast<const float*>(rings + w * kRingBytes) + g * kRec;
      const float sc = r[D] == -CUDART_INF_F ? 0.f : ex2(r[D] - m);  // warps without pages
      l += r[D + 1] * sc;
      if (d < D) acc += r[d] * sc;
    }
    if (whole) {
      if (d < D && g < a.gq) orow[g * D + d] = __float2bfloat16_rn(acc / l);
    } else if (d < D) {
      rec[g * kRec + d] = acc;
    } else {
      rec[g * kRec + D] = m;
      rec[g * kRec + D + 1] = l;
    }
  }
  if (whole) return;

  // ---- count this split in (release); the CTA completing the count merges (acquire)
  __syncthreads();
  int* counter = a.counters + static_cast<size_t>(b) * a.hkv + h;
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(counter, 1);
    __threadfence();
    flag[1] = old == nsplit - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!flag[1]) return;
  const float* recs = a.records + (static_cast<size_t>(b) * a.hkv + h) * a.splits * kState;
  merge_records<G, D>([&](int r) { return recs + static_cast<size_t>(r) * kState; }, nsplit, a.gq,
                      reinterpret_cast<float*>(const_cast<unsigned char*>(rings)), orow);
  if (tid == 0) *counter = 0;
}

template <int G, int D, bool kFused>
__global__ void __launch_bounds__(kGenThreads) decode_generic_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                 const __grid_constant__ CUtensorMap vmap,
                                                                 const GenArgs a) {
  using S = Lay<G, D>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // swizzle atoms need 1024
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kOffBars);
  int* flag = reinterpret_cast<int*>(smem + S::kOffFlag);  // [0] a wait failed, [1] this CTA merges
  int* ids = reinterpret_cast<int*>(smem + S::kOffIds);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int hq0 = h * a.gq;
  const int nq = a.hkv * a.gq;
  if (tid == 0) {  // descriptors ahead of the first copies
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }

  // Every argument buffer may come from the previous kernel in the stream, so the kernel waits
  // for it first -- except in early mode, where lengths, block table and pages are read and the
  // first copies issued while the predecessor finishes; each warp then waits before it reads
  // q / k_new / v_new or writes anything. Dependents are released only after a wait.
  bool waited = !a.early;
  auto wait_once = [&]() {
    if (!waited) {
      grid_dependency_wait();
      allow_dependents();
      waited = true;
    }
  };
  if (!a.early) {
    grid_dependency_wait();
    allow_dependents();
  }

  int sl = __ldg(a.seq_lens + b);
  const int cap = a.max_pages * kPageSize;
  if (sl < 0 || sl > cap) {
    if (tid == 0 && s == 0 && h == 0) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
    sl = sl < 0 ? 0 : cap;
  }
  __nv_bfloat16* orow = a.out + (static_cast<size_t>(b) * nq + hq0) * D;
  if (sl == 0) {
    wait_once();
    if (s == 0)
      for (int i = tid; i < a.gq * D; i += kGenThreads) orow[i] = __float2bfloat16_rn(0.f);
    return;
  }
  const int np = (sl + kPageSize - 1) / kPageSize;
  const int nsplit = (np + a.pps - 1) / a.pps;
  if (s >= nsplit) return;
  // the table row of the new token's position (the RoPE call)
  const float* cs = nullptr;
  if (kFused && a.rope != nullptr) {
    int pos = sl - 1;
    if (pos >= a.rope_max_pos) {  // past the table: reported, clamped to its last row
      if (tid == 0) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
      pos = a.rope_max_pos - 1;
    }
    cs = a.rope + static_cast<size_t>(pos) * D;
  }
  const int p0 = s * a.pps;
  const int p1 = p0 + a.pps < np ? p0 + a.pps : np;

  if (tid < kGenWarps * S::kStages) mbar_init(&full[tid], 1);
  if (tid == 0) flag[0] = 0;
  for (int p = p0 + tid; p < p1; p += kGenThreads) {
    int id = __ldg(a.block_table + static_cast<size_t>(b) * a.max_pages + p);
    if (id < 0 || id >= a.num_pages) {
      set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
      id = -1;  // reported; the page is read as page 0 and nothing is appended to it
    }
    ids[p - p0] = id;
  }
  fence_barrier_init();
  __syncthreads();

  const int nw = p1 - p0 > warp ? (p1 - p0 - warp + kGenWarps - 1) / kGenWarps : 0;
  unsigned char* ring = smem + warp * S::kRing;
  uint64_t* wfull = full + warp * S::kStages;
  auto issue = [&](int i) {  // whole warp: page i of this warp into stage i % kStages
    const int page = p0 + warp + i * kGenWarps;
    const int id = ids[page - p0];
    if (kFused && page == np - 1 && id >= 0) {
      // fused append: this page holds the request's new token; its K and V rows for head h are
      // written first (one 16-byte chunk per lane), then fenced before the warp's tensor copy
      wait_once();  // the new rows come from the predecessor
      constexpr int kRowChunks = D / 8;
      const size_t row = ((static_cast<size_t>(id) * a.hkv + h) * kPageSize + (sl - 1) % kPageSize) * D;
      const size_t src = (static_cast<size_t>(b) * a.hkv + h) * D;
      if (lane < 2 * kRowChunks) {
        const bool is_v = lane >= kRowChunks;
        const int ch = is_v ? lane - kRowChunks : lane;
        const uint4 x = (!is_v && cs != nullptr)
                            ? rope_key_chunk<D>(a.k_new + src, ch, cs)
                            : __ldg(reinterpret_cast<const uint4*>((is_v ? a.v_new : a.k_new) + src) + ch);
        reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(is_v ? a.v_pages : a.k_pages) + row)[ch] = x;
        fence_proxy_async_global();
      }
      __syncwarp();
    }
    if (lane == 0) {
      const int z = (id < 0 ? 0 : id) * a.hkv + h;  // tile index in the pool
      unsigned char* dst = ring + (i % S::kStages) * S::kStage;
      uint64_t* bar = &wfull[i % S::kStages];
      mbar_arrive_expect_tx(bar, S::kStage);
      tma_load_4d(dst, &kmap, 0, 0, 0, z, bar);  // the whole K tile (its D / 64 swizzled blocks)
      tma_load_4d(dst + S::kTile, &vmap, 0, 0, 0, z, bar);
    }
  };
  for (int i = 0; i < S::kStages && i < nw; ++i) issue(i);
  wait_once();  // q comes from the predecessor

  const int r = lane >> 2, c = lane & 3;  // fragment row and column pair
  // Q^T as the B operand: head r, dims 16 ks + 2c (+1) and 16 ks + 8 + 2c (+1)
  uint32_t qf[S::kKS][2];
  {
    const bool live = r < a.gq;
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(a.q + (static_cast<size_t>(b) * nq + hq0 + (live ? r : 0)) * D);
#pragma unroll
    for (int ks = 0; ks < S::kKS; ++ks) {
      qf[ks][0] = live ? __ldg(qrow + 8 * ks + c) : 0u;
      qf[ks][1] = live ? __ldg(qrow + 8 * ks + 4 + c) : 0u;
    }
    if (cs != nullptr) {
      // the RoPE call: rotate the query rows at the new token's position in fp32 (pairs (d, d + D/2) sit
      // in steps ks and ks + kKS/2 of the same lane), each product rounded first, then round to bf16 as
      // the score product's operand
#pragma unroll
      for (int ks = 0; ks < S::kKS / 2; ++ks)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = 16 * ks + 8 * e + 2 * c;
          const float2 cc = make_float2(__ldg(cs + d), __ldg(cs + d + 1));
          const float2 sn = make_float2(__ldg(cs + D / 2 + d), __ldg(cs + D / 2 + d + 1));
          const float2 lo = bf2_to_f2(qf[ks][e]), hi = bf2_to_f2(qf[ks + S::kKS / 2][e]);
          const float2 t1 = __fmul2_rn(hi, sn), t2 = __fmul2_rn(lo, sn);
          const float2 ylo = __ffma2_rn(lo, cc, make_float2(-t1.x, -t1.y));
          const float2 yhi = __ffma2_rn(hi, cc, t2);
          qf[ks][e] = pack_bf16x2(ylo.x, ylo.y);
          qf[ks + S::kKS / 2][e] = pack_bf16x2(yhi.x, yhi.y);
        }
    }
  }
  uint32_t koff[S::kKS], voff[S::kKS];
  mma_offsets<S::kKS>(koff, voff);

  float o[S::kKS][4];  // O^T: dims 16 ks + r (+8) x heads 2c, 2c + 1
#pragma unroll
  for (int ks = 0; ks < S::kKS; ++ks) o[ks][0] = o[ks][1] = o[ks][2] = o[ks][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F;  // running max of heads 2c, 2c + 1 (log2 domain)
  float l0 = 0.f, l1 = 0.f;                      // this lane's part of their running sums
  bool failed = false;
  for (int it = 0; it < nw && !failed; ++it) {
    const int st = it % S::kStages;
    const bool ok = mbar_wait_bounded(&wfull[st], static_cast<uint32_t>(it / S::kStages) & 1u);
    failed = __any_sync(kGenFull, !ok);
    if (failed) {
      if (lane == 0) {
        set_status(a.status, PKV_ERR_DEVICE_TIMEOUT);
        flag[0] = 1;
      }
      break;
    }
    const int page = p0 + warp + it * kGenWarps;
    const int rem = sl - page * kPageSize;
    const int nv = rem < kPageSize ? rem : kPageSize;
    const uint32_t kt = smem_u32(ring + st * S::kStage), vt = kt + S::kTile;

    mma_page<S::kKS>(kt, vt, koff, voff, qf, nv, a.qscale, o, m0, m1, l0, l1);
    __syncwarp();  // the stage is free again
    if (it + S::kStages < nw) issue(it + S::kStages);
  }

  // ---- this warp's state into its drained ring: [G][D + 4] as o, m, l
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    l0 += __shfl_xor_sync(kGenFull, l0, m);
    l1 += __shfl_xor_sync(kGenFull, l1, m);
  }
  float* wst = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int n = 2 * c + j;
    if (n < G) {
#pragma unroll
      for (int ks = 0; ks < S::kKS; ++ks) {
        wst[n * (D + 4) + 16 * ks + r] = o[ks][j];
        wst[n * (D + 4) + 16 * ks + r + 8] = o[ks][2 + j];
      }
      if (r == 0) {
        wst[n * (D + 4) + D] = j ? m1 : m0;
        wst[n * (D + 4) + D + 1] = j ? l1 : l0;
      }
    }
  }
  finish_split<G, D, S::kRing>(a, smem, flag, b, h, s, nsplit, orow);
}

// Splits per (request, KV head) and pages per split for the host sizes: enough
// CTAs to fill the GPU once at the resident CTAs per SM the shape allows, with
// splits of at least 8 pages and at most as many as the merging CTA can weigh
// in its drained rings.
template <int G, int D>
void plan(int batch, int hkv, int max_pages, int num_sms, int& splits, int& pps) {
  const size_t per_sm = 227 * 1024;
  const int resident = static_cast<int>(per_sm / (Lay<G, D>::smem_bytes(1) + 1024));
  // one wave of CTAs (each SM holds all of its CTAs from the start), splits of at least 8 pages
  // (fewer records for short requests)
  const long long want = 1LL * num_sms * (resident > 0 ? resident : 1);
  const long long pairs = static_cast<long long>(batch) * hkv;
  long long sp = (want + pairs - 1) / pairs;
  if (sp > (max_pages + 7) / 8) sp = (max_pages + 7) / 8;
  // the merging CTA keeps two floats per (split, head) in its drained rings
  constexpr int kMaxSplits = (kGenWarps * Lay<G, D>::kRing / 4 - G) / (2 * G);
  if (sp > kMaxSplits) sp = kMaxSplits;
  if (sp < 1) sp = 1;
  pps = static_cast<int>((max_pages + sp - 1) / sp);
  splits = (max_pages + pps - 1) / pps;
}

template <int G, int D>
size_t gen_workspace(int batch, int hkv, int max_pages, int num_sms) {
  int splits = 1, pps = 1;
  plan<G, D>(batch, hkv, max_pages, num_sms, splits, pps);
  size_t off = PKV_STATUS_BYTES;
  off += (static_cast<size_t>(batch) * hkv * 4 + 255) / 256 * 256;
  off += static_cast<size_t>(batch) * hkv * splits * G * (D + 4) * 4;  // records [G][D + 4]
  return off;
}

template <int G, int D>
int gen_launch(const void* q, const void* k_new, const void* v_new, const void* k_pages, const void* v_pages,
               const int32_t* block_table, const int32_t* seq_lens, const float* rope, int rope_max_pos, void* out,
               float scale, int batch, int hkv, int gq, int max_pages, int num_pages, void* workspace, int num_sms,
               cudaStream_t stream, uint32_t flags) {
  int splits = 1, pps = 1;
  plan<G, D>(batch, hkv, max_pages, num_sms, splits, pps);
  const size_t smem = Lay<G, D>::smem_bytes(pps);
  if (smem > 227 * 1024) return PKV_ERR_UNSUPPORTED;
  const bool fused = k_new != nullptr;
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, const GenArgs);
  const Kern kern = fused ? decode_generic_kernel<G, D, true> : decode_generic_kernel<G, D, false>;
  static bool attr_set[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !attr_set[dev][fused ? 1 : 0]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev][fused ? 1 : 0] = true;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  GenArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.early = (flags & PKV_DECODE_EARLY_PREFETCH) ? 1 : 0;
  a.rope = fused ? rope : nullptr;
  a.rope_max_pos = rope_max_pos;
  a.k_pages = static_cast<const __nv_bfloat16*>(k_pages);
  a.v_pages = static_cast<const __nv_bfloat16*>(v_pages);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.qscale = scale * kLog2e;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.hkv = hkv;
  a.gq = gq;
  a.pps = pps;
  a.splits = splits;
  a.status = reinterpret_cast<int*>(ws);
  a.counters = reinterpret_cast<int*>(ws + PKV_STATUS_BYTES);
  a.records = reinterpret_cast<float*>(ws + PKV_STATUS_BYTES + (static_cast<size_t>(batch) * hkv * 4 + 255) / 256 * 256);
  const dim3 grid(static_cast<unsigned>(splits), static_cast<unsigned>(hkv), static_cast<unsigned>(batch));
  CUtensorMap kmap, vmap;
  const int rc = encode_page_maps(k_pages, v_pages, D, num_pages, hkv, &kmap, &vmap);
  if (rc != PKV_OK) return rc;
  return launch_pdl(kern, grid, dim3(kGenThreads), smem, stream, kmap, vmap, a) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // namespace

// Tensor maps of the two pools for the tensor-core kernel: [tiles][16 rows][D]
// with tile = page * hkv + KV head, boxes of 64 dims x 16 rows (128-byte rows,
// 128-byte swizzle).
namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

int encode_page_maps(const void* k_pages, const void* v_pages, int head_dim, int num_pages, int hkv, CUtensorMap* kmap,
              CUtensorMap* vmap) {
  const long long tiles = static_cast<long long>(num_pages) * hkv;
  if (tiles > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // tile coordinates are 32-bit
  EncodeTiledFn enc = encoder();
  if (enc == nullptr) return PKV_ERR_CUDA;
  if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
  const cuuint32_t halves = static_cast<cuuint32_t>(head_dim / 64);
  // (dim within the half, row, half, tile): a tile's halves are 128 bytes apart inside each 2 * head_dim-byte row
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(kPageSize), halves, static_cast<cuuint64_t>(tiles)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(head_dim) * 2, 128,
                                 static_cast<cuuint64_t>(head_dim) * 2 * kPageSize};
  const cuuint32_t box[4] = {64, kPageSize, halves, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const void* pools[2] = {k_pages, v_pages};
  CUtensorMap* maps[2] = {kmap, vmap};
  for (int i = 0; i < 2; ++i)
    if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pools[i]), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
  return PKV_OK;
}

bool decode_generic_supported(int num_q_heads, int num_kv_heads, int head_dim, int page_size) {
  if (num_kv_heads < 1 || num_kv_heads > 65535 || page_size != kPageSize) return false;
  if (num_q_heads % num_kv_heads != 0) return false;
  const int g = num_q_heads / num_kv_heads;
  return g >= 1 && g <= 8 && (head_dim == 64 || head_dim == 128);
}

// The kernel's group size for g query heads per KV head: the next of 1, 2, 4, 8.
static int padded_group(int g) { return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8; }

#define PKV_GEN_DISPATCH(CALL)                     \
  switch (group * 1000 + head_dim) {               \
    case 1064: return CALL(1, 64);                 \
    case 1128: return CALL(1, 128);                \
    case 2064: return CALL(2, 64);                 \
    case 2128: return CALL(2, 128);                \
    case 4064: return CALL(4, 64);                 \
    case 4128: return CALL(4, 128);                \
    case 8064: return CALL(8, 64);                 \
    case 8128: return CALL(8, 128);                \
    default: break;                                \
  }

size_t decode_generic_workspace_bytes(int num_q_heads, int num_kv_heads, int head_dim, int32_t batch,
                                      int32_t max_pages, int num_sms) {
  const int group = padded_group(num_q_heads / num_kv_heads);
#define PKV_GEN_WS(G, D) gen_workspace<G, D>(batch, num_kv_heads, max_pages, num_sms)
  PKV_GEN_DISPATCH(PKV_GEN_WS)
#undef PKV_GEN_WS
  return 0;
}

int launch_decode_generic(const void* q, const void* k_new, const void* v_new, const void* k_pages,
                          const void* v_pages, const int32_t* block_table, const int32_t* seq_lens, const float* rope,
                          int32_t rope_max_pos, void* out, float scale, int num_q_heads, int num_kv_heads,
                          int head_dim, int32_t batch, int32_t max_pages, int32_t num_pages, void* workspace,
                          int num_sms, cudaStream_t stream, uint32_t flags) {
  if (batch == 0) return PKV_OK;
  if (rope != nullptr && k_new == nullptr) return PKV_ERR_NULL_ARG;
  const int gq = num_q_heads / num_kv_heads;
  const int group = padded_group(gq);
#define PKV_GEN_RUN(G, D)                                                                                    \
  gen_launch<G, D>(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, rope, rope_max_pos, out, scale,  \
                   batch, num_kv_heads, gq, max_pages, num_pages, workspace, num_sms, stream, flags)
  PKV_GEN_DISPATCH(PKV_GEN_RUN)
#undef PKV_GEN_RUN
  return PKV_ERR_UNSUPPORTED;
}

#undef PKV_GEN_DISPATCH

}  // namespace pkv
