// decode_generic.cu -- decode attention for cache geometries other than the
// Qwen3 decoder's 16 query / 8 KV heads of dimension 128 (decode.cu serves that
// one): G = num_q_heads / num_kv_heads query heads per KV head with G from 1 to
// 8, head_dim 64 or 128, any number of KV heads, page size 16. A group of 3, 5,
// 6 or 7 heads runs in the kernel for 4 or 8 with the extra query rows zero and
// their outputs not written.
//
// The operation is the one of decode.cu (PagedAttention decoding, "FunASR vLLM
// Inference Engine Guide", section 2): for every request and query head, the
// softmax-weighted mean of the value rows over the cached positions, scores
// scale * <q, k_j>. The pages name other backbones for the same decoder slot
// (Llama-style and larger Qwen3 / OLMo / SmolLM decoders) without their head
// counts, so this path exists to serve whatever geometry the cache descriptor
// gives, at the price of a simpler schedule than decode.cu's.
//
// Schedule:
//  * The grid is (splits, KV heads, requests). CTA (s, h, b) takes pages
//    [s * pps, (s + 1) * pps) of request b, KV head h; pps and the number of
//    splits come from the host sizes (enough CTAs for two waves).
//    CTAs past a request's last page exit at once.
//  * Each of the 4 warps takes every 4th page of the split and keeps a ring of
//    its own (2 stages for head_dim 128, 3 for 64: three CTAs fit an SM): lane 0
//    issues the page's K and V tiles as 1-D bulk copies (cp.async.bulk)
//    completing on the stage's mbarrier, a ring's depth of pages ahead.
//  * Scores: kL = G * head_dim / 64 lanes per token (at least 2), so that each
//    lane keeps its slice of the G query rows (64 floats, pre-scaled by
//    scale * log2(e)) in registers; packed fp32 FMAs over the lane's 16-byte
//    chunks of the key row (in an order rotated by token, so the 32 lanes' reads
//    spread over all shared memory banks), for all G heads from one K read. A
//    transpose-reduce over the kL lanes (halve the heads each round, then sum
//    the copies) leaves each lane the full score of one (token, head). Online
//    softmax in the log2 domain with tokens past seq_len masked; p and the
//    rescale factors go through shared memory. Values: each lane owns
//    head_dim / 32 dims of every head.
//  * The warps' states are merged in shared memory. A request whose pages fit
//    one split writes the bf16 output; otherwise each split writes an fp32
//    record (o, m, l per head), counts itself in (fence, atomic), and the CTA
//    completing the count merges the request's records (log-sum-exp, in split
//    order) and resets the counter.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {
namespace {

constexpr int kGenWarps = 4;
constexpr int kGenThreads = kGenWarps * 32;
constexpr unsigned kGenFull = 0xffffffffu;

template <int G, int D>
struct Gen {
  static constexpr int kTile = kPageSize * D * 2;  // one (page, KV head) K or V tile
  static constexpr int kStage = 2 * kTile;
  static constexpr int kStages = D == 128 ? 2 : 3;   // per warp: 3 CTAs of 4 warps per SM either way
  static constexpr int kRing = kStages * kStage;     // per warp
  static constexpr int kChunks = D / 8;              // 16-byte chunks of a row
  // Score pass: kL lanes per token, so that a lane's slice of the G query rows is
  // 64 floats (kL = G * D / 64, at least 2); kTP tokens per pass, kNP passes per
  // page, kCH 16-byte chunks of the row per lane. kL >= G always.
  static constexpr int kL = G * D / 64 < 2 ? 2 : G * D / 64;
  static constexpr int kTP = 32 / kL;
  static constexpr int kNP = kPageSize / kTP;
  static constexpr int kCH = kChunks / kL;
  static constexpr int kDup = kL / G;                // lanes of a token holding the same head's score
  static_assert(kCH >= 1 && kNP >= 1 && kDup >= 1, "score pass layout");
  static constexpr int kLaneDims = D / 32;           // value dims per lane
  static constexpr int kRec = D + 2;                 // floats per head in a record: o[D], m, l
  static constexpr int kState = G * kRec;            // a warp's or a split's (o, m, l) of all G heads
  static_assert(kState * 4 <= kRing, "a warp's state fits its drained ring");
  // shared memory: rings | full barriers | q (fp32) | p buffers | flags | page ids
  static constexpr int kOffBars = kGenWarps * kRing;
  static constexpr int kOffQ = kOffBars + kGenWarps * kStages * 8;
  static constexpr int kOffP = kOffQ + G * D * 4;
  static constexpr int kOffFlag = kOffP + kGenWarps * (kPageSize + 1) * G * 8;
  static constexpr int kOffIds = kOffFlag + 16;
  static size_t smem_bytes(int pps) { return kOffIds + static_cast<size_t>(pps) * 4; }
};

struct GenArgs {
  const __nv_bfloat16* q;
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
  float* records;  // [batch][hkv][splits][G][D + 2]
};

template <int G, int D>
__global__ void __launch_bounds__(kGenThreads) decode_generic_kernel(const GenArgs a) {
  using S = Gen<G, D>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kOffBars);
  float* qs = reinterpret_cast<float*>(smem + S::kOffQ);
  int* flag = reinterpret_cast<int*>(smem + S::kOffFlag);  // [0] a wait failed, [1] this CTA merges
  int* ids = reinterpret_cast<int*>(smem + S::kOffIds);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int hq0 = h * a.gq;  // first query head of the group
  const int nq = a.hkv * a.gq;

  grid_dependency_wait();
  allow_dependents();

  int sl = __ldg(a.seq_lens + b);
  const int cap = a.max_pages * kPageSize;
  if (sl < 0 || sl > cap) {
    if (tid == 0 && s == 0 && h == 0) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
    sl = sl < 0 ? 0 : cap;
  }
  __nv_bfloat16* orow = a.out + (static_cast<size_t>(b) * nq + hq0) * D;
  if (sl == 0) {  // an empty request (graph-bucket padding): zero rows
    if (s == 0)
      for (int i = tid; i < a.gq * D; i += kGenThreads) orow[i] = __float2bfloat16_rn(0.f);
    return;
  }
  const int np = (sl + kPageSize - 1) / kPageSize;
  const int nsplit = (np + a.pps - 1) / a.pps;
  if (s >= nsplit) return;
  const int p0 = s * a.pps;
  const int p1 = p0 + a.pps < np ? p0 + a.pps : np;

  if (tid < kGenWarps * S::kStages) mbar_init(&full[tid], 1);
  if (tid == 0) flag[0] = 0;
  for (int i = tid; i < G * D; i += kGenThreads)  // padding heads (i / D >= gq) get zero rows
    qs[i] = i < a.gq * D ? __bfloat162float(a.q[(static_cast<size_t>(b) * nq + hq0) * D + i]) * a.qscale : 0.f;
  for (int p = p0 + tid; p < p1; p += kGenThreads) {
    int id = __ldg(a.block_table + static_cast<size_t>(b) * a.max_pages + p);
    if (id < 0 || id >= a.num_pages) {
      set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
      id = 0;  // reported, not read out of bounds
    }
    ids[p - p0] = id;
  }
  fence_barrier_init();
  __syncthreads();

  // ---- this warp's pages: p0 + warp, p0 + warp + 4, ...
  const int nw = p1 - p0 > warp ? (p1 - p0 - warp + kGenWarps - 1) / kGenWarps : 0;
  unsigned char* ring = smem + warp * S::kRing;
  uint64_t* wfull = full + warp * S::kStages;
  auto issue = [&](int i) {  // lane 0: page i of this warp into stage i % S::kStages
    const int id = ids[warp + i * kGenWarps];
    const size_t off = (static_cast<size_t>(id) * a.hkv + h) * (S::kTile / 2);
    unsigned char* dst = ring + (i % S::kStages) * S::kStage;
    mbar_arrive_expect_tx(&wfull[i % S::kStages], S::kStage);
    bulk_g2s(dst, a.k_pages + off, S::kTile, &wfull[i % S::kStages]);
    bulk_g2s(dst + S::kTile, a.v_pages + off, S::kTile, &wfull[i % S::kStages]);
  };
  if (lane == 0)
    for (int i = 0; i < S::kStages && i < nw; ++i) issue(i);

  // score-pass position of this lane: token slot i of a pass, part sp of the row
  const int i = lane / S::kL, sp = lane % S::kL;
  const int h_own = sp / S::kDup;  // head whose scores this lane holds after the reduce
  // the lane's query chunks (rotated by token slot, so that the 32 lanes' K reads
  // spread over all banks): chunk (k) = sp + kL * ((k + i) mod kCH), both as fp32 pairs
  float2 q2[S::kCH][4][G];
#pragma unroll
  for (int k = 0; k < S::kCH; ++k) {
    const int c = sp + S::kL * ((k + i) % S::kCH);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float4 qa = *reinterpret_cast<const float4*>(qs + g * D + c * 8);
      const float4 qb = *reinterpret_cast<const float4*>(qs + g * D + c * 8 + 4);
      q2[k][0][g] = make_float2(qa.x, qa.y);
      q2[k][1][g] = make_float2(qa.z, qa.w);
      q2[k][2][g] = make_float2(qb.x, qb.y);
      q2[k][3][g] = make_float2(qb.z, qb.w);
    }
  }
  // p of every (token, head) as the pair (p, p), then every head's rescale factor
  float2* pb = reinterpret_cast<float2*>(smem + S::kOffP) + warp * (kPageSize + 1) * G;
  float mrun = -CUDART_INF_F, lrun = 0.f;  // of head h_own
  float2 o[G][S::kLaneDims / 2];  // dims lane * kLaneDims .., in pairs
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int k = 0; k < S::kLaneDims / 2; ++k) o[g][k] = make_float2(0.f, 0.f);
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
    const int n_valid = rem < kPageSize ? rem : kPageSize;
    const unsigned char* kt = ring + st * S::kStage;
    const unsigned char* vt = kt + S::kTile;
    // ---- scores: pass ps covers tokens ps * kTP .. ; each lane ends with the score
    // of (token ps * kTP + i, head h_own) after a transpose-reduce over its kL lanes
    float sc[S::kNP];
#pragma unroll
    for (int ps = 0; ps < S::kNP; ++ps) {
      const int tok = ps * S::kTP + i;
      float2 acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < S::kCH; ++k) {
        const int c = sp + S::kL * ((k + i) % S::kCH);
        const uint4 u = *reinterpret_cast<const uint4*>(kt + tok * (D * 2) + c * 16);
        const float2 k0 = bf2_to_f2(u.x), k1 = bf2_to_f2(u.y), k2 = bf2_to_f2(u.z), k3 = bf2_to_f2(u.w);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          acc[g] = __ffma2_rn(q2[k][0][g], k0, acc[g]);
          acc[g] = __ffma2_rn(q2[k][1][g], k1, acc[g]);
          acc[g] = __ffma2_rn(q2[k][2][g], k2, acc[g]);
          acc[g] = __ffma2_rn(q2[k][3][g], k3, acc[g]);
        }
      }
      float v[G];
#pragma unroll
      for (int g = 0; g < G; ++g) v[g] = acc[g].x + acc[g].y;
      // halving rounds (masks kL/2, kL/4, .. down to kDup): keep one half of the heads,
      // send the other to the partner; then sum the kDup copies of the last one
#pragma unroll
      for (int r = 0; (G >> r) > 1; ++r) {
        const int m = S::kL >> (r + 1), n = G >> r;
        const bool up = (sp & m) != 0;
#pragma unroll
        for (int j = 0; j < n / 2; ++j) {
          const float send = up ? v[j] : v[j + n / 2];
          const float keep = up ? v[j + n / 2] : v[j];
          v[j] = keep + __shfl_xor_sync(kGenFull, send, m);
        }
      }
#pragma unroll
      for (int m = S::kDup / 2; m >= 1; m >>= 1) v[0] += __shfl_xor_sync(kGenFull, v[0], m);
      sc[ps] = tok < n_valid ? v[0] : -CUDART_INF_F;
    }
    // ---- online softmax of head h_own over the page's tokens (passes, then token slots)
    float mx = sc[0];
#pragma unroll
    for (int ps = 1; ps < S::kNP; ++ps) mx = fmaxf(mx, sc[ps]);
#pragma unroll
    for (int m = S::kL; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kGenFull, mx, m));
    const float mnew = fmaxf(mrun, mx);
    const float alpha = ex2(mrun - mnew);
    float psum = 0.f;
#pragma unroll
    for (int ps = 0; ps < S::kNP; ++ps) {
      const float p = ex2(sc[ps] - mnew);
      psum += p;
      if (sp % S::kDup == 0) pb[(ps * S::kTP + i) * G + h_own] = make_float2(p, p);
    }
#pragma unroll
    for (int m = S::kL; m < 32; m <<= 1) psum += __shfl_xor_sync(kGenFull, psum, m);
    lrun = lrun * alpha + psum;
    mrun = mnew;
    if (i == 0 && sp % S::kDup == 0) pb[kPageSize * G + h_own] = make_float2(alpha, alpha);
    __syncwarp();
    // ---- values: lane owns dims lane * kLaneDims .. of every head (packed pairs)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 al = pb[kPageSize * G + g];
#pragma unroll
      for (int k = 0; k < S::kLaneDims / 2; ++k) o[g][k] = __fmul2_rn(o[g][k], al);
    }
#pragma unroll
    for (int tt = 0; tt < kPageSize; ++tt) {
      if (tt < n_valid) {
        float2 vv[S::kLaneDims / 2];
        if constexpr (S::kLaneDims == 4) {
          const uint2 u = *reinterpret_cast<const uint2*>(vt + tt * (D * 2) + lane * 8);
          vv[0] = bf2_to_f2(u.x);
          vv[1] = bf2_to_f2(u.y);
        } else {
          vv[0] = bf2_to_f2(*reinterpret_cast<const uint32_t*>(vt + tt * (D * 2) + lane * 4));
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 p = pb[tt * G + g];
#pragma unroll
          for (int k = 0; k < S::kLaneDims / 2; ++k) o[g][k] = __ffma2_rn(p, vv[k], o[g][k]);
        }
      }
    }
    __syncwarp();  // the stage and the p buffer are free again
    if (lane == 0 && it + S::kStages < nw) issue(it + S::kStages);
  }

  // ---- CTA merge of the warp states (each in its own drained ring)
  float* wst = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int k = 0; k < S::kLaneDims / 2; ++k) {
      wst[g * S::kRec + lane * S::kLaneDims + 2 * k] = o[g][k].x;
      wst[g * S::kRec + lane * S::kLaneDims + 2 * k + 1] = o[g][k].y;
    }
  if (i == 0 && sp % S::kDup == 0) {  // one lane per head holds its m and l
    wst[h_own * S::kRec + D] = mrun;
    wst[h_own * S::kRec + D + 1] = lrun;
  }
  __syncthreads();
  if (flag[0] != 0) return;  // a wait failed: copies may still land, write nothing
  const bool whole = nsplit == 1;
  float* rec = a.records + ((static_cast<size_t>(b) * a.hkv + h) * a.splits + s) * S::kState;
  for (int e = tid; e < G * (D + 1); e += kGenThreads) {
    const int g = e / (D + 1), d = e % (D + 1);  // d == D: this head's m and l
    float m = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kGenWarps; ++w)
      m = fmaxf(m, reinterpret_cast<const float*>(smem + w * S::kRing)[g * S::kRec + D]);
    float l = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kGenWarps; ++w) {
      const float* r = reinterpret_cast<const float*>(smem + w * S::kRing) + g * S::kRec;
      const float sc = r[D] == -CUDART_INF_F ? 0.f : ex2(r[D] - m);  // warps without pages
      l += r[D + 1] * sc;
      if (d < D) acc += r[d] * sc;
    }
    if (whole) {
      if (d < D && g < a.gq) orow[g * D + d] = __float2bfloat16_rn(acc / l);
    } else if (d < D) {
      rec[g * S::kRec + d] = acc;
    } else {
      rec[g * S::kRec + D] = m;
      rec[g * S::kRec + D + 1] = l;
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
  const float* recs = a.records + (static_cast<size_t>(b) * a.hkv + h) * a.splits * S::kState;
  for (int e = tid; e < a.gq * D; e += kGenThreads) {
    const int g = e / D, d = e % D;
    float m = -CUDART_INF_F;
    for (int r = 0; r < nsplit; ++r) m = fmaxf(m, recs[r * S::kState + g * S::kRec + D]);
    float l = 0.f, acc = 0.f;
    for (int r = 0; r < nsplit; ++r) {
      const float* x = recs + r * S::kState + g * S::kRec;
      const float sc = ex2(x[D] - m);
      l += x[D + 1] * sc;
      acc += x[d] * sc;
    }
    orow[g * D + d] = __float2bfloat16_rn(acc / l);
  }
  if (tid == 0) *counter = 0;
}

// Splits per (request, KV head) and pages per split for the host sizes: enough
// CTAs to fill the GPU twice at the resident CTAs per SM the shape allows, with
// splits of at least 8 pages.
template <int G, int D>
void plan(int batch, int hkv, int max_pages, int num_sms, int& splits, int& pps) {
  const size_t per_sm = 227 * 1024;
  const int resident = static_cast<int>(per_sm / (Gen<G, D>::smem_bytes(1) + 1024));
  // two waves of CTAs, splits of at least 8 pages (fewer records for short requests)
  const long long want = 2LL * num_sms * (resident > 0 ? resident : 1);
  const long long pairs = static_cast<long long>(batch) * hkv;
  long long sp = (want + pairs - 1) / pairs;
  if (sp > (max_pages + 7) / 8) sp = (max_pages + 7) / 8;
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
  off += static_cast<size_t>(batch) * hkv * splits * Gen<G, D>::kState * 4;
  return off;
}

template <int G, int D>
int gen_launch(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
               const int32_t* seq_lens, void* out, float scale, int batch, int hkv, int gq, int max_pages,
               int num_pages, void* workspace, int num_sms, cudaStream_t stream) {
  int splits = 1, pps = 1;
  plan<G, D>(batch, hkv, max_pages, num_sms, splits, pps);
  const size_t smem = Gen<G, D>::smem_bytes(pps);
  if (smem > 227 * 1024) return PKV_ERR_UNSUPPORTED;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(decode_generic_kernel<G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  GenArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
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
  return launch_pdl(decode_generic_kernel<G, D>, grid, dim3(kGenThreads), smem, stream, a) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // namespace

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

int launch_decode_generic(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                          const int32_t* seq_lens, void* out, float scale, int num_q_heads, int num_kv_heads,
                          int head_dim, int32_t batch, int32_t max_pages, int32_t num_pages, void* workspace,
                          int num_sms, cudaStream_t stream) {
  if (batch == 0) return PKV_OK;
  const int gq = num_q_heads / num_kv_heads;
  const int group = padded_group(gq);
#define PKV_GEN_RUN(G, D)                                                                                   \
  gen_launch<G, D>(q, k_pages, v_pages, block_table, seq_lens, out, scale, batch, num_kv_heads, gq, max_pages, \
                   num_pages, workspace, num_sms, stream)
  PKV_GEN_DISPATCH(PKV_GEN_RUN)
#undef PKV_GEN_RUN
  return PKV_ERR_UNSUPPORTED;
}

#undef PKV_GEN_DISPATCH

}  // namespace pkv
