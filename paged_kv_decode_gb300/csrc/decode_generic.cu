// decode_generic.cu -- decode attention for cache geometries other than the
// Qwen3 decoder's 16 query / 8 KV heads of dimension 128 (decode.cu serves that
// one): G = num_q_heads / num_kv_heads query heads per KV head with G in
// {1, 2, 4, 8}, head_dim 64 or 128, any number of KV heads, page size 16.
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
//    splits come from the host sizes (enough CTAs to fill the GPU twice).
//    CTAs past a request's last page exit at once.
//  * Each of the 4 warps takes every 4th page of the split and keeps a 3-stage
//    ring of its own: lane 0 issues the page's K and V tiles as 1-D bulk copies
//    (cp.async.bulk) completing on the stage's mbarrier, three pages ahead.
//  * Scores: two lanes per token, each over half the row's 16-byte chunks (in
//    an order rotated by token, so the 32 lanes' reads spread over all shared
//    memory banks), for all G query heads of the group from one K read; the
//    query rows sit in shared memory as fp32, pre-scaled by scale * log2(e).
//    Online softmax in the log2 domain with tokens past seq_len masked.
//    Values: each lane owns head_dim / 32 dims of every head.
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
constexpr int kGenStages = 3;
constexpr unsigned kGenFull = 0xffffffffu;

template <int G, int D>
struct Gen {
  static constexpr int kTile = kPageSize * D * 2;  // one (page, KV head) K or V tile
  static constexpr int kStage = 2 * kTile;
  static constexpr int kRing = kGenStages * kStage;  // per warp
  static constexpr int kChunks = D / 8;              // 16-byte chunks of a row
  static constexpr int kLaneChunks = kChunks / 2;    // per lane (two lanes per token)
  static constexpr int kLaneDims = D / 32;           // value dims per lane
  static constexpr int kRec = D + 2;                 // floats per head in a record: o[D], m, l
  static constexpr int kState = G * kRec;            // a warp's or a split's (o, m, l) of all G heads
  static_assert(kState * 4 <= kRing, "a warp's state fits its drained ring");
  // shared memory: rings | full barriers | q (fp32) | p buffers | flags | page ids
  static constexpr int kOffBars = kGenWarps * kRing;
  static constexpr int kOffQ = kOffBars + kGenWarps * kGenStages * 8;
  static constexpr int kOffP = kOffQ + G * D * 4;
  static constexpr int kOffFlag = kOffP + kGenWarps * kPageSize * G * 4;
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
  const int hq0 = h * G;  // first query head of the group
  const int nq = a.hkv * G;

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
      for (int i = tid; i < G * D; i += kGenThreads) orow[i] = __float2bfloat16_rn(0.f);
    return;
  }
  const int np = (sl + kPageSize - 1) / kPageSize;
  const int nsplit = (np + a.pps - 1) / a.pps;
  if (s >= nsplit) return;
  const int p0 = s * a.pps;
  const int p1 = p0 + a.pps < np ? p0 + a.pps : np;

  if (tid < kGenWarps * kGenStages) mbar_init(&full[tid], 1);
  if (tid == 0) flag[0] = 0;
  for (int i = tid; i < G * D; i += kGenThreads)
    qs[i] = __bfloat162float(a.q[(static_cast<size_t>(b) * nq + hq0) * D + i]) * a.qscale;
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
  uint64_t* wfull = full + warp * kGenStages;
  auto issue = [&](int i) {  // lane 0: page i of this warp into stage i % kGenStages
    const int id = ids[warp + i * kGenWarps];
    const size_t off = (static_cast<size_t>(id) * a.hkv + h) * (S::kTile / 2);
    unsigned char* dst = ring + (i % kGenStages) * S::kStage;
    mbar_arrive_expect_tx(&wfull[i % kGenStages], S::kStage);
    bulk_g2s(dst, a.k_pages + off, S::kTile, &wfull[i % kGenStages]);
    bulk_g2s(dst + S::kTile, a.v_pages + off, S::kTile, &wfull[i % kGenStages]);
  };
  if (lane == 0)
    for (int i = 0; i < kGenStages && i < nw; ++i) issue(i);

  const int t = lane >> 1, half = lane & 1;
  float* pb = reinterpret_cast<float*>(smem + S::kOffP) + warp * kPageSize * G;  // [token][head]
  float mrun[G], lrun[G], o[G][S::kLaneDims];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    mrun[g] = -CUDART_INF_F;
    lrun[g] = 0.f;
#pragma unroll
    for (int k = 0; k < S::kLaneDims; ++k) o[g][k] = 0.f;
  }
  bool failed = false;
  for (int i = 0; i < nw && !failed; ++i) {
    const int st = i % kGenStages;
    const bool ok = mbar_wait_bounded(&wfull[st], static_cast<uint32_t>(i / kGenStages) & 1u);
    failed = __any_sync(kGenFull, !ok);
    if (failed) {
      if (lane == 0) {
        set_status(a.status, PKV_ERR_DEVICE_TIMEOUT);
        flag[0] = 1;
      }
      break;
    }
    const int page = p0 + warp + i * kGenWarps;
    const int rem = sl - page * kPageSize;
    const int n_valid = rem < kPageSize ? rem : kPageSize;
    const unsigned char* kt = ring + st * S::kStage;
    const unsigned char* vt = kt + S::kTile;
    // scores of token t for the G heads, from half of the row's chunks
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll
    for (int j = 0; j < S::kLaneChunks; ++j) {
      const int c = 2 * ((j + t) % S::kLaneChunks) + half;
      const uint4 u = *reinterpret_cast<const uint4*>(kt + t * (D * 2) + c * 16);
      const float2 k0 = bf2_to_f2(u.x), k1 = bf2_to_f2(u.y), k2 = bf2_to_f2(u.z), k3 = bf2_to_f2(u.w);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4 qa = *reinterpret_cast<const float4*>(qs + g * D + c * 8);
        const float4 qb = *reinterpret_cast<const float4*>(qs + g * D + c * 8 + 4);
        acc[g] = fmaf(qa.x, k0.x, acc[g]);
        acc[g] = fmaf(qa.y, k0.y, acc[g]);
        acc[g] = fmaf(qa.z, k1.x, acc[g]);
        acc[g] = fmaf(qa.w, k1.y, acc[g]);
        acc[g] = fmaf(qb.x, k2.x, acc[g]);
        acc[g] = fmaf(qb.y, k2.y, acc[g]);
        acc[g] = fmaf(qb.z, k3.x, acc[g]);
        acc[g] = fmaf(qb.w, k3.y, acc[g]);
      }
    }
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float sc = acc[g] + __shfl_xor_sync(kGenFull, acc[g], 1);
      if (t >= n_valid) sc = -CUDART_INF_F;
      float mx = sc;
#pragma unroll
      for (int x = 2; x < 32; x <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kGenFull, mx, x));
      const float mnew = fmaxf(mrun[g], mx);
      alpha[g] = ex2(mrun[g] - mnew);
      const float p = ex2(sc - mnew);
      float ps = p;
#pragma unroll
      for (int x = 2; x < 32; x <<= 1) ps += __shfl_xor_sync(kGenFull, ps, x);
      lrun[g] = lrun[g] * alpha[g] + ps;
      mrun[g] = mnew;
      if (half == 0) pb[t * G + g] = p;
    }
    __syncwarp();
    // values: lane owns dims lane * kLaneDims .. of every head
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int k = 0; k < S::kLaneDims; ++k) o[g][k] *= alpha[g];
    for (int tt = 0; tt < n_valid; ++tt) {
      float v[S::kLaneDims];
      if constexpr (S::kLaneDims == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(vt + tt * (D * 2) + lane * 8);
        const float2 a0 = bf2_to_f2(u.x), a1 = bf2_to_f2(u.y);
        v[0] = a0.x, v[1] = a0.y, v[2] = a1.x, v[3] = a1.y;
      } else {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(vt + tt * (D * 2) + lane * 4);
        const float2 a0 = bf2_to_f2(u);
        v[0] = a0.x, v[1] = a0.y;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = pb[tt * G + g];
#pragma unroll
        for (int k = 0; k < S::kLaneDims; ++k) o[g][k] = fmaf(p, v[k], o[g][k]);
      }
    }
    __syncwarp();  // the stage and the p buffer are free again
    if (lane == 0 && i + kGenStages < nw) issue(i + kGenStages);
  }

  // ---- CTA merge of the warp states (each in its own drained ring)
  float* wst = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int k = 0; k < S::kLaneDims; ++k) wst[g * S::kRec + lane * S::kLaneDims + k] = o[g][k];
    if (lane == 0) {
      wst[g * S::kRec + D] = mrun[g];
      wst[g * S::kRec + D + 1] = lrun[g];
    }
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
      if (d < D) orow[g * D + d] = __float2bfloat16_rn(acc / l);
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
  for (int e = tid; e < G * D; e += kGenThreads) {
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
// CTAs to fill the GPU twice at the resident CTAs per SM the shape allows.
template <int G, int D>
void plan(int batch, int hkv, int max_pages, int num_sms, int& splits, int& pps) {
  const size_t per_sm = 227 * 1024;
  const int resident = static_cast<int>(per_sm / (Gen<G, D>::smem_bytes(1) + 1024));
  const long long want = 2LL * num_sms * (resident > 0 ? resident : 1);
  const long long pairs = static_cast<long long>(batch) * hkv;
  long long sp = (want + pairs - 1) / pairs;
  if (sp > max_pages) sp = max_pages;
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
               const int32_t* seq_lens, void* out, float scale, int batch, int hkv, int max_pages, int num_pages,
               void* workspace, int num_sms, cudaStream_t stream) {
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
  return (g == 1 || g == 2 || g == 4 || g == 8) && (head_dim == 64 || head_dim == 128);
}

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
  const int group = num_q_heads / num_kv_heads;
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
  const int group = num_q_heads / num_kv_heads;
#define PKV_GEN_RUN(G, D)                                                                                        \
  gen_launch<G, D>(q, k_pages, v_pages, block_table, seq_lens, out, scale, batch, num_kv_heads, max_pages, num_pages, \
                   workspace, num_sms, stream)
  PKV_GEN_DISPATCH(PKV_GEN_RUN)
#undef PKV_GEN_RUN
  return PKV_ERR_UNSUPPORTED;
}

#undef PKV_GEN_DISPATCH

}  // namespace pkv
