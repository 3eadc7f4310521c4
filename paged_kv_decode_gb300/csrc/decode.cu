// decode.cu -- batched decode attention over the paged KV cache (split-KV).
//
// Source of the operation: PagedAttention decoding in the LLM engine
// ("FunASR vLLM Inference Engine Guide", section 2 "vLLM Engine Architecture");
// decode is where long-audio serving spends its time ("Optimizing ASR for
// 90-minute multi-speaker audio", section "Time spent: profiling").
//
// The op reads every cached K/V row once and does ~1 FMA per byte, so it is
// bound by HBM bandwidth. Design:
//
//  * Work is the list of (request, KV head, page) triples, ordered by request,
//    then KV head, then page. The kernel is persistent: gridDim.x CTAs (the SM
//    count times the CTAs resident per SM) each take an equal contiguous share
//    of that list, computed on the device from seq_lens, so the grid depends
//    only on host-known sizes (CUDA-graph friendly) and every CTA streams the
//    same number of pages whatever the length mix.
//  * A CTA's share is cut into pieces, one per (request, KV head) it touches.
//    Inside a piece its 4 warps take pages round-robin. Each warp owns a ring
//    of 3 shared-memory stages and fills them itself with 1-D bulk copies
//    (cp.async.bulk, one 4 KiB K tile and one 4 KiB V tile per page) that
//    complete on an mbarrier, so up to 24 KiB per warp is in flight.
//  * Both query heads of the GQA group are computed from one K/V read. Scores
//    use packed fp32 FMAs (two dims per instruction); the softmax is online in
//    the log2 domain (q pre-scaled by scale * log2 e); tokens past seq_len in
//    the last page are masked before they can touch the max or the sum, so
//    unused slots may hold anything, NaN included.
//  * At the end of a piece the warps merge through shared memory. A piece that
//    covers its whole (request, KV head) writes the bf16 output. Otherwise it
//    writes an fp32 partial (m, l, o) and bumps a per-(request, KV head)
//    counter; the CTA that brings the counter to the number of pieces merges
//    all partials (log-sum-exp) and resets the counter to zero.
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_kernels.h"

namespace pkv {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecRing = 3;
constexpr int kDecCtasPerSm = 2;
constexpr int kStageBytes = 2 * kTileBytes;  // K tile + V tile of one (page, KV head)
constexpr int kRec = kHeadDim + 4;           // floats per query-head record: m, l, pad, pad, o[128]
constexpr int kPieceFloats = kGroup * kRec;  // a partial record of one piece (both query heads)
constexpr int kMaxDecodeBatch = 2048;
constexpr unsigned kFull = 0xffffffffu;

constexpr int kSmemRing = kDecWarps * kDecRing * kStageBytes;
constexpr int kSmemBars = kDecWarps * kDecRing * 8;
constexpr int kMergeFloats = kDecWarps * kGroup * kRec;  // one buffer of warp records
constexpr int kSmemMerge = 2 * kMergeFloats * 4;         // double-buffered by piece parity
constexpr int kSmemPbuf = kDecWarps * kPageSize * 4 * 4; // per warp: [16 tokens][p0, p0, p1, p1]
constexpr int kSmemFlag = 16;
constexpr int kSmemFixed = kSmemRing + kSmemBars + kSmemMerge + kSmemPbuf + kSmemFlag;

static size_t decode_smem_bytes(int batch) { return kSmemFixed + static_cast<size_t>(2 * batch + 1) * 4; }

int decode_max_batch() { return kMaxDecodeBatch; }

struct DecodeArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  const int* block_table;
  const int* seq_lens;
  __nv_bfloat16* out;
  float qscale;  // scale * log2(e)
  int batch;
  int max_pages;
  int num_pages;
  int* status;
  int* counters;   // [batch * kKVHeads], zero between calls
  float* partials; // [2 * gridDim.x][kPieceFloats]
};

// A piece: pages [p0, p1) of KV head h of request b; flattened indices [fstart, fend).
struct Piece {
  int b, h, np, p0, p1;
  long long fstart, fend;
};

// Piece of the CTA share [.., hi) that starts at flattened index f.
// pref[b] = page-head triples of requests before b (pref[batch] = total).
__device__ __forceinline__ bool find_piece(long long f, long long hi, const int* pref, int batch, Piece& pc) {
  if (f >= hi) return false;
  int lo_b = 0, hi_b = batch - 1;
  while (lo_b < hi_b) {
    const int mid = (lo_b + hi_b + 1) >> 1;
    if (pref[mid] <= f) lo_b = mid; else hi_b = mid - 1;
  }
  pc.b = lo_b;
  pc.np = (pref[lo_b + 1] - pref[lo_b]) / kKVHeads;
  const long long off = f - pref[lo_b];
  pc.h = static_cast<int>(off / pc.np);
  pc.p0 = static_cast<int>(off % pc.np);
  const long long p1 = pc.p0 + (hi - f);
  pc.p1 = static_cast<int>(p1 < pc.np ? p1 : pc.np);
  pc.fstart = f;
  pc.fend = f + (pc.p1 - pc.p0);
  return true;
}

// CTA whose share [lo(c), lo(c+1)) contains flattened index f, with lo(c) = c * T / G.
__device__ __forceinline__ int cta_of(long long f, long long T, int G) {
  return static_cast<int>(((f + 1) * G + T - 1) / T - 1);
}
__device__ __forceinline__ long long share_lo(int c, long long T, int G) { return static_cast<long long>(c) * T / G; }

// V accumulation for the tokens of one half-warp; kChecked masks tokens >= n_valid.
template <bool kChecked>
__device__ __forceinline__ void pv_tokens(uint32_t vrow0, uint32_t prow0, int t0, int n_valid, float2 (&o)[2][4]) {
#pragma unroll
  for (int tt = 0; tt < 8; ++tt) {
    if (kChecked && t0 + tt >= n_valid) break;
    const uint4 u = lds128(vrow0 + tt * kRowBytes);
    const float4 pp = lds128f(prow0 + tt * 16);
    const float2 ph0 = make_float2(pp.x, pp.y);
    const float2 ph1 = make_float2(pp.z, pp.w);
    const float2 v0 = bf2_to_f2(u.x), v1 = bf2_to_f2(u.y), v2 = bf2_to_f2(u.z), v3 = bf2_to_f2(u.w);
    o[0][0] = __ffma2_rn(ph0, v0, o[0][0]);
    o[0][1] = __ffma2_rn(ph0, v1, o[0][1]);
    o[0][2] = __ffma2_rn(ph0, v2, o[0][2]);
    o[0][3] = __ffma2_rn(ph0, v3, o[0][3]);
    o[1][0] = __ffma2_rn(ph1, v0, o[1][0]);
    o[1][1] = __ffma2_rn(ph1, v1, o[1][1]);
    o[1][2] = __ffma2_rn(ph1, v2, o[1][2]);
    o[1][3] = __ffma2_rn(ph1, v3, o[1][3]);
  }
}

__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemRing);
  float* merge = reinterpret_cast<float*>(smem + kSmemRing + kSmemBars);
  float* pbuf = merge + 2 * kMergeFloats;
  int* flag = reinterpret_cast<int*>(pbuf + kDecWarps * kPageSize * 4);
  int* pref = flag + kSmemFlag / 4;
  int* sl = pref + a.batch + 1;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int batch = a.batch;

  if (tid < kDecWarps * kDecRing) mbar_init(&bars[tid], 1);

  // seq lens (clamped) and the exclusive prefix of page-head triples
  if (warp == 0) {
    int carry = 0;
    const int cap = a.max_pages * kPageSize;
    for (int base = 0; base < batch; base += 32) {
      const int b = base + lane;
      int s = 0;
      if (b < batch) {
        s = __ldg(a.seq_lens + b);
        if (s < 0 || s > cap) {
          set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
          s = s < 0 ? 0 : cap;
        }
        sl[b] = s;
      }
      const int v = ((s + kPageSize - 1) / kPageSize) * kKVHeads;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (b < batch) pref[b] = carry + x - v;
      carry += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) pref[batch] = carry;
  }
  fence_barrier_init();
  __syncthreads();

  // zero output rows of empty requests (graph-bucket padding)
  for (int b = blockIdx.x; b < batch; b += gridDim.x) {
    if (sl[b] == 0) {
      uint4* o = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(b) * kQHeads * kHeadDim);
      for (int i = tid; i < kQHeads * kHeadDim / 8; i += kDecThreads) o[i] = make_uint4(0, 0, 0, 0);
    }
  }

  // Only min(gridDim.x, T) CTAs take a share, so that every share is non-empty
  // and the CTAs between the first and last holder of a (request, KV head) all
  // hold a piece of it.
  const long long T = pref[batch];
  const int G = static_cast<int>(T < gridDim.x ? T : gridDim.x);
  if (static_cast<int>(blockIdx.x) >= G) return;
  const long long lo = share_lo(blockIdx.x, T, G);
  const long long hi = share_lo(blockIdx.x + 1, T, G);
  if (lo >= hi) return;

  unsigned char* my_ring = ring + warp * kDecRing * kStageBytes;
  uint64_t* my_bars = bars + warp * kDecRing;

  // ---------------------------------------------------------------- producer (lane 0)
  // Walks this warp's page sequence (pages p0 + warp, p0 + warp + 4, ... of each
  // piece, pieces in order) kDecRing elements ahead of the consumer.
  Piece pp{};
  int pp_page = 0;
  bool pp_valid = false;
  int pp_id = 0;  // block-table entry of the element the producer points at
  int issued = 0;
  uint64_t policy = 0;

  auto pp_normalize = [&]() {
    while (pp_valid && pp_page >= pp.p1) {
      pp_valid = find_piece(pp.fend, hi, pref, batch, pp);
      pp_page = pp.p0 + warp;
    }
  };
  auto pp_load_id = [&]() {
    if (pp_valid) pp_id = __ldg(a.block_table + static_cast<size_t>(pp.b) * a.max_pages + pp_page);
  };
  auto pp_issue = [&](int slot, int id, int h) {
    if (id < 0 || id >= a.num_pages) {
      set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
      id = 0;
    }
    const size_t off = (static_cast<size_t>(id) * kKVHeads + h) * (kTileBytes / 2);
    unsigned char* dst = my_ring + slot * kStageBytes;
    mbar_arrive_expect_tx(&my_bars[slot], kStageBytes);
    bulk_g2s_hint(dst, a.k_pages + off, kTileBytes, &my_bars[slot], policy);
    bulk_g2s_hint(dst + kTileBytes, a.v_pages + off, kTileBytes, &my_bars[slot], policy);
    ++issued;
  };

  if (lane == 0) {
    policy = policy_evict_first();
    pp_valid = find_piece(lo, hi, pref, batch, pp);
    pp_page = pp.p0 + warp;
    pp_normalize();
    int ids[kDecRing], hs[kDecRing];
    int n0 = 0;
#pragma unroll
    for (int r = 0; r < kDecRing; ++r) {
      if (pp_valid) {
        ids[r] = __ldg(a.block_table + static_cast<size_t>(pp.b) * a.max_pages + pp_page);
        hs[r] = pp.h;
        ++n0;
        pp_page += kDecWarps;
        pp_normalize();
      }
    }
    pp_load_id();
#pragma unroll
    for (int r = 0; r < kDecRing; ++r)
      if (r < n0) pp_issue(r, ids[r], hs[r]);
  }

  // ---------------------------------------------------------------- consumer
  const int qq = lane & 3;         // quarter of the row for the score pass
  const int tp = (lane >> 2) & 1;  // token parity: rotates the chunk order to avoid bank conflicts
  const int head_mine = qq & 1;    // query head whose score this lane ends up holding
  const int t_mine = (qq >> 1) * 8 + (lane >> 2);  // token whose score this lane holds
  const int hf = lane >> 4;        // half-warp: tokens hf*8 .. hf*8+7 for the V pass
  const int dl = lane & 15;        // dims dl*8 .. dl*8+7 for the V pass
  const uint32_t pb = smem_u32(pbuf + warp * kPageSize * 4);

  int k = 0;         // elements of this warp's sequence visited so far
  int consumed = 0;  // elements whose copy completed
  bool failed = false;
  int piece_idx = 0;
  long long f = lo;
  Piece pc;
  while (find_piece(f, hi, pref, batch, pc)) {
    const int b = pc.b;
    const int h = pc.h;

    // query rows of both heads of the group, in this lane's chunk order, pre-scaled
    float2 q2[4][4][2];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * kQHeads + h * kGroup + i) * kHeadDim);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 u = __ldg(qrow + qq + 4 * (j ^ tp));
        const float2 sc = make_float2(a.qscale, a.qscale);
        q2[j][0][i] = __fmul2_rn(bf2_to_f2(u.x), sc);
        q2[j][1][i] = __fmul2_rn(bf2_to_f2(u.y), sc);
        q2[j][2][i] = __fmul2_rn(bf2_to_f2(u.z), sc);
        q2[j][3][i] = __fmul2_rn(bf2_to_f2(u.w), sc);
      }
    }

    float2 mrun = make_float2(-CUDART_INF_F, -CUDART_INF_F);
    float lsum = 0.f;
    float2 o[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = make_float2(0.f, 0.f);

    for (int p = pc.p0 + warp; p < pc.p1; p += kDecWarps) {
      const int slot = k % kDecRing;
      const uint32_t parity = static_cast<uint32_t>(k / kDecRing) & 1u;
      if (!failed) {
        const bool ok = mbar_wait_bounded(&my_bars[slot], parity);
        failed = __any_sync(kFull, !ok);
        if (failed && lane == 0) set_status(a.status, PKV_ERR_DEVICE_TIMEOUT);
        if (!failed) ++consumed;
      }
      if (!failed) {
        const int rem = sl[b] - p * kPageSize;
        const int n_valid = rem < kPageSize ? rem : kPageSize;
        const uint32_t kt = smem_u32(my_ring + slot * kStageBytes);
        const uint32_t vt = kt + kTileBytes;

        // ---- scores: lanes (token group of 4) x (quarter of the row), two passes of 8 tokens
        float2 acc[2][2];
#pragma unroll
        for (int ps = 0; ps < 2; ++ps)
#pragma unroll
          for (int i = 0; i < 2; ++i) acc[ps][i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t coff = (qq + 4 * (j ^ tp)) * 16;
#pragma unroll
          for (int ps = 0; ps < 2; ++ps) {
            const uint4 u = lds128(kt + (ps * 8 + (lane >> 2)) * kRowBytes + coff);
            const float2 k0 = bf2_to_f2(u.x), k1 = bf2_to_f2(u.y), k2 = bf2_to_f2(u.z), k3 = bf2_to_f2(u.w);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              acc[ps][i] = __ffma2_rn(q2[j][0][i], k0, acc[ps][i]);
              acc[ps][i] = __ffma2_rn(q2[j][1][i], k1, acc[ps][i]);
              acc[ps][i] = __ffma2_rn(q2[j][2][i], k2, acc[ps][i]);
              acc[ps][i] = __ffma2_rn(q2[j][3][i], k3, acc[ps][i]);
            }
          }
        }
        const float a00 = acc[0][0].x + acc[0][0].y, a01 = acc[0][1].x + acc[0][1].y;
        const float a10 = acc[1][0].x + acc[1][0].y, a11 = acc[1][1].x + acc[1][1].y;
        // transpose-reduce over the 4 lanes of a token group: lane qq ends with
        // the full score of (pass qq>>1, head qq&1)
        const bool hi_pass = (qq & 2) != 0;
        float keep0 = hi_pass ? a10 : a00, keep1 = hi_pass ? a11 : a01;
        const float send0 = hi_pass ? a00 : a10, send1 = hi_pass ? a01 : a11;
        keep0 += __shfl_xor_sync(kFull, send0, 2);
        keep1 += __shfl_xor_sync(kFull, send1, 2);
        const float keeph = head_mine ? keep1 : keep0;
        const float sendh = head_mine ? keep0 : keep1;
        float s = keeph + __shfl_xor_sync(kFull, sendh, 1);
        if (t_mine >= n_valid) s = -CUDART_INF_F;

        // ---- online softmax (log2 domain)
        float mx = s;
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float mo = __shfl_xor_sync(kFull, mx, 1);
        const float2 mpage = head_mine ? make_float2(mo, mx) : make_float2(mx, mo);
        const float2 mnew = make_float2(fmaxf(mrun.x, mpage.x), fmaxf(mrun.y, mpage.y));
        const float2 alpha = make_float2(ex2(mrun.x - mnew.x), ex2(mrun.y - mnew.y));
        mrun = mnew;
        const float pj = ex2(s - (head_mine ? mnew.y : mnew.x));
        lsum = lsum * (head_mine ? alpha.y : alpha.x) + pj;
        {
          const uint32_t dst = pb + t_mine * 16 + head_mine * 8;
          asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(dst), "f"(pj), "f"(pj) : "memory");
        }
        const float2 ax = make_float2(alpha.x, alpha.x), ay = make_float2(alpha.y, alpha.y);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          o[0][e] = __fmul2_rn(o[0][e], ax);
          o[1][e] = __fmul2_rn(o[1][e], ay);
        }
        __syncwarp();

        // ---- values
        const uint32_t vrow0 = vt + (hf * 8) * kRowBytes + dl * 16;
        const uint32_t prow0 = pb + (hf * 8) * 16;
        if (n_valid == kPageSize) pv_tokens<false>(vrow0, prow0, hf * 8, n_valid, o);
        else pv_tokens<true>(vrow0, prow0, hf * 8, n_valid, o);
      }
      __syncwarp();  // the stage and the p buffer are free again
      if (lane == 0 && !failed && pp_valid) {
        pp_issue(slot, pp_id, pp.h);
        pp_page += kDecWarps;
        pp_normalize();
        pp_load_id();
      }
      ++k;
    }

    // ---- warp totals: combine the two half-warps, sum l over the lanes of each head
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[i][e].x += __shfl_xor_sync(kFull, o[i][e].x, 16);
        o[i][e].y += __shfl_xor_sync(kFull, o[i][e].y, 16);
      }
    float lh = lsum;
    lh += __shfl_xor_sync(kFull, lh, 2);
    lh += __shfl_xor_sync(kFull, lh, 4);
    lh += __shfl_xor_sync(kFull, lh, 8);
    lh += __shfl_xor_sync(kFull, lh, 16);
    const float lother = __shfl_xor_sync(kFull, lh, 1);
    const float l0 = head_mine ? lother : lh;
    const float l1 = head_mine ? lh : lother;

    float* mbuf = merge + (piece_idx & 1) * kMergeFloats;
    float* mw = mbuf + warp * kPieceFloats;
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float4* dst = reinterpret_cast<float4*>(mw + i * kRec + 4 + lane * 8);
        dst[0] = make_float4(o[i][0].x, o[i][0].y, o[i][1].x, o[i][1].y);
        dst[1] = make_float4(o[i][2].x, o[i][2].y, o[i][3].x, o[i][3].y);
      }
    }
    if (lane == 0) {
      mw[0] = mrun.x;
      mw[1] = l0;
      mw[kRec] = mrun.y;
      mw[kRec + 1] = l1;
    }
    __syncthreads();

    // ---- CTA merge of the 4 warp records: thread tid owns dim tid of both heads
    float M[2], L[2], O[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float m = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) m = fmaxf(m, mbuf[w * kPieceFloats + i * kRec]);
      float l = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float* r = mbuf + w * kPieceFloats + i * kRec;
        const float sc = ex2(r[0] - m);
        l += r[1] * sc;
        acc += r[4 + tid] * sc;
      }
      M[i] = m;
      L[i] = l;
      O[i] = acc;
    }
    const bool complete = (pc.p0 == 0 && pc.p1 == pc.np);
    if (complete) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
        a.out[(static_cast<size_t>(b) * kQHeads + h * kGroup + i) * kHeadDim + tid] = __float2bfloat16_rn(O[i] / L[i]);
    } else {
      const long long fseg = pref[b] + static_cast<long long>(h) * pc.np;
      const int cfirst = cta_of(fseg, T, G);
      const int clast = cta_of(fseg + pc.np - 1, T, G);
      const int my_slot = 2 * blockIdx.x + (pc.fstart == lo ? 0 : 1);
      float* rec = a.partials + static_cast<size_t>(my_slot) * kPieceFloats;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        rec[i * kRec + 4 + tid] = O[i];
        if (tid == 0) {
          rec[i * kRec] = M[i];
          rec[i * kRec + 1] = L[i];
        }
      }
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        const int old = atomicAdd(a.counters + b * kKVHeads + h, 1);
        flag[0] = (old == clast - cfirst) ? 1 : 0;
      }
      __syncthreads();
      if (flag[0]) {
        __threadfence();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float m = -CUDART_INF_F;
          for (int c = cfirst; c <= clast; ++c) {
            const int sidx = 2 * c + ((c == cfirst && share_lo(c, T, G) < fseg) ? 1 : 0);
            m = fmaxf(m, __ldcg(a.partials + static_cast<size_t>(sidx) * kPieceFloats + i * kRec));
          }
          float l = 0.f, acc = 0.f;
          for (int c = cfirst; c <= clast; ++c) {
            const int sidx = 2 * c + ((c == cfirst && share_lo(c, T, G) < fseg) ? 1 : 0);
            const float* r = a.partials + static_cast<size_t>(sidx) * kPieceFloats + i * kRec;
            const float sc = ex2(__ldcg(r) - m);
            l += __ldcg(r + 1) * sc;
            acc += __ldcg(r + 4 + tid) * sc;
          }
          a.out[(static_cast<size_t>(b) * kQHeads + h * kGroup + i) * kHeadDim + tid] = __float2bfloat16_rn(acc / l);
        }
        if (tid == 0) a.counters[b * kKVHeads + h] = 0;
      }
    }
    f = pc.fend;
    ++piece_idx;
  }

  // copies still in flight after a timeout: wait for them (bounded) before the CTA exits
  if (failed && lane == 0) {
    for (int e = consumed; e < issued; ++e) {
      if (!mbar_wait_bounded(&my_bars[e % kDecRing], static_cast<uint32_t>(e / kDecRing) & 1u)) break;
    }
  }
}

size_t decode_workspace_bytes(int32_t batch, int num_sms) {
  size_t off = PKV_STATUS_BYTES;
  off += (static_cast<size_t>(batch) * kKVHeads * 4 + 255) / 256 * 256;
  off += static_cast<size_t>(2) * kDecCtasPerSm * num_sms * kPieceFloats * 4;
  return off;
}

int launch_decode(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                  const int32_t* seq_lens, void* out, float scale, int32_t batch, int32_t max_pages,
                  int32_t num_pages, void* workspace, int num_sms, cudaStream_t stream) {
  if (batch == 0) return PKV_OK;
  const size_t smem = decode_smem_bytes(batch);
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(decode_smem_bytes(kMaxDecodeBatch))) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_kernel, kDecThreads, smem) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (occ < 1) return PKV_ERR_UNSUPPORTED;
  if (occ > kDecCtasPerSm) occ = kDecCtasPerSm;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  DecodeArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_pages = static_cast<const __nv_bfloat16*>(k_pages);
  a.v_pages = static_cast<const __nv_bfloat16*>(v_pages);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.qscale = scale * kLog2e;
  a.batch = batch;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.status = reinterpret_cast<int*>(ws);
  a.counters = reinterpret_cast<int*>(ws + PKV_STATUS_BYTES);
  a.partials = reinterpret_cast<float*>(ws + PKV_STATUS_BYTES +
                                        (static_cast<size_t>(batch) * kKVHeads * 4 + 255) / 256 * 256);
  decode_kernel<<<num_sms * occ, kDecThreads, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
