// decode_kernel.cuh -- the batched decode attention kernel over the paged KV
// cache (split-KV), templated on the cache geometry; decode.cu launches it.
//
// Source of the operation: PagedAttention decoding in the LLM engine
// ("FunASR vLLM Inference Engine Guide", section 2 "vLLM Engine Architecture");
// decode is where long-audio serving spends its time ("Optimizing ASR for
// 90-minute multi-speaker audio", section "Time spent: profiling"). For every
// request and query head: the softmax-weighted mean of the value rows over the
// cached positions, scores scale * <q, k_j>. The pages name other backbones for
// the same decoder slot without their head counts, so besides the Qwen3 decoder
// (16 query / 8 KV heads of dimension 128, head counts fixed at compile time)
// the kernel serves head_dim 64 or 128 with 1 to 8 query heads per KV head and
// any KV-head count; a group of 3, 5, 6 or 7 heads runs as 4 or 8 with the
// extra query rows zero and their outputs not written.
//
// The op reads every cached K/V row once and does ~1 FMA per byte per query
// head, so it is bound by HBM bandwidth. Design:
//
//  * Work is the list of (request, KV head, page) triples, ordered by request,
//    then KV head, then page. The kernel is persistent: gridDim.x CTAs (the SM
//    count times the CTAs resident per SM) each take a contiguous share of that
//    list, computed on the device from seq_lens, so the grid depends only on
//    host-known sizes (CUDA-graph friendly). Shares are equal in cost: a page
//    costs 1 and, for batches (the polled merge below), each (request, KV head)
//    that starts inside a share costs kPieceCost more, because a piece boundary
//    stalls the CTA's stream (a warp merge behind a barrier, the refill of the
//    stage ring after it) and a split piece's merge waits on its other holders.
//  * A CTA's share is cut into pieces, one per (request, KV head) it touches.
//    Its consumer warps take the share's pages round-robin (page f of the share
//    goes to consumer (f - lo) mod kCons, across piece boundaries). A producer warp
//    fills each consumer's ring of shared-memory stages with tiled TMA copies
//    (cp.async.bulk.tensor, per page one copy of the K tile and one of the V
//    tile, each head_dim / 64 swizzled 16-row x 64-dim halves, evict-first)
//    that complete on the stage's full barrier; consumers release stages
//    through empty barriers.
//  * All query heads of the GQA group are computed from one K/V read, the two
//    products of a page as warp-level bf16 tensor-core MMAs with fp32
//    accumulation (pkv_mma.cuh): scores S^T = K Q^T with the group's rows as
//    the B operand's first columns (8 columns, rows past the group zero),
//    softmax online in registers in the log2 domain (scale * log2 e applied to
//    the fp32 scores), p rounded to bf16 for the value product O^T += V^T P^T.
//    Tokens past seq_len in the last page are masked in the scores and in the
//    value operand's registers, so unused slots may hold anything, NaN included.
//  * Optional fused append: the consumer warp that takes a request's last page
//    loads the request's new K/V row for that head (with that page's block-table
//    entry) when its piece starts, and once the page is staged writes the row
//    over the slot's copied bytes (swizzled, then a proxy fence before the
//    stage's next tensor copy) and into the pool. The producer copies the page
//    like any other, so in early mode it never waits for the predecessor. With
//    a cos/sin table the whole producer warp writes the row instead, rotating
//    the key (rotary position embedding at the new token's position, pairs
//    (i, i + head_dim / 2), fp32, rounded to bf16); in early mode the chunk's
//    pages before its first new-row page are copied before the warp waits.
//    Each piece's query rows are rotated the same way after they are staged
//    (then rounded to bf16 as the MMA operand).
//  * The query rows of the next piece are copied into shared memory (cp.async)
//    while the current piece streams, so a piece boundary costs no round trip.
//  * At the end of a piece the warps merge through shared memory (at most four
//    query heads per pass). A piece that covers its whole (request, KV head)
//    writes the bf16 output. Otherwise it writes a partial record (m, l, o per
//    head). Only a share's first and last piece can be split, and a pair's
//    holders are consecutive CTAs. The records are merged (log-sum-exp, in an
//    order fixed by the pair alone) in one of two ways, each its own
//    instantiation, chosen by the expected number of holders per pair (grid
//    size over batch x KV heads):
//     - Counted, for few pairs over many CTAs (one long request): fp32
//       records; after its last piece a CTA bumps the pairs' counters (one
//       fence, one round trip) and the CTA that completes a count stages the
//       records in its drained stage ring (cp.async, one round trip per batch),
//       merges them and resets the counter.
//     - Polled, for many pairs over few CTAs each: records of tagged 32-bit
//       words -- o rounded to 16 significant bits, m and l exact as the sum of
//       two such values, a tag in every word's low byte -- written with no
//       fence or atomic. The CTA holding a pair's last page (necessarily its
//       first piece, begun by lower-numbered CTAs) reads the holders' records
//       once its own share is done, again until every word carries the tag,
//       merges them and clears the records for the next call. Its wait relies
//       on the holders having started, which the hardware's dispatch of CTAs
//       in index order gives; the wait is bounded either way.
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_kernels.h"
#include "pkv_mma.cuh"
#include "pkv_tc.cuh"

namespace pkv {

// Launch shape (compile-time; the defaults are the tuned configuration).
#ifndef PKV_DEC_CONSUMERS
#define PKV_DEC_CONSUMERS 4
#endif
#ifndef PKV_DEC_RING
#define PKV_DEC_RING 3  // stages per consumer warp at head_dim 128 (twice as many at 64)
#endif
#ifndef PKV_DEC_CTAS_PER_SM
#define PKV_DEC_CTAS_PER_SM 2
#endif
#ifndef PKV_DEC_ROUND_PAGES  // pages the producer issues per round
#define PKV_DEC_ROUND_PAGES 4
#endif
#ifndef PKV_DEC_PIECE_COST  // pages a (request, KV head) boundary inside a share counts for (polled merge)
#define PKV_DEC_PIECE_COST 32
#endif
constexpr int kCons = PKV_DEC_CONSUMERS;  // consumer warps; one more warp produces
constexpr int kConsThreads = kCons * 32;
constexpr int kDecThreads = kConsThreads + 32;
constexpr int kDecCtasPerSm = PKV_DEC_CTAS_PER_SM;
constexpr int kRoundPages = PKV_DEC_ROUND_PAGES;
constexpr int kMaxDecodeBatch = 1024;
constexpr int kMaxGrid = 2048;  // partial-record slots are sized for this many CTAs
constexpr int kMinShare = 8;    // pages per CTA at least on average (when the step has that many)
constexpr unsigned kFull = 0xffffffffu;
constexpr int kSmemMisc = 32;                // flag words, then the CTA's share bounds
constexpr int kSmemAlign = 1024;             // the ring starts on a 1024-byte boundary (swizzle atoms)
constexpr uint32_t kTag = 0xa5u;             // low byte of a word written by this call
constexpr int kPollMax = 24;                 // polled merge up to this many holders per pair
// A step with few (request, KV head) pairs for the two-CTA grid (the counted
// merge) runs the wide launch shape when the block table can hold at least this
// many (request, KV head, page) triples (batch x max_pages x KV heads); with half
// the CTAs, a pair then has few enough holders for the polled merge. One 40k-token
// request measured 29.25 -> 28.27 us per layer, 16k 14.49 -> 13.57, but 4k 7.30 -> 7.92
// (half the CTAs for a small step), hence the bound.
constexpr long long kWideMinPages = 8192;

struct DecodeArgs {
  const __nv_bfloat16* q;      // [batch][hq][D]
  const __nv_bfloat16* k_new;  // optional fused append: [batch][hkv][D], nullptr = none
  const __nv_bfloat16* v_new;
  const __nv_bfloat16* k_pages;
  const __nv_bfloat16* v_pages;
  const int* block_table;
  const int* seq_lens;
  __nv_bfloat16* out;  // [batch][hq][D]
  const float* rope;  // optional cos/sin table [rope_max_pos][D] fp32 (cos[D/2], sin[D/2]), nullptr = none
  int rope_max_pos;
  float qscale;  // scale * log2(e)
  int early;     // prefetch before the grid dependency (caller guarantees the predecessor leaves
                 // pools, block table and lengths alone)
  int batch;
  int max_pages;
  int num_pages;
  int hkv;  // KV heads (run-time geometries)
  int gq;   // query heads per KV head (run-time geometries; at most the kernel's group)
  int* status;
  int* counters;       // [batch * hkv], zero between calls (counted merge)
  float* partials;     // [2 * gridDim.x][G * (D + 4)] (counted merge)
  uint32_t* tagged;    // [2 * gridDim.x][G * D + 4 * G], no word tagged between calls (polled merge)
};

// Geometry of one instantiation: head_dim D, G query heads per KV head computed
// (1, 2, 4 or 8), whether the head counts are the Qwen3 decoder's 16 / 8 fixed
// at compile time (otherwise DecodeArgs::hkv / gq), and the launch shape: two
// CTAs per SM with kRing stages per consumer, or (kWide, for a few long requests)
// one CTA per SM with twice the stages, so each (request, KV head) has half as
// many holders to merge and each CTA twice the bytes in flight.
template <int D_, int G_, bool kFixed_, bool kWide_ = false>
struct DecGeo {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr bool kFixed = kFixed_;
  static constexpr bool kWide = kWide_;
  static constexpr int kCtasPerSm = kWide ? 1 : kDecCtasPerSm;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "one 8-column MMA tile of heads");
  static_assert(!kFixed || (D == kHeadDim && G == kGroup), "the fixed geometry is 16 / 8 / 128");
  static constexpr int kKS = D / 16;                    // 16-dim steps of both MMA products
  static constexpr int kRing = (D == 128 ? PKV_DEC_RING : 2 * PKV_DEC_RING) * (kWide ? 2 : 1);  // per consumer
  static constexpr int kStages = kCons * kRing;
  static constexpr int kTile = kPageSize * D * 2;       // one (page, KV head) tile of K or V
  static constexpr int kStage = 2 * kTile;              // K tile + V tile
  static constexpr int kRowB = D * 2;                   // one K or V row
  static constexpr int kRec = D + 4;                    // floats per query-head record: m, l, pad, pad, o[D]
  static constexpr int kPiece = G * kRec;               // a counted record of one piece (all heads)
  static constexpr int kPieceB = kPiece * 4;
  static constexpr int kSplitWords = G * D + 4 * G;     // polled record: o[G][D], then m_hi, m_lo, l_hi,
  static constexpr int kSplitB = kSplitWords * 4;       // l_lo of each head
  static constexpr int kMH = G < 4 ? G : 4;             // heads per pass through the merge buffer
  static constexpr int kQBuf = G * D * 2;               // query rows of one (request, KV head)
  static constexpr int kCsB = D * 4;                    // one cos/sin table row
  static constexpr int kSmemRing = kStages * kStage;
  static constexpr int kSmemBars = 2 * kStages * 8;     // full + empty barrier per stage
  static constexpr int kMergeFloats = kCons * kMH * kRec;
  static constexpr int kSmemMerge = kMergeFloats * 4;
  static constexpr int kSmemQ = 2 * kQBuf;              // this piece's rows and the next piece's
  static constexpr int kSmemCs = 2 * kCsB;              // rows for this piece's and the next piece's position
  static constexpr int kSmemFixed = kSmemAlign + kSmemRing + kSmemBars + kSmemMerge + kSmemQ + kSmemCs + kSmemMisc;
  static constexpr int kMergeCap = kSmemRing / kPieceB;  // records staged per batch of a counted merge
  // Lane layout of the record merges: 4-word groups of a record's o, group x at words 4x .. 4x + 3
  // (head 4x / D, dims 4x mod D ..); lane l holds groups l, l + 32, ...
  static constexpr int kGroups = G * D / 4;
  static constexpr int kLW = kGroups >= 32 ? kGroups / 32 : 1;
  static constexpr int kMergeBatch = 16 / kLW > 8 ? 8 : (16 / kLW < 1 ? 1 : 16 / kLW);  // polled records in flight
  static constexpr int kItems = (kMH * D + kConsThreads - 1) / kConsThreads;  // (head, dim) per thread per pass
  static_assert(kRoundPages >= 1 && kRoundPages <= kStages, "a page's previous stage use is in an earlier round");
  static_assert(kSplitB % 16 == 0 && kPieceB % 16 == 0, "16-byte loads, copies and clears of a record");
  static_assert((kSmemRing + kSmemBars) % 16 == 0 && kSmemMerge % 16 == 0 && kQBuf % 16 == 0, "alignment");
  static_assert(kMergeCap >= 1, "a record fits the ring");
  __device__ __forceinline__ static int hkv(const DecodeArgs& a) { return kFixed ? kKVHeads : a.hkv; }
  __device__ __forceinline__ static int gq(const DecodeArgs& a) { return kFixed ? kGroup : a.gq; }
  static size_t smem_bytes(int batch) { return kSmemFixed + static_cast<size_t>(3 * batch + 2) * 4; }
};

// A piece: pages [p0, p1) of KV head h of request b; flattened indices [fstart, fend).
struct Piece {
  int b, h, np, p0, p1;
  long long fstart, fend;
};

// Request b holding flattened index f: the largest b with pref[b] <= f.
__device__ __forceinline__ int request_of(long long f, const int* pref, int batch) {
  int lo_b = 0, hi_b = batch - 1;
  while (lo_b < hi_b) {
    const int mid = (lo_b + hi_b + 1) >> 1;
    if (pref[mid] <= f) lo_b = mid; else hi_b = mid - 1;
  }
  return lo_b;
}
__device__ __forceinline__ int pages_of(int s) { return (s + kPageSize - 1) / kPageSize; }

// Piece of the CTA share [.., hi) that starts at flattened index f.
// pref[b] = page-head triples of requests before b (pref[batch] = total); sl = clamped lengths.
__device__ __forceinline__ bool find_piece(long long f, long long hi, const int* pref, const int* sl, int batch,
                                           Piece& pc) {
  if (f >= hi) return false;
  const int b = request_of(f, pref, batch);
  pc.b = b;
  pc.np = pages_of(sl[b]);
  const long long off = f - pref[b];
  pc.h = static_cast<int>(off / pc.np);
  pc.p0 = static_cast<int>(off % pc.np);
  const long long p1 = pc.p0 + (hi - f);
  pc.p1 = static_cast<int>(p1 < pc.np ? p1 : pc.np);
  pc.fstart = f;
  pc.fend = f + (pc.p1 - pc.p0);
  return true;
}

// The shares. Each (request, KV head) boundary inside a share costs kLam pages
// (the warp merge behind a barrier, the record, the refill of the stage ring
// after it, the merge's wait for the pair's other holders), so a flattened index
// f costs C(f) = f + kLam * (pairs starting in (0, f]), and CTA c holds the
// indices f with floor(c Ctot / n) <= C(f) < floor((c + 1) Ctot / n), Ctot =
// T + kLam * (pairs - 1): lo(c) is the smallest f with C(f) >= floor(c Ctot / n).
// A share that falls inside one boundary's jump is empty; the holders of a pair
// are still consecutive, non-empty shares. With kLam = 0 the shares are equal in
// pages (lo(c) = c T / n). pcp[b] = non-empty pairs before request b. Measured at
// bs16: kLam 0 / 8 / 16 / 24 / 32 / 40 / 64 gave 18.67 / 18.82 / 18.55 / 18.02 /
// 17.91 / 18.02 / 18.95 us per layer; the counted merge (one long request) keeps 0.
template <int kLam>
struct Shares {
  static constexpr int lam = kLam;
  const int* pref;
  const int* pcp;
  const int* sl;
  int batch, hkv, n;
  long long T, Ctot;
  long long q;  // Ctot / n
  int r;        // Ctot mod n
  // T_ and pairs_: pref[batch] and pcp[batch]
  __device__ __forceinline__ void init(const int* pref_, const int* pcp_, const int* sl_, int batch_, int hkv_,
                                       int n_, long long T_, int pairs_) {
    pref = pref_;
    pcp = pcp_;
    sl = sl_;
    batch = batch_;
    hkv = hkv_;
    n = n_;
    T = T_;
    Ctot = T + static_cast<long long>(lam) * (pairs_ > 0 ? pairs_ - 1 : 0);
    if (Ctot < (1LL << 32)) {  // (the usual case: a 32-bit division)
      const unsigned c32 = static_cast<unsigned>(Ctot);
      q = c32 / static_cast<unsigned>(n);
      r = static_cast<int>(c32 - static_cast<unsigned>(q) * static_cast<unsigned>(n));
    } else {
      q = Ctot / n;
      r = static_cast<int>(Ctot - q * n);
    }
  }
  // floor(c Ctot / n) without a 64-bit division (c r < 2^22)
  __device__ __forceinline__ long long y_of(int c) const {
    return c * q + static_cast<unsigned>(c * r) / static_cast<unsigned>(n);
  }
  __device__ __forceinline__ long long cost(long long f) const {  // f < T
    if (kLam == 0) return f;
    const int b = request_of(f, pref, batch);
    return f + static_cast<long long>(lam) * (pcp[b] + (f - pref[b]) / pages_of(sl[b]));
  }
  // first index of CTA c's share: the smallest f with C(f) >= floor(c Ctot / n)
  __device__ __forceinline__ long long lo(int c) const {
    const long long y = y_of(c);
    if (kLam == 0) return y;
    int lb = 0, hb = batch - 1;
    while (lb < hb) {
      const int mid = (lb + hb + 1) >> 1;
      if (pref[mid] + static_cast<long long>(lam) * pcp[mid] <= y) lb = mid; else hb = mid - 1;
    }
    return lo_in(lb, y);
  }
  // the same, given lb: the last request whose first pair costs at most y
  __device__ __forceinline__ long long lo_in(int lb, long long y) const {
    const int np = pages_of(sl[lb]);
    if (np == 0) return pref[lb];
    const long long key = pref[lb] + static_cast<long long>(lam) * pcp[lb];
    // (y - key < (np + lam) * hkv < 2^32: the table bound keeps max_pages * hkv below 2^31)
    long long h = static_cast<unsigned>(y - key) / static_cast<unsigned>(np + lam);
    if (h > hkv - 1) h = hkv - 1;
    const long long s_next = pref[lb] + (h + 1) * np;
    const long long f = y - static_cast<long long>(lam) * (pcp[lb] + h);
    return f < s_next ? f : s_next;
  }
  // the CTA whose share holds index f (< T)
  __device__ __forceinline__ int cta(long long f) const { return static_cast<int>(((cost(f) + 1) * n + Ctot - 1) / Ctot - 1); }
};

// Polled records are 32-bit words: an fp32 value rounded to nearest (even) at
// 15 mantissa bits, with the tag in the freed low byte. Each word is one
// single-copy-atomic access, so a reader that sees the tag sees the value,
// without a fence on the writer's side; a cleared word (zero) carries no tag.
__device__ __forceinline__ uint32_t tag_word(float v) {
  const uint32_t u = __float_as_uint(v);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fffff00u | kTag;  // NaN stays NaN
  return ((u + 0x7fu + ((u >> 8) & 1u)) & 0xffffff00u) | kTag;
}
__device__ __forceinline__ float untag(uint32_t w) { return __uint_as_float(w & 0xffffff00u); }
// v = hi + lo with hi and lo both 24-bit floats: exact for every finite fp32 v
__device__ __forceinline__ void tag_split(float v, uint32_t& hi, uint32_t& lo) {
  hi = tag_word(v);
  lo = tag_word(v - untag(hi));
}
__device__ __forceinline__ void st_word(uint32_t* p, uint32_t w) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(w) : "memory");
}
__device__ __forceinline__ uint4 ld_words4(const uint32_t* p) {
  uint4 r;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}
__device__ __forceinline__ uint32_t ld_word(const uint32_t* p) {
  uint32_t r;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(r) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ bool tagged(uint32_t w) { return (w & 0xffu) == kTag; }

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsThreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Combine the consumer warps' states of heads [h0, h0 + Geo::kMH) in the merge
// buffer ([warp][head - h0][kRec]: m, l, pad, pad, o[D]) for this thread's
// items: item e is (head h0 + x / D, dim x mod D) with x = tid + e * kConsThreads
// (valid when x < kMH * D). States of warps that folded nothing (m = -inf) weigh 0.
template <class Geo>
__device__ __forceinline__ void combine_items(const float* merge, int tid, float (&M)[Geo::kItems],
                                              float (&L)[Geo::kItems], float (&O)[Geo::kItems]) {
#pragma unroll
  for (int e = 0; e < Geo::kItems; ++e) {
    const int x = tid + e * kConsThreads;
    const int hi = x / Geo::D < Geo::kMH ? x / Geo::D : Geo::kMH - 1, d = x % Geo::D;
    float m = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kCons; ++w) m = fmaxf(m, merge[(w * Geo::kMH + hi) * Geo::kRec]);
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kCons; ++w) {
      const float* r = merge + (w * Geo::kMH + hi) * Geo::kRec;
      const float sc = r[0] == -CUDART_INF_F ? 0.f : ex2(r[0] - m);
      l += r[1] * sc;
      o += r[4 + d] * sc;
    }
    M[e] = m;
    L[e] = l;
    O[e] = o;
  }
}

// Write a warp's folded record-merge state (lane layout: group j = lane + 32 j)
// of heads [h0, h0 + kMH) into its merge-buffer slot.
template <class Geo>
__device__ __forceinline__ void store_lane_state(float* mw, int lane, int h0, const float (&fm)[Geo::kLW],
                                                 const float (&fl)[Geo::kLW], const float4 (&fo)[Geo::kLW]) {
#pragma unroll
  for (int j = 0; j < Geo::kLW; ++j) {
    const int x = lane + 32 * j;
    if (x >= Geo::kGroups) continue;
    const int hd = (4 * x) / Geo::D, d = (4 * x) % Geo::D;
    if (hd < h0 || hd >= h0 + Geo::kMH) continue;
    float* r = mw + (hd - h0) * Geo::kRec;
    reinterpret_cast<float4*>(r + 4 + d)[0] = fo[j];
    if (d == 0) {
      r[0] = fm[j];
      r[1] = fl[j];
    }
  }
}

// kFused: a.k_new / a.v_new are given (fused append); kRope: a.rope is given too;
// kPolled: the polled merge, else the counted one. Each combination is its own
// instantiation, so a path carries no code (and no registers) for the others.
template <class Geo, bool kFused, bool kRope, bool kPolled>
__global__ void __launch_bounds__(kDecThreads, Geo::kCtasPerSm) decode_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                             const __grid_constant__ CUtensorMap vmap,
                                                                             const DecodeArgs a) {
  constexpr int D = Geo::D, G = Geo::G, kKS = Geo::kKS, kRing = Geo::kRing, kStages = Geo::kStages;
  constexpr int kRec = Geo::kRec, kMH = Geo::kMH, kLW = Geo::kLW;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((kSmemAlign - (smem_u32(smem_raw) & (kSmemAlign - 1))) & (kSmemAlign - 1));
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Geo::kSmemRing);
  uint64_t* empty = full + kStages;
  float* merge = reinterpret_cast<float*>(smem + Geo::kSmemRing + Geo::kSmemBars);
  unsigned char* qbuf = reinterpret_cast<unsigned char*>(merge + Geo::kMergeFloats);
  unsigned char* csbuf = qbuf + Geo::kSmemQ;
  int* flag = reinterpret_cast<int*>(csbuf + Geo::kSmemCs);  // [0..1] merge flags, [2] a wait failed, [4..5] share
  int* pref = flag + kSmemMisc / 4;
  int* sl = pref + a.batch + 1;
  int* pcp = sl + a.batch;  // [batch + 1] non-empty (request, KV head) pairs before each request

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int batch = a.batch;
  const int hkv = Geo::hkv(a);
  const int gq = Geo::gq(a);
  const int hq = hkv * gq;
  if (tid == kConsThreads) {  // the producer's first lane: descriptors before its first copies
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }

  if (tid < kStages) {
    mbar_init(&full[tid], 1);
    mbar_init(&empty[tid], 1);
  }
  if (tid == kStages) flag[2] = 0;
  // Every argument buffer may come from the previous kernel in the stream, so
  // the kernel waits for it before touching them -- except in early mode, where
  // the caller guarantees that the predecessor writes neither the pools nor the
  // block table nor the lengths: then the length scan, the share decoding and
  // the first page copies overlap the predecessor's tail, and each warp waits
  // only before it reads q / k_new / v_new or writes anything. Dependents are
  // released only after this grid's own wait, so the kernel two launches back
  // has always completed when a successor starts early.
  if (!a.early) {
    grid_dependency_wait();
    allow_dependents();
  }

  // seq lens (clamped) and the exclusive prefix of (KV head, page) pairs per request
  if (warp == 0) {
    int carry = 0, pcarry = 0;
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
      const int v = pages_of(s) * hkv;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (b < batch) pref[b] = carry + x - v;
      carry += __shfl_sync(kFull, x, 31);
      const int w = kPolled && s > 0 ? hkv : 0;  // (the counted instantiation prices no boundary)
      int z = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, z, o);
        if (lane >= o) z += y;
      }
      if (b < batch) pcp[b] = pcarry + z - w;
      pcarry += __shfl_sync(kFull, z, 31);
    }
    if (lane == 0) {
      pref[batch] = carry;
      pcp[batch] = pcarry;
    }
    // This CTA's share bounds, once, by this warp: the request holding each bound is the
    // last one whose first pair costs no more than the bound's cost, counted with ballots
    // over the requests (their costs are non-decreasing); lanes 0 and 1 then place lo(c)
    // and lo(c + 1) inside their requests.
    __syncwarp();
    const long long Tw = carry;
    const long long gw = Tw / kMinShare > 0 ? Tw / kMinShare : 1;
    const int nw = static_cast<int>(gw < gridDim.x ? gw : gridDim.x);
    if (static_cast<int>(blockIdx.x) < nw) {
      Shares<kPolled ? PKV_DEC_PIECE_COST : 0> sw;
      sw.init(pref, pcp, sl, batch, hkv, nw, Tw, pcarry);
      const long long y0 = sw.y_of(blockIdx.x), y1 = sw.y_of(blockIdx.x + 1);
      if (sw.lam == 0) {
        if (lane < 2) flag[4 + lane] = static_cast<int>(lane ? y1 : y0);
      } else {
        int n0 = 0, n1 = 0;
        for (int base = 0; base < batch; base += 32) {
          const int b = base + lane;
          const long long key = b < batch ? pref[b] + static_cast<long long>(sw.lam) * pcp[b] : (1LL << 62);
          n0 += __popc(__ballot_sync(kFull, key <= y0));
          n1 += __popc(__ballot_sync(kFull, key <= y1));
        }
        if (lane < 2) flag[4 + lane] = static_cast<int>(sw.lo_in((lane ? n1 : n0) - 1, lane ? y1 : y0));
      }
    }
  }
  fence_barrier_init();
  __syncthreads();

  // Only min(gridDim.x, T / 8) CTAs (at least one) take a share, so that a share
  // holds 8 pages on average (a tiny step is not spread so thin that its merges
  // dominate); the CTAs between the first and last holder of a (request, KV head)
  // all hold a piece of it.
  const long long T = pref[batch];
  const long long g_want = T / kMinShare > 0 ? T / kMinShare : 1;
  const int nsh = static_cast<int>(g_want < gridDim.x ? g_want : gridDim.x);
  // zero output rows of empty requests (graph-bucket padding): CTA c clears rows
  // c, c + gridDim.x, ...; in early mode only after the grid dependency
  auto zero_empty_rows = [&](int first_thread, int nthreads) {
    for (int b = blockIdx.x; b < batch; b += gridDim.x) {
      if (sl[b] == 0) {
        uint4* o = reinterpret_cast<uint4*>(a.out + static_cast<size_t>(b) * hq * D);
        for (int i = tid - first_thread; i < hq * D / 8; i += nthreads) o[i] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  if (static_cast<int>(blockIdx.x) >= nsh) {
    if (a.early) {
      grid_dependency_wait();
      allow_dependents();
    }
    zero_empty_rows(0, kDecThreads);
    return;
  }
  // the polled instantiation (batches, many short pairs) prices a pair boundary; the counted one
  // (one long request) does not. The share bounds came from warp 0 (T < 2^31: int words)
  const long long lo = flag[4];
  const long long hi = flag[5];

  // ============================================================== producer warp
  // Walks the share 32 flattened indices at a time, one per lane: each lane
  // decodes its (request, KV head, page), loads the block-table entry, and works
  // out which consumer reads the page ((f - lo) mod kCons) and which stage of
  // that consumer's ring it fills (its running page count, from the lanes
  // before it with the same consumer). The lanes then issue their own tensor
  // copies in rounds of kRoundPages consecutive pages (round r of a chunk holds
  // its pages R r .. R r + R - 1, R <= kStages), each lane once its stage's
  // previous use has been consumed. That previous use is the page kStages
  // earlier in the share, issued in an earlier round, so each stage's empty
  // barrier is at most one phase behind the wait and a round waits only on
  // pages of earlier rounds. The assignment follows the share and not the
  // piece: with a piece-relative one a run of one-page pieces piled onto one
  // consumer, and a round could wait on a consumer held at a piece boundary by
  // a page of a later round (a deadlock). Smaller rounds land a CTA's first
  // pages sooner; one SIMT copy instruction per round amortises the issue.
  if (warp == kCons) {
    const uint64_t policy = policy_evict_first();
    const unsigned lt_mask = (1u << lane) - 1u;
    int base[kCons];  // pages handed to each consumer before this chunk
#pragma unroll
    for (int c = 0; c < kCons; ++c) base[c] = 0;
    bool pfail = false;
    bool waited = !a.early;
    for (long long f0 = lo; f0 < hi && !pfail; f0 += 32) {
      const long long f = f0 + lane;
      const bool valid = f < hi;
      int hh = 0, id = 0, c = 0, wslot = -1, bb = 0;
      if (valid) {
        const int b = request_of(f, pref, batch);
        const int np = pages_of(sl[b]);
        const int off = static_cast<int>(f - pref[b]);
        hh = off / np;
        const int p = off % np;
        c = static_cast<int>((f - lo) % kCons);
        bb = b;
        id = __ldg(a.block_table + static_cast<size_t>(b) * a.max_pages + p);
        if (kRope && p == np - 1) wslot = (sl[b] - 1) % kPageSize;  // the new token's slot (rotated append)
      }
      const unsigned same = __match_any_sync(kFull, valid ? c : -1);
      const int idx = __popc(same & lt_mask);  // earlier lanes of this chunk feeding the same consumer
      int my_base = 0;
#pragma unroll
      for (int cc = 0; cc < kCons; ++cc) {
        if (cc == c) my_base = base[cc];
        base[cc] += __popc(__ballot_sync(kFull, valid && c == cc));
      }
      const int k = my_base + idx;
      const int slot = c * kRing + k % kRing;
      const int use = k / kRing;
      const int my_round = lane / kRoundPages;
      int rounds = valid ? my_round + 1 : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) rounds = max(rounds, __shfl_xor_sync(kFull, rounds, o));
      // The chunk's copies, in rounds; only the lanes in [from, to) take part.
      auto issue_rounds = [&](int from, int to) {
        for (int r = 0; r < rounds; ++r) {
          if (valid && my_round == r && !pfail && lane >= from && lane < to) {
            if (use > 0 && !mbar_wait_bounded(&empty[slot], static_cast<uint32_t>(use - 1) & 1u)) {
              set_status(a.status, PKV_ERR_DEVICE_TIMEOUT);
              pfail = true;
            } else {
              const bool id_ok = id >= 0 && id < a.num_pages;
              if (!id_ok) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
              const int pid = id_ok ? id : 0;
              const int z = pid * hkv + hh;  // tile of the pool
              unsigned char* dst = ring + slot * Geo::kStage;
              mbar_arrive_expect_tx(&full[slot], Geo::kStage);
              // one copy per tile: its D / 64 16-row x 64-dim halves, 128-byte swizzled
              tma_load_4d_hint(dst, &kmap, 0, 0, 0, z, &full[slot], policy);
              tma_load_4d_hint(dst + Geo::kTile, &vmap, 0, 0, 0, z, &full[slot], policy);
            }
          }
          __syncwarp();
        }
      };
      // New rows come from the predecessor. Without the rotary embedding the consumer that takes
      // a request's last page writes the new row into the staged page and into the pool, so
      // every page goes out at once, whatever the slot of the new row holds now.
      if (!kRope) {
        issue_rounds(0, 32);
      } else {
        // With it the whole warp writes the rows: every page of this chunk that holds its
        // request's new token gets the token's rotated K row and its V row for that head
        // before any lane copies that page. In early mode the pages before the chunk's first
        // such page are copied first; the rest wait for the predecessor. (Pages go out in
        // share order either way, so a page's stage was issued before it: no round waits on a
        // page it holds back.) Lanes take key pairs (i, i + D/2), i = lane (+ 32 at D = 128),
        // rotated in fp32 as y1 = fma(x1, c, -(x2 s)), y2 = fma(x2, c, x1 s) with each product
        // rounded first, then rounded to bf16.
        const unsigned nmask = __ballot_sync(kFull, valid && wslot >= 0);
        int from = 0;  // lanes already issued
        if (!waited && nmask != 0u) {
          from = __ffs(nmask) - 1;
          issue_rounds(0, from);
          grid_dependency_wait();
          allow_dependents();
          waited = true;
        }
        unsigned amask = __ballot_sync(kFull, valid && wslot >= 0 && id >= 0 && id < a.num_pages);
        if (amask != 0u) {
          while (amask != 0u) {
            const int src = __ffs(amask) - 1;
            amask &= amask - 1u;
            const int rb = __shfl_sync(kFull, bb, src), rh = __shfl_sync(kFull, hh, src);
            const int rpid = __shfl_sync(kFull, id, src), rslot = __shfl_sync(kFull, wslot, src);
            const size_t row = ((static_cast<size_t>(rpid) * hkv + rh) * kPageSize + rslot) * D;
            const size_t srow = (static_cast<size_t>(rb) * hkv + rh) * D;
            __nv_bfloat16* kd = const_cast<__nv_bfloat16*>(a.k_pages) + row;
            int pos = sl[rb] - 1;
            if (pos >= a.rope_max_pos) {  // past the table: reported, clamped to its last row
              if (lane == 0) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
              pos = a.rope_max_pos - 1;
            }
            const float* cs = a.rope + static_cast<size_t>(pos) * D;
#pragma unroll
            for (int t = 0; t < D / 64; ++t) {
              const int i = lane + 32 * t;
              const float x1 = __bfloat162float(a.k_new[srow + i]);
              const float x2 = __bfloat162float(a.k_new[srow + i + D / 2]);
              const float cc = __ldg(cs + i), sn = __ldg(cs + D / 2 + i);
              kd[i] = __float2bfloat16_rn(__fmaf_rn(x1, cc, -__fmul_rn(x2, sn)));
              kd[i + D / 2] = __float2bfloat16_rn(__fmaf_rn(x2, cc, __fmul_rn(x1, sn)));
            }
            if (lane < Geo::kRowB / 16)
              reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(a.v_pages) + row)[lane] =
                  __ldg(reinterpret_cast<const uint4*>(a.v_new + srow) + lane);
          }
          fence_proxy_async_global();  // this lane's row stores before the warp's tensor copies
          __syncwarp();
        }
        issue_rounds(from, 32);
      }
      pfail = __any_sync(kFull, pfail);
    }
    if (!kRope || !waited) {
      grid_dependency_wait();
      allow_dependents();
    }
    return;
  }

  // ============================================================== consumer warps
  const int r = lane >> 2, cq = lane & 3;  // MMA fragment row and column pair of this lane
  uint32_t koff[kKS], voff[kKS];
  mma_offsets<kKS>(koff, voff);

  int k = 0;  // pages of this warp's sequence visited so far
  bool failed = false;

  // Warp 0 stages the query rows of a piece in qbuf[buf] (16-byte chunks, rows
  // past the group's gq not read), so that the next piece's rows are on chip
  // before the current one ends; with a cos/sin table, also the table row of
  // the request's new position.
  const uint32_t qb = smem_u32(qbuf);
  const uint32_t csb = smem_u32(csbuf);
  auto stage_q = [&](const Piece& p, int buf) {
    if (warp == 0) {
      const unsigned char* src =
          reinterpret_cast<const unsigned char*>(a.q + (static_cast<size_t>(p.b) * hq + p.h * gq) * D);
#pragma unroll
      for (int c = lane; c < Geo::kQBuf / 16; c += 32)
        if (c / (D / 8) < gq) cp_async16(qb + buf * Geo::kQBuf + c * 16, src + c * 16);
      if (kRope) {
        const int pos = min(sl[p.b] - 1, a.rope_max_pos - 1);  // a piece's request has sl >= 1
        const unsigned char* cs = reinterpret_cast<const unsigned char*>(a.rope + static_cast<size_t>(pos) * D);
        if (lane < Geo::kCsB / 16) cp_async16(csb + buf * Geo::kCsB + lane * 16, cs + lane * 16);
      }
    }
  };
  // CTAs cfirst .. cfirst + n - 1 hold the pieces of (request b, KV head h); the
  // record of CTA c is in slot 2c, or 2c + 1 when it is the second split piece
  // of c's share (first_has_two: the first holder's share starts before (b, h)).
  Shares<kPolled ? PKV_DEC_PIECE_COST : 0> sh;
  sh.init(pref, pcp, sl, batch, hkv, nsh, T, pcp[batch]);
  auto span_of = [&](int b, int h, int& cfirst, int& n, bool& first_has_two) {
    const int np = pages_of(sl[b]);
    const long long fseg = pref[b] + static_cast<long long>(h) * np;
    cfirst = sh.cta(fseg);
    n = sh.cta(fseg + np - 1) - cfirst + 1;
    first_has_two = sh.lo(cfirst) < fseg;
  };
  // Split pieces whose partial records are written but not yet counted: only
  // the first and the last piece of a share can be split, and both are counted
  // together after the last piece, so that no piece boundary waits on a fence
  // or an atomic.
  int npend = 0;
  int pb0 = 0, ph0 = 0, pc0 = 0, pn0 = 0, pb1 = 0, ph1 = 0, pc1 = 0, pn1 = 0;
  bool pt0 = false, pt1 = false;

  Piece pc;
  bool have = find_piece(lo, hi, pref, sl, batch, pc);
  // Polled merge: the CTA that holds the last page of a split (request, KV head)
  // merges it; that pair can only be its first piece, begun by an earlier CTA.
  const bool merger = kPolled && have && pc.p0 > 0 && pc.p1 == pc.np;
  const int mb = pc.b, mh = pc.h;
  // the merger's holders, worked out now rather than after the stream
  int m_cf = 0, m_n = 0;
  bool m_two = false;
  if (merger) span_of(mb, mh, m_cf, m_n, m_two);
  // in early mode the share, its pieces and the merger's holders above came from the lengths alone;
  // q, the output and the records wait for the predecessor
  if (a.early) {
    grid_dependency_wait();
    allow_dependents();
  }
  zero_empty_rows(0, kConsThreads);
  if (have) stage_q(pc, 0);
  if (warp == 0) cp_async_wait_all();
  consumer_sync();
  for (int j = 0; have; ++j) {
    Piece nx;
    const bool have_next = find_piece(pc.fend, hi, pref, sl, batch, nx);
    if (have_next) stage_q(nx, (j + 1) & 1);
    const int b = pc.b;
    const int h = pc.h;
    const bool complete = (pc.p0 == 0 && pc.p1 == pc.np);
    int sp_cfirst = 0, sp_n = 0;
    bool sp_two = false;
    if (!kPolled && !complete) span_of(b, h, sp_cfirst, sp_n, sp_two);  // before the stream, off the critical path

    // Q^T as the B operand of the score MMA: lane (r, cq) holds head r's dims 16 ks + 2 cq (+1) and
    // 16 ks + 8 + 2 cq (+1); rows r >= gq are zero. With a cos/sin table the staged rows are rotated
    // here (pairs (i, i + D/2) sit in steps ks and ks + kKS/2 of the same lane) in fp32, each product
    // rounded first, then rounded to bf16.
    const uint32_t qcur = qb + (j & 1) * Geo::kQBuf;
    const uint32_t ccur = csb + (j & 1) * Geo::kCsB;
    const bool qrow = r < gq;
    uint32_t qf[kKS][2];
    if constexpr (!kRope) {
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        qf[ks][0] = qrow ? lds32(qcur + r * Geo::kRowB + (16 * ks + 2 * cq) * 2) : 0u;
        qf[ks][1] = qrow ? lds32(qcur + r * Geo::kRowB + (16 * ks + 8 + 2 * cq) * 2) : 0u;
      }
    } else {
      float2 x[kKS][2];
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        x[ks][0] = qrow ? bf2_to_f2(lds32(qcur + r * Geo::kRowB + (16 * ks + 2 * cq) * 2)) : make_float2(0.f, 0.f);
        x[ks][1] = qrow ? bf2_to_f2(lds32(qcur + r * Geo::kRowB + (16 * ks + 8 + 2 * cq) * 2)) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int ks = 0; ks < kKS / 2; ++ks)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = 16 * ks + 8 * e + 2 * cq;  // dims d, d + 1 pair with d + D/2, d + D/2 + 1
          const float2 cs = lds64f(ccur + d * 4), sn = lds64f(ccur + Geo::kCsB / 2 + d * 4);
          const float2 xl = x[ks][e], xh = x[ks + kKS / 2][e];
          const float2 t1 = __fmul2_rn(xh, sn), t2 = __fmul2_rn(xl, sn);
          x[ks][e] = __ffma2_rn(xl, cs, make_float2(-t1.x, -t1.y));
          x[ks + kKS / 2][e] = __ffma2_rn(xh, cs, t2);
        }
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        qf[ks][0] = pack_bf16x2(x[ks][0].x, x[ks][0].y);
        qf[ks][1] = pack_bf16x2(x[ks][1].x, x[ks][1].y);
      }
    }

    float o[kKS][4];  // O^T: dims 16 ks + r (+8) x heads 2 cq, 2 cq + 1
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) o[ks][0] = o[ks][1] = o[ks][2] = o[ks][3] = 0.f;
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;

    const int w0 = static_cast<int>((pc.fstart - lo) % kCons);  // consumer of the piece's first page
    const int p_first = pc.p0 + (warp - w0 + kCons) % kCons;    // this warp's first page of the piece
    // Fused append without the rotary embedding: the warp that takes the request's last page loads
    // the new token's K and V rows for this head now (lane l: 16-byte chunk l of the K row, or of
    // the V row from lane D / 8 on) with that page's block-table entry. Once the page is staged it
    // writes them over the copied slot and into the pool.
    const bool takes_new =
        kFused && !kRope && pc.p1 == pc.np && p_first <= pc.np - 1 && (pc.np - 1 - p_first) % kCons == 0;
    constexpr int kRowChunks = D / 8;
    uint4 nrow = make_uint4(0u, 0u, 0u, 0u);
    int nid = -1;
    if (takes_new) {
      if (lane < 2 * kRowChunks)
        nrow = __ldg(reinterpret_cast<const uint4*>((lane < kRowChunks ? a.k_new : a.v_new) +
                                                    (static_cast<size_t>(b) * hkv + h) * D) +
                     lane % kRowChunks);
      nid = __ldg(a.block_table + static_cast<size_t>(b) * a.max_pages + pc.np - 1);
    }
    for (int p = p_first; p < pc.p1; p += kCons) {
      const int slot = warp * kRing + k % kRing;
      const uint32_t parity = static_cast<uint32_t>(k / kRing) & 1u;
      if (!failed) {
        const bool ok = mbar_wait_bounded(&full[slot], parity);
        failed = __any_sync(kFull, !ok);
        if (failed && lane == 0) {
          set_status(a.status, PKV_ERR_DEVICE_TIMEOUT);
          flag[2] = 1;
        }
      }
      if (!failed) {
        const int rem = sl[b] - p * kPageSize;
        const int n_valid = rem < kPageSize ? rem : kPageSize;
        const uint32_t kt = smem_u32(ring + slot * Geo::kStage);
        if (takes_new && p == pc.np - 1) {
          const int t = (sl[b] - 1) % kPageSize;  // the new token's slot
          if (lane < 2 * kRowChunks) {
            const int c = lane % kRowChunks;
            const int tile = lane < kRowChunks ? 0 : Geo::kTile;
            *reinterpret_cast<uint4*>(ring + slot * Geo::kStage + tile + swz(t, c)) = nrow;
            if (nid >= 0 && nid < a.num_pages) {  // (the producer reports a page id out of the pool)
              __nv_bfloat16* pool = const_cast<__nv_bfloat16*>(lane < kRowChunks ? a.k_pages : a.v_pages);
              reinterpret_cast<uint4*>(pool + ((static_cast<size_t>(nid) * hkv + h) * kPageSize + t) * D)[c] = nrow;
            }
          }
          fence_proxy_async_smem();  // the row stores before the stage's next tensor copy
          __syncwarp();
        }
        mma_page<kKS>(kt, kt + Geo::kTile, koff, voff, qf, n_valid, a.qscale, o, m0, m1, l0, l1);
      }
      __syncwarp();  // the stage and the p buffer are free again
      if (lane == 0 && !failed) mbar_arrive(&empty[slot]);
      ++k;
    }

    // ---- warp states: lane (r, cq) holds heads 2 cq, 2 cq + 1 (MMA columns); l summed over r
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, m);
      l1 += __shfl_xor_sync(kFull, l1, m);
    }
    __nv_bfloat16* orow = a.out + (static_cast<size_t>(b) * hq + h * gq) * D;
    const int my_slot = 2 * blockIdx.x + (pc.fstart == lo ? 0 : 1);
#pragma unroll
    for (int h0 = 0; h0 < G; h0 += kMH) {  // passes of kMH heads through the merge buffer
      float* mw = merge + warp * kMH * kRec;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hd = 2 * cq + e;
        if (hd >= h0 && hd < h0 + kMH) {
          float* rw = mw + (hd - h0) * kRec;
#pragma unroll
          for (int ks = 0; ks < kKS; ++ks) {
            rw[4 + 16 * ks + r] = o[ks][e];
            rw[4 + 16 * ks + r + 8] = o[ks][e + 2];
          }
          if (r == 0) {
            rw[0] = e ? m1 : m0;
            rw[1] = e ? l1 : l0;
          }
        }
      }
      consumer_sync();

      // ---- CTA combine of the warp states for this thread's (head, dim) items
      float M[Geo::kItems], L[Geo::kItems], O[Geo::kItems];
      combine_items<Geo>(merge, tid, M, L, O);
      if (complete) {
#pragma unroll
        for (int e = 0; e < Geo::kItems; ++e) {
          const int x = tid + e * kConsThreads;
          if (x < kMH * D && h0 + x / D < gq) orow[(h0 + x / D) * D + x % D] = __float2bfloat16_rn(O[e] / L[e]);
        }
      } else if constexpr (kPolled) {
        uint32_t* rec = a.tagged + static_cast<size_t>(my_slot) * Geo::kSplitWords;
#pragma unroll
        for (int e = 0; e < Geo::kItems; ++e) {
          const int x = tid + e * kConsThreads;
          if (x < kMH * D) st_word(rec + h0 * D + x, tag_word(O[e]));
        }
        if (tid < 4 * kMH) {  // m_hi, m_lo, l_hi, l_lo of head h0 + tid / 4
          const int hi4 = tid >> 2;
          float m = -CUDART_INF_F;
#pragma unroll
          for (int w = 0; w < kCons; ++w) m = fmaxf(m, merge[(w * kMH + hi4) * kRec]);
          float l = 0.f;
#pragma unroll
          for (int w = 0; w < kCons; ++w) {
            const float* rr = merge + (w * kMH + hi4) * kRec;
            l += rr[1] * (rr[0] == -CUDART_INF_F ? 0.f : ex2(rr[0] - m));
          }
          uint32_t whi, wlo;
          tag_split((tid & 2) ? l : m, whi, wlo);
          st_word(rec + G * D + 4 * h0 + tid, (tid & 1) ? wlo : whi);
        }
      } else {
        float* rec = a.partials + static_cast<size_t>(my_slot) * Geo::kPiece;
#pragma unroll
        for (int e = 0; e < Geo::kItems; ++e) {
          const int x = tid + e * kConsThreads;
          if (x < kMH * D) {
            rec[(h0 + x / D) * kRec + 4 + x % D] = O[e];
            if (x % D == 0) {
              rec[(h0 + x / D) * kRec] = M[e];
              rec[(h0 + x / D) * kRec + 1] = L[e];
            }
          }
        }
      }
      if (h0 + kMH < G) consumer_sync();  // the merge buffer is free for the next heads
    }
    if (!complete && !kPolled) {
      if (npend == 0) {
        pb0 = b, ph0 = h, pc0 = sp_cfirst, pn0 = sp_n, pt0 = sp_two;
      } else {
        pb1 = b, ph1 = h, pc1 = sp_cfirst, pn1 = sp_n, pt1 = sp_two;
      }
      ++npend;
    }
    if (warp == 0) cp_async_wait_all();  // the next piece's query rows have landed
    consumer_sync();                     // merge buffer and qbuf[j & 1] free, qbuf[(j + 1) & 1] visible
    pc = nx;
    have = have_next;
  }

  // Lane layout of the record merges below: lane l folds 4-word groups x = l + 32 j
  // (j < kLW) of each record, group x holding dims 4x mod D .. of head 4x / D.
  auto group_head = [&](int j) { return (4 * (lane + 32 * j)) / D; };
  auto group_ok = [&](int j) { return lane + 32 * j < Geo::kGroups; };
  // Final output of the folded states: each warp's lane state into the merge
  // buffer, kMH heads per pass, combined across warps into the output rows.
  auto finish_pair = [&](int b, int h, const float (&fm)[kLW], const float (&fl)[kLW], const float4 (&fo)[kLW]) {
    __nv_bfloat16* orow = a.out + (static_cast<size_t>(b) * hq + h * gq) * D;
#pragma unroll
    for (int h0 = 0; h0 < G; h0 += kMH) {
      store_lane_state<Geo>(merge + warp * kMH * kRec, lane, h0, fm, fl, fo);
      consumer_sync();
      float M[Geo::kItems], L[Geo::kItems], O[Geo::kItems];
      combine_items<Geo>(merge, tid, M, L, O);
#pragma unroll
      for (int e = 0; e < Geo::kItems; ++e) {
        const int x = tid + e * kConsThreads;
        if (x < kMH * D && h0 + x / D < gq) orow[(h0 + x / D) * D + x % D] = __float2bfloat16_rn(O[e] / L[e]);
      }
      consumer_sync();  // the merge buffer is free again
    }
  };

  if constexpr (kPolled) {
    if (!merger || flag[2] != 0) return;  // (a failed wait: copies may still land, merge nothing)

    // Polled merge (log-sum-exp) of the pair of this CTA's first piece over the
    // records of its n holders. Warp w folds records t = w, w + kCons, ... in that
    // order, with up to kMergeBatch of them loaded at a time (lanes 0 .. 4G - 1
    // also load the m/l words); a record is read again until every word carries
    // the tag. The order depends only on the pair, so the result is the same bits
    // on every call.
    const int cf = m_cf, n = m_n;
    const bool two = m_two;
    auto rec_of = [&](int t) {
      const size_t slot = 2 * static_cast<size_t>(cf + t) + ((t == 0 && two) ? 1 : 0);
      return a.tagged + slot * Geo::kSplitWords;
    };
    float fm[kLW], fl[kLW];
    float4 fo[kLW];
#pragma unroll
    for (int j = 0; j < kLW; ++j) {
      fm[j] = -CUDART_INF_F;
      fl[j] = 0.f;
      fo[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    constexpr int kMB = Geo::kMergeBatch;
    const uint4 tag4 = make_uint4(kTag, kTag, kTag, kTag);
    bool lost = false;  // a record never got its tags (a bounded wait ran out)
    for (int t0 = warp; t0 < n && !lost; t0 += kMB * kCons) {
      uint4 R[kMB][kLW];  // o groups of this lane
      uint32_t W[kMB];    // lanes 0 .. 4G - 1: word lane of the m/l block
      auto load = [&](int rr) {
        const uint32_t* rec = rec_of(t0 + rr * kCons);
#pragma unroll
        for (int j = 0; j < kLW; ++j) R[rr][j] = group_ok(j) ? ld_words4(rec + 4 * (lane + 32 * j)) : tag4;
        W[rr] = lane < 4 * G ? ld_word(rec + G * D + lane) : kTag;
      };
#pragma unroll
      for (int rr = 0; rr < kMB; ++rr)
        if (t0 + rr * kCons < n) load(rr);
#pragma unroll
      for (int rr = 0; rr < kMB; ++rr) {
        if (t0 + rr * kCons >= n) break;
        auto all_tagged = [&]() {
          bool ok = tagged(W[rr]);
#pragma unroll
          for (int j = 0; j < kLW; ++j)
            ok = ok && tagged(R[rr][j].x) && tagged(R[rr][j].y) && tagged(R[rr][j].z) && tagged(R[rr][j].w);
          return __all_sync(kFull, ok);
        };
        if (!all_tagged()) {
          const long long tw = clock64();
          bool ok = false;
          while (!ok) {
            if (clock64() - tw > kWaitLimitCycles) break;
            load(rr);
            ok = all_tagged();
          }
          if (!ok) {
            lost = true;
            break;
          }
        }
        const float ml = untag(W[rr]);
#pragma unroll
        for (int j = 0; j < kLW; ++j) {
          const int hd = group_head(j) < G ? group_head(j) : G - 1;
          const float mr = __shfl_sync(kFull, ml, 4 * hd) + __shfl_sync(kFull, ml, 4 * hd + 1);
          const float lr = __shfl_sync(kFull, ml, 4 * hd + 2) + __shfl_sync(kFull, ml, 4 * hd + 3);
          const float mn = fmaxf(fm[j], mr);
          const float keep = ex2(fm[j] - mn), sc = ex2(mr - mn);
          fl[j] = fl[j] * keep + lr * sc;
          float4& ov = fo[j];
          ov.x = ov.x * keep + untag(R[rr][j].x) * sc;
          ov.y = ov.y * keep + untag(R[rr][j].y) * sc;
          ov.z = ov.z * keep + untag(R[rr][j].z) * sc;
          ov.w = ov.w * keep + untag(R[rr][j].w) * sc;
          fm[j] = mn;
        }
      }
    }
    if (lost && lane == 0) {
      set_status(a.status, PKV_ERR_DEVICE_TIMEOUT);
      flag[2] = 1;
    }
    consumer_sync();
    if (flag[2] != 0) return;
    finish_pair(mb, mh, fm, fl, fo);
    // clear the tags of the merged records for the next call (every read above has completed)
    for (int i = tid; i < n * (Geo::kSplitB / 16); i += kConsThreads) {
      const int t = i / (Geo::kSplitB / 16), c = i % (Geo::kSplitB / 16);
      reinterpret_cast<uint4*>(rec_of(t))[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  } else {
    if (npend == 0) return;

    // Count this CTA's records in (release) and learn whether it completed a count
    // (acquire): the CTA that does merges every record of that (request, KV head).
    if (tid == 0) {
      __threadfence();
      const int old0 = atomicAdd(a.counters + pb0 * hkv + ph0, 1);
      const int old1 = npend > 1 ? atomicAdd(a.counters + pb1 * hkv + ph1, 1) : -1;
      __threadfence();
      flag[0] = old0 == pn0 - 1 ? 1 : 0;
      flag[1] = npend > 1 && old1 == pn1 - 1 ? 1 : 0;
    }
    consumer_sync();
    if (flag[2] != 0) {  // a wait failed: copies may still land in the ring, merge nothing
      if (tid == 0) {
        if (flag[0]) a.counters[pb0 * hkv + ph0] = 0;
        if (flag[1]) a.counters[pb1 * hkv + ph1] = 0;
      }
      return;
    }
    // Final merges (log-sum-exp over the partial records) of the pairs whose count
    // this CTA completed, one pair after the other. A pair's records are staged in
    // the drained stage ring by 16-byte asynchronous copies (one round trip per
    // batch of up to kMergeCap records); record t is folded by warp t % kCons in
    // the lane layout above, and the warps' states are then combined through the
    // merge buffer. Which warp folds which record, and the batch boundaries,
    // depend only on the pair, so the result is the same whichever CTA merges.
    const uint32_t ring_s = smem_u32(ring);
    const float* Rs = reinterpret_cast<const float*>(ring);
    constexpr int kChunks = Geo::kPieceB / 16;
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      if (!flag[i]) continue;
      const int nm = i ? pn1 : pn0, cf = i ? pc1 : pc0;
      const bool two = i ? pt1 : pt0;
      float fm[kLW], fl[kLW];
      float4 fo[kLW];
#pragma unroll
      for (int j = 0; j < kLW; ++j) {
        fm[j] = -CUDART_INF_F;
        fl[j] = 0.f;
        fo[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int t0 = 0; t0 < nm; t0 += Geo::kMergeCap) {
        const int t1 = t0 + Geo::kMergeCap < nm ? t0 + Geo::kMergeCap : nm;
        for (int t = t0 + warp; t < t1; t += kCons) {
          const size_t slot = 2 * static_cast<size_t>(cf + t) + ((t == 0 && two) ? 1 : 0);
          const unsigned char* src = reinterpret_cast<const unsigned char*>(a.partials + slot * Geo::kPiece);
          const uint32_t dst = ring_s + (t - t0) * Geo::kPieceB;
          for (int c = lane; c < kChunks; c += 32) cp_async16(dst + c * 16, src + c * 16);
        }
        cp_async_wait_all();
        consumer_sync();
        const int pfirst = ((warp - t0) % kCons + kCons) % kCons;  // this warp's first record position
#pragma unroll
        for (int j = 0; j < kLW; ++j) {
          if (!group_ok(j)) continue;
          const int hd = group_head(j), d = (4 * (lane + 32 * j)) % D;
          float m = fm[j];
          for (int p = pfirst; p < t1 - t0; p += kCons) m = fmaxf(m, Rs[p * Geo::kPiece + hd * kRec]);
          const float keep = fm[j] == -CUDART_INF_F ? 0.f : ex2(fm[j] - m);
          float l = fl[j] * keep;
          float4 ov = fo[j];
          ov.x *= keep, ov.y *= keep, ov.z *= keep, ov.w *= keep;
#pragma unroll 4
          for (int p = pfirst; p < t1 - t0; p += kCons) {
            const float* rr = Rs + p * Geo::kPiece + hd * kRec;
            const float sc = ex2(rr[0] - m);
            l += rr[1] * sc;
            const float4 v = *reinterpret_cast<const float4*>(rr + 4 + d);  // plain load: schedulable across records
            ov.x += v.x * sc, ov.y += v.y * sc, ov.z += v.z * sc, ov.w += v.w * sc;
          }
          fm[j] = m;
          fl[j] = l;
          fo[j] = ov;
        }
        consumer_sync();  // the ring is free for the next batch
      }
      const int b = i ? pb1 : pb0, h = i ? ph1 : ph0;
      finish_pair(b, h, fm, fl, fo);
      if (tid == 0) a.counters[b * hkv + h] = 0;
    }
  }
}

// Host: launch one instantiation family (a geometry) of the kernel.
struct DecodeLaunch {
  const void* q;
  const void* k_new;
  const void* v_new;
  const void* k_pages;
  const void* v_pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* rope;
  int32_t rope_max_pos;
  void* out;
  float scale;
  int hq, hkv, head_dim;
  int32_t batch, max_pages, num_pages;
  void* workspace;
  int num_sms;
  cudaStream_t stream;
  uint32_t flags;
};

// Launchers of the run-time-geometry instantiations (decode_d64.cu, decode_d128.cu); G is the
// kernel's group (1, 2, 4 or 8).
int launch_decode_d64(const DecodeLaunch& c, int G);
int launch_decode_d128(const DecodeLaunch& c, int G);

// Workspace layout of a decode call: status | counters [batch * hkv] (256-byte
// padded) | counted records [2 * grid][G * (D + 4)] fp32 | polled records
// [2 * grid][G * D + 4 G] words.
inline int decode_grid(int num_sms) {
  return kDecCtasPerSm * num_sms < kMaxGrid ? kDecCtasPerSm * num_sms : kMaxGrid;
}
inline size_t decode_counter_bytes(int32_t batch, int hkv) {
  return (static_cast<size_t>(batch) * hkv * 4 + 255) / 256 * 256;
}

template <class Geo>
int launch_decode_geo(const DecodeLaunch& c) {
  using GeoW = DecGeo<Geo::D, Geo::G, Geo::kFixed, true>;
  if (c.batch == 0) return PKV_OK;
  if (c.rope != nullptr && c.k_new == nullptr) return PKV_ERR_NULL_ARG;
  // Polled merge when a pair is expected to span at most kPollMax CTAs (equal
  // lengths); the counted merge for few pairs over many CTAs. Few pairs and a
  // table that can hold a long step take the wide shape (half the CTAs), whose
  // merge is chosen the same way over its own grid. The record slots are laid out
  // for the two-CTA grid either way.
  const int grid = decode_grid(c.num_sms);
  const long long pairs = static_cast<long long>(c.batch) * c.hkv;
  // (head_dim 64 stays narrow: with one CTA per SM its consumers, four per SM, page too slowly -- one
  // 40k-token request at 16/8/64 measured 19.0 us per layer wide against 17.8 narrow)
  const bool wide = Geo::D == 128 && grid > kPollMax * pairs && pairs * c.max_pages >= kWideMinPages;
  const int grid_used = wide ? (c.num_sms < kMaxGrid ? c.num_sms : kMaxGrid) : grid;
  const bool polled = grid_used <= kPollMax * pairs;
  const size_t smem = wide ? GeoW::smem_bytes(c.batch) : Geo::smem_bytes(c.batch);
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, const DecodeArgs);
  // (the wide rows are never taken at head_dim 64; they name the narrow kernels there so that
  // no wide head_dim-64 instantiation is built)
  using GW = typename std::conditional<Geo::D == 128, GeoW, Geo>::type;
  static const Kern kKerns[4][3] = {
      {decode_kernel<Geo, false, false, false>, decode_kernel<Geo, true, false, false>,
       decode_kernel<Geo, true, true, false>},
      {decode_kernel<Geo, false, false, true>, decode_kernel<Geo, true, false, true>,
       decode_kernel<Geo, true, true, true>},
      {decode_kernel<GW, false, false, false>, decode_kernel<GW, true, false, false>,
       decode_kernel<GW, true, true, false>},
      {decode_kernel<GW, false, false, true>, decode_kernel<GW, true, false, true>,
       decode_kernel<GW, true, true, true>}};
  const int variant = c.k_new == nullptr ? 0 : c.rope == nullptr ? 1 : 2;
  const int shape = (wide ? 2 : 0) + (polled ? 1 : 0);
  const Kern kern = kKerns[shape][variant];
  static bool attr_set[64][4][3] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !attr_set[dev][shape][variant]) {
    const size_t max_smem = wide ? GeoW::smem_bytes(kMaxDecodeBatch) : Geo::smem_bytes(kMaxDecodeBatch);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(max_smem)) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev][shape][variant] = true;
  }
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kDecThreads, smem) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (occ < 1) return PKV_ERR_UNSUPPORTED;
  const int occ_cap = wide ? GeoW::kCtasPerSm : Geo::kCtasPerSm;
  if (occ > occ_cap) occ = occ_cap;

  unsigned char* ws = static_cast<unsigned char*>(c.workspace);
  DecodeArgs a;
  a.q = static_cast<const __nv_bfloat16*>(c.q);
  a.k_new = static_cast<const __nv_bfloat16*>(c.k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(c.v_new);
  a.k_pages = static_cast<const __nv_bfloat16*>(c.k_pages);
  a.v_pages = static_cast<const __nv_bfloat16*>(c.v_pages);
  a.block_table = c.block_table;
  a.seq_lens = c.seq_lens;
  a.out = static_cast<__nv_bfloat16*>(c.out);
  a.rope = c.rope;
  a.rope_max_pos = c.rope_max_pos;
  a.qscale = c.scale * kLog2e;
  a.early = (c.flags & PKV_DECODE_EARLY_PREFETCH) ? 1 : 0;
  a.batch = c.batch;
  a.max_pages = c.max_pages;
  a.num_pages = c.num_pages;
  a.hkv = c.hkv;
  a.gq = c.hq / c.hkv;
  a.status = reinterpret_cast<int*>(ws);
  a.counters = reinterpret_cast<int*>(ws + PKV_STATUS_BYTES);
  a.partials = reinterpret_cast<float*>(ws + PKV_STATUS_BYTES + decode_counter_bytes(c.batch, c.hkv));
  a.tagged = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(a.partials) +
                                         static_cast<size_t>(2) * grid * Geo::kPieceB);
  CUtensorMap kmap, vmap;
  const int rc = encode_page_maps(c.k_pages, c.v_pages, Geo::D, c.num_pages, c.hkv, &kmap, &vmap);
  if (rc != PKV_OK) return rc;
  const int launch_grid = c.num_sms * occ < kMaxGrid ? c.num_sms * occ : kMaxGrid;
  return launch_pdl(kern, dim3(launch_grid), dim3(kDecThreads), smem, c.stream, kmap, vmap, a) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // namespace pkv
