// prefill.cu -- chunked-prefill attention on the 5th-generation tensor cores.
//
// Source of the operation: a long prompt is prefilled in 4096-token chunks,
// one per scheduler step, interleaved with other requests' decode steps
// ("Optimizing ASR for 90-minute multi-speaker audio", section "Chunked
// prefill for long audio"). Row i of a chunk that follows P cached tokens sits
// at absolute position P + i and attends keys 0 .. P + i (bottom-right causal).
//
// This is a dense contraction (about 1300 flop per byte), so it runs on
// tcgen05.mma with accumulators in tensor memory:
//
//  * A CTA owns 128 query rows of one request and one KV head, i.e. two
//    128 x 128 query tiles (the two query heads of the GQA group) that share
//    every K/V tile it loads.
//  * Warp 9 (TMA) loads both query tiles once and then K/V tiles of 128 keys
//    through the block table, one page (16 rows x 64 columns, 128-byte
//    swizzle) per tiled TMA load, into a 2-stage ring.
//  * Warp 8 (MMA) issues, per K/V tile and query head h, S_h = Q_h K^T
//    (M = N = 128, K = 128 in 8 steps of 16) into TMEM, then, once the softmax
//    warps have written P_h back into TMEM, O_h += P_h V with P_h as the
//    tensor-memory A operand and V as an MN-major shared-memory B operand. The
//    issue order PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1) keeps the two heads'
//    softmaxes half a period apart, so one head's MMAs fill the other's softmax.
//  * Warps 0-3 and 4-7 (one warpgroup per query head, one thread per row; 224
//    registers each after a setmaxnreg rebalance, warps 10-11 only donate theirs) read
//    S_h from TMEM, apply the scale and the causal mask, keep the running max
//    and sum, and store P_h = exp2(s - m) as bf16 over S_h's first 64 columns.
//    The O accumulator is rescaled in TMEM only when a row's max grows by more
//    than 2^8 (otherwise the stale max is kept; the final O / l is unchanged).
//  * TMEM: S_0, S_1, O_0, O_1, 128 columns each (512 allocated, 1 CTA per SM).
//  * Work is a list of items (request, KV head, 128-row query tile), each
//    needing 1 + (cached + covered rows) / 128 key tiles. Two schedules, chosen
//    on the device from the lengths: when the largest item is comparable to
//    a CTA's fair share, one CTA per item, dispatched heaviest first (the
//    hardware's dispatch is a longest-first list schedule); when there are
//    many more key tiles than SMs can balance in whole items (long cached
//    prefixes), one persistent CTA per SM takes an equal share of key tiles,
//    cutting items, and the CTA that completes an item merges its partial
//    results (fp16 O / l, fp32 max and sum; log-sum-exp).
#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_kernels.h"
#include "pkv_mma.cuh"
#include "pkv_tc.cuh"

namespace pkv {

constexpr int kPfRows = 128;                 // query rows per CTA
constexpr int kPfKeys = 128;                 // keys per K/V tile
constexpr int kPfPagesPerTile = kPfKeys / kPageSize;
constexpr int kPfMmaWarp = 8;
constexpr int kPfTmaWarp = 9;
constexpr int kPfThreads = 12 * 32;        // 3 warpgroups: softmax head 0, softmax head 1, MMA + TMA (+2 idle)
// Register split: the launch gives every thread 168 registers (12 warps, 3 per
// SM sub-partition); the MMA/TMA warpgroup drops to 56 and the two softmax
// warpgroups rise to 224 ((224 + 224 + 56) * 32 <= 16384 per sub-partition,
// and the CTA total stays 384 * 168).
constexpr int kPfRegsSoftmax = 224;
constexpr int kPfRegsOther = 56;
static_assert(2 * 128 * kPfRegsSoftmax + 128 * kPfRegsOther <= kPfThreads * 168, "register split");
// The mixed-step kernel carries the decode CTAs' code and the decode-page scan as well; there the
// MMA/TMA warpgroup gets 16 more registers and the softmax ones 8 fewer (at 224 / 56 its split schedule
// measured 25 % slower than the prefill kernel's; 216 / 72 was the best of the splits tried).
template <bool kMixed>
struct PfRegs {
  static constexpr int kSoftmax = kMixed ? 216 : kPfRegsSoftmax;
  static constexpr int kOther = kMixed ? 72 : kPfRegsOther;
  static_assert(2 * 128 * kSoftmax + 128 * kOther <= kPfThreads * 168, "register split");
};
constexpr int kPfHalfBytes = kPfRows * 128;  // one 64-column half of a 128-row bf16 tile: 16 KiB
constexpr int kPfStages = 2;
constexpr int kNumBars = 14;
constexpr int kPfMaxSeqs = 1024;  // request prefix sums live in shared memory

// Sizes that depend on the head dimension HD (64 or 128): a 128-row tile of Q,
// K or V is HD / 64 halves of 64 columns (128-byte rows, 128-byte swizzle).
template <int HD>
struct PfDim {
  static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
  static constexpr int kHalves = HD / 64;
  static constexpr int kTileBytes = kHalves * kPfHalfBytes;
  static constexpr int kPageBytes = kPageSize * HD * 2;  // one page of K (or V) of one KV head
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kOffQ = 0;                                 // Q_0, Q_1
  static constexpr int kOffV = kOffQ + 2 * kTileBytes;            // V stages
  static constexpr int kOffK = kOffV + kPfStages * kTileBytes;    // K stages
  static constexpr int kOffBars = kOffK + kPfStages * kTileBytes;
  // + tmem address, fail flag, two merge flags; alignment slack (the request prefix sums follow).
  // head_dim 64 pads the CTA to more than half the SM's shared memory: one CTA per SM, since each
  // holds all 512 TMEM columns
  static constexpr int kSmemBytes =
      (kOffBars + kNumBars * 8 + 16 + 1024) > 120 * 1024 ? (kOffBars + kNumBars * 8 + 16 + 1024) : 120 * 1024;
  // Partial record of a split piece, per query head slot: the piece's normalised output O / l as
  // fp16, 4 dims per 8-byte word laid out [dim / 4][row] (a warp's 32 rows are one coalesced
  // 256-byte line per word), then the rows' running max (log2 units) and sum as fp32.
  static constexpr int kRecO = HD / 4 * kPfRows * 8;
  static constexpr int kRecHeadBytes = kRecO + 2 * kPfRows * 4;
  static constexpr int kRecBytes = 2 * kRecHeadBytes;
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, HD, true);  // B = V tile, MN-major
};

// + the request prefix sums of cost units and of items, the schedule, the CTA's share (lo, hi, U, G), each
// softmax group's pending split pieces and the split schedule's worker count, as 64-bit words
template <int HD>
static size_t pf_smem_bytes(int num_seqs) {
  return PfDim<HD>::kSmemBytes + static_cast<size_t>(2 * (num_seqs + 1) + 1 + 4 + 4 + 1) * 8;
}

// Item mode (no item is split) when the largest item is at least this share
// (in percent) of a CTA's average number of key tiles; split mode otherwise.
#ifndef PKV_PF_ITEM_MODE_PCT
#define PKV_PF_ITEM_MODE_PCT 75
#endif

// TMEM columns
constexpr uint32_t kColS = 0;    // S_h at kColS + 128 h
constexpr uint32_t kColO = 256;  // O_h at kColO + 128 h
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false);  // B = K tile, K-major

// A CTA holds two query-head slots of one KV head: head pair p of KV head g is
// query heads g G + 2p and g G + 2p + 1 (G query heads per KV head). With an
// odd G the last pair has one head; its second slot repeats the first head and
// its output is not written.
struct PrefillArgs {
  const int* block_table;
  const int* prefix_lens;
  const int* cu_q_lens;
  __nv_bfloat16* out;
  int num_seqs;
  int total_q;
  int max_pages;
  int num_pages;
  int tmax;     // query tiles computed per request: ceil(max_q_len / 128)
  int workers;  // split mode: persistent CTAs (one per SM); the grid has max(workers, items) CTAs
  int hq;       // query heads
  int hkv;      // KV heads
  int grp;      // query heads per KV head
  int npair;    // head pairs per KV head: ceil(grp / 2)
  int pairs;    // head pairs per request: hkv * npair
  float scale_log2;
  int* status;
  int* counters;   // [num_seqs][pairs][tmax][2], zero between calls
  unsigned char* records;  // [2 * workers][PfDim::kRecBytes]
  // the mixed step (kMixed): decode requests attended in the same launch, one CTA per (request, KV
  // head) after the pcta prefill CTAs; the same pools, their own block table and lengths
  const __nv_bfloat16* dq;  // [dbatch][16][128]
  const int* dbt;           // [dbatch][dmax_pages]
  const int* dlens;         // [dbatch]
  __nv_bfloat16* dout;      // [dbatch][16][128]
  int dbatch;
  int dmax_pages;
  int dmaxc;     // decode chunks per (request, KV head) at most: ceil(dmax_pages / 64)
  float* drec;   // [dbatch][8][dmaxc][2][132] partial records of chunked pairs
  int* dcnt;     // [dbatch][8] chunk counters, zero between calls
  int pcta;  // prefill CTAs of the grid: max(items, workers)
};

// Head counts of a launch: compile-time constants for the Qwen3 decoder's 16 query / 8 KV heads
// (kFixed; its kernel keeps the register allocation and schedule tuned for it), the launch's
// arguments for other geometries.
template <bool kFixed>
struct PfHeads {
  __device__ __forceinline__ static int hq(const PrefillArgs& a) { return kFixed ? kQHeads : a.hq; }
  __device__ __forceinline__ static int hkv(const PrefillArgs& a) { return kFixed ? kKVHeads : a.hkv; }
  __device__ __forceinline__ static int grp(const PrefillArgs& a) { return kFixed ? kGroup : a.grp; }
  __device__ __forceinline__ static int npair(const PrefillArgs& a) { return kFixed ? (kGroup + 1) / 2 : a.npair; }
  __device__ __forceinline__ static int pairs(const PrefillArgs& a) {
    return kFixed ? kKVHeads * ((kGroup + 1) / 2) : a.pairs;
  }
};

// KV head, first query head, and whether the second slot holds a head of its own, of head pair hp.
template <bool kFixed>
__device__ __forceinline__ void pf_pair_heads(const PrefillArgs& a, int hp, int& g, int& qh0, bool& two) {
  using Hd = PfHeads<kFixed>;
  g = hp / Hd::npair(a);
  const int p = hp - g * Hd::npair(a);
  qh0 = g * Hd::grp(a) + 2 * p;
  two = 2 * p + 1 < Hd::grp(a);
}

struct PfBars {
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t k_full[kPfStages];
  uint64_t v_full[kPfStages];
  uint64_t kv_empty[kPfStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
};
static_assert(sizeof(PfBars) == kNumBars * 8, "barrier block");

// Bounded wait that gives up at once after any wait of the CTA has timed out.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile int* fail, int* status) {
  if (*fail) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *fail = 1;
  set_status(status, PKV_ERR_DEVICE_TIMEOUT);
  return false;
}

// Warp-collective form: every lane waits and the warp agrees on the outcome
// (the tcgen05.ld/st that follow are warp-wide). A phase that has already
// completed costs one try_wait: the CTA's failure flag (a volatile shared load
// in front of every wait) is read only on the slow path. The MMA issuer's
// waits sit between its MMA batches, so their cost is idle tensor-pipe time.
__device__ __forceinline__ bool pf_wait_warp(uint64_t* bar, uint32_t parity, volatile int* fail, int* status) {
  if (__all_sync(0xffffffffu, mbar_try_wait(smem_u32(bar), parity))) return true;
  return __all_sync(0xffffffffu, pf_wait(bar, parity, fail, status));
}
// Two waits with one poll when both phases have already completed.
__device__ __forceinline__ bool pf_wait_warp2(uint64_t* b1, uint32_t p1, uint64_t* b2, uint32_t p2, volatile int* fail,
                                              int* status) {
  if (__all_sync(0xffffffffu, mbar_try_wait(smem_u32(b1), p1) && mbar_try_wait(smem_u32(b2), p2))) return true;
  return pf_wait_warp(b1, p1, fail, status) && pf_wait_warp(b2, p2, fail, status);
}

// Work is a list of items (request n, KV head g, query tile t), ordered by n,
// then g, then t. Query tile t of a request with P cached tokens and qlen chunk
// rows needs n_t = ceil((P + min(128 (t + 1), qlen)) / 128) key tiles. Shares
// are cut in cost units: an item costs kPfItemCost units for its fixed work (the
// query tile load, the pipeline fill and drain, the epilogue) followed by one
// unit per key tile, so a CTA whose share holds many small items gets fewer key
// tiles. A (request, head pair) costs W = sum over its items; pref[n] = pairs * sum
// of W before n. A piece is the part of one item inside a CTA's share that holds key
// tiles: [k0, k1).
#ifndef PKV_PF_ITEM_COST
#define PKV_PF_ITEM_COST 2
#endif
constexpr int kPfItemCost = PKV_PF_ITEM_COST;
struct PfPiece {
  int n, hp, t, k0, k1, nt, q0, qlen, P;  // hp: head pair of the request
  long long fseg, fend;  // the item's cost units start at fseg; the piece ends at fend
};

__device__ __forceinline__ int pf_tiles(int P, int qlen, int t) {
  const int rows = qlen < kPfRows * (t + 1) ? qlen : kPfRows * (t + 1);
  return (P + rows + kPfKeys - 1) / kPfKeys;
}
// Query tiles computed for a request (at most tmax) and the units before tile t
// (tiles before the last are full: n_s = ceil(P / 128) + s + 1).
__device__ __forceinline__ int pf_qtiles(int qlen, int tmax) {
  const int T = (qlen + kPfRows - 1) / kPfRows;
  return T < tmax ? T : tmax;
}
__device__ __forceinline__ long long pf_units_before(int P, int t) {
  const long long c = (P + kPfKeys - 1) / kPfKeys;
  return static_cast<long long>(t) * (c + kPfItemCost) + static_cast<long long>(t) * (t + 1) / 2;
}

// Split mode: a request's items are ordered by KV head, then query tile; the
// first `workers` CTAs (one per SM) each take an equal contiguous share of the
// cost units, cutting through items, whose partial results are merged
// afterwards. (Item mode, CTA b computing item b of each request's items taken
// heaviest first, needs no pieces.)
template <bool kFixed>
__device__ __forceinline__ bool pf_find_piece(long long f, long long hi, const long long* pref, const PrefillArgs& a,
                                              PfPiece& pc) {
  for (; f < hi; f = pc.fend) {
    int lo_n = 0, hi_n = a.num_seqs - 1;
    while (lo_n < hi_n) {
      const int mid = (lo_n + hi_n + 1) >> 1;
      if (pref[mid] <= f) lo_n = mid; else hi_n = mid - 1;
    }
    pc.n = lo_n;
    pc.q0 = __ldg(a.cu_q_lens + lo_n);
    pc.qlen = __ldg(a.cu_q_lens + lo_n + 1) - pc.q0;
    pc.P = __ldg(a.prefix_lens + lo_n);
    const long long W = (pref[lo_n + 1] - pref[lo_n]) / PfHeads<kFixed>::pairs(a);
    const long long off = f - pref[lo_n];
    pc.hp = static_cast<int>(off / W);
    const long long o2 = off - pc.hp * W;
    int lo_t = 0, hi_t = pf_qtiles(pc.qlen, a.tmax) - 1;
    while (lo_t < hi_t) {
      const int mid = (lo_t + hi_t + 1) >> 1;
      if (pf_units_before(pc.P, mid) <= o2) lo_t = mid; else hi_t = mid - 1;
    }
    pc.t = lo_t;
    pc.nt = pf_tiles(pc.P, pc.qlen, pc.t);
    const long long ub = pf_units_before(pc.P, pc.t);
    const long long p0 = o2 - ub;  // position inside the item: fixed-cost units, then key tiles
    const long long p_end = p0 + (hi - f);
    const long long p1 = p_end < kPfItemCost + pc.nt ? p_end : kPfItemCost + pc.nt;
    pc.k0 = static_cast<int>(p0 > kPfItemCost ? p0 - kPfItemCost : 0);
    pc.k1 = static_cast<int>(p1 - kPfItemCost);
    pc.fseg = pref[lo_n] + pc.hp * W + ub;
    pc.fend = f + (p1 - p0);
    if (pc.k1 > pc.k0) return true;
  }
  return false;
}

// CTA whose share [c U / G, (c + 1) U / G) holds unit f.
__device__ __forceinline__ int pf_cta_of(long long f, long long U, int G) {
  return static_cast<int>(((f + 1) * G + U - 1) / U - 1);
}
__device__ __forceinline__ long long pf_share_lo(int c, long long U, int G) { return static_cast<long long>(c) * U / G; }

__device__ __forceinline__ void pf_group_sync(int h) {  // the 128 softmax threads of query head h
  asm volatile("bar.sync %0, 128;" ::"r"(2 + h) : "memory");
}

// A decode page of one KV head costs this fraction of a prefill key tile of SM time (the split
// schedule of the mixed step keeps SMs apart for the decode CTAs in proportion): a key tile of both
// query heads takes about 2 us of an SM; a decode CTA keeps 24 pages (192 KiB) in flight and streams a
// page (8 KiB of K and V) in about 0.09 us. (16, 24, 32 and 64 measured within 2 % of each other.)
#ifndef PKV_MIXED_PAGES_PER_TILE
#define PKV_MIXED_PAGES_PER_TILE 24
#endif
// Pages of one (request, KV head) per decode CTA of the mixed step; longer contexts are cut into
// chunks whose partial results are merged by the CTA that completes the pair's count.
// (64 measured faster than 128 and 256: more CTAs stream at once.)
#ifndef PKV_MIXED_CHUNK_PAGES
#define PKV_MIXED_CHUNK_PAGES 64
#endif
constexpr int kMixChunkPages = PKV_MIXED_CHUNK_PAGES;
constexpr int kMixStages = 3;  // the two K/V stages of the prefill CTA and the Q area
constexpr int kMixRec = kHeadDim + 4;  // floats per head of a partial record: o[128], m, l, 2 pad
static int mixed_chunks_per_pair(int dmax_pages) { return (dmax_pages + kMixChunkPages - 1) / kMixChunkPages; }

// Pages of all (request, KV head) pairs of the mixed step's decode batch (lengths clamped to the
// block table), summed over the warp. Kept out of line: inlined, its code changed the register
// allocation of the prefill roles' loops.
__device__ __noinline__ long long mixed_decode_pages(const int* dlens, int dbatch, int dmax_pages) {
  const int lane = threadIdx.x & 31;
  long long pages = 0;
  for (int base = 0; base < dbatch; base += 32) {
    const int n = base + lane;
    if (n < dbatch) {
      const int len = __ldg(dlens + n);
      const int cl = len < 0 ? 0 : (len > dmax_pages * kPageSize ? dmax_pages * kPageSize : len);
      pages += kKVHeads * ((cl + kPageSize - 1) / kPageSize);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pages += __shfl_xor_sync(0xffffffffu, pages, o);
  return pages;
}

// Decode CTA of the mixed step: decode attention of one chunk of <= 64 pages of one (request b, KV
// head g) pair of the decode batch, in a CTA shaped like the prefill ones. Warp 9 copies the chunk's
// pages, 8 per 128-key tile, into three stages (the prefill K/V stages and the Q area) through the
// decode block table, reading a tile's page ids one tile ahead; warps 0-7 take page w of every tile and
// run the warp-level tensor-core page step of the decode kernels on it (S^T = K Q^T for the group's two
// query heads, online softmax, O^T += V^T P^T; a page's two 64-dim boxes lie 16 KiB apart in a stage),
// then merge their (o, m, l) states through shared memory. A pair in one chunk writes its bf16 rows;
// otherwise the chunk writes a partial record and counts itself in (fence, atomic), and the CTA that
// completes the count merges the pair's records (log-sum-exp, in chunk order) and resets the counter.
// Every consumer warp waits for every tile before it frees the stage (8 arrivals per phase), so none
// runs ahead of the stage ring. Kept out of line, like mixed_decode_pages.
__device__ __noinline__ void mixed_decode_cta(const PrefillArgs& a, const CUtensorMap* kmap,
                                                 const CUtensorMap* vmap, PfBars* bars, unsigned char* sQ,
                                                 unsigned char* sK, unsigned char* sV, volatile int* fail,
                                                 long long* scratch, int warp, int lane) {
  using Dm = PfDim<128>;
  constexpr int kKS = kHeadDim / 16;
  const int tid = threadIdx.x;
  if (tid == 32) {  // the stages' barriers: full ones completed by the copies, empty ones by 8 warps
    for (int st = 0; st < 2; ++st) {
      mbar_init(&bars->k_full[st], 1);
      mbar_init(&bars->v_full[st], 1);
      mbar_init(&bars->kv_empty[st], 8);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->p_full[0], 8);
    *fail = 0;
    fence_barrier_init();
  }
  // ---- which chunk: chunks are ordered by request, KV head, chunk; request b has nc_b chunks per head
  // (at least one: an empty request writes zeros)
  const long long e = static_cast<long long>(blockIdx.x) - a.pcta;
  if (warp == 0) {
    long long carry = 0;
    int found = -1;
    for (int base = 0; base < a.dbatch && found < 0; base += 32) {
      const int n = base + lane;
      long long cnt = 0;
      if (n < a.dbatch) {
        int len = __ldg(a.dlens + n);
        len = len < 0 ? 0 : (len > a.dmax_pages * kPageSize ? a.dmax_pages * kPageSize : len);
        const int np = (len + kPageSize - 1) / kPageSize;
        cnt = kKVHeads * static_cast<long long>(np > 0 ? (np + kMixChunkPages - 1) / kMixChunkPages : 1);
      }
      long long x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const bool mine = n < a.dbatch && e >= carry + x - cnt && e < carry + x;
      const unsigned hit = __ballot_sync(0xffffffffu, mine);
      if (hit != 0u) {
        const int src = __ffs(hit) - 1;
        found = base + src;
        if (lane == src) {
          const long long off = e - (carry + x - cnt);  // chunk index within the request: g * nc + c
          const long long nc = cnt / kKVHeads;
          scratch[0] = n;
          scratch[1] = off / nc;  // g
          scratch[2] = off % nc;  // c
          scratch[3] = nc;
        }
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (found < 0 && lane == 0) scratch[0] = -1;  // past the last chunk
  }
  __syncthreads();
  const int b = static_cast<int>(scratch[0]);
  if (b < 0) return;
  const int g = static_cast<int>(scratch[1]), ci = static_cast<int>(scratch[2]), nc = static_cast<int>(scratch[3]);
  int len = __ldg(a.dlens + b);
  const int cap = a.dmax_pages * kPageSize;
  if (len < 0 || len > cap) {
    if (tid == 0 && g == 0 && ci == 0) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
    len = len < 0 ? 0 : cap;
  }
  const int np = (len + kPageSize - 1) / kPageSize;
  const int pg0 = ci * kMixChunkPages;                                    // the chunk's first page
  const int pg1 = np < pg0 + kMixChunkPages ? np : pg0 + kMixChunkPages;  // and its end
  const int ntl = pg1 > pg0 ? (pg1 - pg0 + kPfPagesPerTile - 1) / kPfPagesPerTile : 0;
  __nv_bfloat16* orow = a.dout + (static_cast<size_t>(b) * kQHeads + kGroup * g) * kHeadDim;
  // stage s: K and V tiles and their barriers (the third stage is the Q area, on the S/P barriers)
  auto kst = [&](int st) { return st < 2 ? sK + st * Dm::kTileBytes : sQ; };
  auto vst = [&](int st) { return st < 2 ? sV + st * Dm::kTileBytes : sQ + Dm::kTileBytes; };
  auto kfull = [&](int st) { return st < 2 ? &bars->k_full[st] : &bars->s_full[0]; };
  auto vfull = [&](int st) { return st < 2 ? &bars->v_full[st] : &bars->s_full[1]; };
  auto empty = [&](int st) { return st < 2 ? &bars->kv_empty[st] : &bars->p_full[0]; };

  if (warp == kPfTmaWarp) {
    // ------------------------------------------------------------------ page copies
    auto page_id = [&](int j) {  // this lane's page of tile j (-1: none or outside the pool)
      const int pg = pg0 + j * kPfPagesPerTile + lane;
      int id = -1;
      if (lane < kPfPagesPerTile && pg < pg1) {
        id = __ldg(a.dbt + static_cast<size_t>(b) * a.dmax_pages + pg);
        if (id < 0 || id >= a.num_pages) {
          set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
          id = -1;
        }
      }
      return id;
    };
    int id_next = ntl > 0 ? page_id(0) : -1;
    for (int j = 0; j < ntl; ++j) {
      const int st = j % kMixStages;
      const int use = j / kMixStages;
      const int id = id_next;
      if (j + 1 < ntl) id_next = page_id(j + 1);  // the next tile's ids while this one waits for its stage
      if (use > 0 && !pf_wait_warp(empty(st), static_cast<uint32_t>(use - 1) & 1u, fail, a.status)) break;
      const bool valid = id >= 0;
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      const uint32_t bytes = static_cast<uint32_t>(__popc(vmask)) * static_cast<uint32_t>(Dm::kPageBytes);
      if (lane == 0) {
        mbar_arrive_expect_tx(kfull(st), bytes);
        mbar_arrive_expect_tx(vfull(st), bytes);
      }
      __syncwarp();
      if (valid) {
        const int row = (id * kKVHeads + g) * kPageSize;
        unsigned char* kd = kst(st) + lane * (kPageSize * 128);
        unsigned char* vd = vst(st) + lane * (kPageSize * 128);
        tma_load_2d(kd, kmap, 0, row, kfull(st));
        tma_load_2d(kd + kPfHalfBytes, kmap, 64, row, kfull(st));
        tma_load_2d(vd, vmap, 0, row, vfull(st));
        tma_load_2d(vd + kPfHalfBytes, vmap, 64, row, vfull(st));
      }
    }
  }

  constexpr int kRec = kMixRec;
  float* st_all = reinterpret_cast<float*>(sK);  // the warps' states, once every stage is drained
  if (warp < 8) {
    // ------------------------------------------------------------------ consumers: page w of every tile
    const int r = lane >> 2, c = lane & 3;
    uint32_t qf[kKS][2];  // Q^T as the B operand: head r of the group (rows r >= 2 zero)
    {
      const bool live = r < kGroup;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          a.dq + (static_cast<size_t>(b) * kQHeads + kGroup * g + (live ? r : 0)) * kHeadDim);
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        qf[ks][0] = live ? __ldg(qrow + 8 * ks + c) : 0u;
        qf[ks][1] = live ? __ldg(qrow + 8 * ks + 4 + c) : 0u;
      }
    }
    uint32_t koff[kKS], voff[kKS];
    mma_offsets<kKS, kPfHalfBytes>(koff, voff);
    float o[kKS][4];
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) o[ks][0] = o[ks][1] = o[ks][2] = o[ks][3] = 0.f;
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
    bool ok = true;
    for (int j = 0; j < ntl; ++j) {
      const int st = j % kMixStages;
      const uint32_t ph = static_cast<uint32_t>(j / kMixStages) & 1u;
      ok = ok && pf_wait_warp(kfull(st), ph, fail, a.status) && pf_wait_warp(vfull(st), ph, fail, a.status);
      const int p = pg0 + j * kPfPagesPerTile + warp;
      if (ok && p < pg1) {
        const int rem = len - p * kPageSize;
        const uint32_t kt = smem_u32(kst(st) + warp * (kPageSize * 128));
        const uint32_t vt = smem_u32(vst(st) + warp * (kPageSize * 128));
        mma_page<kKS>(kt, vt, koff, voff, qf, rem < kPageSize ? rem : kPageSize, a.scale_log2, o, m0, m1, l0, l1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(empty(st));
    }
#pragma unroll
    for (int m = 4; m < 32; m <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, m);
      l1 += __shfl_xor_sync(0xffffffffu, l1, m);
    }
    // every stage is drained (each warp waited for every tile), so stage 0 holds the states:
    // [warp][head][128 + 4] floats
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (c == 0) {  // lanes c == 0 hold heads 0 and 1 of the group
      float* wst = st_all + warp * kGroup * kRec;
#pragma unroll
      for (int n = 0; n < kGroup; ++n) {
#pragma unroll
        for (int ks = 0; ks < kKS; ++ks) {
          wst[n * kRec + 16 * ks + r] = o[ks][n];
          wst[n * kRec + 16 * ks + r + 8] = o[ks][2 + n];
        }
        if (r == 0) {
          wst[n * kRec + kHeadDim] = n ? m1 : m0;
          wst[n * kRec + kHeadDim + 1] = n ? l1 : l0;
        }
      }
    }
  }
  __syncthreads();
  if (*fail) return;
  // ---- merge the 8 warps' states: one thread per (head, dim); the chunk's result is (O, M, L) with
  // O = sum_w o_w 2^(m_w - M), L = sum_w l_w 2^(m_w - M), M = max_w m_w (log2 units)
  float* rec = a.drec + ((static_cast<size_t>(b) * kKVHeads + g) * a.dmaxc + ci) * (kGroup * kRec);
  if (tid < 256) {
    const int n = tid >> 7, d = tid & 127;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < 8; ++w) M = fmaxf(M, st_all[(w * kGroup + n) * kRec + kHeadDim]);
    float L = 0.f, O = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float* ws = st_all + (w * kGroup + n) * kRec;
        const float ew = ex2(ws[kHeadDim] - M);  // a warp without pages: m = -inf, weight 0
        L += ws[kHeadDim + 1] * ew;
        O += ws[d] * ew;
      }
    }
    if (nc == 1) {
      orow[n * kHeadDim + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);  // an empty request: zeros
    } else {
      rec[n * kRec + d] = O;
      if (d == 0) {
        rec[n * kRec + kHeadDim] = M;
        rec[n * kRec + kHeadDim + 1] = L;
      }
    }
  }
  if (nc == 1) return;
  // ---- count the chunk in (release); the CTA completing the pair's count merges (acquire)
  __syncthreads();
  volatile int* merge_flag = reinterpret_cast<volatile int*>(scratch + 4);
  int* counter = a.dcnt + static_cast<size_t>(b) * kKVHeads + g;
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(counter, 1);
    __threadfence();
    *merge_flag = old == nc - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!*merge_flag) return;
  if (tid < 256) {
    const int n = tid >> 7, d = tid & 127;
    const float* recs = a.drec + (static_cast<size_t>(b) * kKVHeads + g) * a.dmaxc * (kGroup * kRec);
    float M = -CUDART_INF_F;
    for (int k = 0; k < nc; ++k) M = fmaxf(M, __ldcg(recs + (k * kGroup + n) * kRec + kHeadDim));
    float L = 0.f, O = 0.f;
    for (int k = 0; k < nc; ++k) {  // chunk order: the same bits whichever CTA merges
      const float* rk = recs + (k * kGroup + n) * kRec;
      const float mk = __ldcg(rk + kHeadDim);
      const float ek = mk == -CUDART_INF_F ? 0.f : ex2(mk - M);
      L += __ldcg(rk + kHeadDim + 1) * ek;
      O += __ldcg(rk + d) * ek;
    }
    orow[n * kHeadDim + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
  }
  if (tid == 0) *counter = 0;
}

template <int HD, bool kFixed, bool kMixed>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // 1024-byte aligned for 128-byte swizzle atoms
  using Dm = PfDim<HD>;
  using Hd = PfHeads<kFixed>;
  static_assert(!kMixed || (HD == 128 && kFixed), "the mixed step serves the 16/8/128 geometry");
  PfBars* bars = reinterpret_cast<PfBars*>(smem + Dm::kOffBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Dm::kOffBars + kNumBars * 8);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2]
  long long* pref = reinterpret_cast<long long*>(tmem_slot + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  grid_dependency_wait();
  allow_dependents();
  if constexpr (kMixed) {
    // the mixed step: CTAs past the prefill ones attend a chunk of a decode (request, KV head) each
    // (a path of their own, so the prefill roles keep their registers)
    if (static_cast<int>(blockIdx.x) >= a.pcta) {
      mixed_decode_cta(a, &kmap, &vmap, bars, smem + Dm::kOffQ, smem + Dm::kOffK, smem + Dm::kOffV, fail, pref, warp,
                       lane);
      return;
    }
  }

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bars->s_full[h], 1);
      mbar_init(&bars->p_full[h], 128);
      mbar_init(&bars->o_done[h], 1);
    }
    *fail = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    // units per request (pairs W_n; 0 for a request whose shape is out of bounds) and their exclusive prefix
    long long carry = 0, icarry = 0, tiles_all = 0;
    int nt_max = 0;
    long long* ipref = pref + a.num_seqs + 2;
    const long long cap = static_cast<long long>(a.max_pages) * kPageSize;
    for (int base = 0; base < a.num_seqs; base += 32) {
      const int n = base + lane;
      long long w8 = 0, items = 0;
      if (n < a.num_seqs) {
        const int q0 = __ldg(a.cu_q_lens + n), q1 = __ldg(a.cu_q_lens + n + 1);
        const int P = __ldg(a.prefix_lens + n);
        const int qlen = q1 - q0;
        const int T = qlen > 0 ? pf_qtiles(qlen, a.tmax) : 0;
        const long long rows = qlen < kPfRows * T ? qlen : static_cast<long long>(kPfRows) * T;
        if (P < 0 || q0 < 0 || qlen < 0 || q1 > a.total_q || static_cast<long long>(P) + rows > cap) {
          set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
        } else if (T > 0) {
          // a chunk longer than the caller's max_q_len bound: its rows past the first tmax query
          // tiles are not computed, so the call reports it
          if (qlen > static_cast<long long>(kPfRows) * a.tmax) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
          const int nt_last = pf_tiles(P, qlen, T - 1);
          w8 = Hd::pairs(a) * (pf_units_before(P, T - 1) + kPfItemCost + nt_last);
          tiles_all += w8 - static_cast<long long>(Hd::pairs(a)) * kPfItemCost * T;
          items = static_cast<long long>(Hd::pairs(a)) * T;
          nt_max = nt_max > nt_last ? nt_max : nt_last;
        }
      }
      long long x = w8, xi = items;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        const long long yi = __shfl_up_sync(0xffffffffu, xi, o);
        if (lane >= o) {
          x += y;
          xi += yi;
        }
      }
      if (n < a.num_seqs) {
        pref[n] = carry + x - w8;
        ipref[n] = icarry + xi - items;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
      icarry += __shfl_sync(0xffffffffu, xi, 31);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tiles_all += __shfl_xor_sync(0xffffffffu, tiles_all, o);
      nt_max = max(nt_max, __shfl_xor_sync(0xffffffffu, nt_max, o));
    }
    // the mixed step: decode pages of all pairs (their CTAs follow the prefill ones)
    const long long dec_pages = kMixed ? mixed_decode_pages(a.dlens, a.dbatch, a.dmax_pages) : 0;
    if (lane == 0) {
      pref[a.num_seqs] = carry;
      ipref[a.num_seqs] = icarry;
      const bool items_mode =
          100LL * nt_max * a.workers >= static_cast<long long>(PKV_PF_ITEM_MODE_PCT) * tiles_all;
      pref[a.num_seqs + 1] = items_mode;
      // Split schedule of the mixed step: leave k SMs to the decode CTAs, k in proportion to the decode
      // pages' share of the SM time (item mode needs none: the decode CTAs fill the SMs its tail frees).
      long long workers = a.workers;
      if (kMixed && !items_mode && dec_pages > 0) {
        const long long dec_tiles = (dec_pages + PKV_MIXED_PAGES_PER_TILE - 1) / PKV_MIXED_PAGES_PER_TILE;
        long long k = (static_cast<long long>(a.workers) * dec_tiles + dec_tiles + tiles_all - 1) / (dec_tiles + tiles_all);
        k = k < 1 ? 1 : (k > a.workers / 2 ? a.workers / 2 : k);
        workers = a.workers - k;
      }
      pref[2 * a.num_seqs + 11] = workers;
    }
  }
  if (warp == kPfMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  unsigned char* sQ = smem + Dm::kOffQ;
  unsigned char* sV = smem + Dm::kOffV;
  unsigned char* sK = smem + Dm::kOffK;

  const bool item_mode = pref[a.num_seqs + 1] != 0;

  if (item_mode) {
    // ================================================================ item mode: CTA b computes item b
    const long long* ipref = pref + a.num_seqs + 2;
    const long long b = blockIdx.x;
    if (b < ipref[a.num_seqs]) {
      int n = 0, hi_n = a.num_seqs - 1;
      while (n < hi_n) {
        const int mid = (n + hi_n + 1) >> 1;
        if (ipref[mid] <= b) n = mid; else hi_n = mid - 1;
      }
      const int q0 = __ldg(a.cu_q_lens + n);
      const int qlen = __ldg(a.cu_q_lens + n + 1) - q0;
      const int P = __ldg(a.prefix_lens + n);
      const int jj = static_cast<int>(b - ipref[n]);
      const int tile = pf_qtiles(qlen, a.tmax) - 1 - jj / Hd::pairs(a);  // heaviest first
      int g, qh0;
      bool two;
      pf_pair_heads<kFixed>(a, jj % Hd::pairs(a), g, qh0, two);
      const int i0 = tile * kPfRows;
      const int rows_here = qlen - i0 < kPfRows ? qlen - i0 : kPfRows;
      const int kv_end = P + i0 + rows_here;  // in bounds: the length scan dropped out-of-bounds requests
      const int n_tiles = (kv_end + kPfKeys - 1) / kPfKeys;
      const int n_pages = (kv_end + kPageSize - 1) / kPageSize;
    if (warp == kPfTmaWarp) {
      // ------------------------------------------------------------------ TMA producer
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kOther));
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full, 2 * Dm::kTileBytes);
        for (int h = 0; h < 2; ++h)
          for (int half = 0; half < Dm::kHalves; ++half)
            tma_load_3d(sQ + h * Dm::kTileBytes + half * kPfHalfBytes, &qmap, half * 64, qh0 + (two ? h : 0),
                        q0 + i0, &bars->q_full);
      }
      // this lane's page id of the first key tile, then of each next tile one tile ahead (the
      // block-table read is not on the path from a stage's release to its copies)
      int id_next = lane < kPfPagesPerTile && lane < n_pages
                        ? __ldg(a.block_table + static_cast<size_t>(n) * a.max_pages + lane) : 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j & 1;
        const int use = j >> 1;
        const int pg = j * kPfPagesPerTile + lane;
        const int id_cur = id_next;
        if (j + 1 < n_tiles && lane < kPfPagesPerTile && pg + kPfPagesPerTile < n_pages)
          id_next = __ldg(a.block_table + static_cast<size_t>(n) * a.max_pages + pg + kPfPagesPerTile);
        if (use > 0 && !pf_wait_warp(&bars->kv_empty[st], static_cast<uint32_t>(use - 1) & 1u, fail, a.status)) break;
        bool valid = lane < kPfPagesPerTile && pg < n_pages;
        int id = 0;
        if (valid) {
          id = id_cur;
          if (id < 0 || id >= a.num_pages) {
            set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
            valid = false;
          }
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        const uint32_t bytes = static_cast<uint32_t>(__popc(vmask)) * static_cast<uint32_t>(Dm::kPageBytes);
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->k_full[st], bytes);
          mbar_arrive_expect_tx(&bars->v_full[st], bytes);
        }
        __syncwarp();
        if (valid) {
          const int row = (id * Hd::hkv(a) + g) * kPageSize;
          unsigned char* kd = sK + st * Dm::kTileBytes + lane * (kPageSize * 128);
          unsigned char* vd = sV + st * Dm::kTileBytes + lane * (kPageSize * 128);
  #pragma unroll
          for (int half = 0; half < Dm::kHalves; ++half)  // K first: the QK MMA waits only for K
            tma_load_2d(kd + half * kPfHalfBytes, &kmap, 64 * half, row, &bars->k_full[st]);
  #pragma unroll
          for (int half = 0; half < Dm::kHalves; ++half)
            tma_load_2d(vd + half * kPfHalfBytes, &vmap, 64 * half, row, &bars->v_full[st]);
        }
      }
    } else if (warp == kPfMmaWarp) {
      // ------------------------------------------------------------------ MMA issuer
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kOther));
      // Issue order QK_0(0) QK_1(0) | PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1) | ...: the
      // two heads' softmaxes run half a period apart, so while one head's softmax
      // works the other head's PV and next QK keep the tensor pipe busy. QK_h(j+1)
      // overwrites S_h, which holds P_h(j), so it waits for PV_h(j) (o_done) --
      // which also keeps O_h out of the softmax's way while it may rescale it.
      auto issue_qk = [&](int j, int h) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t qa = smem_u32(sQ + h * Dm::kTileBytes);
          const uint32_t kb = smem_u32(sK + (j & 1) * Dm::kTileBytes);
  #pragma unroll
          for (int s = 0; s < HD / 16; ++s) {
            const uint32_t off = (s >> 2) * kPfHalfBytes + (s & 3) * 32;
            mma_ss(tmem + kColS + 128 * h, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                   kIdescQK, s > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[h]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int j, int h) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vb = smem_u32(sV + (j & 1) * Dm::kTileBytes);
  #pragma unroll
          for (int s = 0; s < 8; ++s) {
            mma_ts(tmem + kColO + 128 * h, tmem + kColS + 128 * h + 8 * s,
                   sdesc_sw128(vb + s * 2048, kPfHalfBytes, 1024), Dm::kIdescPV, (j > 0 || s > 0) ? 1u : 0u);
          }
          mma_commit(&bars->o_done[h]);
        }
        __syncwarp();
      };
      bool ok = pf_wait_warp(&bars->q_full, 0, fail, a.status) && pf_wait_warp(&bars->k_full[0], 0, fail, a.status);
      if (ok) {
        issue_qk(0, 0);
        issue_qk(0, 1);
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int st = j & 1;
        const uint32_t ph = static_cast<uint32_t>(j >> 1) & 1u;
        const bool next = j + 1 < n_tiles;
        const uint32_t ph_next = static_cast<uint32_t>((j + 1) >> 1) & 1u;
        if (!pf_wait_warp2(&bars->v_full[st], ph, &bars->p_full[0], static_cast<uint32_t>(j) & 1u, fail, a.status))
          break;
        if (j == n_tiles - 1 && kv_end < (j + 1) * kPfKeys) {
          // keys past the end: zero their V rows (unused slots may hold NaN and 0 * NaN = NaN)
          const int r0 = kv_end - j * kPfKeys;
          uint4* vbase = reinterpret_cast<uint4*>(sV + st * Dm::kTileBytes);
          for (int idx = r0 * 8 + lane; idx < kPfKeys * 8; idx += 32) {
  #pragma unroll
            for (int half = 0; half < Dm::kHalves; ++half) vbase[half * (kPfHalfBytes / 16) + idx] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        const uint32_t pj = static_cast<uint32_t>(j) & 1u;
        issue_pv(j, 0);
        if (next) {
          if (!pf_wait_warp2(&bars->k_full[st ^ 1], ph_next, &bars->o_done[0], pj, fail, a.status))
            break;
          issue_qk(j + 1, 0);
        }
        if (!pf_wait_warp(&bars->p_full[1], pj, fail, a.status)) break;
        issue_pv(j, 1);
        if (lane == 0) mma_commit(&bars->kv_empty[st]);
        __syncwarp();
        if (next) {
          if (!pf_wait_warp(&bars->o_done[1], pj, fail, a.status)) break;
          issue_qk(j + 1, 1);
        }
      }
    } else if (warp < 8) {
      // ------------------------------------------------------------------ softmax warpgroups
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kSoftmax));
      const int h = warp >> 2;
      const int quarter = warp & 3;
      const int r = quarter * 32 + lane;  // row of the tile = TMEM lane
      const int lim_row = P + i0 + r;     // last visible key of this row (causal)
      const int lim = lim_row < kv_end - 1 ? lim_row : kv_end - 1;
      const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      float m_used = -CUDART_INF_F;
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (!pf_wait_warp(&bars->s_full[h], static_cast<uint32_t>(j) & 1u, fail, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[4][32];
  #pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(t_row + kColS + 128 * h + 32 * c, sr[c]);
        tmem_ld_wait();
        const bool diag = j * kPfKeys + kPfKeys - 1 > P + i0;
        // row max over the raw scores (the scale is positive, so it keeps the order)
        float mx = -CUDART_INF_F;
        if (diag) {
  #pragma unroll
          for (int c = 0; c < 4; ++c)
  #pragma unroll
            for (int e = 0; e < 32; ++e) {
              if (j * kPfKeys + 32 * c + e > lim) sr[c][e] = __float_as_uint(-CUDART_INF_F);
              mx = fmaxf(mx, __uint_as_float(sr[c][e]));
            }
        } else {
  #pragma unroll
          for (int c = 0; c < 4; ++c)
  #pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sr[c][e]));
        }
        const float m_new = fmaxf(m_used, mx);
        const bool first = m_used == -CUDART_INF_F;
        const bool grow = first || (m_new - m_used) * a.scale_log2 > 8.f;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = first ? 0.f : (grow ? ex2((m_used - m_new) * a.scale_log2) : 1.f);
          if (j > 0) {
  #pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              uint32_t orr[32];
              tmem_ld32(t_row + kColO + 128 * h + 32 * c, orr);
              tmem_ld_wait();
  #pragma unroll
              for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
              tmem_st32(t_row + kColO + 128 * h + 32 * c, orr);
            }
            tmem_st_wait();
          }
          if (grow) {
            l *= alpha;
            m_used = m_new;
          }
        }
        // P = 2^(s * scale * log2 e - m * scale * log2 e) as bf16 pairs over S's first 64 columns
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nm2 = make_float2(-m_used * a.scale_log2, -m_used * a.scale_log2);
        float2 l2 = make_float2(0.f, 0.f);
  #pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          uint32_t pk[32];
  #pragma unroll
          for (int c2 = 0; c2 < 2; ++c2)
  #pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 t = __ffma2_rn(make_float2(__uint_as_float(sr[2 * hc + c2][e]),
                                                      __uint_as_float(sr[2 * hc + c2][e + 1])),
                                          sc2, nm2);
              const float2 pp = make_float2(ex2(t.x), ex2(t.y));
              l2 = __fadd2_rn(l2, pp);
              pk[c2 * 16 + (e >> 1)] = pack_bf16x2(pp.x, pp.y);
            }
          tmem_st32(t_row + kColS + 128 * h + 32 * hc, pk);
        }
        l += l2.x + l2.y;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_cta(&bars->p_full[h]);
      }
      if (ok && pf_wait_warp(&bars->o_done[h], static_cast<uint32_t>(n_tiles - 1) & 1u, fail, a.status)) {
        tc_fence_after();
        const float inv = 1.f / l;
        const bool write = r < rows_here && (h == 0 || two);
        __nv_bfloat16* orow = a.out + (static_cast<size_t>(q0 + i0 + r) * Hd::hq(a) + qh0 + h) * HD;
  #pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32(t_row + kColO + 128 * h + 32 * c, orr);
          tmem_ld_wait();
          if (write) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(orr[8 * q + 0]) * inv, __uint_as_float(orr[8 * q + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(orr[8 * q + 2]) * inv, __uint_as_float(orr[8 * q + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(orr[8 * q + 4]) * inv, __uint_as_float(orr[8 * q + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(orr[8 * q + 6]) * inv, __uint_as_float(orr[8 * q + 7]) * inv);
              dst[q] = v;
            }
          }
        }
      }
    } else {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kOther));  // idle warps 10-11
    }

    }
  } else {
    // ================================================================ split mode: shares of key tiles
    // Only min(workers, U) CTAs take a share, so every share is non-empty.
    const long long U = pref[a.num_seqs];
    const long long nw = pref[2 * a.num_seqs + 11];  // persistent workers (fewer in a mixed step)
    const int G = static_cast<int>(U < nw ? U : nw);
    const bool active = static_cast<int>(blockIdx.x) < G;
    const long long lo = active ? pf_share_lo(blockIdx.x, U, G) : 0;
    const long long hi = active ? pf_share_lo(blockIdx.x + 1, U, G) : 0;
    // the softmax warps re-read these from shared memory instead of keeping them live
    volatile long long* share = pref + 2 * a.num_seqs + 3;  // lo, hi, U, G
    volatile long long* pend_f = share + 4;                 // [head][2]: start units of split pieces not yet counted
  if (!active) {
    } else if (warp == kPfTmaWarp) {
      // ------------------------------------------------------------------ TMA producer
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kOther));
      int gj = 0;  // key tiles of this CTA so far
      int pi = 0;
      PfPiece pc;
      bool run = true;
      for (long long f = lo; run && pf_find_piece<kFixed>(f, hi, pref, a, pc); f = pc.fend, ++pi) {
        // this piece's query tiles, once the previous piece's QK MMAs are done with the buffer
        if (pi > 0 && !pf_wait_warp(&bars->q_empty, static_cast<uint32_t>(pi - 1) & 1u, fail, a.status)) break;
        if (lane == 0) {
          int g, qh0;
          bool two;
          pf_pair_heads<kFixed>(a, pc.hp, g, qh0, two);
          mbar_arrive_expect_tx(&bars->q_full, 2 * Dm::kTileBytes);
          for (int h = 0; h < 2; ++h)
            for (int half = 0; half < Dm::kHalves; ++half)
              tma_load_3d(sQ + h * Dm::kTileBytes + half * kPfHalfBytes, &qmap, half * 64, qh0 + (two ? h : 0),
                          pc.q0 + pc.t * kPfRows, &bars->q_full);
        }
        const int rows = pc.qlen < kPfRows * (pc.t + 1) ? pc.qlen : kPfRows * (pc.t + 1);
        const int n_pages = (pc.P + rows + kPageSize - 1) / kPageSize;
        // this lane's page id of the piece's first key tile, then of each next tile one tile ahead
        int id_next = lane < kPfPagesPerTile && pc.k0 * kPfPagesPerTile + lane < n_pages
                          ? __ldg(a.block_table + static_cast<size_t>(pc.n) * a.max_pages + pc.k0 * kPfPagesPerTile + lane)
                          : 0;
        for (int k = pc.k0; k < pc.k1; ++k, ++gj) {
          const int st = gj & 1;
          const int use = gj >> 1;
          const int pg = k * kPfPagesPerTile + lane;
          const int id_cur = id_next;
          if (k + 1 < pc.k1 && lane < kPfPagesPerTile && pg + kPfPagesPerTile < n_pages)
            id_next = __ldg(a.block_table + static_cast<size_t>(pc.n) * a.max_pages + pg + kPfPagesPerTile);
          if (use > 0 && !pf_wait_warp(&bars->kv_empty[st], static_cast<uint32_t>(use - 1) & 1u, fail, a.status)) {
            run = false;
            break;
          }
          bool valid = lane < kPfPagesPerTile && pg < n_pages;
          int id = 0;
          if (valid) {
            id = id_cur;
            if (id < 0 || id >= a.num_pages) {
              set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
              valid = false;
            }
          }
          const unsigned vmask = __ballot_sync(0xffffffffu, valid);
          const uint32_t bytes = static_cast<uint32_t>(__popc(vmask)) * static_cast<uint32_t>(Dm::kPageBytes);
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars->k_full[st], bytes);
            mbar_arrive_expect_tx(&bars->v_full[st], bytes);
          }
          __syncwarp();
          if (valid) {
            const int row = (id * Hd::hkv(a) + pc.hp / Hd::npair(a)) * kPageSize;
            unsigned char* kd = sK + st * Dm::kTileBytes + lane * (kPageSize * 128);
            unsigned char* vd = sV + st * Dm::kTileBytes + lane * (kPageSize * 128);
  #pragma unroll
            for (int half = 0; half < Dm::kHalves; ++half)  // K first: the QK MMA waits only for K
              tma_load_2d(kd + half * kPfHalfBytes, &kmap, 64 * half, row, &bars->k_full[st]);
  #pragma unroll
            for (int half = 0; half < Dm::kHalves; ++half)
              tma_load_2d(vd + half * kPfHalfBytes, &vmap, 64 * half, row, &bars->v_full[st]);
          }
        }
      }
    } else if (warp == kPfMmaWarp) {
      // ------------------------------------------------------------------ MMA issuer
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kOther));
      // Issue order QK_0(0) QK_1(0) | PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1) | ... over
      // the CTA's key tiles (across pieces): the two heads' softmaxes run half a
      // period apart, so while one head's softmax works the other head's PV and
      // next QK keep the tensor pipe busy. QK_h(j+1) overwrites S_h, which holds
      // P_h(j), so it waits for PV_h(j) (o_done) -- which also keeps O_h out of
      // the softmax's way while it rescales it or reads it at the end of a piece.
      auto issue_qk = [&](int st, int h) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t qa = smem_u32(sQ + h * Dm::kTileBytes);
          const uint32_t kb = smem_u32(sK + st * Dm::kTileBytes);
  #pragma unroll
          for (int s = 0; s < HD / 16; ++s) {
            const uint32_t off = (s >> 2) * kPfHalfBytes + (s & 3) * 32;
            mma_ss(tmem + kColS + 128 * h, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                   kIdescQK, s > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[h]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int st, int h, bool acc) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vb = smem_u32(sV + st * Dm::kTileBytes);
  #pragma unroll
          for (int s = 0; s < 8; ++s) {
            mma_ts(tmem + kColO + 128 * h, tmem + kColS + 128 * h + 8 * s,
                   sdesc_sw128(vb + s * 2048, kPfHalfBytes, 1024), Dm::kIdescPV, (acc || s > 0) ? 1u : 0u);
          }
          mma_commit(&bars->o_done[h]);
        }
        __syncwarp();
      };
      auto commit_q_empty = [&]() {
        if (lane == 0) mma_commit(&bars->q_empty);
        __syncwarp();
      };
      PfPiece cur, nxt;
      bool ok = pf_find_piece<kFixed>(lo, hi, pref, a, cur);
      bool have_nxt = ok && pf_find_piece<kFixed>(cur.fend, hi, pref, a, nxt);
      ok = ok && pf_wait_warp(&bars->q_full, 0, fail, a.status) && pf_wait_warp(&bars->k_full[0], 0, fail, a.status);
      if (ok) {
        issue_qk(0, 0);
        issue_qk(0, 1);
        if (cur.k1 - cur.k0 == 1) commit_q_empty();
      }
      int gj = 0, j = 0, pi = 0;
      while (ok) {
        const int st = gj & 1;
        const uint32_t ph = static_cast<uint32_t>(gj >> 1) & 1u;
        const uint32_t pj = static_cast<uint32_t>(gj) & 1u;
        const int ntiles = cur.k1 - cur.k0;
        const bool next_in = j + 1 < ntiles;
        const bool next = next_in || have_nxt;
        const int k = cur.k0 + j;
        if (!pf_wait_warp2(&bars->v_full[st], ph, &bars->p_full[0], pj, fail, a.status)) break;
        const int rows = cur.qlen < kPfRows * (cur.t + 1) ? cur.qlen : kPfRows * (cur.t + 1);
        const int kv_end = cur.P + rows;
        if (k == cur.nt - 1 && kv_end < (k + 1) * kPfKeys) {
          // keys past the end: zero their V rows (unused slots may hold NaN and 0 * NaN = NaN)
          const int r0 = kv_end - k * kPfKeys;
          uint4* vbase = reinterpret_cast<uint4*>(sV + st * Dm::kTileBytes);
          for (int idx = r0 * 8 + lane; idx < kPfKeys * 8; idx += 32) {
  #pragma unroll
            for (int half = 0; half < Dm::kHalves; ++half) vbase[half * (kPfHalfBytes / 16) + idx] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        issue_pv(st, 0, j > 0);
        if (next) {
          if (!next_in && !pf_wait_warp(&bars->q_full, static_cast<uint32_t>(pi + 1) & 1u, fail, a.status)) break;
          if (!pf_wait_warp2(&bars->k_full[st ^ 1], static_cast<uint32_t>((gj + 1) >> 1) & 1u, &bars->o_done[0], pj,
                             fail, a.status))
            break;
          issue_qk(st ^ 1, 0);
        }
        if (!pf_wait_warp(&bars->p_full[1], pj, fail, a.status)) break;
        issue_pv(st, 1, j > 0);
        if (lane == 0) mma_commit(&bars->kv_empty[st]);
        __syncwarp();
        if (!next) break;
        if (!pf_wait_warp(&bars->o_done[1], pj, fail, a.status)) break;
        issue_qk(st ^ 1, 1);
        // that was the last QK of its piece: the query buffer may be refilled
        if (next_in ? j + 2 == ntiles : nxt.k1 - nxt.k0 == 1) commit_q_empty();
        ++gj;
        if (next_in) {
          ++j;
        } else {
          cur = nxt;
          have_nxt = pf_find_piece<kFixed>(cur.fend, hi, pref, a, nxt);
          j = 0;
          ++pi;
        }
      }
    } else if (warp < 8) {
      // ------------------------------------------------------------------ softmax warpgroups
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kSoftmax));
      const int h = warp >> 2;
      const int quarter = warp & 3;
      const int r = quarter * 32 + lane;  // row of the tile = TMEM lane
      const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      if (quarter == 0 && lane == 0) {
        share[0] = lo;
        share[1] = hi;
        share[2] = U;
        share[3] = G;
        pend_f[2 * h] = -1;
        pend_f[2 * h + 1] = -1;
      }
      pf_group_sync(h);  // both warpgroups write the same values
      bool ok = true;
      int gj = 0;
      long long f = share[0];
      while (true) {
        // only the scalars the key-tile loop needs stay live across it (the piece is
        // looked up again for the end-of-piece work)
        int kb, ke, lim, diag_from;
        {
          PfPiece pc;
          if (!pf_find_piece<kFixed>(f, share[1], pref, a, pc)) break;
          const int i0 = pc.t * kPfRows;
          const int rows = pc.qlen < i0 + kPfRows ? pc.qlen : i0 + kPfRows;
          const int lim_row = pc.P + i0 + r;  // last visible key of this row (causal)
          lim = lim_row < pc.P + rows - 1 ? lim_row : pc.P + rows - 1;
          diag_from = pc.P + i0;
          kb = pc.k0;
          ke = pc.k1;
        }
        float m_used = -CUDART_INF_F;
        float l = 0.f;
        for (int k = kb; k < ke; ++k, ++gj) {
          if (ok && !pf_wait_warp(&bars->s_full[h], static_cast<uint32_t>(gj) & 1u, fail, a.status)) ok = false;
          if (!ok) continue;
          tc_fence_after();
          uint32_t sr[4][32];
  #pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(t_row + kColS + 128 * h + 32 * c, sr[c]);
          tmem_ld_wait();
          const bool diag = k * kPfKeys + kPfKeys - 1 > diag_from;
          // row max over the raw scores (the scale is positive, so it keeps the order)
          float mx = -CUDART_INF_F;
          if (diag) {
  #pragma unroll
            for (int c = 0; c < 4; ++c)
  #pragma unroll
              for (int e = 0; e < 32; ++e) {
                if (k * kPfKeys + 32 * c + e > lim) sr[c][e] = __float_as_uint(-CUDART_INF_F);
                mx = fmaxf(mx, __uint_as_float(sr[c][e]));
              }
          } else {
  #pragma unroll
            for (int c = 0; c < 4; ++c)
  #pragma unroll
              for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sr[c][e]));
          }
          const float m_new = fmaxf(m_used, mx);
          const bool first = m_used == -CUDART_INF_F;
          const bool grow = first || (m_new - m_used) * a.scale_log2 > 8.f;
          if (__any_sync(0xffffffffu, grow)) {
            const float alpha = first ? 0.f : (grow ? ex2((m_used - m_new) * a.scale_log2) : 1.f);
            if (k > kb) {
  #pragma unroll
              for (int c = 0; c < HD / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(t_row + kColO + 128 * h + 32 * c, orr);
                tmem_ld_wait();
  #pragma unroll
                for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                tmem_st32(t_row + kColO + 128 * h + 32 * c, orr);
              }
              tmem_st_wait();
            }
            if (grow) {
              l *= alpha;
              m_used = m_new;
            }
          }
          // P = 2^(s * scale * log2 e - m * scale * log2 e) as bf16 pairs over S's first 64 columns;
          // a row with no visible key yet (a piece that starts past key 0) gets P = 0
          const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
          const float mo = m_used == -CUDART_INF_F ? 0.f : -m_used * a.scale_log2;
          const float2 nm2 = make_float2(mo, mo);
          float2 l2 = make_float2(0.f, 0.f);
  #pragma unroll
          for (int c = 0; c < 4; ++c) {  // scores 32c .. 32c+31 -> P columns 16c .. 16c+15
            uint32_t pk[16];
  #pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 t =
                  __ffma2_rn(make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sc2, nm2);
              const float2 pp = make_float2(ex2(t.x), ex2(t.y));
              l2 = __fadd2_rn(l2, pp);
              pk[e >> 1] = pack_bf16x2(pp.x, pp.y);
            }
            tmem_st16(t_row + kColS + 128 * h + 16 * c, pk);
          }
          l += l2.x + l2.y;
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_cta(&bars->p_full[h]);
        }
        // ---- end of the piece: O_h is complete once PV_h of its last key tile is done
        if (ok && !pf_wait_warp(&bars->o_done[h], static_cast<uint32_t>(gj - 1) & 1u, fail, a.status)) ok = false;
        if (ok) tc_fence_after();
        asm volatile("" : "+l"(f));  // look the piece up again rather than keep it live
        PfPiece pc;
        pf_find_piece<kFixed>(f, share[1], pref, a, pc);
        const int i0 = pc.t * kPfRows;
        const int rows_here = (pc.qlen < i0 + kPfRows ? pc.qlen : i0 + kPfRows) - i0;
        int pg_, qh0;
        bool two;
        pf_pair_heads<kFixed>(a, pc.hp, pg_, qh0, two);
        const bool write = r < rows_here && (h == 0 || two);
        __nv_bfloat16* orow = a.out + (static_cast<size_t>(pc.q0 + i0 + r) * Hd::hq(a) + qh0 + h) * HD;
        if (pc.k0 == 0 && pc.k1 == pc.nt) {
          if (ok) {
            const float inv = 1.f / l;
  #pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              uint32_t orr[32];
              tmem_ld32(t_row + kColO + 128 * h + 32 * c, orr);
              tmem_ld_wait();
              if (write) {
                uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
  #pragma unroll
                for (int q = 0; q < 4; ++q) {
                  uint4 v;
                  v.x = pack_bf16x2(__uint_as_float(orr[8 * q + 0]) * inv, __uint_as_float(orr[8 * q + 1]) * inv);
                  v.y = pack_bf16x2(__uint_as_float(orr[8 * q + 2]) * inv, __uint_as_float(orr[8 * q + 3]) * inv);
                  v.z = pack_bf16x2(__uint_as_float(orr[8 * q + 4]) * inv, __uint_as_float(orr[8 * q + 5]) * inv);
                  v.w = pack_bf16x2(__uint_as_float(orr[8 * q + 6]) * inv, __uint_as_float(orr[8 * q + 7]) * inv);
                  dst[q] = v;
                }
              }
            }
          }
        } else {
          // Split piece (only a share's first and last piece can be): write this
          // CTA's partial record of the row now, count it after the last piece.
          unsigned char* rec = a.records +
                               static_cast<size_t>(2 * blockIdx.x + (f == share[0] ? 0 : 1)) * Dm::kRecBytes +
                               h * Dm::kRecHeadBytes;
          uint2* ro = reinterpret_cast<uint2*>(rec);
          float* rml = reinterpret_cast<float*>(rec + Dm::kRecO);
          const float inv = l > 0.f ? 1.f / l : 0.f;  // a row with no visible key in the piece has l = 0
          if (ok) {
  #pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              uint32_t orr[32];
              tmem_ld32(t_row + kColO + 128 * h + 32 * c, orr);
              tmem_ld_wait();
  #pragma unroll
              for (int q = 0; q < 8; ++q) {
                // O / l is a convex combination of V rows; fp16 holds it (clamped to the fp16 range)
                auto h16 = [&](int e) { return fminf(fmaxf(__uint_as_float(orr[e]) * inv, -65504.f), 65504.f); };
                const __half2 lo2 = __floats2half2_rn(h16(4 * q), h16(4 * q + 1));
                const __half2 hi2 = __floats2half2_rn(h16(4 * q + 2), h16(4 * q + 3));
                ro[(c * 8 + q) * kPfRows + r] =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&lo2), *reinterpret_cast<const uint32_t*>(&hi2));
              }
            }
          }
          rml[r] = m_used == -CUDART_INF_F ? -CUDART_INF_F : m_used * a.scale_log2;
          rml[kPfRows + r] = l;
          if (quarter == 0 && lane == 0) pend_f[2 * h + (f == share[0] ? 0 : 1)] = f;
        }
        f = pc.fend;
      }
      // ---- count the split pieces' records in (one fence, one round trip); the
      // CTA that completes an item's count merges the records of all its holders
      // (log-sum-exp) and resets the counter. The barriers run whatever ok is.
      pf_group_sync(h);  // this head's records and pend_f are written
      const long long pf0 = pend_f[2 * h], pf1 = pend_f[2 * h + 1];
      if (pf0 >= 0 || pf1 >= 0) {
        const long long Us = share[2];
        const int Gs = static_cast<int>(share[3]);
        if (quarter == 0 && lane == 0) {
          int flags = 0;
          __threadfence();
          int old[2] = {-1, -1}, want[2] = {0, 0};
  #pragma unroll
          for (int i = 0; i < 2; ++i) {
            const long long fi = i == 0 ? pf0 : pf1;
            if (fi < 0) continue;
            PfPiece pc;
            pf_find_piece<kFixed>(fi, share[1], pref, a, pc);
            want[i] = pf_cta_of(pc.fseg + kPfItemCost + pc.nt - 1, Us, Gs) - pf_cta_of(pc.fseg + kPfItemCost, Us, Gs);
            old[i] = atomicAdd(a.counters + ((static_cast<size_t>(pc.n) * Hd::pairs(a) + pc.hp) * a.tmax + pc.t) * 2 + h, 1);
          }
          __threadfence();
          if (pf0 >= 0 && old[0] == want[0]) flags |= 1;
          if (pf1 >= 0 && old[1] == want[1]) flags |= 2;
          merge_flag[h] = flags;
        }
        pf_group_sync(h);
        const int flags = merge_flag[h];
  #pragma unroll 1
        for (int i = 0; i < 2; ++i) {
          if (!((flags >> i) & 1)) continue;
          PfPiece pc;
          pf_find_piece<kFixed>(i == 0 ? pf0 : pf1, share[1], pref, a, pc);
          const int holders0 = pf_cta_of(pc.fseg + kPfItemCost, Us, Gs);
          const int nhold = pf_cta_of(pc.fseg + kPfItemCost + pc.nt - 1, Us, Gs) - holders0 + 1;
          const bool first_has_two = pf_share_lo(holders0, Us, Gs) < pc.fseg;
          auto rec_of = [&](int j) {
            const int c = holders0 + j;
            return a.records + static_cast<size_t>(2 * c + ((j == 0 && first_has_two) ? 1 : 0)) * Dm::kRecBytes +
                   h * Dm::kRecHeadBytes;
          };
          float M = -CUDART_INF_F;
          for (int j = 0; j < nhold; ++j)
            M = fmaxf(M, __ldcg(reinterpret_cast<const float*>(rec_of(j) + Dm::kRecO) + r));
          const int i0 = pc.t * kPfRows;
          int pg_, qh0;
          bool two;
          pf_pair_heads<kFixed>(a, pc.hp, pg_, qh0, two);
          const bool write = r < (pc.qlen < i0 + kPfRows ? pc.qlen : i0 + kPfRows) - i0 && (h == 0 || two);
          __nv_bfloat16* orow = a.out + (static_cast<size_t>(pc.q0 + i0 + r) * Hd::hq(a) + qh0 + h) * HD;
          float L = 0.f;
  #pragma unroll 1
          for (int half = 0; half < Dm::kHalves; ++half) {  // dims 64 half .. 64 half + 63
            float acc[64];
  #pragma unroll
            for (int e = 0; e < 64; ++e) acc[e] = 0.f;
            float lsum = 0.f;
  #pragma unroll 2
            for (int j = 0; j < nhold; ++j) {
              const unsigned char* rj = rec_of(j);
              const float m_j = __ldcg(reinterpret_cast<const float*>(rj + Dm::kRecO) + r);
              const float l_j = __ldcg(reinterpret_cast<const float*>(rj + Dm::kRecO) + kPfRows + r);
              const float w = m_j == -CUDART_INF_F ? 0.f : ex2(m_j - M) * l_j;  // the record holds O / l
              lsum += w;
              const uint2* oj = reinterpret_cast<const uint2*>(rj) + (16 * half) * kPfRows + r;
  #pragma unroll
              for (int q = 0; q < 16; ++q) {
                const uint2 u = __ldcg(oj + q * kPfRows);
                const float2 a01 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
                const float2 a23 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
                acc[4 * q] += w * a01.x;
                acc[4 * q + 1] += w * a01.y;
                acc[4 * q + 2] += w * a23.x;
                acc[4 * q + 3] += w * a23.y;
              }
            }
            if (half == 0) L = lsum;
            const float inv = 1.f / L;
            if (write) {
              uint4* dst = reinterpret_cast<uint4*>(orow + 64 * half);
  #pragma unroll
              for (int q = 0; q < 8; ++q) {
                uint4 v;
                v.x = pack_bf16x2(acc[8 * q + 0] * inv, acc[8 * q + 1] * inv);
                v.y = pack_bf16x2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv);
                v.z = pack_bf16x2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv);
                v.w = pack_bf16x2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv);
                dst[q] = v;
              }
            }
          }
          if (quarter == 0 && lane == 0)
            a.counters[((static_cast<size_t>(pc.n) * Hd::pairs(a) + pc.hp) * a.tmax + pc.t) * 2 + h] = 0;
        }
      }
    } else {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PfRegs<kMixed>::kOther));  // idle warps 10-11
    }

  }

  tc_fence_before();
  __syncthreads();
  if (warp == kPfMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------------ host
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

// Workspace: status header, split counters [num_seqs][head pairs][tmax][2], then
// two partial records per CTA of the persistent grid (one CTA per SM).
static int pf_pairs(int hq, int hkv) { return hkv * ((hq / hkv + 1) / 2); }
static size_t pf_counter_bytes(int32_t num_seqs, int32_t max_q_len, int pairs) {
  const size_t tmax = (static_cast<size_t>(max_q_len) + kPfRows - 1) / kPfRows;
  return (static_cast<size_t>(num_seqs) * pairs * tmax * 2 * 4 + 255) / 256 * 256;
}
static size_t pf_rec_bytes(int hd) { return hd == 64 ? PfDim<64>::kRecBytes : PfDim<128>::kRecBytes; }

bool prefill_supported(int num_q_heads, int num_kv_heads, int head_dim, int page_size) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || page_size != kPageSize) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  if (num_q_heads % num_kv_heads != 0) return false;
  const int g = num_q_heads / num_kv_heads;
  return g >= 1 && g <= 8;
}

size_t prefill_workspace_bytes(int num_q_heads, int num_kv_heads, int head_dim, int32_t num_seqs, int32_t max_q_len,
                               int num_sms) {
  return PKV_STATUS_BYTES + pf_counter_bytes(num_seqs, max_q_len, pf_pairs(num_q_heads, num_kv_heads)) +
         static_cast<size_t>(2) * num_sms * pf_rec_bytes(head_dim);
}

// The mixed step's decode part after the prefill workspace: chunk counters [dec_batch][8] (256-byte
// padded), then the partial records [dec_batch][8][chunks][2][132] floats.
static size_t mixed_counter_bytes(int32_t dec_batch) {
  return (static_cast<size_t>(dec_batch) * kKVHeads * 4 + 255) / 256 * 256;
}
size_t mixed_workspace_bytes(int32_t num_seqs, int32_t max_q_len, int32_t dec_batch, int32_t dec_max_pages,
                             int num_sms) {
  const int maxc = mixed_chunks_per_pair(dec_max_pages);
  return prefill_workspace_bytes(kQHeads, kKVHeads, kHeadDim, num_seqs, max_q_len, num_sms) +
         mixed_counter_bytes(dec_batch) +
         static_cast<size_t>(dec_batch) * kKVHeads * (maxc > 1 ? maxc : 0) * kGroup * kMixRec * 4;
}
int prefill_max_seqs() { return kPfMaxSeqs; }

template <int HD, bool kFixed, bool kMixed>
static int launch_prefill_hd(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             PrefillArgs a, int num_seqs, long long items, int num_sms, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(prefill_kernel<HD, kFixed, kMixed>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(pf_smem_bytes<HD>(kPfMaxSeqs))) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  // one CTA per SM fits (TMEM and shared memory); split mode uses the first num_sms CTAs (fewer in a mixed
  // step) as persistent workers, item mode one CTA per item; the mixed step's decode CTAs follow, one per
  // chunk of <= 64 pages of a (decode request, KV head), as many as the longest request can need
  a.pcta = static_cast<int>(items > num_sms ? items : num_sms);
  const long long grid =
      static_cast<long long>(a.pcta) + (kMixed ? static_cast<long long>(a.dbatch) * kKVHeads * a.dmaxc : 0);
  if (grid > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
  return launch_pdl(prefill_kernel<HD, kFixed, kMixed>, dim3(static_cast<unsigned>(grid)), dim3(kPfThreads),
                    pf_smem_bytes<HD>(num_seqs), stream, qmap, kmap, vmap, a) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

int launch_prefill(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                   const int32_t* prefix_lens, const int32_t* cu_q_lens, int32_t num_seqs, int32_t total_q,
                   void* out, float scale, int num_q_heads, int num_kv_heads, int head_dim, int32_t max_pages,
                   int32_t max_q_len, int32_t num_pages, void* workspace, cudaStream_t stream,
                   const MixedDecode* dec) {
  const bool mixed = dec != nullptr && dec->batch > 0;
  if (!mixed && (num_seqs == 0 || max_q_len == 0 || total_q == 0)) return PKV_OK;
  if (mixed && !(num_q_heads == kQHeads && num_kv_heads == kKVHeads && head_dim == kHeadDim))
    return PKV_ERR_UNSUPPORTED;
  if (!prefill_supported(num_q_heads, num_kv_heads, head_dim, kPageSize)) return PKV_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return PKV_ERR_CUDA;
  const cuuint64_t hd = static_cast<cuuint64_t>(head_dim);

  CUtensorMap qmap, kmap, vmap;
  {
    // (a mixed step may have no chunk rows: the map then covers one row it never reads)
    const cuuint64_t rows = total_q > 0 ? static_cast<cuuint64_t>(total_q) : 1;
    const cuuint64_t dims[3] = {hd, static_cast<cuuint64_t>(num_q_heads), rows};
    const cuuint64_t strides[2] = {hd * 2, static_cast<cuuint64_t>(num_q_heads) * hd * 2};
    const cuuint32_t box[3] = {64, 1, kPfRows};
    const cuuint32_t estr[3] = {1, 1, 1};
    // (without chunk rows the map points at the K pool: it needs a valid address and is never read)
    void* qbase = total_q > 0 && q != nullptr ? const_cast<void*>(q) : const_cast<void*>(k_pages);
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, qbase, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {hd, static_cast<cuuint64_t>(num_pages) * num_kv_heads * kPageSize};
    const cuuint64_t strides[1] = {hd * 2};
    const cuuint32_t box[2] = {64, kPageSize};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(k_pages), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
    if (enc(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(v_pages), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
  }

  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  PrefillArgs a;
  a.block_table = block_table;
  a.prefix_lens = prefix_lens;
  a.cu_q_lens = cu_q_lens;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.tmax = (max_q_len + kPfRows - 1) / kPfRows;
  a.workers = num_sms;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.grp = num_q_heads / num_kv_heads;
  a.npair = (a.grp + 1) / 2;
  a.pairs = num_kv_heads * a.npair;
  a.scale_log2 = scale * kLog2e;
  a.status = reinterpret_cast<int*>(ws);
  a.counters = reinterpret_cast<int*>(ws + PKV_STATUS_BYTES);
  a.records = ws + PKV_STATUS_BYTES + pf_counter_bytes(num_seqs, max_q_len, a.pairs);
  a.dq = mixed ? static_cast<const __nv_bfloat16*>(dec->q) : nullptr;
  a.dbt = mixed ? dec->block_table : nullptr;
  a.dlens = mixed ? dec->seq_lens : nullptr;
  a.dout = mixed ? static_cast<__nv_bfloat16*>(dec->out) : nullptr;
  a.dbatch = mixed ? dec->batch : 0;
  a.dmax_pages = mixed ? dec->max_pages : 1;
  a.dmaxc = mixed_chunks_per_pair(a.dmax_pages);
  {
    unsigned char* dws = ws + prefill_workspace_bytes(num_q_heads, num_kv_heads, head_dim, num_seqs, max_q_len, num_sms);
    a.dcnt = mixed ? reinterpret_cast<int*>(dws) : nullptr;
    a.drec = mixed ? reinterpret_cast<float*>(dws + mixed_counter_bytes(a.dbatch)) : nullptr;
  }
  a.pcta = 0;
  const long long items = static_cast<long long>(num_seqs) * a.pairs * a.tmax;
  if (mixed) return launch_prefill_hd<128, true, true>(qmap, kmap, vmap, a, num_seqs, items, num_sms, stream);
  if (head_dim == 64)
    return launch_prefill_hd<64, false, false>(qmap, kmap, vmap, a, num_seqs, items, num_sms, stream);
  if (num_q_heads == kQHeads && num_kv_heads == kKVHeads)  // the Qwen3 decoder: head counts fixed at compile time
    return launch_prefill_hd<128, true, false>(qmap, kmap, vmap, a, num_seqs, items, num_sms, stream);
  return launch_prefill_hd<128, false, false>(qmap, kmap, vmap, a, num_seqs, items, num_sms, stream);
}

}  // namespace pkv
