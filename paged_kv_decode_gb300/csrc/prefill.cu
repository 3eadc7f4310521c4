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
//  * Grid: (query tile x KV head, request), dispatched longest causal tiles first.
#include <cuda.h>
#include <math_constants.h>

#include "pkv_device.cuh"
#include "pkv_kernels.h"
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
constexpr int kPfHalfBytes = kPfRows * 128;  // one 64-column half of a 128 x 128 bf16 tile: 16 KiB
constexpr int kPfTileBytes = 2 * kPfHalfBytes;
constexpr int kPfStages = 2;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                                   // Q_0, Q_1
constexpr int kOffV = kOffQ + 2 * kPfTileBytes;            // V stages
constexpr int kOffK = kOffV + kPfStages * kPfTileBytes;    // K stages
constexpr int kOffBars = kOffK + kPfStages * kPfTileBytes;
constexpr int kNumBars = 13;
constexpr int kPfSmemBytes = kOffBars + kNumBars * 8 + 16 + 1024;  // + tmem address, fail flag, alignment slack

// TMEM columns
constexpr uint32_t kColS = 0;    // S_h at kColS + 128 h
constexpr uint32_t kColO = 256;  // O_h at kColO + 128 h
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false);  // B = K tile, K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, true);   // B = V tile, MN-major

struct PrefillArgs {
  const int* block_table;
  const int* prefix_lens;
  const int* cu_q_lens;
  __nv_bfloat16* out;
  int total_q;
  int max_pages;
  int num_pages;
  float scale_log2;
  int* status;
};

struct PfBars {
  uint64_t q_full;
  uint64_t k_full[kPfStages];
  uint64_t v_full[kPfStages];
  uint64_t kv_empty[kPfStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
};
static_assert(sizeof(PfBars) == kNumBars * 8, "barrier block");

// Share of the softmax exponentials (pairs out of every 4) evaluated on the FMA
// pipe instead of the MUFU unit. With the raw-score max and packed FMAs the
// softmax is bound by FMA-pipe issue rather than by MUFU, and any share > 0
// measured slower on a GB300 (0: 670/986/1090, 1: 629/919/1005 TFLOP/s for a
// 4096-row chunk after 0/8192/32768 cached tokens), so the default is 0.
#ifndef PKV_PF_POLY_PAIRS
#define PKV_PF_POLY_PAIRS 0
#endif
constexpr int kPfPolyPairsOf4 = PKV_PF_POLY_PAIRS;

// 2^t for a pair of t <= 8 (t = -inf gives about 2^-125) without the MUFU unit:
// Cody-Waite range reduction 2^t = 2^n * 2^f with n = round(t) (the 1.5 * 2^23
// addition rounds t to an integer in the low mantissa bits) and f in [-1/2, 1/2],
// 2^f from a degree-3 polynomial fitted by the Remez exchange for relative
// error (max 7.5e-5; exp2_poly_fit.py reproduces the constants), and 2^n
// applied by adding n to the exponent field.
__device__ __forceinline__ float2 exp2_poly2(float2 t) {
  constexpr float kRound = 12582912.f;  // 1.5 * 2^23
  constexpr float c0 = 0.9999280571937561f, c1 = 0.6932609677314758f, c2 = 0.2426111251115799f,
                  c3 = 0.0551716685295105f;
  t.x = fmaxf(t.x, -125.f);
  t.y = fmaxf(t.y, -125.f);
  const float2 j = __fadd2_rn(t, make_float2(kRound, kRound));
  const float2 n = __fadd2_rn(j, make_float2(-kRound, -kRound));
  const float2 f = __ffma2_rn(n, make_float2(-1.f, -1.f), t);
  float2 p = __ffma2_rn(make_float2(c3, c3), f, make_float2(c2, c2));
  p = __ffma2_rn(p, f, make_float2(c1, c1));
  p = __ffma2_rn(p, f, make_float2(c0, c0));
  return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(j.x) << 23)),
                     __int_as_float(__float_as_int(p.y) + (__float_as_int(j.y) << 23)));
}

// Bounded wait that gives up at once after any wait of the CTA has timed out.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile int* fail, int* status) {
  if (*fail) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *fail = 1;
  set_status(status, PKV_ERR_DEVICE_TIMEOUT);
  return false;
}

// Warp-collective form: every lane waits and the warp agrees on the outcome
// (the tcgen05.ld/st that follow are warp-wide).
__device__ __forceinline__ bool pf_wait_warp(uint64_t* bar, uint32_t parity, volatile int* fail, int* status) {
  return __all_sync(0xffffffffu, pf_wait(bar, parity, fail, status));
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // 1024-byte aligned for 128-byte swizzle atoms
  PfBars* bars = reinterpret_cast<PfBars*>(smem + kOffBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBars + kNumBars * 8);
  volatile int* fail = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // CTAs are dispatched in blockIdx.x order: walk (query tile, KV head) pairs
  // tile-major from the last tile, so every head's longest causal tiles start first.
  const int n_qtiles = gridDim.x / kKVHeads;
  const int tile = n_qtiles - 1 - static_cast<int>(blockIdx.x) / kKVHeads;
  const int g = static_cast<int>(blockIdx.x) % kKVHeads;  // KV head
  const int n = blockIdx.y;                                 // request

  grid_dependency_wait();
  allow_dependents();

  const int q0 = __ldg(a.cu_q_lens + n);
  const int q1 = __ldg(a.cu_q_lens + n + 1);
  const int P = __ldg(a.prefix_lens + n);
  const int qlen = q1 - q0;
  const int i0 = tile * kPfRows;
  if (i0 >= qlen) return;
  const int rows_here = qlen - i0 < kPfRows ? qlen - i0 : kPfRows;
  const long long kv_end_ll = static_cast<long long>(P) + i0 + rows_here;  // keys 0 .. kv_end-1 are needed
  if (P < 0 || q0 < 0 || q1 > a.total_q || kv_end_ll > static_cast<long long>(a.max_pages) * kPageSize) {
    if (tid == 0) set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
    return;
  }
  const int kv_end = static_cast<int>(kv_end_ll);
  const int n_tiles = (kv_end + kPfKeys - 1) / kPfKeys;
  const int n_pages = (kv_end + kPageSize - 1) / kPageSize;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
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
  if (warp == kPfMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  unsigned char* sQ = smem + kOffQ;
  unsigned char* sV = smem + kOffV;
  unsigned char* sK = smem + kOffK;


  if (warp == kPfTmaWarp) {
    // ------------------------------------------------------------------ TMA producer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPfRegsOther));
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->q_full, 2 * kPfTileBytes);
      for (int h = 0; h < 2; ++h)
        for (int half = 0; half < 2; ++half)
          tma_load_3d(sQ + h * kPfTileBytes + half * kPfHalfBytes, &qmap, half * 64, 2 * g + h, q0 + i0,
                      &bars->q_full);
    }
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j & 1;
      const int use = j >> 1;
      if (use > 0 && !pf_wait_warp(&bars->kv_empty[st], static_cast<uint32_t>(use - 1) & 1u, fail, a.status)) break;
      const int pg = j * kPfPagesPerTile + lane;
      bool valid = lane < kPfPagesPerTile && pg < n_pages;
      int id = 0;
      if (valid) {
        id = __ldg(a.block_table + static_cast<size_t>(n) * a.max_pages + pg);
        if (id < 0 || id >= a.num_pages) {
          set_status(a.status, PKV_ERR_OUT_OF_BOUNDS);
          valid = false;
        }
      }
      const unsigned vmask = __ballot_sync(0xffffffffu, valid);
      const uint32_t bytes = static_cast<uint32_t>(__popc(vmask)) * 2u * (kPageSize * 128u);
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->k_full[st], bytes);
        mbar_arrive_expect_tx(&bars->v_full[st], bytes);
      }
      __syncwarp();
      if (valid) {
        const int row = (id * kKVHeads + g) * kPageSize;
        unsigned char* kd = sK + st * kPfTileBytes + lane * (kPageSize * 128);
        unsigned char* vd = sV + st * kPfTileBytes + lane * (kPageSize * 128);
        tma_load_2d(kd, &kmap, 0, row, &bars->k_full[st]);
        tma_load_2d(kd + kPfHalfBytes, &kmap, 64, row, &bars->k_full[st]);
        tma_load_2d(vd, &vmap, 0, row, &bars->v_full[st]);
        tma_load_2d(vd + kPfHalfBytes, &vmap, 64, row, &bars->v_full[st]);
      }
    }
  } else if (warp == kPfMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPfRegsOther));
    // Issue order QK_0(0) QK_1(0) | PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1) | ...: the
    // two heads' softmaxes run half a period apart, so while one head's softmax
    // works the other head's PV and next QK keep the tensor pipe busy. QK_h(j+1)
    // overwrites S_h, which holds P_h(j), so it waits for PV_h(j) (o_done) --
    // which also keeps O_h out of the softmax's way while it may rescale it.
    auto issue_qk = [&](int j, int h) {
      tc_fence_after();
      if (lane == 0) {
        const uint32_t qa = smem_u32(sQ + h * kPfTileBytes);
        const uint32_t kb = smem_u32(sK + (j & 1) * kPfTileBytes);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
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
        const uint32_t vb = smem_u32(sV + (j & 1) * kPfTileBytes);
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          mma_ts(tmem + kColO + 128 * h, tmem + kColS + 128 * h + 8 * s,
                 sdesc_sw128(vb + s * 2048, kPfHalfBytes, 1024), kIdescPV, (j > 0 || s > 0) ? 1u : 0u);
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
      if (!pf_wait_warp(&bars->v_full[st], ph, fail, a.status)) break;
      if (j == n_tiles - 1 && kv_end < (j + 1) * kPfKeys) {
        // keys past the end: zero their V rows (unused slots may hold NaN and 0 * NaN = NaN)
        const int r0 = kv_end - j * kPfKeys;
        uint4* vbase = reinterpret_cast<uint4*>(sV + st * kPfTileBytes);
        for (int idx = r0 * 8 + lane; idx < kPfKeys * 8; idx += 32) {
          vbase[idx] = make_uint4(0, 0, 0, 0);
          vbase[kPfHalfBytes / 16 + idx] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const uint32_t pj = static_cast<uint32_t>(j) & 1u;
      if (!pf_wait_warp(&bars->p_full[0], pj, fail, a.status)) break;
      issue_pv(j, 0);
      if (next) {
        if (!pf_wait_warp(&bars->k_full[st ^ 1], ph_next, fail, a.status) ||
            !pf_wait_warp(&bars->o_done[0], pj, fail, a.status))
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPfRegsSoftmax));
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
          for (int c = 0; c < 4; ++c) {
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
            float2 pp;
            if (((e >> 1) & 3) < kPfPolyPairsOf4) {
              pp = exp2_poly2(t);
            } else {
              pp = make_float2(ex2(t.x), ex2(t.y));
            }
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
      const bool write = r < rows_here;
      __nv_bfloat16* orow = a.out + (static_cast<size_t>(q0 + i0 + r) * kQHeads + 2 * g + h) * kHeadDim;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPfRegsOther));  // idle warps 10-11
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

size_t prefill_workspace_bytes(int32_t, int32_t, int) { return PKV_STATUS_BYTES; }

int launch_prefill(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table,
                   const int32_t* prefix_lens, const int32_t* cu_q_lens, int32_t num_seqs, int32_t total_q,
                   void* out, float scale, int32_t max_pages, int32_t max_q_len, int32_t num_pages, void* workspace,
                   cudaStream_t stream) {
  if (num_seqs == 0 || max_q_len == 0 || total_q == 0) return PKV_OK;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return PKV_ERR_CUDA;

  CUtensorMap qmap, kmap, vmap;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(kQHeads),
                                static_cast<cuuint64_t>(total_q)};
    const cuuint64_t strides[2] = {kHeadDim * 2, static_cast<cuuint64_t>(kQHeads) * kHeadDim * 2};
    const cuuint32_t box[3] = {64, 1, kPfRows};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PKV_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim),
                                static_cast<cuuint64_t>(num_pages) * kKVHeads * kPageSize};
    const cuuint64_t strides[1] = {kHeadDim * 2};
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

  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmemBytes) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  PrefillArgs a;
  a.block_table = block_table;
  a.prefix_lens = prefix_lens;
  a.cu_q_lens = cu_q_lens;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.total_q = total_q;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.scale_log2 = scale * kLog2e;
  a.status = static_cast<int*>(workspace);
  const dim3 grid(((max_q_len + kPfRows - 1) / kPfRows) * kKVHeads, num_seqs);
  return launch_pdl(prefill_kernel, grid, dim3(kPfThreads), static_cast<size_t>(kPfSmemBytes), stream, qmap, kmap,
                    vmap, a) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}

}  // namespace pkv
