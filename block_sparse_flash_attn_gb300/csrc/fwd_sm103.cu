// Block-sparse flash-attention forward for sm_103a (GB300).
//
// What it computes: for every query tile (128 rows of one (batch, head)) and
// every live key block of that tile (the plan's CSR list), the exact softmax
// attention over all live keys, O = softmax(scale * Q K^T + mask) V, plus the
// natural-log LSE per row.  The operation is the one of "Writing Pallas
// Kernels for JAX: Stepping Outside the XLA Safety Net" (section "Writing the
// Kernel Logic: Load, Compute, Store": scaled scores, masked to -inf, softmax,
// product with V) made exact across key blocks the flash-attention way
// ("Pallas-Triton kernels and kernel auto-tuning", section "Flash Attention").
// Dead key blocks are never loaded (the mask's purpose in "Writing the Kernel
// Logic": only the small 128x128 block is ever materialised).
//
// GB300 design (one persistent CTA per SM, 384 threads = 3 warpgroups):
//   warps 0-3  softmax + epilogue for query slot 0 (TMEM lanes 0..127)
//   warps 4-7  softmax + epilogue for query slot 1
//   warp  8    TMA producer and tile scheduler (one elected lane)
//   warp  9    tcgen05 MMA issuer (one elected lane), TMEM owner
//   warps 10-11 idle (they complete warpgroup 2 so it can hand its
//              registers to the softmax warpgroups with setmaxnreg)
// Two query tiles are in flight per CTA so the tensor core works on one slot
// while the other slot's softmax runs.  Tensor memory (512 columns):
//   S0 = [0,128), S1 = [128,256): fp32 scores, overwritten in place by the
//   bf16 probabilities P (columns 0..63 of the slot's S region);
//   O0 = [256,384), O1 = [384,512): fp32 output accumulators.
// Shared memory: Q tile per slot, a ring of K/V tiles (each 128 x D bf16,
// 128-byte swizzled by TMA, read by tcgen05.mma through matrix descriptors).
//
// Per slot and tile with n live key blocks the MMA warp runs
//   S(0); then for j = 1..n-1: [wait P(j-1)] O += P(j-1) V(j-1); S(j);
//   finally [wait P(n-1)] O += P(n-1) V(n-1); signal O ready.
// Because tcgen05 ops of one thread complete in order, "S(j) done" also
// means "PV(j-1) done", so the softmax may rescale O right after seeing S(j).
// Online softmax in base 2 with lazy rescale: the running max m only moves
// when a block's max exceeds it by more than 8 (log2 units), so P <= 256 and
// the O rescale (a TMEM round trip) is rare after the first block.
//
// Every wait is bounded (globaltimer); on expiry the kernel records a timeout
// in the status word, every role leaves its loop, outstanding TMA loads and
// MMAs are drained (again with a limit) and TMEM is freed before exit.
#include <cstdint>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace bsattn {
namespace {

constexpr int kThreads = 384;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kRegsSoftmax = 208;  // 2 x 128 x 208 + 128 x 88 = 384 x 168 (launch budget)
constexpr int kRegsOther = 88;
constexpr float kTau = 8.0f;
// Every kPolyEvery-th pair of probabilities in a block without causal masking
// is computed by the FMA-pipe polynomial instead of the MUFU ex2 (0 = never).
#ifndef BSATTN_POLY_EVERY
#define BSATTN_POLY_EVERY 0
#endif
constexpr int kPolyEvery = BSATTN_POLY_EVERY;
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kDrainNs = 200ull * 1000 * 1000;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kBlock * D * 2;  // one 128 x D bf16 tile
  static constexpr int kBoxes = D / 64;              // 64-column (128-byte) TMA boxes
  static constexpr int kBoxBytes = kBlock * 128;     // 16 KB per box
  static constexpr int kStages = (D == 128) ? 4 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
  static constexpr int kSmem = kBarOff + 1024;
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, true);
};

// One scheduled tile as the producer publishes it to the MMA and softmax roles.
struct TileInfo {
  int t;     // tile id (b*H + h)*nb + qb, or -1 when no tiles are left
  int r0;    // first CSR entry of the tile
  int n;     // live key blocks
  int diag;  // causal and the last live block is the diagonal one
};

struct __align__(16) Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t tq_full[2][2];
  uint64_t tq_empty[2][2];
  uint64_t drain;
  TileInfo tq[2][2];
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainNs) return;
  }
}

__device__ __forceinline__ void raise_internal(volatile int* abort_flag, int* status) {
  *abort_flag = 1;
  atomicOr(status, kStatusInternal);
}

// ---------------------------------------------------------------------------
// warp 8: tile scheduler + TMA producer
// ---------------------------------------------------------------------------
template <int D>
__device__ void run_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const FwdParams& p, Bars* bars,
                             uint32_t q_base, uint32_t ring_base, volatile int* abort_flag) {
  using C = Cfg<D>;
  const uint64_t lim = p.timeout_ns;
  int it = 0;
  int tq_cnt[2] = {0, 0}, q_cnt[2] = {0, 0};
  int jn[2] = {0, 0}, n[2] = {0, 0}, rp[2] = {0, 0}, hrow[2] = {0, 0};
  bool active[2] = {true, true};
  bool ok = true;

  auto push = [&](const CUtensorMap* tm, int kb, int s) -> bool {
    if (kb < 0 || kb >= p.nb) {
      raise_internal(abort_flag, p.status);
      return false;
    }
    const int st = it % C::kStages;
    const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
    if (!wait_bounded(smem_u32(&bars->empty[st]), ph ^ 1u, abort_flag, p.status, lim))
      return false;
    const uint32_t fb = smem_u32(&bars->full[st]);
    mbar_arrive_expect_tx(fb, C::kTileBytes);
    const uint32_t dst = ring_base + st * C::kTileBytes;
#pragma unroll
    for (int c = 0; c < C::kBoxes; ++c)
      tma_load_2d(dst + c * C::kBoxBytes, tm, fb, c * 64, hrow[s] + kb * kBlock);
    ++it;
    return true;
  };

  while (ok && (active[0] || active[1])) {
    for (int s = 0; s < 2 && ok; ++s) {
      if (!active[s]) continue;
      if (jn[s] == 0) {
        const int e = tq_cnt[s] & 1;
        const uint32_t ph = (uint32_t)(tq_cnt[s] >> 1) & 1u;
        if (!wait_bounded(smem_u32(&bars->tq_empty[s][e]), ph ^ 1u, abort_flag, p.status, lim)) {
          ok = false;
          break;
        }
        const int idx = atomicAdd(p.counter, 1);
        const int t = idx < p.n_live ? p.tile_order[idx] : -1;
        int r0 = 0, cnt = 0, bh = 0, qb = 0, diag = 0;
        if (t >= 0) {
          r0 = p.row_ptr[t];
          cnt = p.row_ptr[t + 1] - r0;
          bh = t / p.nb;
          qb = t - bh * p.nb;
          if (cnt <= 0 || cnt > p.nb) {
            raise_internal(abort_flag, p.status);
            ok = false;
            break;
          }
          diag = (p.causal && p.col_idx[r0 + cnt - 1] == qb) ? 1 : 0;
        }
        volatile int* slot = reinterpret_cast<volatile int*>(&bars->tq[s][e]);
        slot[0] = t;
        slot[1] = r0;
        slot[2] = cnt;
        slot[3] = diag;
        mbar_arrive(smem_u32(&bars->tq_full[s][e]));
        ++tq_cnt[s];
        if (t < 0) {
          active[s] = false;
          continue;
        }
        rp[s] = r0;
        n[s] = cnt;
        hrow[s] = bh * p.S;
        const uint32_t qph = ((uint32_t)q_cnt[s] & 1u) ^ 1u;
        if (!wait_bounded(smem_u32(&bars->q_empty[s]), qph, abort_flag, p.status, lim)) {
          ok = false;
          break;
        }
        ++q_cnt[s];
        const uint32_t qbar = smem_u32(&bars->q_full[s]);
        mbar_arrive_expect_tx(qbar, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c)
          tma_load_2d(q_base + s * C::kTileBytes + c * C::kBoxBytes, tm_q, qbar, c * 64,
                      hrow[s] + qb * kBlock);
        if (!push(tm_k, p.col_idx[r0], s)) {
          ok = false;
          break;
        }
        jn[s] = 1;
      } else {
        if (!push(tm_v, p.col_idx[rp[s] + jn[s] - 1], s)) {
          ok = false;
          break;
        }
        if (jn[s] < n[s]) {
          if (!push(tm_k, p.col_idx[rp[s] + jn[s]], s)) {
            ok = false;
            break;
          }
          ++jn[s];
        } else {
          jn[s] = 0;
        }
      }
    }
  }
  if (!ok) {
    // Let every TMA load this warp issued land before the CTA exits.
    for (int i = (it > C::kStages ? it - C::kStages : 0); i < it; ++i)
      wait_drain(smem_u32(&bars->full[i % C::kStages]), (uint32_t)(i / C::kStages) & 1u);
    for (int s = 0; s < 2; ++s)
      if (q_cnt[s] > 0) wait_drain(smem_u32(&bars->q_full[s]), (uint32_t)(q_cnt[s] - 1) & 1u);
  }
}

// ---------------------------------------------------------------------------
// warp 9: tcgen05 MMA issuer
// ---------------------------------------------------------------------------
template <int D>
__device__ void run_mma(const FwdParams& p, Bars* bars, uint32_t tmem, uint32_t q_base,
                        uint32_t ring_base, volatile int* abort_flag) {
  using C = Cfg<D>;
  const uint64_t lim = p.timeout_ns;
  int it = 0;
  int tq_cnt[2] = {0, 0}, q_cnt[2] = {0, 0}, p_cnt[2] = {0, 0};
  int jn[2] = {0, 0}, n[2] = {0, 0};
  bool active[2] = {true, true};
  bool ok = true;

  auto pop = [&](uint32_t& addr, uint32_t& empty_bar) -> bool {
    const int st = it % C::kStages;
    const uint32_t ph = (uint32_t)(it / C::kStages) & 1u;
    if (!wait_bounded(smem_u32(&bars->full[st]), ph, abort_flag, p.status, lim)) return false;
    addr = ring_base + st * C::kTileBytes;
    empty_bar = smem_u32(&bars->empty[st]);
    ++it;
    return true;
  };

  // S[s] = Q[s] K^T : M=128, N=128, K=D in steps of 16 (32 bytes inside a
  // 128-byte swizzle row; a new 64-column box every 4 steps).  A negative
  // scale is applied as -Q (instruction-descriptor negate bit) so the
  // softmax always sees a non-negative multiplier.
  const uint32_t idesc_s = C::kIdescS | (p.neg_scale ? (1u << 13) : 0u);
  auto issue_s = [&](int s, uint32_t kaddr) {
    const uint32_t qaddr = q_base + s * C::kTileBytes;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * C::kBoxBytes + (kk & 3) * 32;
      const uint64_t ad = smem_desc_sw128(qaddr + off, 16, 1024);
      const uint64_t bd = smem_desc_sw128(kaddr + off, 16, 1024);
      mma_ss(tmem + s * 128, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
    }
  };
  // O[s] (+)= P[s] V : M=128, N=D, K=128 keys in steps of 16.  P is read from
  // TMEM (bf16 pairs, 8 columns per step); V is MN-major (D contiguous):
  // 8-key groups 1024 bytes apart, 64-column boxes 16 KB apart.
  auto issue_pv = [&](int s, uint32_t vaddr, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t bd = smem_desc_sw128(vaddr + kk * 2048, C::kBoxBytes, 1024);
      mma_ts(tmem + 256 + s * 128, tmem + s * 128 + kk * 8, bd, C::kIdescO,
             (accumulate || kk > 0) ? 1u : 0u);
    }
  };

  while (ok && (active[0] || active[1])) {
    for (int s = 0; s < 2 && ok; ++s) {
      if (!active[s]) continue;
      if (jn[s] == 0) {
        const int e = tq_cnt[s] & 1;
        const uint32_t ph = (uint32_t)(tq_cnt[s] >> 1) & 1u;
        if (!wait_bounded(smem_u32(&bars->tq_full[s][e]), ph, abort_flag, p.status, lim)) {
          ok = false;
          break;
        }
        const volatile int* slot = reinterpret_cast<const volatile int*>(&bars->tq[s][e]);
        const int t = slot[0];
        const int cnt = slot[2];
        mbar_arrive(smem_u32(&bars->tq_empty[s][e]));
        ++tq_cnt[s];
        if (t < 0) {
          active[s] = false;
          continue;
        }
        n[s] = cnt;
        if (!wait_bounded(smem_u32(&bars->q_full[s]), (uint32_t)q_cnt[s] & 1u, abort_flag,
                          p.status, lim)) {
          ok = false;
          break;
        }
        ++q_cnt[s];
        uint32_t kaddr, eb;
        if (!pop(kaddr, eb)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(s, kaddr);
        mma_commit(eb);
        if (n[s] == 1) mma_commit(smem_u32(&bars->q_empty[s]));
        mma_commit(smem_u32(&bars->s_full[s]));
        jn[s] = 1;
      } else {
        if (!wait_bounded(smem_u32(&bars->p_full[s]), (uint32_t)p_cnt[s] & 1u, abort_flag,
                          p.status, lim)) {
          ok = false;
          break;
        }
        ++p_cnt[s];
        uint32_t vaddr, eb;
        if (!pop(vaddr, eb)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(s, vaddr, jn[s] > 1);
        mma_commit(eb);
        if (jn[s] < n[s]) {
          uint32_t kaddr, eb2;
          if (!pop(kaddr, eb2)) {
            ok = false;
            break;
          }
          issue_s(s, kaddr);
          mma_commit(eb2);
          if (jn[s] == n[s] - 1) mma_commit(smem_u32(&bars->q_empty[s]));
          mma_commit(smem_u32(&bars->s_full[s]));
          ++jn[s];
        } else {
          mma_commit(smem_u32(&bars->o_full[s]));
          jn[s] = 0;
        }
      }
    }
  }
  // Every MMA issued so far must finish before TMEM is released.
  mma_commit(smem_u32(&bars->drain));
  wait_drain(smem_u32(&bars->drain), 0);
}

// ---------------------------------------------------------------------------
// warps 0-7: softmax + epilogue (one thread per query row of the slot)
// ---------------------------------------------------------------------------
template <int D, bool OUT_F32>
__device__ void write_empty_tiles(const FwdParams& p) {
  using OutT = typename std::conditional<OUT_F32, float, uint16_t>::type;
  const int tid = threadIdx.x;  // 0..255
  constexpr int kVec = 16 / sizeof(OutT);
  for (int e = blockIdx.x; e < p.n_empty; e += gridDim.x) {
    const int t = p.empty_tiles[e];
    const int bh = t / p.nb;
    const int qb = t - bh * p.nb;
    const size_t row0 = (size_t)bh * p.S + (size_t)qb * kBlock;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<OutT*>(p.out) + row0 * D);
    const int nvec = kBlock * D / kVec;
    for (int i = tid; i < nvec; i += 256) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < kBlock) p.lse[row0 + tid] = -__int_as_float(0x7f800000);
  }
}

// The softmax warps execute warp-collective tcgen05.ld/st, so every lane of a
// warp must take the same path after a wait: the outcome is made uniform.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint64_t limit_ns) {
  const bool ok = wait_bounded(bar, parity, abort_flag, status, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// Probabilities of one 128-column row slice: p = 2^(s*sl - m), rounded to
// bf16 pairs into pr[]; returns the running sums of the unrounded (a32) and of
// the rounded (ar) values in four independent pairs of accumulators.
template <bool POLY>
__device__ __forceinline__ void softmax_exp(const uint32_t* sr, uint32_t* pr, float sl, float nm,
                                            float (&a32)[8], float (&ar)[8]) {
#pragma unroll
  for (int q = 0; q < 64; ++q) {
    float x0, x1;
    fma2(x0, x1, __uint_as_float(sr[2 * q]), __uint_as_float(sr[2 * q + 1]), sl, sl, nm, nm);
    float p0, p1;
    if (POLY && kPolyEvery > 0 && (q % (kPolyEvery > 0 ? kPolyEvery : 1)) == kPolyEvery - 1) {
      exp2_poly2(p0, p1, x0, x1);
    } else {
      p0 = ex2_approx(x0);
      p1 = ex2_approx(x1);
    }
    const uint32_t pk = pack_bf16x2(p0, p1);
    pr[q] = pk;
    const int k = (q & 3) * 2;
    add2(a32[k], a32[k + 1], a32[k], a32[k + 1], p0, p1);
    add2(ar[k], ar[k + 1], ar[k], ar[k + 1], __uint_as_float(pk << 16),
         __uint_as_float(pk & 0xFFFF0000u));
  }
}

__device__ __forceinline__ float row_max128(const uint32_t* sr) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = fmaxf(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
#pragma unroll
  for (int c = 16; c < 128; c += 16) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      a[i] = max3(a[i], __uint_as_float(sr[c + 2 * i]), __uint_as_float(sr[c + 2 * i + 1]));
  }
  return fmaxf(max3(a[0], a[1], a[2]), max3(max3(a[3], a[4], a[5]), a[6], a[7]));
}

template <int D, bool OUT_F32>
__device__ void run_softmax(const FwdParams& p, Bars* bars, uint32_t tmem,
                            volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int s = warp >> 2;             // query slot
  const int sub = warp & 3;            // TMEM sub-partition: lanes 32*sub .. 32*sub+31
  const int r = sub * 32 + lane;       // row of the query tile owned by this thread
  const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
  const uint32_t tS = tmem + s * 128 + lane_off;
  const uint32_t tO = tmem + 256 + s * 128 + lane_off;
  const float sl = p.scale_log2;       // > 0 (see FwdParams)
  const uint32_t kNegInf = 0xff800000u;
  const uint64_t lim = p.timeout_ns;

  write_empty_tiles<D, OUT_F32>(p);

  int tq_cnt = 0, s_cnt = 0, o_cnt = 0;
  for (;;) {
    const int e = tq_cnt & 1;
    const uint32_t ph = (uint32_t)(tq_cnt >> 1) & 1u;
    if (!wait_warp(smem_u32(&bars->tq_full[s][e]), ph, abort_flag, p.status, lim)) return;
    const volatile int* slot = reinterpret_cast<const volatile int*>(&bars->tq[s][e]);
    const int t = slot[0];
    const int n = slot[2];
    const int diag_last = slot[3];
    mbar_arrive(smem_u32(&bars->tq_empty[s][e]));
    ++tq_cnt;
    if (t < 0) return;
    const int bh = t / p.nb;
    const int qb = t - bh * p.nb;

    float m = __uint_as_float(kNegInf);  // running max of scale*log2(e)*score (lazy)
    float a32[8], ar[8];                 // unrounded (LSE) and rounded (O) row sums
#pragma unroll
    for (int i = 0; i < 8; ++i) a32[i] = ar[i] = 0.f;
    for (int jb = 0; jb < n; ++jb) {
      if (!wait_warp(smem_u32(&bars->s_full[s]), (uint32_t)s_cnt & 1u, abort_flag, p.status,
                     lim))
        return;
      ++s_cnt;
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld32(tS + 0, sr + 0);
      tmem_ld32(tS + 32, sr + 32);
      tmem_ld32(tS + 64, sr + 64);
      tmem_ld32(tS + 96, sr + 96);
      tmem_wait_ld();
      reg_fence(sr, 128);
      const bool diag = diag_last && jb == n - 1;
      if (diag) {  // causal diagonal tile: key c is allowed for query row r iff c <= r
#pragma unroll
        for (int c = 0; c < 128; ++c) sr[c] = (c > r) ? kNegInf : sr[c];
      }
      const float xm = row_max128(sr) * sl;
      const bool need = xm > m + kTau;  // always true on the first block (m = -inf)
      float f = 1.f;
      if (need) {
        f = ex2_approx(m - xm);  // 0 when m = -inf
        m = xm;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          a32[i] *= f;
          ar[i] *= f;
        }
      }
      uint32_t pr[64];
      if (diag) softmax_exp<false>(sr, pr, sl, -m, a32, ar);
      else softmax_exp<true>(sr, pr, sl, -m, a32, ar);
      tmem_st32(tS + 0, pr);
      tmem_st32(tS + 32, pr + 32);

      // O rescale when this row's max moved (PV(jb-1) is complete: S(jb) was
      // committed after it).
      if (jb > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t orr[32];
          tmem_ld32(tO + c0, orr);
          tmem_wait_ld();
          reg_fence(orr, 32);
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * f);
          tmem_st32(tO + c0, orr);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full[s]));
    }

    // epilogue: O = O_acc / l, LSE = ln2 * (m + log2 l32)
    if (!wait_warp(smem_u32(&bars->o_full[s]), (uint32_t)o_cnt & 1u, abort_flag, p.status, lim))
      return;
    ++o_cnt;
    tc_fence_after();
    const float l = ((ar[0] + ar[1]) + (ar[2] + ar[3])) + ((ar[4] + ar[5]) + (ar[6] + ar[7]));
    const float l32 =
        ((a32[0] + a32[1]) + (a32[2] + a32[3])) + ((a32[4] + a32[5]) + (a32[6] + a32[7]));
    const size_t row = (size_t)bh * p.S + (size_t)qb * kBlock + r;
    const float inv_l = 1.0f / l;
    p.lse[row] = (m + __log2f(l32)) * 0.69314718055994530942f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t orr[32];
      tmem_ld32(tO + c0, orr);
      tmem_wait_ld();
      reg_fence(orr, 32);
      if constexpr (OUT_F32) {
        float* dst = reinterpret_cast<float*>(p.out) + row * D + c0;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          st_global_v4(dst + i, __float_as_uint(__uint_as_float(orr[i]) * inv_l),
                       __float_as_uint(__uint_as_float(orr[i + 1]) * inv_l),
                       __float_as_uint(__uint_as_float(orr[i + 2]) * inv_l),
                       __float_as_uint(__uint_as_float(orr[i + 3]) * inv_l));
      } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + row * D + c0;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv_l,
                              __uint_as_float(orr[2 * i + 1]) * inv_l);
#pragma unroll
        for (int i = 0; i < 16; i += 4) st_global_v4(dst + 2 * i, pk[i], pk[i + 1], pk[i + 2], pk[i + 3]);
      }
    }
    tc_fence_before();
  }
}

template <int D, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    bsattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128B-swizzled tiles want 1024-byte alignment
  Bars* bars = reinterpret_cast<Bars*>(smem_raw + (base - raw) + C::kBarOff);
  const uint32_t q_base = base + C::kQOff;
  const uint32_t ring_base = base + C::kRingOff;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->q_full[s]), 1);
      mbar_init(smem_u32(&bars->q_empty[s]), 1);
      mbar_init(smem_u32(&bars->s_full[s]), 1);
      mbar_init(smem_u32(&bars->p_full[s]), 128);
      mbar_init(smem_u32(&bars->o_full[s]), 1);
      for (int e = 0; e < 2; ++e) {
        mbar_init(smem_u32(&bars->tq_full[s][e]), 1);
        mbar_init(smem_u32(&bars->tq_empty[s][e]), 1 + 128);
      }
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;

  if (warp >= 8) {
    regs_dec<kRegsOther>();
    if (warp == kWarpLoad && lane == 0)
      run_producer<D>(&tm_q, &tm_k, &tm_v, p, bars, q_base, ring_base, abort_flag);
    else if (warp == kWarpMma && lane == 0)
      run_mma<D>(p, bars, tmem, q_base, ring_base, abort_flag);
  } else {
    regs_inc<kRegsSoftmax>();
    run_softmax<D, OUT_F32>(p, bars, tmem, abort_flag);
  }
  __syncwarp();  // reconverge each warp before the CTA-wide barrier

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // The last CTA to finish rewinds the tile counter for the next launch on
  // this workspace (every CTA has stopped claiming tiles by now).
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.done, 1) == (int)gridDim.x - 1) {
      atomicExch(p.counter, 0);
      atomicExch(p.done, 0);
      __threadfence();
    }
  }
}

__global__ void selftest_wait_kernel(unsigned long long timeout_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the wait must end through its time limit.
  wait_bounded(smem_u32(&bar), 0, &abort_flag, status, timeout_ns);
  __syncthreads();
}

template <int D, bool OUT_F32>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int grid, cudaStream_t stream) {
  const size_t smem = Cfg<D>::kSmem + 1024;
  cudaError_t e = cudaFuncSetAttribute(bsattn_fwd_kernel<D, OUT_F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  bsattn_fwd_kernel<D, OUT_F32><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_smem_bytes(int D) {
  return D == 64 ? Cfg<64>::kSmem + 1024 : Cfg<128>::kSmem + 1024;
}

cudaError_t launch_fwd(int D, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t stream) {
  if (D == 64) {
    return out_f32 ? launch_one<64, true>(tq, tk, tv, p, grid, stream)
                   : launch_one<64, false>(tq, tk, tv, p, grid, stream);
  }
  return out_f32 ? launch_one<128, true>(tq, tk, tv, p, grid, stream)
                 : launch_one<128, false>(tq, tk, tv, p, grid, stream);
}

cudaError_t launch_selftest_wait(unsigned long long timeout_ns, int* d_status,
                                 cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(timeout_ns, d_status);
  return cudaGetLastError();
}

}  // namespace bsattn
