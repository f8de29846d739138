// Block-sparse flash-attention backward for sm_103a (GB300).
//
// What it computes: the gradients dQ, dK, dV of the forward operation
// O = softmax(scale * Q K^T + mask) V over the same live blocks.  "Writing
// Pallas Kernels for JAX: Stepping Outside the XLA Safety Net" (section "The
// Empathy of the Void") notes that a hand-written attention kernel needs its
// own gradient definitions; these are the derivative of that article's
// forward operation (sections "Designing the Block Specification" and
// "Writing the Kernel Logic: Load, Compute, Store"), formed blockwise the way
// flash attention forms the exact softmax ("Pallas-Triton kernels and kernel
// auto-tuning", section "Flash Attention"):
//
//   P_ij  = exp(scale q_i.k_j - LSE_i)         (recomputed from the saved LSE)
//   dP_ij = dO_i . v_j,   Dl_i = dO_i . O_i,   dS_ij = P_ij (dP_ij - Dl_i)
//   dV_j  = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j
//
// GB300 design: two kernels, neither with atomics (several key tiles feed
// each dQ row and several query tiles each dK/dV row; fp32 reductions for
// either were measured to bound the whole pass by L2 atomic throughput).
//
// bsattn_bwd_kernel (dK, dV): one CTA per key tile (128 keys of one (batch,
// head)), 288 threads: eight CUDA-core warps (two per TMEM sub-partition,
// warps 4h .. 4h+3 working on half h of each query block: queries 64h ..
// 64h+63) and one copy / MMA warp.  It walks the plan's transposed list (the
// live query blocks of its key block) and keeps dV and dK in tensor memory.
// Per query block and half h, with keys as TMEM lanes:
//   S^T_h = K Q_h^T, dP^T_h = V dO_h^T                 (tcgen05, N = 64, operands in smem)
//   P^T = 2^(S^T scale log2 e - LSE log2 e), dS^T = P^T (dP^T - Dl)   (CUDA cores)
//   P^T (bf16) goes back to tensor memory over S^T_h (queries 64h + 2c,
//   64h + 2c + 1 in column 64h + c: each half writes inside the scores it read);
//   dS^T (bf16) goes to shared memory
//   dV += P^T_h dO_h   (A from tensor memory, B = dO read MN-major, K = 64)
//   dK += dS^T_h Q_h   (A = dS^T, B = Q read MN-major, K = 64)
// Each step has a barrier per half, so the CUDA cores work on one half while
// the tensor core computes the other half's products: half 0's P^T / dS^T
// overlaps S^T_1 and dP^T_1, half 1's overlaps dV, dK of half 0 and the next
// block's S^T_0, dP^T_0.  Q and dO are double-buffered: the next query
// block's tiles load once the previous block's products are done with them.
//
// bsattn_bwd_dq_kernel (dQ): one CTA per query tile, walking the forward
// plan's list of live key blocks with queries as TMEM lanes: S = Q K^T and
// dP = dO V^T recomputed, dS = P (dP - Dl) to shared memory, dQ += dS K in
// tensor memory (K and V double-buffered), dQ written once at the end; the
// same 288 threads and per-half pipeline as the dK/dV kernel, halves of the
// key block (keys 64h .. 64h+63) instead of the query block.
//
// Every mbarrier wait is bounded; on expiry the status word records a
// timeout and the CTA drains its copies and MMAs before it frees tensor memory.
#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace bsattn {
namespace {

constexpr uint32_t kBwdTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634074f;
constexpr int kMaxKvGroup = 64;  // query heads per K/V head the dK/dV kernel walks

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = kBlock * D * 2;  // one 128 x D bf16 tile
  static constexpr int kBoxes = D / 64;              // 64-column (128-byte) TMA boxes
  static constexpr int kBoxBytes = kBlock * 128;     // 16 KB per box
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;     // two buffers
  static constexpr int kdOOff = kQOff + 2 * kTileBytes;  // two buffers
  static constexpr int kdSOff = kdOOff + 2 * kTileBytes;  // 128 x 128 bf16: two boxes
  static constexpr int kBarOff = kdSOff + 2 * kBoxBytes;
  static constexpr int kGrpOff = kBarOff + 128;  // per query head of the group: list start, prefix
  static constexpr int kSmem = kGrpOff + 4 * (2 * kMaxKvGroup + 1) + 124;
  // S^T = K Q^T and dP^T = V dO^T, per half of the query block: M = 128 keys,
  // N = 64 queries, both K-major
  static constexpr uint32_t kIdescT = idesc_bf16_f32(128, 64, false);
  // dV += P^T dO and dK += dS^T Q: M = 128 keys, N = D, B MN-major
  static constexpr uint32_t kIdescKV = idesc_bf16_f32(128, D, true);
  // tensor-memory columns
  static constexpr uint32_t kTS = 0;         // S^T (fp32), then P^T (bf16) in [0,32) and [64,96)
  static constexpr uint32_t kTdP = 128;      // dP^T (fp32)
  static constexpr uint32_t kTdV = 256;      // dV accumulator (D columns)
  static constexpr uint32_t kTdK = 256 + D;  // dK accumulator (D columns)
};
static_assert(BwdCfg<128>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");
static_assert(BwdCfg<128>::kTdK + 128 <= kBwdTmemCols, "tensor memory exceeded");

// The dK/dV kernel works on each query block in two halves h (queries
// 64h .. 64h+63), with a barrier per half for every step, so that one half's
// CUDA-core work overlaps the tensor core's work on the other half.
struct __align__(8) BwdBars {
  uint64_t kv_full;      // K and V of the key tile loaded
  uint64_t qd_full[2];   // Q and dO of a query block loaded (by buffer)
  uint64_t st_done[2];   // S^T and dP^T of half h computed
  uint64_t pds_done[2];  // P^T (tensor memory) and dS^T (shared memory) of half h written
  uint64_t grad_done[2]; // dV and dK updated with half h
  uint64_t drain;        // every MMA issued so far complete
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 128, "barrier block must fit its 128-byte region");
constexpr int kBwdKvThreads = 288;  // dK/dV kernel: 8 CUDA-core warps and an MMA / copy warp

// Dl_i = dO_i . O_i (fp32 over the stored O and dO); one warp per row.
template <int D, bool O_F32>
__global__ void bwd_prep_kernel(const void* __restrict__ o, const uint16_t* __restrict__ dout,
                                float* __restrict__ dl, long long rows) {
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr int kPer = D / 32;  // elements per lane: 4 (D = 128) or 2 (D = 64)
  const size_t base = (size_t)row * D + (size_t)lane * kPer;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const float g = __uint_as_float((uint32_t)dout[base + e] << 16);
    float x;
    if constexpr (O_F32)
      x = reinterpret_cast<const float*>(o)[base + e];
    else
      x = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(o)[base + e] << 16);
    acc = fmaf(g, x, acc);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 16);
  acc += __shfl_xor_sync(0xffffffffu, acc, 8);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (lane == 0) dl[row] = acc;
}

__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* status, uint64_t limit_ns) {
  const bool ok = wait_bounded(bar, parity, abort_flag, status, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait used while draining (no abort check: the copies and MMAs in
// flight finish on their own; the limit only guards against a broken state).
__device__ __forceinline__ void bwd_drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return;
}

template <int D>
__global__ void __launch_bounds__(kBwdKvThreads, 1)
    bsattn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = BwdCfg<D>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int kMmaWarp = 8;   // warps 0-7: CUDA-core work, half h = warps 4h .. 4h+3
  const int tile = blockIdx.x;  // (b * Hkv + hk) * nb + kb: a key tile of K/V head hk
  const int kvbh = tile / p.nb;
  const int kb = tile - kvbh * p.nb;
  const int g = p.kv_group;     // query heads reading this K/V head
  const int hkv = p.H / g;      // K/V heads per batch entry
  const int bh0 = (kvbh / hkv) * p.H + (kvbh % hkv) * g;  // its first query head b*H + hk*g
  const int krow0 = kvbh * p.S + kb * kBlock;             // first key row of the tile

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  // The CTA walks the transposed lists of the group's query heads one after
  // the other: head bh0 + i contributes entries [g_st[i], g_st[i+1]) of the
  // walk, starting at row_idx[g_c0[i]].
  int* g_c0 = reinterpret_cast<int*>(smem_raw + (base - raw) + C::kGrpOff);
  int* g_st = g_c0 + kMaxKvGroup;
  if (tid < g) {
    const int t = (bh0 + tid) * p.nb + kb;
    g_c0[tid] = p.col_ptr[t];
    g_st[tid + 1] = p.col_ptr[t + 1] - p.col_ptr[t];
  }
  __syncthreads();
  if (tid == 0) {
    g_st[0] = 0;
    for (int i = 0; i < g; ++i) g_st[i + 1] += g_st[i];
  }
  __syncthreads();
  const int n = g_st[g];
  // entry j of the walk: query head (b*H + h) and query block
  auto entry = [&](int j, int& bhq, int& qbj) {
    int gi = 0;
    while (gi + 1 < g && g_st[gi + 1] <= j) ++gi;
    bhq = bh0 + gi;
    qbj = p.row_idx[g_c0[gi] + (j - g_st[gi])];
  };
  if (n <= 0) {  // no live query block: dK = dV = 0
    float4* dk4 = reinterpret_cast<float4*>(p.dk + (size_t)krow0 * D);
    float4* dv4 = reinterpret_cast<float4*>(p.dv + (size_t)krow0 * D);
    for (int i = tid; i < kBlock * D / 4; i += kBwdKvThreads) {
      dk4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      dv4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  // The plan's lists must hold valid query blocks; anything else is an internal error.
  bool bad = n > p.nb * g;
  for (int gi = 0; !bad && gi < g; ++gi) bad = g_st[gi + 1] - g_st[gi] > p.nb;
  for (int i = tid; !bad && i < n; i += kBwdKvThreads) {
    int bhq = 0, qb = 0;
    entry(i, bhq, qb);
    bad = qb < 0 || qb >= p.nb || (p.causal && qb < kb);
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(p.status, kStatusInternal);
    return;
  }

  BwdBars* bars = reinterpret_cast<BwdBars*>(smem_raw + (base - raw) + C::kBarOff);
  const uint64_t lim = p.timeout_ns;
  volatile int* abort_flag = &bars->abort_flag;

  if (tid == 0) {
    mbar_init(smem_u32(&bars->kv_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->qd_full[i]), 1);
      mbar_init(smem_u32(&bars->st_done[i]), 1);
      mbar_init(smem_u32(&bars->pds_done[i]), 4);  // the half's four warps
      mbar_init(smem_u32(&bars->grad_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&bars->tmem_base), kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;

  if (warp == kMmaWarp) {
    // ---- copies and MMAs (elected lane): per block j, for each half h,
    // S^T_h = K Q_h^T and dP^T_h = V dO_h^T once the half's buffers are free
    // (dV, dK of the previous block's half h complete), then, once the CUDA
    // cores have written P^T_h and dS^T_h, dV += P^T_h dO_h and dK += dS^T_h Q_h.
    auto load_tile = [&](const CUtensorMap* tm, uint32_t dst, uint32_t bar, int row) {
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c) tma_load_2d(dst + c * C::kBoxBytes, tm, bar, c * 64, row);
    };
    auto load_qd = [&](int i) {  // Q and dO of entry i into buffer i % 2
      const int b = i & 1;
      const uint32_t bar = smem_u32(&bars->qd_full[b]);
      int bhq = 0, qbi = 0;
      entry(i, bhq, qbi);
      const int row = bhq * p.S + qbi * kBlock;
      mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
      load_tile(&tm_q, base + C::kQOff + b * C::kTileBytes, bar, row);
      load_tile(&tm_do, base + C::kdOOff + b * C::kTileBytes, bar, row);
    };
    int n_issued = 0, n_waited = 0;  // Q-dO loads issued / awaited
    if (elect_one()) {
      const uint32_t bar = smem_u32(&bars->kv_full);
      mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
      load_tile(&tm_k, base + C::kKOff, bar, krow0);
      load_tile(&tm_v, base + C::kVOff, bar, krow0);
      load_qd(0);
      if (n > 1) load_qd(1);
    }
    __syncwarp();
    n_issued = n > 1 ? 2 : 1;
    ok = bwd_wait(smem_u32(&bars->kv_full), 0, abort_flag, p.status, lim);
    const bool kv_ok = ok;
    const uint64_t kd = smem_desc_sw128(base + C::kKOff, 16, 1024);
    const uint64_t vd = smem_desc_sw128(base + C::kVOff, 16, 1024);
    const uint64_t ds_k = smem_desc_sw128(base + C::kdSOff, 16, 1024);
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1;
      ok = bwd_wait(smem_u32(&bars->qd_full[b]), (uint32_t)(j >> 1) & 1u, abort_flag, p.status,
                    lim);
      if (!ok) break;
      n_waited = j + 1;
      for (int h = 0; ok && h < 2; ++h) {
        if (j > 0) {  // half h of the previous block multiplied: its columns and dS^T free
          ok = bwd_wait(smem_u32(&bars->grad_done[h]), (uint32_t)(j - 1) & 1u, abort_flag,
                        p.status, lim);
          if (!ok) break;
          if (h == 1 && j + 1 < n) {  // the previous block's buffers are free: next Q, dO
            if (elect_one()) load_qd(j + 1);
            __syncwarp();
            n_issued = j + 2;
          }
        }
        tc_fence_after();
        if (elect_one()) {
          // queries 64h .. 64h+63: rows 64h.. of the Q and dO tiles (8 KB into each box)
          const uint32_t rows_h = (uint32_t)h * 64u * 128u;
          const uint64_t qd = smem_desc_sw128(base + C::kQOff + b * C::kTileBytes + rows_h, 16, 1024);
          const uint64_t dd = smem_desc_sw128(base + C::kdOOff + b * C::kTileBytes + rows_h, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::kTS + 64u * h, kd + off, qd + off, C::kIdescT, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::kTdP + 64u * h, vd + off, dd + off, C::kIdescT, kk > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars->st_done[h]));
        }
        __syncwarp();
      }
      for (int h = 0; ok && h < 2; ++h) {
        ok = bwd_wait(smem_u32(&bars->pds_done[h]), (uint32_t)j & 1u, abort_flag, p.status, lim);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint32_t qoff = base + C::kQOff + b * C::kTileBytes;
          const uint32_t dooff = base + C::kdOOff + b * C::kTileBytes;
          const uint64_t do_mn = smem_desc_sw128(dooff, C::kBoxBytes, 1024);
          const uint64_t q_mn = smem_desc_sw128(qoff, C::kBoxBytes, 1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * h + k4;                       // queries 16kk .. 16kk+15
            const uint32_t mn = (uint32_t)(kk * 2048) >> 4;  // 16 rows of 128 bytes
            const uint32_t km = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
            const uint32_t pcol = 64u * h + 8u * k4;  // P^T of queries 16kk .. in bf16 pairs
            mma_ts(tmem + C::kTdV, tmem + C::kTS + pcol, do_mn + mn, C::kIdescKV, acc);
            mma_ss(tmem + C::kTdK, ds_k + km, q_mn + mn, C::kIdescKV, acc);
          }
          mma_commit(smem_u32(&bars->grad_done[h]));
        }
        __syncwarp();
      }
    }
    // Drain: every copy issued and every MMA issued completes before tensor
    // memory is freed and the CTA exits.
    if (!kv_ok) bwd_drain_wait(smem_u32(&bars->kv_full), 0, lim);
    for (int i = n_waited; i < n_issued; ++i)
      bwd_drain_wait(smem_u32(&bars->qd_full[i & 1]), (uint32_t)(i >> 1) & 1u, lim);
    if (elect_one()) mma_commit(smem_u32(&bars->drain));
    __syncwarp();
    bwd_drain_wait(smem_u32(&bars->drain), 0, lim);
  } else {
    // ---- P^T and dS^T of half h (queries 64h .. 64h+63), one key row (TMEM
    // lane) per thread, 32 queries at a time.  P^T (bf16 pairs) goes over
    // the scores just read: queries 64h + 2c, 64h + 2c + 1 in column 64h + c.
    // dS^T (bf16) goes to shared memory, 128-byte swizzled like a TMA tile:
    // row r, 16-byte chunk c of 64-query box h at h * 16 KB + r * 128 +
    // ((c ^ (r mod 8)) * 16).
    const int h = warp >> 2;
    const int r = tid & (kBlock - 1);  // TMEM lane: key row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes
    const float sl = p.scale_log2;
    const uint32_t tS = tmem + C::kTS + lane_off;
    const uint32_t tdP = tmem + C::kTdP + lane_off;
    const uint32_t sdS = base + C::kdSOff;
    // LSE (log2 units) and Dl of the half's queries 64h + lane and 64h + 32 +
    // lane of entry j, loaded one entry ahead by every warp for itself and
    // passed between lanes by shuffles (no barrier between the warps)
    float la_next = 0.f, lb_next = 0.f, da_next = 0.f, db_next = 0.f;
    auto fetch = [&](int i) {
      int bhq = 0, qbi = 0;
      entry(i, bhq, qbi);
      const int qrow = bhq * p.S + qbi * kBlock + 64 * h + lane;
      la_next = p.lse[qrow] * kLog2e;
      lb_next = p.lse[qrow + 32] * kLog2e;
      da_next = p.dl[qrow];
      db_next = p.dl[qrow + 32];
    };
    fetch(0);
    for (int j = 0; j < n; ++j) {
      int bhj = 0, qb = 0;
      entry(j, bhj, qb);
      const float la = la_next, lb = lb_next, da = da_next, db = db_next;
      if (j + 1 < n) fetch(j + 1);
      ok = bwd_wait(smem_u32(&bars->st_done[h]), (uint32_t)j & 1u, abort_flag, p.status, lim);
      if (!ok) break;
      tc_fence_after();
      const bool diag = p.causal && qb == kb;  // key r is allowed for query q iff r <= q
#pragma unroll 1
      for (int ch = 2 * h; ch < 2 * h + 2; ++ch) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tS + ch * 32, sv);
        tmem_ld32(tdP + ch * 32, dp);
        tmem_wait_ld();
        reg_fence(sv, 32);
        reg_fence(dp, 32);
        const float lsrc = (ch & 1) ? lb : la;  // queries 64h + 32 (ch & 1) + lane
        const float dsrc = (ch & 1) ? db : da;
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int q = ch * 32 + i;
          const float l0 = __shfl_sync(0xffffffffu, lsrc, i);
          const float l1 = __shfl_sync(0xffffffffu, lsrc, i + 1);
          const float d0l = __shfl_sync(0xffffffffu, dsrc, i);
          const float d1l = __shfl_sync(0xffffffffu, dsrc, i + 1);
          float p0 = ex2_approx(fmaf(__uint_as_float(sv[i]), sl, -l0));
          float p1 = ex2_approx(fmaf(__uint_as_float(sv[i + 1]), sl, -l1));
          if (diag) {
            p0 = r > q ? 0.f : p0;
            p1 = r > q + 1 ? 0.f : p1;
          }
          const float d0 = p0 * (__uint_as_float(dp[i]) - d0l);
          const float d1 = p1 * (__uint_as_float(dp[i + 1]) - d1l);
          pk[i >> 1] = pack_bf16x2(p0, p1);
          dk[i >> 1] = pack_bf16x2(d0, d1);
        }
        tmem_st32_16(tS + (uint32_t)(64 * (ch >> 1) + 16 * (ch & 1)), pk);
        const uint32_t rowa = sdS + (uint32_t)(ch >> 1) * C::kBoxBytes + (uint32_t)r * 128u;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t c = (uint32_t)((ch & 1) * 4 + u);
          st_shared_v4(rowa + ((c ^ (uint32_t)(r & 7)) << 4), dk[4 * u], dk[4 * u + 1],
                       dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();  // the warp's P^T and dS^T are written
      if (lane == 0) mbar_arrive(smem_u32(&bars->pds_done[h]));
    }
  }
  // Every role has left its loop; the MMA warp drained all copies and MMAs.
  const bool all_ok = __syncthreads_and(ok);
  tc_fence_after();
  if (all_ok && warp < kMmaWarp) {  // dV and dK (times scale), one key row and half the columns
    const int r = tid & (kBlock - 1);
    const int half = warp >> 2;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float* dvr = p.dv + (size_t)(krow0 + r) * D;
    float* dkr = p.dk + (size_t)(krow0 + r) * D;
#pragma unroll 1
    for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
      uint32_t v[32], k[32];
      tmem_ld32(tmem + C::kTdV + lane_off + c, v);
      tmem_ld32(tmem + C::kTdK + lane_off + c, k);
      tmem_wait_ld();
      reg_fence(v, 32);
      reg_fence(k, 32);
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        st_global_v4(dvr + c + i, v[i], v[i + 1], v[i + 2], v[i + 3]);
        st_global_v4(dkr + c + i, __float_as_uint(__uint_as_float(k[i]) * p.scale),
                     __float_as_uint(__uint_as_float(k[i + 1]) * p.scale),
                     __float_as_uint(__uint_as_float(k[i + 2]) * p.scale),
                     __float_as_uint(__uint_as_float(k[i + 3]) * p.scale));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// dQ kernel layout: Q, dO once per tile; K and V double-buffered; dS with
// queries as rows.
template <int D>
struct DqCfg {
  static constexpr int kTileBytes = kBlock * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kBlock * 128;
  static constexpr int kQOff = 0;
  static constexpr int kdOOff = kTileBytes;
  static constexpr int kKOff = 2 * kTileBytes;   // two buffers
  static constexpr int kVOff = 4 * kTileBytes;   // two buffers
  static constexpr int kdSOff = 6 * kTileBytes;  // 128 queries x 128 keys bf16: two boxes
  static constexpr int kBarOff = kdSOff + 2 * kBoxBytes;
  static constexpr int kSmem = kBarOff + 256;
  // S = Q K^T and dP = dO V^T, per half of the key block: M = 128 queries,
  // N = 64 keys, both K-major
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false);
  // dQ += dS K: M = 128 queries, N = D, B (K) read MN-major
  static constexpr uint32_t kIdescQ = idesc_bf16_f32(128, D, true);
  static constexpr uint32_t kTS = 0;     // S (fp32)
  static constexpr uint32_t kTdP = 128;  // dP (fp32)
  static constexpr uint32_t kTdQ = 256;  // dQ accumulator (D columns)
};
static_assert(DqCfg<128>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");

// The dQ kernel works on each key block in two halves h (keys 64h .. 64h+63)
// with a barrier per half for every step, as the dK/dV kernel does.
struct __align__(8) DqBars {
  uint64_t qd_full;      // Q and dO of the tile loaded
  uint64_t kv_full[2];   // K and V of a key block loaded (by buffer)
  uint64_t st_done[2];   // S and dP of half h computed
  uint64_t ds_done[2];   // dS of half h written
  uint64_t grad_done[2]; // dQ updated with half h
  uint64_t drain;        // every MMA issued so far complete
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(DqBars) <= 256, "barrier block must fit its 256-byte region");

template <int D>
__global__ void __launch_bounds__(kBwdKvThreads, 1)
    bsattn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = DqCfg<D>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int kMmaWarp = 8;   // warps 0-7: CUDA-core work, half h = warps 4h .. 4h+3
  const int tile = blockIdx.x;  // (b * H + h) * nb + qb
  const int bh = tile / p.nb;
  const int qb = tile - bh * p.nb;
  const int r0 = p.row_ptr[tile];
  const int n = p.row_ptr[tile + 1] - r0;
  const int qrow0 = bh * p.S + qb * kBlock;  // first query row of the tile
  const int kvbh =  // the K/V head it attends with
      p.kv_group > 1 ? (bh / p.H) * (p.H / p.kv_group) + (bh % p.H) / p.kv_group : bh;
  if (n <= 0) {  // no live key block: dQ = 0
    float4* dq4 = reinterpret_cast<float4*>(p.dq + (size_t)qrow0 * D);
    for (int i = tid; i < kBlock * D / 4; i += kBwdKvThreads)
      dq4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  bool bad = n > p.nb;
  for (int i = tid; !bad && i < n; i += kBwdKvThreads) {
    const int kb = p.col_idx[r0 + i];
    bad = kb < 0 || kb >= p.nb || (p.causal && kb > qb);
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(p.status, kStatusInternal);
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  DqBars* bars = reinterpret_cast<DqBars*>(smem_raw + (base - raw) + C::kBarOff);
  const uint64_t lim = p.timeout_ns;
  volatile int* abort_flag = &bars->abort_flag;
  if (tid == 0) {
    mbar_init(smem_u32(&bars->qd_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->kv_full[i]), 1);
      mbar_init(smem_u32(&bars->st_done[i]), 1);
      mbar_init(smem_u32(&bars->ds_done[i]), 4);  // the half's four warps
      mbar_init(smem_u32(&bars->grad_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&bars->tmem_base), kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  bool ok = true;

  if (warp == kMmaWarp) {
    // ---- copies and MMAs (elected lane): per key block j, for each half h,
    // S_h = Q K_h^T and dP_h = dO V_h^T once the half's columns and dS are
    // free (dQ of the previous block's half h complete), then, once the CUDA
    // cores have written dS_h, dQ += dS_h K_h.
    auto load_tile = [&](const CUtensorMap* tm, uint32_t dst, uint32_t bar, int row) {
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c) tma_load_2d(dst + c * C::kBoxBytes, tm, bar, c * 64, row);
    };
    auto load_kv = [&](int i) {  // K and V of key block number i into buffer i % 2
      const int b = i & 1;
      const uint32_t bar = smem_u32(&bars->kv_full[b]);
      const int row = kvbh * p.S + p.col_idx[r0 + i] * kBlock;
      mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
      load_tile(&tm_k, base + C::kKOff + b * C::kTileBytes, bar, row);
      load_tile(&tm_v, base + C::kVOff + b * C::kTileBytes, bar, row);
    };
    if (elect_one()) {
      const uint32_t bar = smem_u32(&bars->qd_full);
      mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
      load_tile(&tm_q, base + C::kQOff, bar, qrow0);
      load_tile(&tm_do, base + C::kdOOff, bar, qrow0);
      load_kv(0);
      if (n > 1) load_kv(1);
    }
    __syncwarp();
    int n_issued = n > 1 ? 2 : 1, n_waited = 0;
    ok = bwd_wait(smem_u32(&bars->qd_full), 0, abort_flag, p.status, lim);
    const bool qd_ok = ok;
    const uint64_t qd = smem_desc_sw128(base + C::kQOff, 16, 1024);
    const uint64_t dd = smem_desc_sw128(base + C::kdOOff, 16, 1024);
    const uint64_t ds_k = smem_desc_sw128(base + C::kdSOff, 16, 1024);
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1;
      ok = bwd_wait(smem_u32(&bars->kv_full[b]), (uint32_t)(j >> 1) & 1u, abort_flag, p.status,
                    lim);
      if (!ok) break;
      n_waited = j + 1;
      for (int h = 0; ok && h < 2; ++h) {
        if (j > 0) {  // half h of the previous block multiplied: its columns and dS free
          ok = bwd_wait(smem_u32(&bars->grad_done[h]), (uint32_t)(j - 1) & 1u, abort_flag,
                        p.status, lim);
          if (!ok) break;
          if (h == 1 && j + 1 < n) {  // the previous block's K, V are free: next K, V
            if (elect_one()) load_kv(j + 1);
            __syncwarp();
            n_issued = j + 2;
          }
        }
        tc_fence_after();
        if (elect_one()) {
          // keys 64h .. 64h+63: rows 64h.. of the K and V tiles (8 KB into each box)
          const uint32_t rows_h = (uint32_t)h * 64u * 128u;
          const uint64_t kd = smem_desc_sw128(base + C::kKOff + b * C::kTileBytes + rows_h, 16, 1024);
          const uint64_t vd = smem_desc_sw128(base + C::kVOff + b * C::kTileBytes + rows_h, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::kTS + 64u * h, qd + off, kd + off, C::kIdescS, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::kTdP + 64u * h, dd + off, vd + off, C::kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars->st_done[h]));
        }
        __syncwarp();
      }
      for (int h = 0; ok && h < 2; ++h) {
        ok = bwd_wait(smem_u32(&bars->ds_done[h]), (uint32_t)j & 1u, abort_flag, p.status, lim);
        if (!ok) break;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t k_mn = smem_desc_sw128(base + C::kKOff + b * C::kTileBytes, C::kBoxBytes,
                                                1024);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * h + k4;  // keys 16kk .. 16kk+15
            const uint32_t km = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
            const uint32_t mn = (uint32_t)(kk * 2048) >> 4;
            mma_ss(tmem + C::kTdQ, ds_k + km, k_mn + mn, C::kIdescQ, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&bars->grad_done[h]));
        }
        __syncwarp();
      }
    }
    // Drain copies and MMAs in flight.
    if (!qd_ok) bwd_drain_wait(smem_u32(&bars->qd_full), 0, lim);
    for (int i = n_waited; i < n_issued; ++i)
      bwd_drain_wait(smem_u32(&bars->kv_full[i & 1]), (uint32_t)(i >> 1) & 1u, lim);
    if (elect_one()) mma_commit(smem_u32(&bars->drain));
    __syncwarp();
    bwd_drain_wait(smem_u32(&bars->drain), 0, lim);
  } else {
    // ---- dS = P (dP - Dl) of half h (keys 64h .. 64h+63), one query row and
    // 32 keys at a time, to shared memory (bf16, 128-byte swizzled: row r,
    // 16-byte chunk c of 64-key box h at h * 16 KB + r * 128 + ((c ^ (r mod 8)) * 16)).
    const int h = warp >> 2;
    const int r = tid & (kBlock - 1);  // TMEM lane: query row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float l2 = p.lse[qrow0 + r] * kLog2e;  // this row's LSE in log2 units
    const float dlr = p.dl[qrow0 + r];
    const float sl = p.scale_log2;
    const uint32_t tS = tmem + C::kTS + lane_off;
    const uint32_t tdP = tmem + C::kTdP + lane_off;
    const uint32_t sdS = base + C::kdSOff;
    for (int j = 0; j < n; ++j) {
      const int kb = p.col_idx[r0 + j];
      ok = bwd_wait(smem_u32(&bars->st_done[h]), (uint32_t)j & 1u, abort_flag, p.status, lim);
      if (!ok) break;
      tc_fence_after();
      const bool diag = p.causal && kb == qb;  // key c is allowed for query r iff c <= r
#pragma unroll 1
      for (int ch = 2 * h; ch < 2 * h + 2; ++ch) {
        uint32_t sv[32], dp[32];
        tmem_ld32(tS + ch * 32, sv);
        tmem_ld32(tdP + ch * 32, dp);
        tmem_wait_ld();
        reg_fence(sv, 32);
        reg_fence(dp, 32);
        uint32_t dk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int c = ch * 32 + i;
          float p0 = ex2_approx(fmaf(__uint_as_float(sv[i]), sl, -l2));
          float p1 = ex2_approx(fmaf(__uint_as_float(sv[i + 1]), sl, -l2));
          if (diag) {
            p0 = c > r ? 0.f : p0;
            p1 = c + 1 > r ? 0.f : p1;
          }
          dk[i >> 1] = pack_bf16x2(p0 * (__uint_as_float(dp[i]) - dlr),
                                   p1 * (__uint_as_float(dp[i + 1]) - dlr));
        }
        const uint32_t rowa = sdS + (uint32_t)(ch >> 1) * C::kBoxBytes + (uint32_t)r * 128u;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t c = (uint32_t)((ch & 1) * 4 + u);
          st_shared_v4(rowa + ((c ^ (uint32_t)(r & 7)) << 4), dk[4 * u], dk[4 * u + 1],
                       dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();  // the warp's dS is written (and its S, dP reads are complete)
      if (lane == 0) mbar_arrive(smem_u32(&bars->ds_done[h]));
    }
  }
  const bool all_ok = __syncthreads_and(ok);
  tc_fence_after();
  if (all_ok && warp < kMmaWarp) {  // dQ times scale, one query row and half of the columns
    const int r = tid & (kBlock - 1);
    const int half = warp >> 2;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float* dqr = p.dq + (size_t)(qrow0 + r) * D;
#pragma unroll 1
    for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + C::kTdQ + lane_off + c, v);
      tmem_wait_ld();
      reg_fence(v, 32);
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        st_global_v4(dqr + c + i, __float_as_uint(__uint_as_float(v[i]) * p.scale),
                     __float_as_uint(__uint_as_float(v[i + 1]) * p.scale),
                     __float_as_uint(__uint_as_float(v[i + 2]) * p.scale),
                     __float_as_uint(__uint_as_float(v[i + 3]) * p.scale));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

template <int D>
cudaError_t launch_bwd_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, int grid,
                            cudaStream_t stream) {
  static std::atomic<bool> opted_in[64];
  const size_t smem = DqCfg<D>::kSmem + 1024;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bsattn_bwd_dq_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  bsattn_bwd_dq_kernel<D><<<grid, kBwdKvThreads, smem, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, int grid,
                         cudaStream_t stream) {
  static std::atomic<bool> opted_in[64];
  const size_t smem = BwdCfg<D>::kSmem + 1024;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bsattn_bwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  bsattn_bwd_kernel<D><<<grid, kBwdKvThreads, smem, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_prep(int D, bool o_f32, const void* o, const void* dout, float* dl,
                            long long rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;  // 8 warps (rows) per 256-thread block
  const uint16_t* g = static_cast<const uint16_t*>(dout);
  if (D == 128) {
    if (o_f32) bwd_prep_kernel<128, true><<<(unsigned)blocks, 256, 0, stream>>>(o, g, dl, rows);
    else bwd_prep_kernel<128, false><<<(unsigned)blocks, 256, 0, stream>>>(o, g, dl, rows);
  } else {
    if (o_f32) bwd_prep_kernel<64, true><<<(unsigned)blocks, 256, 0, stream>>>(o, g, dl, rows);
    else bwd_prep_kernel<64, false><<<(unsigned)blocks, 256, 0, stream>>>(o, g, dl, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  return D == 128 ? launch_bwd_t<128>(tq, tk, tv, tdo, p, grid, stream)
                  : launch_bwd_t<64>(tq, tk, tv, tdo, p, grid, stream);
}

cudaError_t launch_bwd_dq(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                          int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  return D == 128 ? launch_bwd_dq_t<128>(tq, tk, tv, tdo, p, grid, stream)
                  : launch_bwd_dq_t<64>(tq, tk, tv, tdo, p, grid, stream);
}

}  // namespace bsattn
