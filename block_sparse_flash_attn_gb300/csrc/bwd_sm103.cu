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
// head)), 320 threads: eight CUDA-core warps (two per TMEM sub-partition,
// warps 4h .. 4h+3 working on half h of each query block: queries 64h ..
// 64h+63), an MMA warp and a load warp.  It walks the plan's transposed list
// (the live query blocks of its key block) and keeps dV and dK in tensor
// memory.  Per query block and half h, with keys as TMEM lanes:
//   S^T_h = K Q_h^T, dP^T_h = V dO_h^T                 (tcgen05, N = 64, operands in smem)
//   P^T = 2^(S^T scale log2 e - LSE log2 e), dS^T = P^T (dP^T - Dl)   (CUDA cores)
//   P^T and dS^T (bf16) go back to tensor memory over S^T_h and dP^T_h
//   (queries 64h + 2c, 64h + 2c + 1 in column 64h + c: each half writes
//   inside the values it read)
//   dV += P^T_h dO_h   (A = P^T from tensor memory, B = dO read MN-major, K = 64)
//   dK += dS^T_h Q_h   (A = dS^T from tensor memory, B = Q read MN-major, K = 64)
// The MMA warp interleaves the halves (gradients of half 0 of block j, S^T_0
// of block j + 1, gradients of half 1, S^T_1 of block j + 1), so that each
// half's CUDA-core phase overlaps the other half's products.  A thread that
// issues MMAs is held for about as long as they run, so the MMA warp does
// nothing but wait and issue; the load warp streams Q_h and dO_h (64-row TMA
// boxes, two buffers per half) as the gradient steps free their buffers.
//
// bsattn_bwd_dq_kernel (dQ): one CTA per query tile, walking the forward
// plan's list of live key blocks with queries as TMEM lanes: S = Q K^T and
// dP = dO V^T recomputed, dS = P (dP - Dl) back to tensor memory over dP,
// dQ += dS K in tensor memory (K_h and V_h streamed by the load warp), dQ
// written once at the end; the same 320 threads and interleaved halves as
// the dK/dV kernel, halves of the key block (keys 64h .. 64h+63) instead of
// the query block.
//
// Every mbarrier wait is bounded; on expiry the status word records a
// timeout and the CTA drains its copies and MMAs before it frees tensor memory.
#include <atomic>
#include <cstdint>
#include <type_traits>

#include "bwd.h"
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
  static constexpr int kHalfBoxBytes = kBoxBytes / 2;  // 64 rows of one box
  static constexpr int kHalfBytes = kTileBytes / 2;    // 64 rows of one tile
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;       // two buffers
  static constexpr int kdOOff = kQOff + 2 * kTileBytes;  // two buffers
  static constexpr int kVecBytes = 2 * 64 * 4;  // per CUDA-core warp: LSE and Dl of 64 queries
  static constexpr int kVecOff = kdOOff + 2 * kTileBytes;
  static constexpr int kBarOff = kVecOff + 8 * kVecBytes;
  static constexpr int kGrpOff = kBarOff + 256;  // per query head of the group: list start, prefix
  static constexpr int kSmem = kGrpOff + 4 * (2 * kMaxKvGroup + 1) + 124;
  // S^T = K Q^T and dP^T = V dO^T, per half of the query block: M = 128 keys,
  // N = 64 queries, both K-major
  static constexpr uint32_t kIdescT = idesc_bf16_f32(128, 64, false);
  // dV += P^T dO and dK += dS^T Q: M = 128 keys, A from tensor memory, N = D, B MN-major
  static constexpr uint32_t kIdescKV = idesc_bf16_f32(128, D, true);
  // tensor-memory columns
  static constexpr uint32_t kTS = 0;         // S^T (fp32)
  static constexpr uint32_t kTdP = 128;      // dP^T (fp32)
  static constexpr uint32_t kTdV = 256;      // dV accumulator (D columns)
  static constexpr uint32_t kTdK = 256 + D;  // dK accumulator (D columns)
  // P^T and dS^T (bf16 pairs, 32 columns per half): at D = 64 in columns of
  // their own, so that the next block's S^T_h may be computed while the
  // gradient step still reads them; at D = 128 (no columns left) over the
  // half's S^T and dP^T columns, so S^T_h of the next block waits for it.
  static constexpr bool kSep = D == 64;
  static constexpr uint32_t kTP = kSep ? 256 + 2 * D : kTS;          // half h: + (kSep ? 32 : 64) h
  static constexpr uint32_t kTdS = kSep ? 256 + 2 * D + 64 : kTdP;
  static constexpr uint32_t kHalfStride = kSep ? 32 : 64;
};
static_assert(BwdCfg<128>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");
static_assert(BwdCfg<128>::kTdK + 128 <= kBwdTmemCols, "tensor memory exceeded");

// Barriers of the dK/dV kernel, per half h of each query block (queries
// 64h .. 64h+63) where the halves have their own.
struct __align__(8) BwdBars {
  uint64_t kv_full;        // K and V of the key tile loaded
  // Q_h and dO_h of a query block loaded (by half, buffer); at D = 128 also
  // the previous block's gradient step of the half complete (its operands
  // sit where the next S^T_h goes): two arrivals, the copy's and the commit's
  uint64_t qd_full[2][2];
  uint64_t qd_empty[2][2]; // the gradients of the block in that buffer complete (by half)
  uint64_t st_done[2];     // S^T and dP^T of half h computed
  uint64_t pds_done[2];    // P^T and dS^T of half h written (tensor memory)
  uint64_t drain;          // every MMA issued so far complete
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block must fit its 256-byte region");
// Both kernels: 8 CUDA-core warps, an MMA warp and a load warp.
constexpr int kBwdKvThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;


// Dl_i = dO_i . O_i (fp32 over the stored O and dO).  Each lane takes 8
// consecutive elements of a row with 16-byte loads (D / 8 lanes per row,
// 32 / (D / 8) rows per warp); the lanes of a row add their partial sums.
template <int D, bool O_F32>
__global__ void bwd_prep_kernel(const void* __restrict__ o, const uint16_t* __restrict__ dout,
                                float* __restrict__ dl, long long rows) {
  constexpr int kLanes = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanes;
  // The backward kernel is launched as this kernel's programmatic dependent:
  // it may start now; its warps that read Dl wait for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long gwarp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long row = gwarp * kRowsPerWarp + lane / kLanes;
  float acc = 0.f;
  if (row < rows) {
    const size_t base = (size_t)row * D + (size_t)(lane % kLanes) * 8;
    const uint4 gv = *reinterpret_cast<const uint4*>(dout + base);
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    float x[8];
    if constexpr (O_F32) {
      const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(o) + base);
      const float4 b =
          *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(o) + base + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
      const uint4 ov = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(o) + base);
      const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(ow[e] << 16);
        x[2 * e + 1] = __uint_as_float(ow[e] & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(gw[e] << 16), x[2 * e], acc);
      acc = fmaf(__uint_as_float(gw[e] & 0xFFFF0000u), x[2 * e + 1], acc);
    }
  }
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && lane % kLanes == 0) dl[row] = acc;
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

// Accumulator rows out to global memory, coalesced: the warp's 32 TMEM lanes
// (rows row0 .. row0+31 of `out`, row stride D floats), columns c .. c+31,
// times `scale`.  Each thread holds one row after tcgen05.ld; the 32 x 32 fp32
// piece goes through this warp's 4 KB of shared memory (16-byte chunk q of
// row r at r * 128 + ((q ^ (r mod 8)) * 16), conflict-free both ways) and
// leaves as full 128-byte lines, four rows per warp-wide store.
template <int D>
__device__ __forceinline__ void store_rows32(uint32_t taddr, float scale, float* out, int row0,
                                             int c, uint32_t scratch, int lane) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_wait_ld();
  reg_fence(v, 32);
  const uint32_t mine = scratch + (uint32_t)lane * 128u;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    st_shared_v4(mine + (((uint32_t)q ^ (uint32_t)(lane & 7)) << 4),
                 __float_as_uint(__uint_as_float(v[4 * q]) * scale),
                 __float_as_uint(__uint_as_float(v[4 * q + 1]) * scale),
                 __float_as_uint(__uint_as_float(v[4 * q + 2]) * scale),
                 __float_as_uint(__uint_as_float(v[4 * q + 3]) * scale));
  __syncwarp();
  const int q = lane & 7;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int r = it * 4 + (lane >> 3);
    uint32_t w[4];
    ld_shared_v4(scratch + (uint32_t)r * 128u + (((uint32_t)q ^ (uint32_t)(r & 7)) << 4), w);
    st_global_v4(out + (size_t)(row0 + r) * D + c + 4 * q, w[0], w[1], w[2], w[3]);
  }
  __syncwarp();  // the piece is read before the next one is written
}

// One CTA of dK, dV: key tile number `cta` of the launch order.
template <int D>
__device__ __forceinline__ void bwd_kv_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                           const CUtensorMap& tm_v, const CUtensorMap& tm_do,
                                           const BwdParams& p, int cta) {
  using C = BwdCfg<D>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // warps 0-7: CUDA-core work, half h = warps 4h .. 4h+3; kMmaWarp, kLoadWarp
  // (b * Hkv + hk) * nb + kb: a key tile of K/V head hk; long tiles first
  const int tile = p.kv_group == 1 ? p.kv_order[cta] : cta;
  const int kvbh = tile / p.nb;
  const int kb = tile - kvbh * p.nb;
  const int g = p.kv_group;     // query heads reading this K/V head
  const int hkv = p.H / g;      // K/V heads per batch entry
  const int bh0 = (kvbh / hkv) * p.H + (kvbh % hkv) * g;  // its first query head b*H + hk*g
  const int krow0 = kvbh * p.S + kb * kBlock;             // first key row of the tile

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  BwdBars* bars = reinterpret_cast<BwdBars*>(sbase + C::kBarOff);
  const uint64_t lim = p.timeout_ns;
  volatile int* abort_flag = &bars->abort_flag;
  // Barriers first, then the tile's K and V: they need nothing but the tile,
  // so their load overlaps the list and tensor-memory set-up below.
  if (tid == 0) {
    mbar_init(smem_u32(&bars->kv_full), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&bars->qd_full[h][0]), C::kSep ? 1 : 2);
      mbar_init(smem_u32(&bars->qd_full[h][1]), C::kSep ? 1 : 2);
      mbar_init(smem_u32(&bars->qd_empty[h][0]), 1);
      mbar_init(smem_u32(&bars->qd_empty[h][1]), 1);
      mbar_init(smem_u32(&bars->st_done[h]), 1);
      mbar_init(smem_u32(&bars->pds_done[h]), 4);  // the half's four warps
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    const uint32_t bar = smem_u32(&bars->kv_full);
    mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c) {
        const uint32_t off = (uint32_t)(hh * C::kHalfBoxBytes + c * C::kBoxBytes);
        tma_load_2d(base + C::kKOff + off, &tm_k, bar, c * 64, krow0 + 64 * hh);
        tma_load_2d(base + C::kVOff + off, &tm_v, bar, c * 64, krow0 + 64 * hh);
      }
  }
  // The CTA walks the transposed lists of the group's query heads one after
  // the other: head bh0 + i contributes entries [g_st[i], g_st[i+1]) of the
  // walk, starting at row_idx[g_c0[i]].
  int* g_c0 = reinterpret_cast<int*>(sbase + C::kGrpOff);
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
    if (tid == 0) bwd_drain_wait(smem_u32(&bars->kv_full), 0, lim);  // the K/V copy lands first
    return;
  }
  // The plan's lists must hold valid query blocks; anything else is an
  // internal error.  The list lengths are checked here; each entry is
  // checked where the load warp reads it (and never used out of range).
  bool bad = n > p.nb * g;
  for (int gi = 0; !bad && gi < g; ++gi) bad = g_st[gi + 1] - g_st[gi] > p.nb;
  if (__syncthreads_or(bad)) {
    if (tid == 0) {
      atomicOr(p.status, kStatusInternal);
      bwd_drain_wait(smem_u32(&bars->kv_full), 0, lim);
    }
    return;
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
    // ---- MMAs (one elected lane), in one fixed order per block j:
    //   dV, dK += half 0 of block j;  S^T_0, dP^T_0 of block j + 1;
    //   dV, dK += half 1 of block j;  S^T_1, dP^T_1 of block j + 1.
    // At D = 128, S^T_h of block j + 1 overwrites the tensor-memory operands
    // of the gradient step before it, so it waits (on its readiness barrier)
    // until that step is complete.  The order also fixes the order in which
    // dV and dK accumulate (the gradients repeat bit for bit).  The issuing lane is held for about as long as its
    // MMAs run, so it does nothing else: the loads are the load warp's.
    const uint64_t kd = smem_desc_sw128(base + C::kKOff, 16, 1024);
    const uint64_t vd = smem_desc_sw128(base + C::kVOff, 16, 1024);
    auto issue_st = [&](int h, int j) {  // S^T_h = K Q_h^T, dP^T_h = V dO_h^T of block j
      tc_fence_after();
      if (elect_one()) {
        const uint32_t off = (uint32_t)((j & 1) * C::kTileBytes + h * C::kHalfBoxBytes);
        const uint64_t qd = smem_desc_sw128(base + C::kQOff + off, 16, 1024);
        const uint64_t dd = smem_desc_sw128(base + C::kdOOff + off, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kTS + 64u * h, kd + o, qd + o, C::kIdescT, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kTdP + 64u * h, vd + o, dd + o, C::kIdescT, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->st_done[h]));
      }
      __syncwarp();
    };
    auto issue_grad = [&](int h, int j) {  // dV += P^T_h dO_h, dK += dS^T_h Q_h of block j
      tc_fence_after();
      if (elect_one()) {
        const uint32_t qoff = base + C::kQOff + (j & 1) * C::kTileBytes;
        const uint32_t dooff = base + C::kdOOff + (j & 1) * C::kTileBytes;
        const uint64_t do_mn = smem_desc_sw128(dooff, C::kBoxBytes, 1024);
        const uint64_t q_mn = smem_desc_sw128(qoff, C::kBoxBytes, 1024);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * h + k4;                       // queries 16kk .. 16kk+15
          const uint32_t mn = (uint32_t)(kk * 2048) >> 4;  // 16 rows of 128 bytes
          const uint32_t acc = (j > 0 || h > 0 || k4 > 0) ? 1u : 0u;
          const uint32_t pcol = C::kHalfStride * h + 8u * k4;  // P^T, dS^T of queries 16kk ..
          mma_ts(tmem + C::kTdV, tmem + C::kTP + pcol, do_mn + mn, C::kIdescKV, acc);
          mma_ts(tmem + C::kTdK, tmem + C::kTdS + pcol, q_mn + mn, C::kIdescKV, acc);
        }
        mma_commit(smem_u32(&bars->qd_empty[h][j & 1]));
        // at D = 128 the next S^T_h overwrites this step's operands: its
        // readiness barrier waits for this step too
        if (!C::kSep && j + 1 < n) mma_commit(smem_u32(&bars->qd_full[h][(j + 1) & 1]));
      }
      __syncwarp();
    };
    ok = bwd_wait(smem_u32(&bars->kv_full), 0, abort_flag, p.status, lim);
    for (int h = 0; ok && h < 2; ++h) {
      ok = bwd_wait(smem_u32(&bars->qd_full[h][0]), 0, abort_flag, p.status, lim);
      if (ok) issue_st(h, 0);
    }
    for (int j = 0; ok && j < n; ++j) {
      for (int h = 0; ok && h < 2; ++h) {
        // At D = 64 the next S^T_h depends on its Q_h, dO_h only: both
        // barriers are tested first and the two steps issued back to back.
        if (C::kSep && j + 1 < n)
          ok = bwd_wait(smem_u32(&bars->qd_full[h][(j + 1) & 1]), (uint32_t)((j + 1) >> 1) & 1u,
                        abort_flag, p.status, lim);
        ok = ok && bwd_wait(smem_u32(&bars->pds_done[h]), (uint32_t)j & 1u, abort_flag, p.status,
                            lim);
        if (!ok) break;
        issue_grad(h, j);
        if (j + 1 < n) {
          if (!C::kSep)
            ok = bwd_wait(smem_u32(&bars->qd_full[h][(j + 1) & 1]),
                          (uint32_t)((j + 1) >> 1) & 1u, abort_flag, p.status, lim);
          if (ok) issue_st(h, j + 1);
        }
      }
    }
    // Every MMA issued completes before tensor memory is freed.
    if (elect_one()) mma_commit(smem_u32(&bars->drain));
    __syncwarp();
    bwd_drain_wait(smem_u32(&bars->drain), 0, lim);
  } else if (warp == kLoadWarp) {
    // ---- loads (one elected lane): K and V once; then, in the order of the
    // walk, Q_h and dO_h of entry i into buffer i % 2 of half h once the
    // gradients of entry i - 2's half h are complete.
    auto load_half = [&](const CUtensorMap* tm, uint32_t dst, uint32_t bar, int row) {
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c)
        tma_load_2d(dst + c * C::kBoxBytes, tm, bar, c * 64, row);
    };
    // First Q/dO row of each entry, 32 entries per window held one per lane;
    // the next window is loaded a window ahead.
    auto window_rows = [&](int w0) {
      int row = 0;
      if (w0 + lane < n) {
        int bhq = 0, qbi = 0;
        entry(w0 + lane, bhq, qbi);
        if (qbi < 0 || qbi >= p.nb || (p.causal && qbi < kb)) {  // not a valid list entry
          atomicOr(p.status, kStatusInternal);
          *abort_flag = 1;
          qbi = 0;
        }
        row = bhq * p.S + qbi * kBlock;
      }
      return row;
    };
    int win0 = 0;
    int row_cur = window_rows(0), row_next = window_rows(32);
    // (K and V were loaded by thread 0 at the start)
    int loaded[2] = {0, 0};  // entries 0 .. loaded[h] - 1 loaded for half h
    for (int i = 0; ok && i < n; ++i) {
      while (i >= win0 + 32) {
        win0 += 32;
        row_cur = row_next;
        row_next = window_rows(win0 + 32);
      }
      const int row0 = __shfl_sync(0xffffffffu, row_cur, i - win0);
      const int b = i & 1;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (i >= 2) {
          ok = bwd_wait(smem_u32(&bars->qd_empty[h][b]), (uint32_t)((i >> 1) - 1) & 1u,
                        abort_flag, p.status, lim);
          if (!ok) break;
        }
        if (elect_one()) {
          const uint32_t bar = smem_u32(&bars->qd_full[h][b]);
          const uint32_t off = (uint32_t)(b * C::kTileBytes + h * C::kHalfBoxBytes);
          mbar_arrive_expect_tx(bar, 2 * C::kHalfBytes);
          if (!C::kSep && i == 0) mbar_arrive(bar);  // no gradient step before the first block
          load_half(&tm_q, base + C::kQOff + off, bar, row0 + 64 * h);
          load_half(&tm_do, base + C::kdOOff + off, bar, row0 + 64 * h);
        }
        __syncwarp();
        loaded[h] = i + 1;
      }
    }
    // Every copy issued lands before the CTA exits.
    bwd_drain_wait(smem_u32(&bars->kv_full), 0, lim);
    for (int h = 0; h < 2; ++h)  // the last one or two entries loaded
      for (int i = loaded[h] > 2 ? loaded[h] - 2 : 0; i < loaded[h]; ++i)
        bwd_drain_wait(smem_u32(&bars->qd_full[h][i & 1]), (uint32_t)(i >> 1) & 1u, lim);
  } else if (warp < kMmaWarp) {
    // ---- P^T and dS^T of half h (queries 64h .. 64h+63), one key row (TMEM
    // lane) per thread, 32 queries at a time; both go back to tensor memory
    // as bf16 pairs over the fp32 values just read: queries 64h + 2c and
    // 64h + 2c + 1 in column 64h + c of the S^T (P^T) and dP^T (dS^T) columns.
    // LSE (log2 units) and Dl of the half's 64 queries sit in a shared vector
    // of this warp (written by the warp for itself, read as broadcasts).
    const int h = warp >> 2;
    const int r = tid & (kBlock - 1);  // TMEM lane: key row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes
    const float sl = p.scale_log2;
    const uint64_t sl2 = f2_pack(sl, sl);
    const uint32_t tS = tmem + C::kTS + lane_off;
    const uint32_t tdP = tmem + C::kTdP + lane_off;
    float* vl = reinterpret_cast<float*>(sbase + C::kVecOff + warp * C::kVecBytes);  // [64] -LSE log2 e
    float* vd = vl + 64;                                                             // [64] -Dl
    // LSE and Dl of the half's queries 64h + lane and 64h + 32 + lane of
    // entry i, loaded one entry ahead
    float la_next = 0.f, lb_next = 0.f, da_next = 0.f, db_next = 0.f;
    int qb_next = 0;
    auto fetch = [&](int i) {
      int bhq = 0;
      entry(i, bhq, qb_next);
      if (qb_next < 0 || qb_next >= p.nb) qb_next = 0;  // reported by the load warp
      const int qrow = bhq * p.S + qb_next * kBlock + 64 * h + lane;
      la_next = -p.lse[qrow] * kLog2e;  // held negated: the loop adds them
      lb_next = -p.lse[qrow + 32] * kLog2e;
      da_next = -p.dl[qrow];
      db_next = -p.dl[qrow + 32];
    };
    // Dl is the row-term kernel's output: that grid must be complete (this
    // kernel may have been launched before it finished).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    fetch(0);
    for (int j = 0; j < n; ++j) {
      const int qb = qb_next;
      vl[lane] = la_next;
      vl[lane + 32] = lb_next;
      vd[lane] = da_next;
      vd[lane + 32] = db_next;
      __syncwarp();
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
        // -LSE log2 e and -Dl of the chunk's queries
        const float4* l4 = reinterpret_cast<const float4*>(vl + 32 * (ch & 1));
        const float4* d4 = reinterpret_cast<const float4*>(vd + 32 * (ch & 1));
        uint32_t pk[16], dk[16];
        // the causal diagonal block in its own copy of the loop, so that the
        // loop of every other block has no test in it; pairs of queries with
        // packed f32x2 arithmetic
        auto chunk = [&](auto diag_c) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 l = l4[i >> 2];  // same address in every lane: a broadcast
            const float4 d = d4[i >> 2];
            const uint64_t nl[2] = {f2_pack(l.x, l.y), f2_pack(l.z, l.w)};
            const uint64_t nd[2] = {f2_pack(d.x, d.y), f2_pack(d.z, d.w)};
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const uint64_t x2 = f2_fma(
                  f2_pack(__uint_as_float(sv[i + e]), __uint_as_float(sv[i + e + 1])), sl2,
                  nl[e >> 1]);
              float x0, x1;
              f2_unpack(x2, x0, x1);
              float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              if constexpr (decltype(diag_c)::value) {
                p0 = r > ch * 32 + i + e ? 0.f : p0;
                p1 = r > ch * 32 + i + e + 1 ? 0.f : p1;
              }
              const uint64_t dd2 = f2_add(
                  f2_pack(__uint_as_float(dp[i + e]), __uint_as_float(dp[i + e + 1])), nd[e >> 1]);
              float d0, d1;
              f2_unpack(f2_mul(f2_pack(p0, p1), dd2), d0, d1);
              pk[(i + e) >> 1] = pack_bf16x2(p0, p1);
              dk[(i + e) >> 1] = pack_bf16x2(d0, d1);
            }
          }
        };
        if (diag)
          chunk(std::true_type{});
        else
          chunk(std::false_type{});
        const uint32_t col = C::kHalfStride * h + 16u * (ch & 1);
        tmem_st32_16(tmem + C::kTP + lane_off + col, pk);
        tmem_st32_16(tmem + C::kTdS + lane_off + col, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // the warp's P^T and dS^T are written (and its vectors read)
      if (lane == 0) mbar_arrive(smem_u32(&bars->pds_done[h]));
    }
  }
  // Every role has left its loop; the MMA thread drained all copies and MMAs.
  const bool all_ok = __syncthreads_and(ok);
  tc_fence_after();
  if (all_ok && warp < kMmaWarp) {  // dV and dK (times scale): the warp's 32 key rows, half the columns
    const int half = warp >> 2;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int row0 = krow0 + (warp & 3) * 32;
    // every copy and MMA is complete: the Q buffers serve as scratch, 4 KB per warp
    const uint32_t scratch = base + C::kQOff + (uint32_t)warp * 4096u;
#pragma unroll 1
    for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32) {
      store_rows32<D>(tmem + C::kTdV + lane_off + c, 1.0f, p.dv, row0, c, scratch, lane);
      store_rows32<D>(tmem + C::kTdK + lane_off + c, p.scale, p.dk, row0, c, scratch, lane);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// dQ kernel layout: Q, dO once per tile; K and V double-buffered by halves.
template <int D>
struct DqCfg {
  static constexpr int kTileBytes = kBlock * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kBlock * 128;
  static constexpr int kHalfBoxBytes = kBoxBytes / 2;    // 64 rows of one box
  static constexpr int kHalfBytes = kTileBytes / 2;      // 64 rows of one tile
  static constexpr int kQOff = 0;
  static constexpr int kdOOff = kTileBytes;
  static constexpr int kKOff = 2 * kTileBytes;   // two buffers
  static constexpr int kVOff = 4 * kTileBytes;   // two buffers
  static constexpr int kBarOff = 6 * kTileBytes;
  static constexpr int kSmem = kBarOff + 256;
  // S = Q K^T and dP = dO V^T, per half of the key block: M = 128 queries,
  // N = 64 keys, both K-major
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false);
  // dQ += dS K: M = 128 queries, A = dS from tensor memory, N = D, B (K) read MN-major
  static constexpr uint32_t kIdescQ = idesc_bf16_f32(128, D, true);
  static constexpr uint32_t kTS = 0;     // S (fp32)
  static constexpr uint32_t kTdP = 128;  // dP (fp32)
  static constexpr uint32_t kTdQ = 256;  // dQ accumulator (D columns)
  // dS (bf16 pairs) in columns of its own, 32 per half: the next key block's
  // S_h may be computed while the dQ step still reads them
  static constexpr uint32_t kTdS = 384;
};
static_assert(DqCfg<128>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");

// The dQ kernel works on each key block in two halves h (keys 64h .. 64h+63),
// interleaved as the dK/dV kernel's halves are.
struct __align__(8) DqBars {
  uint64_t qd_full;        // Q and dO of the tile loaded
  uint64_t kv_full[2][2];  // K_h and V_h of a key block loaded (by half, buffer)
  uint64_t kv_empty[2][2]; // dQ has taken the key block in that buffer (by half)
  uint64_t st_done[2];     // S and dP of half h computed
  uint64_t ds_done[2];     // dS of half h written
  uint64_t drain;          // every MMA issued so far complete
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(DqBars) <= 256, "barrier block must fit its 256-byte region");

// One CTA of dQ: query tile number `cta` of the launch order.
template <int D>
__device__ __forceinline__ void bwd_dq_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                           const CUtensorMap& tm_v, const CUtensorMap& tm_do,
                                           const BwdParams& p, int cta) {
  using C = DqCfg<D>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // warps 0-7: CUDA-core work, half h = warps 4h .. 4h+3; kMmaWarp, kLoadWarp
  // (b * H + h) * nb + qb: the forward plan's tiles, long ones first, then the empty ones
  const int tile = cta < p.n_live ? p.tile_order[cta] : p.empty_tiles[cta - p.n_live];
  const int bh = tile / p.nb;
  const int qb = tile - bh * p.nb;
  const int qrow0 = bh * p.S + qb * kBlock;  // first query row of the tile
  const int kvbh =  // the K/V head it attends with
      p.kv_group > 1 ? (bh / p.H) * (p.H / p.kv_group) + (bh % p.H) / p.kv_group : bh;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  DqBars* bars = reinterpret_cast<DqBars*>(smem_raw + (base - raw) + C::kBarOff);
  const uint64_t lim = p.timeout_ns;
  volatile int* abort_flag = &bars->abort_flag;
  const bool live = cta < p.n_live;  // the empty tiles come last
  // Barriers first, then (for a live tile) its Q and dO: they need nothing
  // but the tile, so their load overlaps the set-up below.
  if (tid == 0) {
    mbar_init(smem_u32(&bars->qd_full), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&bars->kv_full[h][0]), 1);
      mbar_init(smem_u32(&bars->kv_full[h][1]), 1);
      mbar_init(smem_u32(&bars->kv_empty[h][0]), 1);
      mbar_init(smem_u32(&bars->kv_empty[h][1]), 1);
      mbar_init(smem_u32(&bars->st_done[h]), 1);
      mbar_init(smem_u32(&bars->ds_done[h]), 4);  // the half's four warps
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    if (live) {
      const uint32_t bar = smem_u32(&bars->qd_full);
      mbar_arrive_expect_tx(bar, 2 * C::kTileBytes);
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int c = 0; c < C::kBoxes; ++c) {
          const uint32_t off = (uint32_t)(hh * C::kHalfBoxBytes + c * C::kBoxBytes);
          tma_load_2d(base + C::kQOff + off, &tm_q, bar, c * 64, qrow0 + 64 * hh);
          tma_load_2d(base + C::kdOOff + off, &tm_do, bar, c * 64, qrow0 + 64 * hh);
        }
    }
  }
  const int r0 = p.row_ptr[tile];
  const int n = p.row_ptr[tile + 1] - r0;
  if (n <= 0) {  // no live key block: dQ = 0
    float4* dq4 = reinterpret_cast<float4*>(p.dq + (size_t)qrow0 * D);
    for (int i = tid; i < kBlock * D / 4; i += kBwdKvThreads)
      dq4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0 && live) bwd_drain_wait(smem_u32(&bars->qd_full), 0, lim);
    return;
  }
  // The list length is checked here; each entry where the load warp reads it.
  const bool bad = n > p.nb;
  if (__syncthreads_or(bad || !live)) {  // a tile with blocks sits among the live ones
    if (tid == 0) {
      atomicOr(p.status, kStatusInternal);
      if (live) bwd_drain_wait(smem_u32(&bars->qd_full), 0, lim);
    }
    return;
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
    // ---- MMAs (one elected lane), in one fixed order per key block j:
    //   dQ += half 0 of block j;  S_0, dP_0 of block j + 1;
    //   dQ += half 1 of block j;  S_1, dP_1 of block j + 1,
    // as in the dK/dV kernel (dQ accumulates in a fixed order; the loads are
    // the load warp's).  dS has columns of its own, so S_h of the next block
    // waits for its K_h, V_h only; the commit of that S also covers the dQ
    // step before it, which the half's warps wait on before they write dS.
    const uint64_t qd = smem_desc_sw128(base + C::kQOff, 16, 1024);
    const uint64_t dd = smem_desc_sw128(base + C::kdOOff, 16, 1024);
    auto issue_st = [&](int h, int j) {  // S_h = Q K_h^T, dP_h = dO V_h^T of key block j
      tc_fence_after();
      if (elect_one()) {
        const uint32_t off = (uint32_t)((j & 1) * C::kTileBytes + h * C::kHalfBoxBytes);
        const uint64_t kd = smem_desc_sw128(base + C::kKOff + off, 16, 1024);
        const uint64_t vd = smem_desc_sw128(base + C::kVOff + off, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kTS + 64u * h, qd + o, kd + o, C::kIdescS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t o = (uint32_t)((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::kTdP + 64u * h, dd + o, vd + o, C::kIdescS, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->st_done[h]));
      }
      __syncwarp();
    };
    auto issue_grad = [&](int h, int j) {  // dQ += dS_h K_h of key block j
      tc_fence_after();
      if (elect_one()) {
        const uint64_t k_mn =
            smem_desc_sw128(base + C::kKOff + (j & 1) * C::kTileBytes, C::kBoxBytes, 1024);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * h + k4;  // keys 16kk .. 16kk+15
          const uint32_t mn = (uint32_t)(kk * 2048) >> 4;
          mma_ts(tmem + C::kTdQ, tmem + C::kTdS + 32u * h + 8u * k4, k_mn + mn, C::kIdescQ,
                 (j > 0 || h > 0 || k4 > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->kv_empty[h][j & 1]));
      }
      __syncwarp();
    };
    ok = bwd_wait(smem_u32(&bars->qd_full), 0, abort_flag, p.status, lim);
    for (int h = 0; ok && h < 2; ++h) {
      ok = bwd_wait(smem_u32(&bars->kv_full[h][0]), 0, abort_flag, p.status, lim);
      if (ok) issue_st(h, 0);
    }
    for (int j = 0; ok && j < n; ++j) {
      for (int h = 0; ok && h < 2; ++h) {
        // both barriers first, then the two steps back to back
        if (j + 1 < n)
          ok = bwd_wait(smem_u32(&bars->kv_full[h][(j + 1) & 1]), (uint32_t)((j + 1) >> 1) & 1u,
                        abort_flag, p.status, lim);
        ok = ok && bwd_wait(smem_u32(&bars->ds_done[h]), (uint32_t)j & 1u, abort_flag, p.status,
                            lim);
        if (!ok) break;
        issue_grad(h, j);
        if (j + 1 < n) issue_st(h, j + 1);
      }
    }
    if (elect_one()) mma_commit(smem_u32(&bars->drain));
    __syncwarp();
    bwd_drain_wait(smem_u32(&bars->drain), 0, lim);
  } else if (warp == kLoadWarp) {
    // ---- loads (one elected lane): Q and dO once; then K_h and V_h of key
    // block i into buffer i % 2 of half h once dQ has taken block i - 2's half h.
    auto load_half = [&](const CUtensorMap* tm, uint32_t dst, uint32_t bar, int row) {
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c)
        tma_load_2d(dst + c * C::kBoxBytes, tm, bar, c * 64, row);
    };
    // First K/V row of each key block of the list, 32 per window held one per
    // lane; the next window is loaded a window ahead.
    auto window_rows = [&](int w0) {
      if (w0 + lane >= n) return 0;
      int kbi = p.col_idx[r0 + w0 + lane];
      if (kbi < 0 || kbi >= p.nb || (p.causal && kbi > qb)) {  // not a valid list entry
        atomicOr(p.status, kStatusInternal);
        *abort_flag = 1;
        kbi = 0;
      }
      return kvbh * p.S + kbi * kBlock;
    };
    int win0 = 0;
    int row_cur = window_rows(0), row_next = window_rows(32);
    // (Q and dO were loaded by thread 0 at the start)
    int loaded[2] = {0, 0};  // key blocks 0 .. loaded[h] - 1 loaded for half h
    for (int i = 0; ok && i < n; ++i) {
      while (i >= win0 + 32) {
        win0 += 32;
        row_cur = row_next;
        row_next = window_rows(win0 + 32);
      }
      const int row0 = __shfl_sync(0xffffffffu, row_cur, i - win0);
      const int b = i & 1;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (i >= 2) {
          ok = bwd_wait(smem_u32(&bars->kv_empty[h][b]), (uint32_t)((i >> 1) - 1) & 1u,
                        abort_flag, p.status, lim);
          if (!ok) break;
        }
        if (elect_one()) {
          const uint32_t bar = smem_u32(&bars->kv_full[h][b]);
          const uint32_t off = (uint32_t)(b * C::kTileBytes + h * C::kHalfBoxBytes);
          mbar_arrive_expect_tx(bar, 2 * C::kHalfBytes);
          load_half(&tm_k, base + C::kKOff + off, bar, row0 + 64 * h);
          load_half(&tm_v, base + C::kVOff + off, bar, row0 + 64 * h);
        }
        __syncwarp();
        loaded[h] = i + 1;
      }
    }
    // Every copy issued lands before the CTA exits.
    bwd_drain_wait(smem_u32(&bars->qd_full), 0, lim);
    for (int h = 0; h < 2; ++h)  // the last one or two key blocks loaded
      for (int i = loaded[h] > 2 ? loaded[h] - 2 : 0; i < loaded[h]; ++i)
        bwd_drain_wait(smem_u32(&bars->kv_full[h][i & 1]), (uint32_t)(i >> 1) & 1u, lim);
  } else if (warp < kMmaWarp) {
    // ---- dS = P (dP - Dl) of half h (keys 64h .. 64h+63), one query row and
    // 32 keys at a time, back to tensor memory as bf16 pairs over the dP just
    // read: keys 64h + 2c and 64h + 2c + 1 in column 64h + c of the dP columns.
    const int h = warp >> 2;
    const int r = tid & (kBlock - 1);  // TMEM lane: query row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float l2 = p.lse[qrow0 + r] * kLog2e;  // this row's LSE in log2 units
    const uint64_t nl2 = f2_pack(-l2, -l2);
    // Dl is the row-term kernel's output: that grid must be complete (this
    // kernel may have been launched before it finished).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float dlr = p.dl[qrow0 + r];
    const uint64_t nd2 = f2_pack(-dlr, -dlr);
    const float sl = p.scale_log2;
    const uint64_t sl2 = f2_pack(sl, sl);
    const uint32_t tS = tmem + C::kTS + lane_off;
    const uint32_t tdP = tmem + C::kTdP + lane_off;
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
        // the causal diagonal block in its own copy of the loop
        auto chunk = [&](auto diag_c) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {  // pairs of keys with packed f32x2 arithmetic
            const uint64_t x2 =
                f2_fma(f2_pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), sl2, nl2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if constexpr (decltype(diag_c)::value) {
              const int c = ch * 32 + i;
              p0 = c > r ? 0.f : p0;
              p1 = c + 1 > r ? 0.f : p1;
            }
            const uint64_t dd2 =
                f2_add(f2_pack(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])), nd2);
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(p0, p1), dd2), d0, d1);
            dk[i >> 1] = pack_bf16x2(d0, d1);
          }
        };
        if (diag)
          chunk(std::true_type{});
        else
          chunk(std::false_type{});
        tmem_st32_16(tmem + C::kTdS + lane_off + (uint32_t)(32 * h + 16 * (ch & 1)), dk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // the warp's dS is written (and its S, dP reads are complete)
      if (lane == 0) mbar_arrive(smem_u32(&bars->ds_done[h]));
    }
  }
  const bool all_ok = __syncthreads_and(ok);
  tc_fence_after();
  if (all_ok && warp < kMmaWarp) {  // dQ times scale: the warp's 32 query rows, half the columns
    const int half = warp >> 2;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int row0 = qrow0 + (warp & 3) * 32;
    // every copy and MMA is complete: the K buffers serve as scratch, 4 KB per warp
    const uint32_t scratch = base + C::kKOff + (uint32_t)warp * 4096u;
#pragma unroll 1
    for (int c = half * (D / 2); c < (half + 1) * (D / 2); c += 32)
      store_rows32<D>(tmem + C::kTdQ + lane_off + c, p.scale, p.dq, row0, c, scratch, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// The backward pass in one launch: CTAs 0 .. n_kv-1 compute dK, dV (key
// tiles, longest first), the rest dQ (query tiles, longest first), so that
// the hardware's CTA scheduler fills the end of the one with the other.
template <int D>
__global__ void __launch_bounds__(kBwdKvThreads, 1)
    bsattn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do, const BwdParams p, int n_kv) {
  if ((int)blockIdx.x < n_kv)
    bwd_kv_cta<D>(tm_q, tm_k, tm_v, tm_do, p, (int)blockIdx.x);
  else
    bwd_dq_cta<D>(tm_q, tm_k, tm_v, tm_do, p, (int)blockIdx.x - n_kv);
}

template <int D>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, int n_kv, int n_q,
                         cudaStream_t stream) {
  static std::atomic<bool> opted_in[64];
  const size_t smem = (BwdCfg<D>::kSmem > DqCfg<D>::kSmem ? BwdCfg<D>::kSmem : DqCfg<D>::kSmem) + 1024;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bsattn_bwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  // A programmatic dependent of the row-term kernel launched just before it
  // on the stream: the CTAs start while that kernel finishes; the warps that
  // read its output (Dl) wait for it with griddepcontrol.wait.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_kv + n_q));
  cfg.blockDim = dim3(kBwdKvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bsattn_bwd_kernel<D>, tq, tk, tv, tdo, p, n_kv);
}

}  // namespace

cudaError_t launch_bwd_prep(int D, bool o_f32, const void* o, const void* dout, float* dl,
                            long long rows, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long long per_block = 8 * (32 / (D / 8));  // 8 warps, 32 / (D / 8) rows each
  const long long blocks = (rows + per_block - 1) / per_block;
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
                       const CUtensorMap& tdo, const BwdParams& p, int n_kv, int n_q,
                       cudaStream_t stream) {
  if (n_kv + n_q <= 0) return cudaSuccess;
  return D == 128 ? launch_bwd_t<128>(tq, tk, tv, tdo, p, n_kv, n_q, stream)
                  : launch_bwd_t<64>(tq, tk, tv, tdo, p, n_kv, n_q, stream);
}

}  // namespace bsattn
