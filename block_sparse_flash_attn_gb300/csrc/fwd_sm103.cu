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
// GB300 design (one persistent CTA per SM, 512 threads = 4 warpgroups, one
// query tile in the softmax at a time):
//   warps 0-7  softmax (and the LSE).  Each warp covers 16 query rows (TMEM
//              lanes); lanes 0..15 own key columns 0..63 of every block (O
//              columns [0, D/2)), lanes 16..31 the same rows' columns 64..127
//              (O columns [D/2, D)); tcgen05 16x32bx2 accesses put both halves
//              of a row in one warp, so row max and sums combine by shuffle.
//   warp  8    TMA producer of K and V (elected lane)
//   warp  9    tcgen05 issuer of S = Q K^T (elected lane), tensor-memory owner
//   warp  10   tile scheduler: claims the next tile when the producer asks
//              for it (a few blocks before the current tile's end),
//              publishes it (CSR range and first key blocks) in a 2-slot
//              queue and loads its Q (elected lane)
//   warp  11   tcgen05 issuer of O += P V (elected lane)
//   warps 12-15 epilogue: one thread per query row reads O from tensor
//              memory, divides it by the row's rounded sum and stores it,
//              while the softmax warps already work on the next tile
// Tensor memory (512 columns allocated): three score buffers S[0] = [0,128),
// S[1] = [128,256), S[2] = [256,384) and the fp32 output accumulator
// O = [384, 384+D) (at D = 64 followed by 16 columns of the rounded row sum,
// see Cfg::kOnes).  Block g (counted over the CTA's whole run) uses
// S[g % 3]; its bf16 probabilities P overwrite the scores already read
// (keys 0..63 -> columns 0..31, keys 64..127 -> columns 64..95).  S(g+3) goes
// into block g's buffer once O += P(g) V(g) is complete, so the scores of
// the next blocks are computed while the softmax works on block g: the chain
// softmax -> PV -> next S spans three blocks and hides behind the tensor
// core's own work.  Shared memory: Q buffers and 3-stage rings of K and V
// tiles (128 x D bf16 each, 128-byte swizzled by TMA, read by tcgen05.mma
// through matrix descriptors): at D = 128 one Q (224 KB), at D = 64 two.
//
// The producer sees the CTA's tiles as one stream of key blocks and loads K
// two blocks ahead of V along it; the scheduler warp loads each tile's Q as
// soon as the Q buffer is free.  Along the same stream one MMA warp issues
// S(g) as soon as K(g) is loaded and PV(g-3) is complete, another issues
// PV(g) as soon as P(g) is written and V(g) loaded; a tile's first PV starts
// a fresh O.  The commit after S(g) frees K(g)'s ring stage and is the
// softmax's "S(g) ready" signal; the commit after PV(g) frees V(g)'s stage
// and is "PV(g) done", which the softmax waits for only before an O rescale
// and the epilogue warps for a tile's last block.  The next tile's first PV,
// the one that overwrites O, waits until the epilogue warps have read O.
// Online softmax in base 2 with lazy rescale: the running max m only moves
// when a block's max exceeds it by more than 8 (log2 units), so P <= 256 and
// the O rescale is rare.  O is normalised by the row sum of the bf16-rounded
// P that multiplied V (so the weights on V sum to one even when a single key
// dominates a row); the LSE uses the fp32 sum of the unrounded P.
//
// Every wait is bounded (globaltimer); on expiry the kernel records a timeout
// in the status word, every role leaves its loop, outstanding TMA loads and
// MMAs are drained (again with a limit) and TMEM is freed before exit.
#include <atomic>
#include <cstdint>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace bsattn {
namespace {

constexpr int kThreads = 512;
constexpr int kSoftmaxThreads = 256;
constexpr int kSoftmaxWarps = kSoftmaxThreads / 32;
constexpr int kWarpLoad = 8;
constexpr int kWarpMmaS = 9;  // also allocates and frees tensor memory
constexpr int kWarpSched = 10;
constexpr int kWarpMmaPV = 11;
constexpr int kWarpEpi0 = 12;  // warps 12-15: epilogue (TMEM sub-partitions 0-3)
constexpr int kEpiWarps = 4;
constexpr uint32_t kEpiBarrier = 1;  // named barrier of the epilogue warps
// Waits off the critical path (the scheduler's wait for a request, the
// epilogue leader's waits) test the barrier about this often (ns) and sleep
// in between: a spinning warp takes issue slots from the softmax warps.
constexpr uint32_t kSleepNs = 200;
// The producer asks for the next tile when its K cursor has this many blocks
// of the current tile left: claiming a tile (four dependent global reads)
// and loading its Q take about as long as this many blocks' MMAs.
constexpr int kClaimAhead = 4;
// Launch budget 512 x 128 registers; the two role warpgroups hand part of
// their share to the two softmax warpgroups: 256 x 208 + 256 x 48 = 512 x 128.
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 48;
constexpr float kTau = 8.0f;
// A row whose probabilities, formed against a stale reference, sum to more
// than this over one block is redone with the block's max as reference.
constexpr float kGrowSum = 4294967296.0f;  // 2^32
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns: three score buffers S[0..2] (128 each; the bf16 P
// of a block overwrites its scores) and the output accumulator O (D).
constexpr int kSBufs = 3;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 384;
static_assert(kTmemS + kSBufs * 128 <= kTmemO && kTmemO + 128 <= kTmemCols &&
                  kTmemO + 64 + 16 <= kTmemCols,
              "tensor memory columns");
constexpr unsigned long long kDrainNs = 200ull * 1000 * 1000;
constexpr int kMaxDevices = 64;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kBlock * D * 2;  // one 128 x D bf16 tile
  static constexpr int kBoxes = D / 64;              // 64-column (128-byte) TMA boxes
  static constexpr int kBoxBytes = kBlock * 128;     // 16 KB per box
  // Ring depths and Q buffers: D = 128 fills 224 KB with one Q tile and
  // three stages of each ring; D = 64 has two Q tiles and three stages.
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 3;
  static constexpr int kQStages = D == 128 ? 1 : 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQStages * kTileBytes;
  // V region: the PV MMA's B operand (MN-major) has its 64-wide column
  // groups kVGroup bytes apart: group c of stage s sits at
  // kVOff + c * kVGroup + s * kBoxBytes.
  static constexpr int kVGroup = kVStages * kBoxBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  // Row sum of the rounded P (the O denominator): at D = 64 the tensor core
  // accumulates it next to O, the PV MMA multiplying P by [V | ones] (N =
  // D + 16; the ones tile of each V stage sits one column group after the
  // stage's V, at kOnesOff + s * kBoxBytes); at D = 128 the 16 extra tensor-
  // memory columns are not free, and the softmax threads add it up.
  static constexpr bool kOnes = D == 64;
  static constexpr int kPvN = kOnes ? D + 16 : D;
  static constexpr int kOnesOff = kVOff + kBoxes * kVGroup;
  static constexpr int kBarOff = kOnesOff + (kOnes ? kVStages * kBoxBytes : 0);
  static constexpr int kSmem = kBarOff + 2048;  // barriers, tile queue, 1/l
  static constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false);
  static constexpr uint32_t kIdescO = idesc_bf16_f32(128, kPvN, true);
};

constexpr int kSlotCols = 32;  // key blocks of a tile published with it
constexpr int kMaxStages = 3;  // deepest K / V ring of any Cfg

// One scheduled tile as the scheduler warp publishes it to the producer, MMA
// and softmax warps.
struct TileInfo {
  int t;     // tile id (b*H + h)*nb + qb, or -1 when no tiles are left
  int r0;    // first CSR entry of the tile
  int n;     // live key blocks
  int diag;  // causal and the last live block is the diagonal one
  int cols[kSlotCols];  // its first min(n, 32) key blocks (CSR col_idx[r0 ..])
};

struct __align__(16) Bars {
  uint64_t k_full[kMaxStages];   // K ring stage loaded
  uint64_t k_empty[kMaxStages];  // S(g) complete: K stage free, S(g) ready for the softmax
  uint64_t v_full[kMaxStages];   // V ring stage loaded
  uint64_t v_empty[kMaxStages];  // PV(g) complete: V stage free, O holds block g
  uint64_t q_full[2];
  uint64_t q_empty[2];  // the tile's last S complete: Q buffer free
  // every softmax warp wrote its rows of P(g), indexed by g % kSBufs: the
  // softmax can run up to kSBufs blocks ahead of the PV issue, and P(g +
  // kSBufs) needs S(g + kSBufs), i.e. PV(g) complete, so a barrier never
  // completes a phase for a later block before its waiter saw the earlier one
  uint64_t p_full[kSBufs];
  uint64_t tq_full[2];  // tile queue slot published
  uint64_t tq_empty[2]; // slot read by the producer, both MMA warps, every softmax warp, epilogue leader
  uint64_t drain;       // all MMAs of both issuers complete (one commit from each)
  uint64_t req;         // the producer asks for the next tile (once per tile)
  uint64_t epi_full;    // the softmax handed a tile's O over to the epilogue warps
  uint64_t o_free;      // the epilogue warps read O (and inv_l): the next tile may overwrite it
  TileInfo tq[2];
  uint32_t tmem_base;
  int abort_flag;
  int epi_tile[2];       // tile the epilogue warps write next (by tile parity); < 0: stop
  float inv_l[kBlock];  // D = 128: 1 / (rounded row sum) of the tile being written out
};
static_assert(sizeof(Bars) <= 2048, "barrier block must fit its 2 KB region");
static_assert(Cfg<128>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");
static_assert(Cfg<64>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");
static_assert(Cfg<128>::kKStages <= kMaxStages && Cfg<64>::kKStages <= kMaxStages &&
                  Cfg<128>::kVStages <= kMaxStages && Cfg<64>::kVStages <= kMaxStages,
              "ring depth");

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

// Every role runs with its whole warp converged (warp-collective tcgen05.ld/st
// in the softmax; uniform bookkeeping in the producer and MMA warps, which
// issue their single-thread instructions from an elected lane), so every lane
// must take the same path after a wait: the outcome is made uniform.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint64_t limit_ns) {
  const bool ok = wait_bounded(bar, parity, abort_flag, status, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// wait_warp for waits off the critical path: sleeps about `sleep_ns` between tests
__device__ __forceinline__ bool wait_warp_idle(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int* status,
                                               uint64_t limit_ns, uint32_t sleep_ns) {
  const bool ok = wait_bounded_idle(bar, parity, abort_flag, status, limit_ns, sleep_ns);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// warp 10: tile scheduler
// ---------------------------------------------------------------------------
// Claims tiles from the global counter (in the plan's tile order).  The first
// tile is claimed at once, every later one when the producer asks for it
// (`req`, a few key blocks before the producer needs it), so a CTA never
// holds a claimed tile long before it can start it: tiles stay with the SMs
// that free up first, which keeps the end of the run balanced.  Each tile is
// published in the 2-slot queue with its first key blocks, then its Q is
// loaded into the tile's Q buffer; the claim's chain of dependent global
// reads (counter, tile order, CSR row pointers, column indices) and the Q
// load are thus off the producer's and the MMA warp's path.  Ends after
// publishing the "no tiles left" entry.
template <int D>
__device__ void run_scheduler(const CUtensorMap* tm_q, const FwdParams& p, Bars* bars,
                              uint32_t smem_base, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.timeout_ns;
  const int rows = p.n_live + p.n_empty;
  int qc = 0;  // Q tiles loaded
  bool ok = true;
  for (int i = 0; ok; ++i) {
    const int e = i & 1;
    // the producer asks a few blocks ahead of need: this wait sleeps between tests
    if (i > 0 && !wait_warp_idle(smem_u32(&bars->req), (uint32_t)(i - 1) & 1u, abort_flag,
                                 p.status, lim, kSleepNs)) {
      ok = false;
      break;
    }
    if (!wait_warp(smem_u32(&bars->tq_empty[e]), ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag,
                   p.status, lim)) {
      ok = false;
      break;
    }
    int idx = 0;
    if (lane == 0) idx = atomicAdd(p.counter, 1);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    const int t = idx < p.n_live ? p.tile_order[idx] : -1;
    int r0 = 0, cnt = 0, diag = 0;
    if (t >= 0) {
      if (t >= rows) {
        raise_internal(abort_flag, p.status);
        ok = false;
        break;
      }
      r0 = p.row_ptr[t];
      cnt = p.row_ptr[t + 1] - r0;
      if (cnt <= 0 || cnt > p.nb) {
        raise_internal(abort_flag, p.status);
        ok = false;
        break;
      }
      diag = (p.causal && p.col_idx[r0 + cnt - 1] == t % p.nb) ? 1 : 0;
      if (lane < cnt) bars->tq[e].cols[lane] = p.col_idx[r0 + lane];
    }
    if (lane == 0) {
      volatile TileInfo* slot = &bars->tq[e];
      slot->t = t;
      slot->r0 = r0;
      slot->n = cnt;
      slot->diag = diag;
    }
    __syncwarp();  // every lane's writes to the slot precede the arrive
    if (lane == 0) mbar_arrive(smem_u32(&bars->tq_full[e]));
    __syncwarp();
    if (t < 0) break;
    // the tile's Q, once its buffer is free (the last S of the tile before
    // the previous one is complete)
    const int qs = qc % C::kQStages;
    if (!wait_warp(smem_u32(&bars->q_empty[qs]), ((uint32_t)(qc / C::kQStages) & 1u) ^ 1u, abort_flag,
                   p.status, lim)) {
      ok = false;
      break;
    }
    if (elect_one()) {
      const int bh = t / p.nb;
      const int row = bh * p.S + (t - bh * p.nb) * kBlock;
      const uint32_t full = smem_u32(&bars->q_full[qs]);
      const uint32_t dst = smem_base + C::kQOff + qs * C::kTileBytes;
      mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c)
        tma_load_2d(dst + c * C::kBoxBytes, tm_q, full, c * 64, row);
    }
    __syncwarp();
    ++qc;
  }
  if (!ok) {
    // Let the Q loads this warp issued land before the CTA exits.
    for (int i = (qc > C::kQStages ? qc - C::kQStages : 0); i < qc; ++i)
      wait_drain(smem_u32(&bars->q_full[i % C::kQStages]), (uint32_t)(i / C::kQStages) & 1u);
  }
}

// Reads tile-queue slot `tqc % 2` (waiting until it is published) and marks
// it read.  Returns false when the wait failed.
__device__ __forceinline__ bool take_tile(Bars* bars, int tqc, const FwdParams& p,
                                          volatile int* abort_flag, int& t, int& r0, int& n,
                                          int& col, uint32_t sleep_ns = 0) {
  const int lane = threadIdx.x & 31;
  const int e = tqc & 1;
  const uint32_t bar = smem_u32(&bars->tq_full[e]);
  const uint32_t par = (uint32_t)(tqc >> 1) & 1u;
  if (!(sleep_ns ? wait_warp_idle(bar, par, abort_flag, p.status, p.timeout_ns, sleep_ns)
                 : wait_warp(bar, par, abort_flag, p.status, p.timeout_ns)))
    return false;
  const volatile TileInfo* slot = &bars->tq[e];
  t = slot->t;
  r0 = slot->r0;
  n = slot->n;
  col = (t >= 0 && lane < n && lane < kSlotCols) ? slot->cols[lane] : 0;
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&bars->tq_empty[e]));
  __syncwarp();
  return true;
}

// ---------------------------------------------------------------------------
// warp 8: TMA producer
// ---------------------------------------------------------------------------
// Two cursors over the CTA's block stream: the K cursor runs two blocks ahead
// of the V cursor, matching the MMA warp's order S(g+2) after PV(g).  Each
// ring is loaded in its consumption order.  When the K cursor has
// kClaimAhead blocks of its tile left (or enters a shorter tile) it asks the
// scheduler for the next tile.
template <int D>
__device__ void run_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const FwdParams& p, Bars* bars,
                             uint32_t smem_base, volatile int* abort_flag) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.timeout_ns;
  int kc = 0, vc = 0, tqc = 0;  // K / V tiles loaded, tiles taken
  bool ok = true, more = true;
  int k_ask = 0;  // K cursor's remaining-block count at which to ask for the next tile
  // K cursor: position in its tile; `k_col` holds, in lane i, the key block
  // of the tile's entry 32 * (k_j / 32) + i.
  int k_rem = 0, k_j = 0, k_r0 = 0, k_hrow = 0, k_col = 0;
  // key rows of blocks whose K is loaded and V not yet (at most two)
  int f0 = 0, f1 = 0, nf = 0;

  // One TMA tile (128 rows x D) into a buffer, completion on `full`, after
  // `empty` says the buffer's previous contents were consumed.
  auto load_tile = [&](const CUtensorMap* tm, uint32_t dst, uint32_t box_stride, uint32_t full,
                       uint32_t empty, uint32_t empty_parity, int row) -> bool {
    if (!wait_warp(empty, empty_parity, abort_flag, p.status, lim)) return false;
    if (elect_one()) {
      mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kBoxes; ++c) tma_load_2d(dst + c * box_stride, tm, full, c * 64, row);
    }
    __syncwarp();
    return true;
  };
  auto next_k = [&]() -> bool {
    if (k_rem == 0) {
      if (!more) return true;
      int t = 0;
      if (!take_tile(bars, tqc, p, abort_flag, t, k_r0, k_rem, k_col)) return false;
      ++tqc;
      if (t < 0) {
        more = false;
        k_rem = 0;
        return true;
      }
      // K/V rows of the tile's head (its group's K/V head under grouped-query attention)
      const int bh = t / p.nb;
      const int kvbh =
          p.kv_group > 1 ? (bh / p.H) * (p.H / p.kv_group) + (bh % p.H) / p.kv_group : bh;
      k_hrow = kvbh * p.S;
      k_j = 0;
      k_ask = k_rem - 1 < kClaimAhead ? k_rem - 1 : kClaimAhead;
    } else if ((k_j & 31) == 0) {  // next 32 entries of the tile's CSR list
      k_col = (lane < k_rem) ? p.col_idx[k_r0 + k_j + lane] : 0;
    }
    const int kb = __shfl_sync(0xffffffffu, k_col, k_j & 31);
    if (kb < 0 || kb >= p.nb) {
      raise_internal(abort_flag, p.status);
      return false;
    }
    const int row = k_hrow + kb * kBlock;
    const int st = kc % C::kKStages;
    if (!load_tile(tm_k, smem_base + C::kKOff + st * C::kTileBytes, C::kBoxBytes,
                   smem_u32(&bars->k_full[st]), smem_u32(&bars->k_empty[st]),
                   ((uint32_t)(kc / C::kKStages) & 1u) ^ 1u, row))
      return false;
    ++kc;
    ++k_j;
    --k_rem;
    if (k_rem == k_ask) {
      if (elect_one()) mbar_arrive(smem_u32(&bars->req));
      __syncwarp();
    }
    if (nf == 0) f0 = row; else f1 = row;
    ++nf;
    return true;
  };
  auto load_v = [&](int row) -> bool {
    const int st = vc % C::kVStages;
    if (!load_tile(tm_v, smem_base + C::kVOff + st * C::kBoxBytes, C::kVGroup,
                   smem_u32(&bars->v_full[st]), smem_u32(&bars->v_empty[st]),
                   ((uint32_t)(vc / C::kVStages) & 1u) ^ 1u, row))
      return false;
    ++vc;
    return true;
  };

  ok = next_k();
  if (ok) ok = next_k();
  while (ok && nf > 0) {
    const int row = f0;
    f0 = f1;
    --nf;
    ok = load_v(row);
    if (ok) ok = next_k();
  }
  if (!ok) {
    // Let every TMA load this warp issued land before the CTA exits.
    for (int i = (kc > C::kKStages ? kc - C::kKStages : 0); i < kc; ++i)
      wait_drain(smem_u32(&bars->k_full[i % C::kKStages]), (uint32_t)(i / C::kKStages) & 1u);
    for (int i = (vc > C::kVStages ? vc - C::kVStages : 0); i < vc; ++i)
      wait_drain(smem_u32(&bars->v_full[i % C::kVStages]), (uint32_t)(i / C::kVStages) & 1u);
  }
}

// ---------------------------------------------------------------------------
// warps 9 and 12: tcgen05 MMA issue, one warp per product (elected lane)
// ---------------------------------------------------------------------------
// tcgen05.mma issue returns only about when the tensor core has taken the
// instruction, so a single issuing thread that also waits on barriers leaves
// the tensor core idle during every wait.  Two warps issue instead, one per
// product, each waiting only on its own operands, so while one waits the
// other keeps the tensor core busy.  Each warp's commits track only its own
// MMAs.
//
// S = Q K^T : M=128, N=128, K=D in steps of 16 (32 bytes inside a 128-byte
// swizzle row; a new 64-column box every 4 steps).  S(g) goes into S[g % 3]
// once K(g) is loaded and PV(g-3), which read P(g-3) out of that buffer, is
// complete; its commit frees the K stage and tells the softmax that S(g) is
// ready.  A negative scale is applied as -Q (instruction-descriptor negate
// bit) so the softmax always sees a non-negative multiplier.  After a tile's
// last S the Q buffer is released.
template <int D>
__device__ void run_mma_s(const FwdParams& p, Bars* bars, uint32_t tmem, uint32_t smem_base,
                          volatile int* abort_flag) {
  using C = Cfg<D>;
  const uint64_t lim = p.timeout_ns;
  const uint32_t idesc_s = C::kIdescS | (p.neg_scale ? (1u << 13) : 0u);
  int kc = 0, qc = 0, tqc = 0;  // S issued, tiles' Q used, tiles taken
  bool ok = true;
  while (ok) {
    int t = 0, r0 = 0, n = 0, col = 0;
    if (!take_tile(bars, tqc, p, abort_flag, t, r0, n, col)) break;
    ++tqc;
    if (t < 0) break;
    const int qs = qc % C::kQStages;
    if (!wait_warp(smem_u32(&bars->q_full[qs]), (uint32_t)(qc / C::kQStages) & 1u, abort_flag,
                   p.status, lim))
      break;
    ++qc;
    const uint64_t qd = smem_desc_sw128(smem_base + C::kQOff + qs * C::kTileBytes, 16, 1024);
    for (int j = 0; j < n; ++j) {
      if (kc >= kSBufs) {  // PV(kc-3) complete: S[kc % 3] holds nothing needed any more
        const int pv = kc - kSBufs;
        if (!wait_warp(smem_u32(&bars->v_empty[pv % C::kVStages]),
                       (uint32_t)(pv / C::kVStages) & 1u, abort_flag, p.status, lim)) {
          ok = false;
          break;
        }
      }
      const int st = kc % C::kKStages;
      if (!wait_warp(smem_u32(&bars->k_full[st]), (uint32_t)(kc / C::kKStages) & 1u, abort_flag,
                     p.status, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
        // descriptors advance by adding the byte offset >> 4 to the start-address field
        const uint64_t kd = smem_desc_sw128(smem_base + C::kKOff + st * C::kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + kTmemS + (kc % kSBufs) * 128, qd + off, kd + off, idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->k_empty[st]));
        if (j == n - 1) mma_commit(smem_u32(&bars->q_empty[qs]));  // the tile's last S: Q free
      }
      __syncwarp();
      ++kc;
    }
  }
  // Every MMA issued here must finish before TMEM is released.
  if (elect_one()) mma_commit(smem_u32(&bars->drain));
  __syncwarp();
  wait_drain(smem_u32(&bars->drain), 0);
}

// O (+)= P V : M=128, N=D, K=128 keys in steps of 16.  P(g) is read from
// S[g % 3] (bf16 pairs, 8 columns per step; keys 0..63 at columns 0..31,
// keys 64..127 at columns 64..95); B is MN-major (D contiguous): 8-key
// groups 1024 bytes apart, 64-wide column groups kVGroup apart.  A tile's
// first PV starts a fresh O.  The commit frees V's ring stage and tells the
// softmax and the S issuer that PV(g) is done.
template <int D>
__device__ void run_mma_pv(const FwdParams& p, Bars* bars, uint32_t tmem, uint32_t smem_base,
                           volatile int* abort_flag) {
  using C = Cfg<D>;
  const uint64_t lim = p.timeout_ns;
  int vc = 0, tqc = 0, ntile = 0;  // PV issued, tiles taken, tiles started
  bool ok = true;
  while (ok) {
    int t = 0, r0 = 0, n = 0, col = 0;
    if (!take_tile(bars, tqc, p, abort_flag, t, r0, n, col)) break;
    ++tqc;
    if (t < 0) break;
    // the tile's first PV overwrites O: the epilogue warps must have read the
    // previous tile's O
    if (ntile > 0 && !wait_warp(smem_u32(&bars->o_free), (uint32_t)(ntile - 1) & 1u, abort_flag,
                                p.status, lim))
      break;
    ++ntile;
    for (int j = 0; j < n; ++j) {
      // P(vc) in (one barrier per score buffer, see Bars::p_full)
      if (!wait_warp(smem_u32(&bars->p_full[vc % kSBufs]), (uint32_t)(vc / kSBufs) & 1u, abort_flag,
                     p.status, lim)) {
        ok = false;
        break;
      }
      const int st = vc % C::kVStages;
      if (!wait_warp(smem_u32(&bars->v_full[st]), (uint32_t)(vc / C::kVStages) & 1u, abort_flag,
                     p.status, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (elect_one()) {
        const uint64_t vd = smem_desc_sw128(smem_base + C::kVOff + st * C::kBoxBytes, C::kVGroup,
                                            1024);
        const uint32_t pbuf = tmem + kTmemS + (vc % kSBufs) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t pcol = (kk < 4) ? kk * 8 : 64 + (kk - 4) * 8;  // keys 16kk .. 16kk+15
          mma_ts(tmem + kTmemO, pbuf + pcol, vd + (uint32_t)(kk * 2048 >> 4), C::kIdescO,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->v_empty[st]));
      }
      __syncwarp();
      ++vc;
    }
  }
  if (elect_one()) mma_commit(smem_u32(&bars->drain));
  __syncwarp();
  wait_drain(smem_u32(&bars->drain), 0);
}

// ---------------------------------------------------------------------------
// warps 0-7: softmax + epilogue
// ---------------------------------------------------------------------------
template <int D, bool OUT_F32>
__device__ void write_empty_tiles(const FwdParams& p) {
  using OutT = typename std::conditional<OUT_F32, float, uint16_t>::type;
  const int tid = threadIdx.x;  // 0..kSoftmaxThreads-1
  constexpr int kVec = 16 / sizeof(OutT);
  for (int e = blockIdx.x; e < p.n_empty; e += gridDim.x) {
    const int t = p.empty_tiles[e];
    const int bh = t / p.nb;
    const int qb = t - bh * p.nb;
    const size_t row0 = (size_t)bh * p.S + (size_t)qb * kBlock;
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<OutT*>(p.out) + row0 * D);
    const int nvec = kBlock * D / kVec;
    for (int i = tid; i < nvec; i += kSoftmaxThreads) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < kBlock) p.lse[row0 + tid] = -__int_as_float(0x7f800000);
  }
}

// Probabilities of one 64-column half row: p = 2^(s*sl - m), rounded to bf16
// pairs into pr[] (the A operand of the PV product).  Accumulates the row sum
// of the fp32 p (for the LSE) in a2, two partial sums in one f32x2 pair, and,
// when ROUNDED, r32 of the bf16-rounded p that multiply V (the O denominator,
// so that the weights on V sum to one even when a single key dominates a
// row), again in two partial sums.  sl2 = (sl, sl), nm2 = (-m, -m).
template <bool ROUNDED>
__device__ __forceinline__ void softmax_exp64(const uint32_t* sr, uint32_t* pr, uint64_t sl2,
                                              uint64_t nm2, uint64_t& a2, float (&r32)[2]) {
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * q]), __uint_as_float(sr[2 * q + 1])), sl2, nm2),
              x0, x1);
    const float p0 = ex2_approx(x0);
    const float p1 = ex2_approx(x1);
    pr[q] = pack_bf16x2(p0, p1);
    a2 = f2_add(a2, f2_pack(p0, p1));
    if (ROUNDED) add_bf16x2_f32(r32[0], r32[1], pr[q]);
  }
}

__device__ __forceinline__ float row_max64(const uint32_t* sr) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = fmaxf(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]));
#pragma unroll
  for (int c = 16; c < 64; c += 16) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      a[i] = max3(a[i], __uint_as_float(sr[c + 2 * i]), __uint_as_float(sr[c + 2 * i + 1]));
  }
  return fmaxf(max3(a[0], a[1], a[2]), max3(max3(a[3], a[4], a[5]), a[6], a[7]));
}

template <int D, bool OUT_F32>
__device__ void run_softmax(const FwdParams& p, Bars* bars, uint32_t tmem,
                            volatile int* abort_flag) {
  using C = Cfg<D>;
  constexpr int DH = D / 2;            // O columns owned by this thread
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = warp & 3;            // TMEM sub-partition: lanes 32*sub .. 32*sub+31
  const int lh = (warp >> 2) & 1;      // which 16 lanes of the sub-partition this warp covers
  const int ch = lane >> 4;            // column half: keys [64ch, 64ch+64), O cols [DH ch, DH ch+DH)
  const int r = sub * 32 + lh * 16 + (lane & 15);  // query row (TMEM lane) of this thread
  // 16x32bx2 accesses: lanes 0..15 of the warp take the address's columns,
  // lanes 16..31 the same rows 64 (or DH) columns further on.
  const uint32_t lane_off = (uint32_t)(sub * 32 + lh * 16) << 16;
  const uint32_t tO = tmem + kTmemO + lane_off;
  const float sl = p.scale_log2;       // > 0 (see FwdParams)
  const uint64_t sl2 = f2_pack(sl, sl);
  const uint32_t kNegInf = 0xff800000u;
  const uint64_t lim = p.timeout_ns;

  write_empty_tiles<D, OUT_F32>(p);

  int tq_cnt = 0, g = 0;  // g: blocks processed by this CTA (selects S buffer / ring stages)
  int ntile = 0;          // tiles handed to the epilogue warps
  for (;;) {
    const int e = tq_cnt & 1;
    const uint32_t ph = (uint32_t)(tq_cnt >> 1) & 1u;
    if (!wait_warp(smem_u32(&bars->tq_full[e]), ph, abort_flag, p.status, lim)) return;
    const volatile int* slot = reinterpret_cast<const volatile int*>(&bars->tq[e]);
    const int t = slot[0];
    const int n = slot[2];
    const int diag_last = slot[3];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars->tq_empty[e]));
    ++tq_cnt;
    if (t < 0) return;
    const int bh = t / p.nb;
    const int qb = t - bh * p.nb;

    float m = __uint_as_float(kNegInf);  // running max of scale*log2(e)*score (lazy)
    uint64_t a2 = 0;            // partial sums of this half row: fp32 p (an f32x2 pair)
    float r32[2] = {0.f, 0.f};  // and bf16-rounded p
    for (int jb = 0; jb < n; ++jb, ++g) {
      const int b = g % kSBufs;  // P barrier of this block
      // S(g) ready = its commit released K(g)'s stage
      if (!wait_warp(smem_u32(&bars->k_empty[g % C::kKStages]), (uint32_t)(g / C::kKStages) & 1u,
                     abort_flag, p.status, lim))
        return;
      tc_fence_after();
      const uint32_t tS = tmem + kTmemS + (g % kSBufs) * 128 + lane_off;  // S buffer of this block
      uint32_t sr[64];
      tmem_ld16x2_32<64>(tS + 0, sr + 0);
      tmem_ld16x2_32<64>(tS + 32, sr + 32);
      tmem_wait_ld();
      reg_fence(sr, 64);
      const bool diag = diag_last && jb == n - 1;
      if (diag) {  // causal diagonal tile: key c is allowed for query row r iff c <= r
#pragma unroll
        for (int c = 0; c < 64; ++c) sr[c] = (ch * 64 + c > r) ? kNegInf : sr[c];
      }
      // After a tile's first block the probabilities are formed against the
      // current reference m without a max pass (any common reference gives
      // the exact softmax).  Only when a row's sum over the block shows that
      // its scores rose far above m (kGrowSum) -- or on the tile's first
      // block, where m = -inf -- is the block redone with its max, by the
      // lazy rule, as the new reference.
      uint32_t pr[32];
      uint64_t b2 = 0;  // this block's sums
      float br32[2] = {0.f, 0.f};
      bool redo = jb == 0;
      if (!redo) {
        softmax_exp64<!C::kOnes>(sr, pr, sl2, f2_pack(-m, -m), b2, br32);
        float b0, b1;
        f2_unpack(b2, b0, b1);
        float bs = b0 + b1;
        bs += __shfl_xor_sync(0xffffffffu, bs, 16);  // the other half of the row
        redo = __any_sync(0xffffffffu, !(bs <= kGrowSum));  // also catches inf / NaN
      }
      bool need = false;
      float f = 1.f;
      if (redo) {
        float mx = row_max64(sr);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // the other half of the row
        const float xm = mx * sl;
        need = xm > m + kTau;  // always true on the first block (m = -inf)
        if (need) {
          f = ex2_approx(m - xm);  // 0 when m = -inf
          m = xm;
          a2 = f2_mul(a2, f2_pack(f, f));
          r32[0] *= f;
          r32[1] *= f;
        }
        b2 = 0;
        br32[0] = br32[1] = 0.f;
        softmax_exp64<!C::kOnes>(sr, pr, sl2, f2_pack(-m, -m), b2, br32);
      }
      a2 = f2_add(a2, b2);
      r32[0] += br32[0];
      r32[1] += br32[1];
      tmem_st16x2_32<64>(tS, pr);  // P over the scores just read (keys 0..63 -> cols 0..31, 64..127 -> 64..95)

      // O rescale (this thread's columns) when a row's max moved: first wait
      // until PV(g-1) has landed in O (PV(g) is not issued before P(g)).
      if (jb > 0 && __any_sync(0xffffffffu, need)) {
        if (!wait_warp(smem_u32(&bars->v_empty[(g - 1) % C::kVStages]),
                       (uint32_t)((g - 1) / C::kVStages) & 1u, abort_flag, p.status, lim))
          return;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) {
          uint32_t orr[32];
          tmem_ld16x2_32<DH>(tO + c0, orr);
          tmem_wait_ld();
          reg_fence(orr, 32);
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * f);
          tmem_st16x2_32<DH>(tO + c0, orr);
        }
        if constexpr (C::kOnes) {  // the row-sum column read at the end scales with O
          uint32_t rs[1];
          tmem_ld16x2_1<1>(tO + D, rs);
          tmem_wait_ld();
          reg_fence(rs, 1);
          rs[0] = __float_as_uint(__uint_as_float(rs[0]) * f);
          tmem_st16x2_1<1>(tO + D, rs);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();  // the warp's stores of P(g) are complete (each lane waited for its own)
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[b]));
    }

    // Hand the tile over to the epilogue warps and go straight on to the next
    // tile: the LSE is written here; at D = 128 the O denominator 1/l goes
    // through shared memory (at D = 64 it sits in tensor memory next to O).
    float a0, a1;
    f2_unpack(a2, a0, a1);
    float l32 = a0 + a1;  // fp32 sum of the unrounded P: the LSE
    l32 += __shfl_xor_sync(0xffffffffu, l32, 16);  // the other half of the row
    const size_t row = (size_t)bh * p.S + (size_t)qb * kBlock + r;
    if (ch == 0) p.lse[row] = (m + __log2f(l32)) * 0.69314718055994530942f;
    // The epilogue warps are done with the previous tile (its 1/l is read):
    // this keeps the softmax at most one tile ahead of them, so a later tile's
    // epi_full phase can never complete before they waited for this one.
    if (ntile > 0 && !wait_warp(smem_u32(&bars->o_free), (uint32_t)(ntile - 1) & 1u, abort_flag,
                                p.status, lim))
      return;
    if constexpr (!C::kOnes) {
      float l = r32[0] + r32[1];  // sum of the rounded P: the O denominator
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (ch == 0) bars->inv_l[r] = 1.0f / l;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars->epi_full));
    ++ntile;
    // Compiler barrier between tiles: nothing of the next tile's setup is
    // scheduled into this one.  Without it the block loop above compiles to
    // code that runs about 15 % slower per block.
    asm volatile("" ::: "memory");
  }
}

// ---------------------------------------------------------------------------
// warps 12-15: epilogue, one thread per query row (TMEM lane)
// ---------------------------------------------------------------------------
// For each tile the softmax hands over: wait for its last PV, read O row by
// row (16 columns at a time), divide by the rounded row sum and store it;
// then release O for the next tile's first PV.  Only the leader warp takes
// tiles and waits (sleeping between tests); it passes the tile on through
// shared memory and a named barrier, where the other three warps wait
// without issuing.  The leader reaches the barrier on every path, with a
// negative tile to stop, so the four warps always leave together.
template <int D, bool OUT_F32>
__device__ void run_epilogue(const FwdParams& p, Bars* bars, uint32_t tmem,
                             volatile int* abort_flag) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;  // query row of the tile = TMEM lane
  const uint32_t tO = tmem + kTmemO + ((uint32_t)((warp & 3) * 32) << 16);
  const uint64_t lim = p.timeout_ns;
  int tqc = 0, g = 0, ntile = 0;  // (leader) tiles taken, blocks of the stream passed; tiles written
  for (;;) {
    if (warp == kWarpEpi0) {
      int t = 0, r0 = 0, n = 0, col = 0;
      bool ok = take_tile(bars, tqc, p, abort_flag, t, r0, n, col, kSleepNs);
      ++tqc;
      if (ok && t >= 0) {
        const int gl = g + n - 1;  // the tile's last block
        g += n;
        // the softmax is done with the tile (its LSE written, 1/l in shared
        // memory at D = 128), and the tile's last PV has landed in O
        ok = wait_warp_idle(smem_u32(&bars->epi_full), (uint32_t)ntile & 1u, abort_flag, p.status,
                            lim, kSleepNs) &&
             wait_warp_idle(smem_u32(&bars->v_empty[gl % C::kVStages]),
                            (uint32_t)(gl / C::kVStages) & 1u, abort_flag, p.status, lim, kSleepNs);
      }
      if (lane == 0) bars->epi_tile[ntile & 1] = ok ? t : -1;
    }
    named_bar_sync(kEpiBarrier, kEpiWarps * 32);
    const int t = *reinterpret_cast<volatile int*>(&bars->epi_tile[ntile & 1]);
    if (t < 0) return;
    tc_fence_after();
    float inv_l = 0.f;
    if constexpr (!C::kOnes) inv_l = bars->inv_l[r];
    if constexpr (C::kOnes) {  // rounded row sum accumulated by the tensor core in column D
      uint32_t rs[1];
      tmem_ld32_1(tO + D, rs);
      tmem_wait_ld();
      reg_fence(rs, 1);
      inv_l = 1.0f / __uint_as_float(rs[0]);
    }
    const int bh = t / p.nb;
    const size_t row = (size_t)bh * p.S + (size_t)(t - bh * p.nb) * kBlock + r;
    // Each thread writes its own row: 32-byte stores (one full sector each)
    // when the output is 32-byte aligned, else 16-byte ones.
    const bool wide = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 16) {
      uint32_t orr[16];
      tmem_ld32_16(tO + c0, orr);
      tmem_wait_ld();
      reg_fence(orr, 16);
      if constexpr (OUT_F32) {
        float* dst = reinterpret_cast<float*>(p.out) + row * D + c0;
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(orr[i]) * inv_l);
        if (wide) {
          st_global_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(v));
          st_global_v8(dst + 8, *reinterpret_cast<const uint32_t(*)[8]>(v + 8));
        } else {
#pragma unroll
          for (int i = 0; i < 16; i += 4) st_global_v4(dst + i, v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      } else {
        uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + row * D + c0;
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pk[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv_l,
                              __uint_as_float(orr[2 * i + 1]) * inv_l);
        if (wide) {
          st_global_v8(dst, pk);
        } else {
          st_global_v4(dst, pk[0], pk[1], pk[2], pk[3]);
          st_global_v4(dst + 8, pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
    tc_fence_before();
    __syncwarp();  // every lane's reads of O are complete
    if (lane == 0) mbar_arrive(smem_u32(&bars->o_free));
    ++ntile;
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
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(smem_u32(&bars->k_full[i]), 1);
      mbar_init(smem_u32(&bars->k_empty[i]), 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(smem_u32(&bars->v_full[i]), 1);
      mbar_init(smem_u32(&bars->v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->q_full[i]), 1);
      mbar_init(smem_u32(&bars->q_empty[i]), 1);
    }
    // the softmax warps arrive once per warp (elected lane, after __syncwarp)
    for (int i = 0; i < kSBufs; ++i) mbar_init(smem_u32(&bars->p_full[i]), kSoftmaxWarps);
    mbar_init(smem_u32(&bars->drain), 2);
    mbar_init(smem_u32(&bars->req), 1);
    mbar_init(smem_u32(&bars->epi_full), kSoftmaxWarps);
    mbar_init(smem_u32(&bars->o_free), kEpiWarps);
    for (int e = 0; e < 2; ++e) {
      mbar_init(smem_u32(&bars->tq_full[e]), 1);
      mbar_init(smem_u32(&bars->tq_empty[e]), 3 + kSoftmaxWarps + 1);
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMmaS) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if constexpr (C::kOnes) {  // bf16 1.0 tiles read by the PV MMA (generic-proxy writes, then a proxy fence)
    uint4* ones = reinterpret_cast<uint4*>(smem_raw + (base - raw) + C::kOnesOff);
    for (int i = threadIdx.x; i < C::kVStages * C::kBoxBytes / 16; i += kThreads)
      ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

  if (warp >= kSoftmaxThreads / 32) {
    regs_dec<kRegsOther>();
    if (warp == kWarpLoad)
      run_producer<D>(&tm_q, &tm_k, &tm_v, p, bars, base, abort_flag);
    else if (warp == kWarpMmaS)
      run_mma_s<D>(p, bars, tmem, base, abort_flag);
    else if (warp == kWarpMmaPV)
      run_mma_pv<D>(p, bars, tmem, base, abort_flag);
    else if (warp >= kWarpEpi0)
      run_epilogue<D, OUT_F32>(p, bars, tmem, abort_flag);
    else if (warp == kWarpSched)
      run_scheduler<D>(&tm_q, p, bars, base, abort_flag);
  } else {
    regs_inc<kRegsSoftmax>();
    run_softmax<D, OUT_F32>(p, bars, tmem, abort_flag);
  }
  __syncwarp();  // reconverge each warp before the CTA-wide barrier

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaS) {
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
  // The shared-memory opt-in is set once per device (it costs host time on
  // every call otherwise); a failed attempt is retried on the next call.
  static std::atomic<bool> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(bsattn_fwd_kernel<D, OUT_F32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
  }
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
