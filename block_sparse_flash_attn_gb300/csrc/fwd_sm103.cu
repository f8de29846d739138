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
// core's own work.  Shared memory: Q buffers and rings of K and V tiles
// (128 x D each, 128-byte swizzled by TMA, read by tcgen05.mma through matrix
// descriptors); see Cfg for the depths of each configuration.
//
// Precision: S = Q K^T in bf16 (e4m3 with FP8 inputs) with fp32 accumulation;
// P V in bf16 at D = 128, in fp16 at D = 64 and with FP8 inputs, so that the
// rounding of P, the largest error term, is 2^-11 instead of 2^-8 where the
// logits are wide.  V reaches fp16 in one of two ways: converted once per
// call into an fp16 copy that the kernel loads (v16_convert_kernel and its
// e4m3 twin, FwdParams::v_pre), or tile by tile in shared memory by the four
// epilogue warps (bf16 -> fp16 in place, e4m3 -> fp16 from a staging ring).
//
// The producer sees the CTA's tiles as one stream of key blocks and loads K
// two blocks ahead of V along it; the scheduler warp loads each tile's Q as
// soon as the Q buffer is free.  With 64-key blocks (kdiv = 2) a block of the
// stream is a pair of consecutive entries of the tile's list, loaded as the
// two 64-row halves of one stage (an odd tail repeats its one entry and the
// softmax masks the copy).  Along the stream one MMA warp issues S(g) as soon
// as K(g) is loaded and PV(g-3) is complete, another issues PV(g) as soon as
// P(g) is written and V(g) loaded (and converted); a tile's first PV starts a
// fresh O.  The commit after S(g) frees K(g)'s ring stage and signals "S(g)
// ready" (s_full); the commit after PV(g) frees V(g)'s stage and signals
// "PV(g) done" (pv_done), which the S issuer waits for before reusing a score
// buffer, the softmax before an O rescale and the epilogue warps for a
// tile's last block.  The next tile's first PV, the one that overwrites O,
// waits until the epilogue warps have read O.
// Online softmax in base 2 with lazy rescale: the running max m only moves
// when a block's max exceeds it by more than 8 (log2 units), so P <= 256 and
// the O rescale is rare.  O is normalised by the row sum of the rounded P
// that multiplied V (so the weights on V sum to one even when a single key
// dominates a row); the LSE uses the fp32 sum of the unrounded P.  A row with
// no allowed key (possible inside a live tile only with 64-key blocks under
// causal) gets O = 0 and LSE = -inf.
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
#ifndef BSATTN_CLAIM_AHEAD
#define BSATTN_CLAIM_AHEAD 4
#endif
constexpr int kClaimAhead = BSATTN_CLAIM_AHEAD;
// Launch budget 512 x 128 registers; the two role warpgroups hand part of
// their share to the two softmax warpgroups: 256 x 208 + 256 x 48 = 512 x 128.
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 48;
constexpr float kTau = 8.0f;
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

#ifndef BSATTN_D128_QSTAGES
#define BSATTN_D128_QSTAGES 1
#endif
#ifndef BSATTN_D128_KSTAGES
#define BSATTN_D128_KSTAGES 3
#endif
#ifndef BSATTN_D128_VSTAGES
#define BSATTN_D128_VSTAGES 3
#endif

// IN8: Q, K, V are e4m3 (FP8), at D = 128 only.  Q and K tiles are then 16 KB
// (one 128-byte row per key or query), S = Q K^T runs as kind::f8f6f4 MMAs
// (K = 32 per instruction), and P V runs in fp16 (P as well): each e4m3 V tile
// lands in its own staging ring, from which the epilogue warps convert it to
// the fp16 V tile that the P V product reads, unless V was converted to fp16
// before the launch (then the fp16 tiles are loaded directly).
template <int D, bool IN8 = false>
struct Cfg {
  static_assert(!IN8 || D == 128, "e4m3 inputs at head_dim 128 only");
  static constexpr bool kIn8 = IN8;
  static constexpr int kTileBytes = kBlock * D * 2;  // one 128 x D bf16 / fp16 tile (V for P V)
  static constexpr int kBoxes = D / 64;              // 64-column (128-byte) boxes of such a tile
  static constexpr int kBoxBytes = kBlock * 128;     // 16 KB per box
  // Q and K tiles as loaded: bf16 (kBoxes boxes), or e4m3 (one 128-byte box)
  static constexpr int kQKBytes = IN8 ? kBlock * D : kTileBytes;
  static constexpr int kQKBoxes = IN8 ? 1 : kBoxes;
  // Ring depths and Q buffers: at D = 128 seven 32 KB tiles fill 224 KB
  // (Q buffers + K stages + V stages = 7); D = 64 has two Q tiles and three
  // stages of each ring; e4m3 has two 16 KB Q tiles, three 16 KB K stages,
  // three 16 KB e4m3 V stages and three 32 KB fp16 V stages (224 KB).
  static constexpr int kKStages = IN8 ? 3 : D == 128 ? BSATTN_D128_KSTAGES : 3;
  static constexpr int kVStages = IN8 ? 3 : D == 128 ? BSATTN_D128_VSTAGES : 3;
  static constexpr int kQStages = IN8 ? 2 : D == 128 ? BSATTN_D128_QSTAGES : 2;
  static constexpr int kV8Stages = IN8 ? 3 : 0;  // e4m3 V staging ring
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQStages * kQKBytes;
  static constexpr int kV8Off = kKOff + kKStages * kQKBytes;
  // V region: the PV MMA's B operand (MN-major) has its 64-wide column
  // groups kVGroup bytes apart: group c of stage s sits at
  // kVOff + c * kVGroup + s * kBoxBytes.
  static constexpr int kVGroup = kVStages * kBoxBytes;
  static constexpr int kVOff = kV8Off + kV8Stages * kBoxBytes;
  // Row sum of the rounded P (the O denominator): at D = 64 the tensor core
  // accumulates it next to O, the PV MMA multiplying P by [V | ones] (N =
  // D + 16; the ones tile of each V stage sits one column group after the
  // stage's V, at kOnesOff + s * kBoxBytes); at D = 128 the 16 extra tensor-
  // memory columns are not free, and the softmax threads add it up.
  static constexpr bool kOnes = D == 64;
  static constexpr int kPvN = kOnes ? D + 16 : D;
  // P V in fp16 (P and V rounded to 11 significant bits instead of bf16's 8)
  // at D = 64 and with e4m3 inputs (V converted before the launch, or by the
  // epilogue warps in shared memory); at D = 128 with bf16 inputs P V stays
  // in bf16.
  static constexpr bool kF16PV = D == 64 || IN8;
  // A half row's block sum above this (formed against a stale reference)
  // makes the softmax redo the block with its max; in fp16 it also keeps every
  // P below fp16's largest finite value: each P <= its half's sum <= 2^15.
  static constexpr float kGrowSum = kF16PV ? 32768.0f : 4294967296.0f;
  static constexpr int kOnesOff = kVOff + kBoxes * kVGroup;
  static constexpr int kBarOff = kOnesOff + (kOnes ? kVStages * kBoxBytes : 0);
  static constexpr int kSmem = kBarOff + 2048;  // barriers, tile queue, 1/l
  // S = Q K^T: bf16 (kind::f16, K = 16 per MMA) or e4m3 (kind::f8f6f4, K =
  // 32 per MMA; e4m3 has the same format code, 0, there as f16 has in kind::f16)
  static constexpr int kSMmas = IN8 ? 4 : D / 16;
  static constexpr uint32_t kIdescS = idesc_f16kind_f32(128, 128, false, false, IN8);
  static constexpr uint32_t kIdescO = idesc_f16kind_f32(128, kPvN, true, false, kF16PV);
};

constexpr int kSlotCols = 32;  // key blocks of a tile published with it
constexpr int kMaxStages = 3;  // deepest K / V ring of any Cfg

// One scheduled tile as the scheduler warp publishes it to the producer, MMA
// and softmax warps.
struct TileInfo {
  int t;     // tile id (b*H + h)*nb + qb, or -1 when no tiles are left
  int bh;    // its head b*H + h and query block qb (t = bh*nb + qb)
  int qb;
  int r0;    // first CSR entry of the tile
  int n;     // blocks of the stream: live key blocks (64-key blocks: their pairs)
  int diag;  // causal and the last live block is the diagonal one (128-key blocks)
  int n64;   // CSR entries of the tile (= n for 128-key blocks)
  int last2[2];  // 64-key blocks: the key blocks of entries n64-2 and n64-1 (-1: none)
  int cols[kSlotCols];  // its first min(n64, 32) CSR entries (col_idx[r0 ..])
};

struct __align__(16) Bars {
  uint64_t k_full[kMaxStages];   // K ring stage loaded
  uint64_t k_empty[kMaxStages];  // S(g) complete: K stage free
  uint64_t v_full[kMaxStages];   // V ring stage loaded
  uint64_t v_empty[kMaxStages];  // PV(g) complete: V stage free, O holds block g
  uint64_t v_conv[kMaxStages];   // fp16 P V: the four epilogue warps converted V(g) to fp16
  uint64_t v8_full[kMaxStages];  // e4m3 inputs: V(g) staged (TMA)
  uint64_t v8_empty[kMaxStages]; // e4m3 inputs: V(g) converted, the staging stage is free
  uint64_t q_full[2];
  uint64_t q_empty[2];  // the tile's last S complete: Q buffer free
  // every softmax warp wrote its rows of P(g), indexed by g % kSBufs: the
  // softmax can run up to kSBufs blocks ahead of the PV issue, and P(g +
  // kSBufs) needs S(g + kSBufs), i.e. PV(g) complete, so a barrier never
  // completes a phase for a later block before its waiter saw the earlier one
  uint64_t p_full[kSBufs];
  // S(g) complete (the softmax may read it) and PV(g) complete (S buffer g %
  // kSBufs may take S(g + kSBufs)), indexed by g % kSBufs: a phase of these can
  // only complete once the waiter is done with the previous one (S(g + 3)
  // needs PV(g), which needs P(g) from the softmax; PV(g + 3) needs S(g + 3),
  // which the S issuer has not issued while it waits for PV(g)), so their
  // parity waits never alias, whatever the ring depths; a wait on a ring
  // stage's own barrier could, when that ring is shallower than kSBufs.
  uint64_t s_full[kSBufs];
  uint64_t pv_done[kSBufs];
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
  int epi_n[2];          // and its live key blocks
  float inv_l[kBlock];  // D = 128: 1 / (rounded row sum) of the tile being written out
};
static_assert(sizeof(Bars) <= 2048, "barrier block must fit its 2 KB region");
static_assert(Cfg<128>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");
static_assert(Cfg<64>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");
static_assert(Cfg<128, true>::kSmem + 1024 <= 232448, "shared memory per CTA (227 KB) exceeded");
static_assert(Cfg<128>::kKStages <= kMaxStages && Cfg<64>::kKStages <= kMaxStages &&
                  Cfg<128>::kVStages <= kMaxStages && Cfg<64>::kVStages <= kMaxStages &&
                  Cfg<128, true>::kKStages <= kMaxStages &&
                  Cfg<128, true>::kV8Stages <= kMaxStages,
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
template <int D, bool IN8, bool KB64>
__device__ void run_scheduler(const CUtensorMap* tm_q, const FwdParams& p, Bars* bars,
                              uint32_t smem_base, volatile int* abort_flag) {
  using C = Cfg<D, IN8>;
  constexpr int kKdiv = KB64 ? 2 : 1;  // 128 / kKdiv keys per key block
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
    int r0 = 0, cnt = 0, diag = 0, l0 = -1, l1 = -1;
    const int bh = t >= 0 ? t / p.nb : 0;
    const int qb = t - bh * p.nb;
    if (t >= 0) {
      if (t >= rows) {
        raise_internal(abort_flag, p.status);
        ok = false;
        break;
      }
      r0 = p.row_ptr[t];
      cnt = p.row_ptr[t + 1] - r0;
      if (cnt <= 0 || cnt > p.nb * kKdiv) {
        raise_internal(abort_flag, p.status);
        ok = false;
        break;
      }
      if constexpr (!KB64) {
        diag = (p.causal && p.col_idx[r0 + cnt - 1] == qb) ? 1 : 0;
      } else {
        l0 = cnt >= 2 ? p.col_idx[r0 + cnt - 2] : -1;
        l1 = p.col_idx[r0 + cnt - 1];
      }
      if (lane < cnt && lane < kSlotCols) bars->tq[e].cols[lane] = p.col_idx[r0 + lane];
    }
    if (lane == 0) {
      volatile TileInfo* slot = &bars->tq[e];
      slot->t = t;
      slot->bh = bh;
      slot->qb = qb;
      slot->r0 = r0;
      slot->n = KB64 ? (cnt + 1) / 2 : cnt;
      slot->diag = diag;
      slot->n64 = cnt;
      slot->last2[0] = l0;
      slot->last2[1] = l1;
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
      const int row = bh * p.S + qb * kBlock;
      const uint32_t full = smem_u32(&bars->q_full[qs]);
      const uint32_t dst = smem_base + C::kQOff + qs * C::kQKBytes;
      mbar_arrive_expect_tx(full, C::kQKBytes);
#pragma unroll
      for (int c = 0; c < C::kQKBoxes; ++c)
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
                                          int& col, uint32_t sleep_ns = 0, int* n64 = nullptr) {
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
  const int ne = slot->n64;
  if (n64) *n64 = ne;
  col = (t >= 0 && lane < ne && lane < kSlotCols) ? slot->cols[lane] : 0;
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
template <int D, bool IN8, bool KB64>
__device__ void run_producer(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const FwdParams& p, Bars* bars,
                             uint32_t smem_base, volatile int* abort_flag) {
  using C = Cfg<D, IN8>;
  constexpr int kKdiv = KB64 ? 2 : 1;  // 128 / kKdiv keys per key block
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.timeout_ns;
  int kc = 0, vc = 0, tqc = 0;  // K / V tiles loaded, tiles taken
  bool ok = true, more = true;
  int k_ask = 0;  // K cursor's remaining-block count at which to ask for the next tile
  // K cursor: position in its tile (stream blocks); `k_col` holds, in lane i,
  // the key block of the tile's CSR entry 32 * (e / 32) + i, e the cursor's
  // first entry (64-key blocks: stream block j is entries 2j and 2j + 1).
  int k_rem = 0, k_j = 0, k_r0 = 0, k_hrow = 0, k_col = 0, k_n64 = 0;
  // key rows of blocks whose K is loaded and V not yet (at most two); with
  // 64-key blocks, the rows of the block's two halves
  int f0 = 0, f1 = 0, g0 = 0, g1 = 0, nf = 0;
  constexpr bool halves = KB64;
  constexpr uint32_t kHalfBytes = 64 * 128;  // 64 rows of a 128-byte-row box

  // One TMA tile (128 rows x D) into a buffer, completion on `full`, after
  // `empty` says the buffer's previous contents were consumed; with 64-key
  // blocks as two 64-row halves from rows `row` and `row2` (the tensor map's
  // box is then 64 rows high).
  // `nbox` boxes of 128-byte rows, `bytes` in all (bf16: D / 64 boxes; e4m3: one).
  auto load_tile = [&](const CUtensorMap* tm, uint32_t dst, uint32_t box_stride, uint32_t full,
                       uint32_t empty, uint32_t empty_parity, int row, int row2, int nbox,
                       uint32_t bytes) -> bool {
    if (!wait_warp(empty, empty_parity, abort_flag, p.status, lim)) return false;
    if (elect_one()) {
      mbar_arrive_expect_tx(full, bytes);
      for (int c = 0; c < nbox; ++c) {
        tma_load_2d(dst + c * box_stride, tm, full, c * 64, row);
        if constexpr (halves) tma_load_2d(dst + c * box_stride + kHalfBytes, tm, full, c * 64, row2);
      }
    }
    __syncwarp();
    return true;
  };
  auto next_k = [&]() -> bool {
    if (k_rem == 0) {
      if (!more) return true;
      int t = 0;
      if (!take_tile(bars, tqc, p, abort_flag, t, k_r0, k_rem, k_col, 0, &k_n64)) return false;
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
    } else {
      const int e = halves ? 2 * k_j : k_j;
      if ((e & 31) == 0)  // next 32 entries of the tile's CSR list
        k_col = (lane < k_n64 - e) ? p.col_idx[k_r0 + e + lane] : 0;
    }
    const int e = halves ? 2 * k_j : k_j;
    const int kb = __shfl_sync(0xffffffffu, k_col, e & 31);
    // the second half: the next entry, or (odd tail) the first half again,
    // whose scores the softmax masks
    int kb2 = kb;
    if (halves && e + 1 < k_n64) kb2 = __shfl_sync(0xffffffffu, k_col, (e + 1) & 31);
    const int nbk = p.nb * kKdiv;
    if (kb < 0 || kb >= nbk || kb2 < 0 || kb2 >= nbk) {
      raise_internal(abort_flag, p.status);
      return false;
    }
    const int krows = kBlock / kKdiv;
    const int row = k_hrow + kb * krows, row2 = k_hrow + kb2 * krows;
    const int st = kc % C::kKStages;
    if (!load_tile(tm_k, smem_base + C::kKOff + st * C::kQKBytes, C::kBoxBytes,
                   smem_u32(&bars->k_full[st]), smem_u32(&bars->k_empty[st]),
                   ((uint32_t)(kc / C::kKStages) & 1u) ^ 1u, row, row2, C::kQKBoxes,
                   C::kQKBytes))
      return false;
    ++kc;
    ++k_j;
    --k_rem;
    if (k_rem == k_ask) {
      if (elect_one()) mbar_arrive(smem_u32(&bars->req));
      __syncwarp();
    }
    if (nf == 0) {
      f0 = row;
      g0 = row2;
    } else {
      f1 = row;
      g1 = row2;
    }
    ++nf;
    return true;
  };
  auto load_v = [&](int row, int row2) -> bool {
    if constexpr (C::kIn8) {
      if (!p.v_pre) {  // into the e4m3 staging ring, free once converted
        const int st = vc % C::kV8Stages;
        if (!load_tile(tm_v, smem_base + C::kV8Off + st * C::kBoxBytes, C::kBoxBytes,
                       smem_u32(&bars->v8_full[st]), smem_u32(&bars->v8_empty[st]),
                       ((uint32_t)(vc / C::kV8Stages) & 1u) ^ 1u, row, row2, 1, C::kBoxBytes))
          return false;
        ++vc;
        return true;
      }
    }
    // bf16 V, or V converted to fp16 before the launch: straight into the ring
    // the P V product reads
    const int st = vc % C::kVStages;
    if (!load_tile(tm_v, smem_base + C::kVOff + st * C::kBoxBytes, C::kVGroup,
                   smem_u32(&bars->v_full[st]), smem_u32(&bars->v_empty[st]),
                   ((uint32_t)(vc / C::kVStages) & 1u) ^ 1u, row, row2, C::kBoxes,
                   C::kTileBytes))
      return false;
    ++vc;
    return true;
  };

  ok = next_k();
  if (ok) ok = next_k();
  while (ok && nf > 0) {
    const int row = f0, row2 = g0;
    f0 = f1;
    g0 = g1;
    --nf;
    ok = load_v(row, row2);
    if (ok) ok = next_k();
  }
  if (!ok) {
    // Let every TMA load this warp issued land before the CTA exits.
    for (int i = (kc > C::kKStages ? kc - C::kKStages : 0); i < kc; ++i)
      wait_drain(smem_u32(&bars->k_full[i % C::kKStages]), (uint32_t)(i / C::kKStages) & 1u);
    bool staged = false;  // e4m3 V went to the staging ring
    if constexpr (C::kIn8) {
      staged = !p.v_pre;
      if (staged)
        for (int i = (vc > C::kV8Stages ? vc - C::kV8Stages : 0); i < vc; ++i)
          wait_drain(smem_u32(&bars->v8_full[i % C::kV8Stages]),
                     (uint32_t)(i / C::kV8Stages) & 1u);
    }
    if (!staged)
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
template <int D, bool IN8>
__device__ void run_mma_s(const FwdParams& p, Bars* bars, uint32_t tmem, uint32_t smem_base,
                          volatile int* abort_flag) {
  using C = Cfg<D, IN8>;
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
    const uint64_t qd = smem_desc_sw128(smem_base + C::kQOff + qs * C::kQKBytes, 16, 1024);
    for (int j = 0; j < n; ++j) {
      if (kc >= kSBufs) {  // PV(kc-3) complete: S[kc % 3] holds nothing needed any more
        const int pv = kc - kSBufs;
        if (!wait_warp(smem_u32(&bars->pv_done[pv % kSBufs]), (uint32_t)(pv / kSBufs) & 1u,
                       abort_flag, p.status, lim)) {
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
        const uint64_t kd = smem_desc_sw128(smem_base + C::kKOff + st * C::kQKBytes, 16, 1024);
        // 32 bytes of K per MMA (16 bf16 or 32 e4m3), a new 64-column box every 4
#pragma unroll
        for (int kk = 0; kk < C::kSMmas; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4;
          if constexpr (C::kIn8)
            mma_ss_f8(tmem + kTmemS + (kc % kSBufs) * 128, qd + off, kd + off, idesc_s,
                      kk > 0 ? 1u : 0u);
          else
            mma_ss(tmem + kTmemS + (kc % kSBufs) * 128, qd + off, kd + off, idesc_s,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars->k_empty[st]));
        mma_commit(smem_u32(&bars->s_full[kc % kSBufs]));
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
template <int D, bool IN8>
__device__ void run_mma_pv(const FwdParams& p, Bars* bars, uint32_t tmem, uint32_t smem_base,
                           volatile int* abort_flag) {
  using C = Cfg<D, IN8>;
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
      // V(vc) loaded (fp16 P V: and converted to fp16 by the epilogue warps,
      // unless V was converted before the launch)
      if (!wait_warp(smem_u32((C::kF16PV && !p.v_pre) ? &bars->v_conv[st] : &bars->v_full[st]),
                     (uint32_t)(vc / C::kVStages) & 1u, abort_flag, p.status, lim)) {
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
        mma_commit(smem_u32(&bars->pv_done[vc % kSBufs]));
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

// 2^x for a pair of fp32 x on the FMA and integer pipes, without the MUFU
// unit: Cody-Waite range reduction x = n + f with n = round(x)
// and f in [-1/2, 1/2] (rounding by adding 1.5 * 2^23), 2^f by a cubic fitted
// for least maximum relative error on [-1/2, 1/2] (Lawson's iteration; error
// <= 7.5e-5, far below the bf16 rounding of P), and 2^n added to the exponent
// field (the integer n sits in the low bits of x + 1.5 * 2^23).  x is clamped
// to [-126, 126]: below, 2^x is negligible next to the row's largest term
// (>= 2^-8; a masked score, -inf, gives 2^-126 instead of 0, which no fp32
// sum of such terms can register); above, the result stays huge, so the
// caller's block-sum test still sees it.
// Measured on GB300: every split tried (6 to 16 of 32 pairs) is slower than
// none (the exponential phase is not bound by the MUFU rate there), so the
// default is 0 and the polynomial path is a tuning option.
#ifndef BSATTN_EXP2_POLY_PAIRS
#define BSATTN_EXP2_POLY_PAIRS 0
#endif
constexpr int kPolyPairs = BSATTN_EXP2_POLY_PAIRS;  // of each 32 pairs per half row
constexpr float kExp2C0 = 0.99992808f, kExp2C1 = 0.69326102f, kExp2C2 = 0.24261111f,
                kExp2C3 = 0.05517149f;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ void exp2_poly_pair(uint64_t x2, float& y0, float& y1) {
  float x0, x1;
  f2_unpack(x2, x0, x1);
  x0 = fminf(fmaxf(x0, -126.0f), 126.0f);
  x1 = fminf(fmaxf(x1, -126.0f), 126.0f);
  const uint64_t xc = f2_pack(x0, x1);
  const uint64_t t = f2_add(xc, f2_pack(kRoundMagic, kRoundMagic));   // magic + round(x)
  const uint64_t nf = f2_add(t, f2_pack(-kRoundMagic, -kRoundMagic));  // round(x), exact
  const uint64_t f = f2_fma(nf, f2_pack(-1.0f, -1.0f), xc);            // x - round(x), exact
  uint64_t p = f2_fma(f2_pack(kExp2C3, kExp2C3), f, f2_pack(kExp2C2, kExp2C2));
  p = f2_fma(p, f, f2_pack(kExp2C1, kExp2C1));
  p = f2_fma(p, f, f2_pack(kExp2C0, kExp2C0));
  float p0, p1, t0, t1;
  f2_unpack(p, p0, p1);
  f2_unpack(t, t0, t1);
  y0 = __uint_as_float(__float_as_uint(p0) + (__float_as_uint(t0) << 23));
  y1 = __uint_as_float(__float_as_uint(p1) + (__float_as_uint(t1) << 23));
}

// Probabilities of one 64-column half row: p = 2^(s*sl - m), rounded to bf16
// (F16: fp16) pairs into pr[] (the A operand of the PV product).  POLY of the 32 pairs,
// spread evenly, take their exponentials from exp2_poly_pair, the others from
// the MUFU unit.  Accumulates the row sum
// of the fp32 p (for the LSE) in a2, two partial sums in one f32x2 pair, and,
// when ROUNDED, r32 of the bf16-rounded p that multiply V (the O denominator,
// so that the weights on V sum to one even when a single key dominates a
// row), again in two partial sums.  sl2 = (sl, sl), nm2 = (-m, -m).
template <bool ROUNDED, int POLY, bool F16>
__device__ __forceinline__ void softmax_exp64(const uint32_t* sr, uint32_t* pr, uint64_t sl2,
                                              uint64_t nm2, uint64_t& a2, float (&r32)[2]) {
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    const uint64_t x2 =
        f2_fma(f2_pack(__uint_as_float(sr[2 * q]), __uint_as_float(sr[2 * q + 1])), sl2, nm2);
    float p0, p1;
    if (((q + 1) * POLY) / 32 != (q * POLY) / 32) {
      exp2_poly_pair(x2, p0, p1);
    } else {
      float x0, x1;
      f2_unpack(x2, x0, x1);
      p0 = ex2_approx(x0);
      p1 = ex2_approx(x1);
    }
    pr[q] = F16 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
    a2 = f2_add(a2, f2_pack(p0, p1));
    if (ROUNDED) {
      if (F16)
        add_f16x2_f32(r32[0], r32[1], pr[q]);
      else
        add_bf16x2_f32(r32[0], r32[1], pr[q]);
    }
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

template <int D, bool OUT_F32, bool IN8, bool KB64>
__device__ void run_softmax(const FwdParams& p, Bars* bars, uint32_t tmem,
                            volatile int* abort_flag) {
  using C = Cfg<D, IN8>;
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
  int sb = 0;             // g % kSBufs: S buffer (and P barrier) of block g
  uint32_t sph = 0;       // (g / kSBufs) & 1: phase of s_full[sb] for block g
  int ntile = 0;          // tiles handed to the epilogue warps
  for (;;) {
    const int e = tq_cnt & 1;
    const uint32_t ph = (uint32_t)(tq_cnt >> 1) & 1u;
    if (!wait_warp(smem_u32(&bars->tq_full[e]), ph, abort_flag, p.status, lim)) return;
    const volatile TileInfo* slot = &bars->tq[e];
    const int t = slot->t;
    const int bh = slot->bh;
    const int qb = slot->qb;
    const int n = slot->n;
    const int diag_last = slot->diag;
    const int n64 = slot->n64;
    const int last_a = slot->last2[0], last_b = slot->last2[1];
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars->tq_empty[e]));
    ++tq_cnt;
    if (t < 0) return;

    float m = __uint_as_float(kNegInf);  // running max of scale*log2(e)*score (lazy)
    uint64_t a2 = 0;            // partial sums of this half row: fp32 p (an f32x2 pair)
    float r32[2] = {0.f, 0.f};  // and bf16-rounded p
    for (int jb = 0; jb < n; ++jb, ++g) {
      // S(g) ready
      if (!wait_warp(smem_u32(&bars->s_full[sb]), sph, abort_flag, p.status, lim)) return;
      tc_fence_after();
      const uint32_t tS = tmem + kTmemS + sb * 128 + lane_off;  // S buffer of this block
      // Keys c (0..63) of this thread's half of the block with c > klim are
      // masked: the causal diagonal of 128-key blocks (key 64 ch + c allowed
      // for query row r iff it is <= r); with 64-key blocks in pairs, the
      // missing second half of an odd tail (all masked) and, under causal,
      // the halves among the tile's last two entries that reach past the
      // tile's first query (key 64 kb + c allowed iff <= 128 qb + r).
      const bool diag = diag_last && jb == n - 1;  // warp-uniform
      int klim = diag ? r - 64 * ch : 63;
      bool masked = diag;
      if constexpr (KB64) {
        const int e64 = 2 * jb + ch;
        if (e64 >= n64) {
          klim = -1;
        } else if (p.causal && e64 >= n64 - 2) {
          const int kb = e64 == n64 - 1 ? last_b : last_a;
          klim = min(63, qb * kBlock + r - kb * 64);
        }
        masked = __any_sync(0xffffffffu, klim < 63);
      }
      uint32_t pr[32];
      uint64_t b2 = 0;  // this block's sums
      float br32[2] = {0.f, 0.f};
      // This thread's 64 scores of the block, masked as above.
      auto load_scores = [&](uint32_t (&sr)[64]) {
        tmem_ld16x2_32<64>(tS + 0, sr + 0);
        tmem_ld16x2_32<64>(tS + 32, sr + 32);
        tmem_wait_ld();
        reg_fence(sr, 64);
        if (masked) {
#pragma unroll
          for (int c = 0; c < 64; ++c) sr[c] = (c > klim) ? kNegInf : sr[c];
        }
      };
      // Masked scores need exact zeros, which the MUFU exponential gives.
      auto exp_pass = [&](const uint32_t (&sr)[64], float mref) {
        if constexpr (kPolyPairs == 0) {
          softmax_exp64<!C::kOnes, 0, C::kF16PV>(sr, pr, sl2, f2_pack(-mref, -mref), b2, br32);
        } else {
          if (masked)
            softmax_exp64<!C::kOnes, 0, C::kF16PV>(sr, pr, sl2, f2_pack(-mref, -mref), b2, br32);
          else
            softmax_exp64<!C::kOnes, kPolyPairs, C::kF16PV>(sr, pr, sl2, f2_pack(-mref, -mref),
                                                            b2, br32);
        }
      };
      // After a tile's first block the probabilities are formed against the
      // current reference m without a max pass (any common reference gives
      // the exact softmax).  Only when a half row's sum over the block shows that
      // its scores rose far above m (C::kGrowSum) -- or on the tile's first
      // block, where m = -inf -- is the block redone with its max, by the
      // lazy rule, as the new reference.  The redo reads the scores again
      // from tensor memory (P has not overwritten them yet), so the scores
      // need not stay in registers past the first pass.
      // A row with no allowed key so far (m = -inf: possible with 64-key
      // blocks under causal) always takes the redo path, with reference 0.
      bool redo = jb == 0 || (KB64 && __any_sync(0xffffffffu, m == __uint_as_float(kNegInf)));
      if (!redo) {
        uint32_t sr[64];
        load_scores(sr);
        exp_pass(sr, m);
        // Each half row is tested on its own sum (no exchange with the other
        // half on this path): a P element never exceeds its half's sum, so
        // the bound that C::kGrowSum keeps on P holds all the same.
        float b0, b1;
        f2_unpack(b2, b0, b1);
        redo = __any_sync(0xffffffffu, !(b0 + b1 <= C::kGrowSum));  // also catches inf / NaN
      }
      bool need = false;     // this thread's row takes a new reference max
      bool rescale = false;  // some row of the warp does (set on the redo path only)
      float f = 1.f;
      if (redo) {
        uint32_t sr[64];
        load_scores(sr);
        float mx = row_max64(sr);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // the other half of the row
        const float xm = mx * sl;
        need = xm > m + kTau;  // always true on the first block (m = -inf)
        rescale = __any_sync(0xffffffffu, need);
        if (need) {
          f = ex2_approx(m - xm);  // 0 when m = -inf
          m = xm;
          a2 = f2_mul(a2, f2_pack(f, f));
          r32[0] *= f;
          r32[1] *= f;
        }
        b2 = 0;
        br32[0] = br32[1] = 0.f;
        exp_pass(sr, (KB64 && m == __uint_as_float(kNegInf)) ? 0.f : m);
      }
      a2 = f2_add(a2, b2);
      r32[0] += br32[0];
      r32[1] += br32[1];
      tmem_st16x2_32<64>(tS, pr);  // P over the scores just read (keys 0..63 -> cols 0..31, 64..127 -> 64..95)

      // O rescale (this thread's columns) when a row's max moved: first wait
      // until PV(g-1) has landed in O (PV(g) is not issued before P(g)).
      if (jb > 0 && rescale) {
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
      if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[sb]));
      if (++sb == kSBufs) {
        sb = 0;
        sph ^= 1u;
      }
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
      if (ch == 0) bars->inv_l[r] = l > 0.f ? 1.0f / l : 0.f;  // no allowed key: O = 0
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
// One tile's O, this thread's row: read O from tensor memory 16 columns at a
// time, divide by the row's rounded sum and store it.  Each thread writes its
// own row: 32-byte stores (one full sector each) when the output is 32-byte
// aligned, else 16-byte ones.
template <int D, bool OUT_F32>
__device__ __forceinline__ void write_o_row(const FwdParams& p, const Bars* bars, uint32_t tO,
                                            int r, int t) {
  using C = Cfg<D>;
  float inv_l = 0.f;
  if constexpr (!C::kOnes) inv_l = bars->inv_l[r];
  if constexpr (C::kOnes) {  // rounded row sum accumulated by the tensor core in column D
    uint32_t rs[1];
    tmem_ld32_1(tO + D, rs);
    tmem_wait_ld();
    reg_fence(rs, 1);
    const float l = __uint_as_float(rs[0]);
    inv_l = l > 0.f ? 1.0f / l : 0.f;  // no allowed key in the row: O = 0
  }
  inv_l *= p.v_scale;  // 1, or the scale of e4m3 V (attention is linear in V)
  const int bh = t / p.nb;
  const size_t row = (size_t)bh * p.S + (size_t)(t - bh * p.nb) * kBlock + r;
  const bool wide = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 16) {
    uint32_t orr[16];
    tmem_ld32_16(tO + c0, orr);
    tmem_wait_ld();
    reg_fence(orr, 16);
    if constexpr (OUT_F32) {
      float* dst = reinterpret_cast<float*>(p.out) + row * D + c0;
#pragma unroll
      for (int i = 0; i < 16; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * inv_l);
      if (wide) {
        st_global_v8(dst, *reinterpret_cast<const uint32_t(*)[8]>(orr));
        st_global_v8(dst + 8, *reinterpret_cast<const uint32_t(*)[8]>(orr + 8));
      } else {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          st_global_v4(dst + i, orr[i], orr[i + 1], orr[i + 2], orr[i + 3]);
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
}

// For each tile the softmax hands over: wait for its last PV, write O (one
// thread per query row = TMEM lane); then release O for the next tile's first
// PV.  Only the leader warp takes tiles and waits (sleeping between tests);
// it passes the tile on through shared memory and a named barrier, where the
// other three warps wait without issuing.  The leader reaches the barrier on
// every path, with a negative tile to stop, so the four warps always leave
// together.
template <int D, bool OUT_F32, bool IN8>
__device__ void run_epilogue(const FwdParams& p, Bars* bars, uint32_t tmem,
                             volatile int* abort_flag) {
  using C = Cfg<D, IN8>;
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
    write_o_row<D, OUT_F32>(p, bars, tO, r, t);
    tc_fence_before();
    __syncwarp();  // every lane's reads of O are complete
    if (lane == 0) mbar_arrive(smem_u32(&bars->o_free));
    ++ntile;
  }
}

// This warp's quarter of one V tile (128 keys x 64 columns, one 16 KB
// 128-byte-swizzled box) converted from bf16 to fp16 in place: the layout
// does not change, element by element.  bf16 converts to fp16 exactly for
// 2^-14 <= |v| <= 65504 (below, to fp16's subnormals, off by < 2^-25);
// `rmax` collects, per 16-bit half, the largest fp16 exponent field seen, so
// that an infinity or NaN (a |v| too large for fp16, or a non-finite v) can
// be reported.
__device__ __forceinline__ void convert_v_quarter(uint32_t stage, int wq, int lane,
                                                  uint32_t& rmax) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = stage + (uint32_t)((wq * 256 + i * 32 + lane) * 16);
    uint32_t w[4];
    ld_shared_v4(a, w);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      w[j] = pack_f16x2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
      rmax = max_u16x2(rmax, w[j] & 0x7C007C00u);
    }
    st_shared_v4(a, w[0], w[1], w[2], w[3]);
  }
}

// This warp's quarter of one e4m3 V tile (128 keys x 128 columns, one 16 KB
// box of 128-byte rows, 128-byte swizzled as TMA wrote it) converted to the
// fp16 V tile of the P V product (two 64-column boxes `group` bytes apart,
// 128-byte swizzled as the MMA's descriptor reads them).  e4m3 converts to
// fp16 exactly.  Two 16-byte chunks are loaded at once (their latencies
// overlap), then each is converted and stored (measured on the e4m3 random
// 10 % workload: one chunk at a time 1077 TFLOP/s, two 1338, four 1309,
// eight 1326).  `nan8` collects, per byte,
// bit 7 set for an e4m3 NaN (0x7F / 0xFF: the 7 low bits all ones, so that
// adding 1 to them carries into bit 7).
__device__ __forceinline__ void convert_v8_quarter(uint32_t src, uint32_t dst, uint32_t group,
                                                   int wq, int lane, uint32_t& nan8) {
#pragma unroll 1
  for (int i0 = 0; i0 < 8; i0 += 2) {
    uint32_t w[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = wq * 256 + (i0 + j) * 32 + lane;
      const uint32_t r = (uint32_t)idx >> 3, c = (uint32_t)idx & 7u;  // key row, 16-byte chunk
      ld_shared_v4(src + r * 128u + ((c ^ (r & 7u)) << 4), w[j]);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int idx = wq * 256 + (i0 + j) * 32 + lane;
      const uint32_t r = (uint32_t)idx >> 3, c = (uint32_t)idx & 7u;
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        nan8 |= ((w[j][e] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
        e4m3x4_to_f16x4(w[j][e], h[2 * e], h[2 * e + 1]);
      }
      // columns 16c .. 16c+15 -> box c / 4, its 16-byte chunks 2 (c % 4) and 2 (c % 4) + 1
      const uint32_t box = dst + (c >> 2) * group + r * 128u;
      const uint32_t j0 = 2u * (c & 3u);
      st_shared_v4(box + ((j0 ^ (r & 7u)) << 4), h[0], h[1], h[2], h[3]);
      st_shared_v4(box + (((j0 + 1u) ^ (r & 7u)) << 4), h[4], h[5], h[6], h[7]);
    }
  }
}

// The epilogue warps when P V runs in fp16 (D = 64, or e4m3 inputs) and V was
// not converted before the launch: besides
// writing each tile's O (as run_epilogue does), they convert every V tile of
// the CTA's block stream to fp16 after its load, each warp a quarter, and
// announce it on v_conv (four arrivals): in place at D = 64; with e4m3 inputs
// from the staging ring into the fp16 ring, once the fp16 stage's previous
// tile has been multiplied (its PV complete), freeing the staging stage.  Blocks are converted in stream order.  Before a
// tile's O is written, all of the tile's V tiles are converted (its PVs need
// them); while waiting for the tile's last PV, a warp also converts the next
// tiles' V tiles as soon as they are loaded, so the next tile's first PV does
// not wait for the conversion after O is released.  Each warp decides alone
// when its rows of O can be written (the softmax's hand-over and the last PV
// are both complete), so no barrier joins them there.
template <int D, bool OUT_F32, bool IN8>
__device__ void run_epilogue_convert(const FwdParams& p, Bars* bars, uint32_t tmem,
                                     uint32_t smem_base, volatile int* abort_flag) {
  using C = Cfg<D, IN8>;
  static_assert(C::kBoxes == 1 || C::kIn8, "one 64-column box per bf16 V tile");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;  // query row of the tile = TMEM lane
  const uint32_t tO = tmem + kTmemO + ((uint32_t)(wq * 32) << 16);
  const uint64_t lim = p.timeout_ns;
  int tqc = 0;    // (leader) tiles taken
  int known = 0;  // blocks of the stream in the tiles seen so far
  int cg = 0;     // blocks whose V this warp has converted
  int ntile = 0;  // tiles taken
  uint32_t rmax = 0;  // D = 64: per half, the largest fp16 exponent field converted
  uint32_t nan8 = 0;  // e4m3: NaN bytes seen
  bool ok = true;     // false once a wait of this warp failed
  auto convert_next = [&]() {
    const int st = cg % C::kVStages;
    if constexpr (C::kIn8) {
      const int s8 = cg % C::kV8Stages;
      convert_v8_quarter(smem_base + C::kV8Off + s8 * C::kBoxBytes,
                         smem_base + C::kVOff + st * C::kBoxBytes, C::kVGroup, wq, lane, nan8);
      fence_proxy_async_smem();  // the tensor core reads what these generic stores wrote
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars->v_conv[st]));
        mbar_arrive(smem_u32(&bars->v8_empty[s8]));
      }
    } else {
      convert_v_quarter(smem_base + C::kVOff + st * C::kBoxBytes, wq, lane, rmax);
      fence_proxy_async_smem();  // the tensor core reads what these generic stores wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->v_conv[st]));
    }
    ++cg;
  };
  // V(g) can be converted: loaded (e4m3: staged, and the fp16 stage's
  // previous tile multiplied).  Non-blocking, warp-uniform.
  auto v_loaded = [&](int g) -> bool {
    bool rdy = false;
    if (lane == 0) {
      if constexpr (C::kIn8)
        rdy = mbar_test_wait(smem_u32(&bars->v8_full[g % C::kV8Stages]),
                             (uint32_t)(g / C::kV8Stages) & 1u) &&
              (g < C::kVStages ||
               mbar_test_wait(smem_u32(&bars->v_empty[(g - C::kVStages) % C::kVStages]),
                              (uint32_t)((g - C::kVStages) / C::kVStages) & 1u));
      else
        rdy = mbar_test_wait(smem_u32(&bars->v_full[g % C::kVStages]),
                             (uint32_t)(g / C::kVStages) & 1u);
    }
    return __shfl_sync(0xffffffffu, rdy, 0);
  };
  // The same, waiting (bounded) until it holds.
  auto wait_v = [&](int g) -> bool {
    if constexpr (C::kIn8) {
      if (!wait_warp(smem_u32(&bars->v8_full[g % C::kV8Stages]), (uint32_t)(g / C::kV8Stages) & 1u,
                     abort_flag, p.status, lim))
        return false;
      return g < C::kVStages ||
             wait_warp(smem_u32(&bars->v_empty[(g - C::kVStages) % C::kVStages]),
                       (uint32_t)((g - C::kVStages) / C::kVStages) & 1u, abort_flag, p.status, lim);
    } else {
      return wait_warp(smem_u32(&bars->v_full[g % C::kVStages]), (uint32_t)(g / C::kVStages) & 1u,
                       abort_flag, p.status, lim);
    }
  };
  // Every warp reaches the named barrier once per tile taken, on every path:
  // a warp whose wait failed (abort flag raised) skips the rest of each
  // iteration, and the leader's next take_tile then fails too and publishes
  // the stop value, so the four warps always leave together.
  for (;;) {
    if (warp == kWarpEpi0) {
      int t = 0, r0 = 0, n = 0, col = 0;
      const bool got = ok && take_tile(bars, tqc, p, abort_flag, t, r0, n, col, kSleepNs);
      ++tqc;
      if (lane == 0) {
        bars->epi_tile[ntile & 1] = got ? t : -1;
        bars->epi_n[ntile & 1] = n;
      }
    }
    named_bar_sync(kEpiBarrier, kEpiWarps * 32);
    const int t = *reinterpret_cast<volatile int*>(&bars->epi_tile[ntile & 1]);
    const int n = *reinterpret_cast<volatile int*>(&bars->epi_n[ntile & 1]);
    ++ntile;
    if (t < 0) break;
    if (!ok) continue;
    known += n;
    // the tile's V tiles (those not converted ahead already)
    while (cg < known) {
      if (!wait_v(cg)) {
        ok = false;
        break;
      }
      convert_next();
    }
    if (!ok) continue;
    // wait for the softmax's hand-over and the tile's last PV; meanwhile
    // convert the following V tiles as they arrive
    const int gl = known - 1;
    const uint32_t tpar = (uint32_t)(ntile - 1) & 1u;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      bool rdy = false;
      if (lane == 0)
        rdy = mbar_test_wait(smem_u32(&bars->epi_full), tpar) &&
              mbar_test_wait(smem_u32(&bars->v_empty[gl % C::kVStages]),
                             (uint32_t)(gl / C::kVStages) & 1u);
      if (__shfl_sync(0xffffffffu, rdy, 0)) break;
      if (v_loaded(cg)) {
        convert_next();
        continue;
      }
      if (*abort_flag || globaltimer_ns() - t0 > lim) {
        if (lane == 0 && !*abort_flag) {
          *abort_flag = 1;
          atomicOr(p.status, kStatusTimeout);
        }
        ok = false;
        break;
      }
      __nanosleep(kSleepNs);
    }
    __syncwarp();
    if (!ok) continue;
    tc_fence_after();
    write_o_row<D, OUT_F32>(p, bars, tO, r, t);
    tc_fence_before();
    __syncwarp();  // every lane's reads of O are complete
    if (lane == 0) mbar_arrive(smem_u32(&bars->o_free));
  }
  // A V entry that is not finite in fp16 (|v| > 65504, or inf / NaN) was converted.
  const bool bad = (rmax & 0xFFFFu) == 0x7C00u || (rmax >> 16) == 0x7C00u || nan8 != 0u;
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kStatusRange);
}

template <int D, bool OUT_F32, bool IN8, bool KB64>
__global__ void __launch_bounds__(kThreads, 1)
    bsattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<D, IN8>;
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
      mbar_init(smem_u32(&bars->v_conv[i]), kEpiWarps);  // one arrival per epilogue warp
    }
    for (int i = 0; i < C::kV8Stages; ++i) {
      mbar_init(smem_u32(&bars->v8_full[i]), 1);
      mbar_init(smem_u32(&bars->v8_empty[i]), kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->q_full[i]), 1);
      mbar_init(smem_u32(&bars->q_empty[i]), 1);
    }
    // the softmax warps arrive once per warp (elected lane, after __syncwarp)
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(smem_u32(&bars->p_full[i]), kSoftmaxWarps);
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
    }
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
  if constexpr (C::kOnes) {  // 1.0 tiles read by the PV MMA (generic-proxy writes, then a proxy fence)
    constexpr uint32_t one2 = C::kF16PV ? 0x3C003C00u : 0x3F803F80u;  // fp16 / bf16 pairs of 1.0
    uint4* ones = reinterpret_cast<uint4*>(smem_raw + (base - raw) + C::kOnesOff);
    for (int i = threadIdx.x; i < C::kVStages * C::kBoxBytes / 16; i += kThreads)
      ones[i] = make_uint4(one2, one2, one2, one2);
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
      run_producer<D, IN8, KB64>(&tm_q, &tm_k, &tm_v, p, bars, base, abort_flag);
    else if (warp == kWarpMmaS)
      run_mma_s<D, IN8>(p, bars, tmem, base, abort_flag);
    else if (warp == kWarpMmaPV)
      run_mma_pv<D, IN8>(p, bars, tmem, base, abort_flag);
    else if (warp >= kWarpEpi0) {
      if constexpr (C::kF16PV) {
        if (!p.v_pre)  // V tiles arrive in bf16 or e4m3: these warps convert them
          run_epilogue_convert<D, OUT_F32, IN8>(p, bars, tmem, base, abort_flag);
        else
          run_epilogue<D, OUT_F32, IN8>(p, bars, tmem, abort_flag);
      } else {
        run_epilogue<D, OUT_F32, IN8>(p, bars, tmem, abort_flag);
      }
    }
    else if (warp == kWarpSched)
      run_scheduler<D, IN8, KB64>(&tm_q, p, bars, base, abort_flag);
  } else {
    regs_inc<kRegsSoftmax>();
    run_softmax<D, OUT_F32, IN8, KB64>(p, bars, tmem, abort_flag);
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

template <int D, bool OUT_F32, bool IN8, bool KB64>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int grid, cudaStream_t stream) {
  const size_t smem = Cfg<D, IN8>::kSmem + 1024;
  // The shared-memory opt-in is set once per device (it costs host time on
  // every call otherwise); a failed attempt is retried on the next call.
  static std::atomic<bool> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(bsattn_fwd_kernel<D, OUT_F32, IN8, KB64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
  }
  bsattn_fwd_kernel<D, OUT_F32, IN8, KB64><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

// The fp16 copy of V that head_dim 64's P V product reads (FwdParams::v_pre):
// 8 values per thread and step, 16-byte loads and stores, grid-stride.  bf16
// converts to fp16 exactly for 2^-14 <= |v| <= 65504 (below, to fp16's
// subnormals, off by < 2^-25); a larger or non-finite value becomes an fp16
// infinity or NaN and raises kStatusRange, as the in-kernel conversion does.
__global__ void __launch_bounds__(256) v16_convert_kernel(const uint4* __restrict__ v,
                                                          uint4* __restrict__ v16, long long n16,
                                                          int* status) {
  uint32_t emax = 0;  // per 16-bit half, the largest fp16 exponent field written
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 w = __ldg(v + i);
    uint32_t o[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[j] = pack_f16x2(__uint_as_float(o[j] << 16), __uint_as_float(o[j] & 0xFFFF0000u));
      emax = max_u16x2(emax, o[j] & 0x7C007C00u);
    }
    v16[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  const bool bad = (emax & 0xFFFFu) == 0x7C00u || (emax >> 16) == 0x7C00u;
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusRange);
}

// The same for e4m3 V (the FP8 forward): 16 values per thread and step, each
// converted exactly; an e4m3 NaN (0x7F / 0xFF) becomes an fp16 NaN and raises
// kStatusRange, as the in-kernel conversion does.
__global__ void __launch_bounds__(256) v16_convert_e4m3_kernel(const uint4* __restrict__ v8,
                                                               uint4* __restrict__ v16,
                                                               long long n16, int* status) {
  uint32_t emax = 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 w = __ldg(v8 + i);
    const uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      e4m3x4_to_f16x4(in[j], o[2 * j], o[2 * j + 1]);
      emax = max_u16x2(emax, o[2 * j] & 0x7C007C00u);
      emax = max_u16x2(emax, o[2 * j + 1] & 0x7C007C00u);
    }
    v16[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
    v16[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  const bool bad = (emax & 0xFFFFu) == 0x7C00u || (emax >> 16) == 0x7C00u;
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusRange);
}

}  // namespace

cudaError_t launch_v16_convert_e4m3(const void* v8, void* v16, long long n, int* status,
                                    int grid, cudaStream_t stream) {
  const long long n16 = n / 16;
  if (n16 <= 0) return cudaSuccess;
  const long long blocks = (n16 + 255) / 256;
  const int g = (int)(blocks < 8LL * grid ? blocks : 8LL * grid);  // grid-stride beyond that
  v16_convert_e4m3_kernel<<<g, 256, 0, stream>>>(static_cast<const uint4*>(v8),
                                                 static_cast<uint4*>(v16), n16, status);
  return cudaGetLastError();
}

cudaError_t launch_v16_convert(const void* v, void* v16, long long n, int* status, int grid,
                               cudaStream_t stream) {
  const long long n16 = n / 8;
  if (n16 <= 0) return cudaSuccess;
  const long long blocks = (n16 + 255) / 256;
  const int g = (int)(blocks < 8LL * grid ? blocks : 8LL * grid);  // grid-stride beyond that
  v16_convert_kernel<<<g, 256, 0, stream>>>(static_cast<const uint4*>(v), static_cast<uint4*>(v16),
                                          n16, status);
  return cudaGetLastError();
}

size_t fwd_smem_bytes(int D) {
  return D == 64 ? Cfg<64>::kSmem + 1024 : Cfg<128>::kSmem + 1024;
}

// The kernel is compiled per head_dim, output type, input type and key-block
// size (64-key blocks add per-block work to the softmax and the producer that
// 128-key plans should not pay).
template <int D, bool IN8, bool KB64>
cudaError_t launch_out(bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t stream) {
  return out_f32 ? launch_one<D, true, IN8, KB64>(tq, tk, tv, p, grid, stream)
                 : launch_one<D, false, IN8, KB64>(tq, tk, tv, p, grid, stream);
}

cudaError_t launch_fwd(int D, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t stream,
                       bool in8) {
  const bool kb64 = p.kdiv == 2;
  if (in8) {
    if (D != 128) return cudaErrorInvalidValue;
    return kb64 ? launch_out<128, true, true>(out_f32, tq, tk, tv, p, grid, stream)
                : launch_out<128, true, false>(out_f32, tq, tk, tv, p, grid, stream);
  }
  if (D == 64)
    return kb64 ? launch_out<64, false, true>(out_f32, tq, tk, tv, p, grid, stream)
                : launch_out<64, false, false>(out_f32, tq, tk, tv, p, grid, stream);
  return kb64 ? launch_out<128, false, true>(out_f32, tq, tk, tv, p, grid, stream)
              : launch_out<128, false, false>(out_f32, tq, tk, tv, p, grid, stream);
}

cudaError_t launch_selftest_wait(unsigned long long timeout_ns, int* d_status,
                                 cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(timeout_ns, d_status);
  return cudaGetLastError();
}

}  // namespace bsattn
