/*
 * bsattn.h -- C ABI of the block-sparse flash-attention forward pass for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (per batch b, head h, query row i, with S keys):
 *
 *   allowed(j) = M[b][h][i/128][j/128] != 0  and  (not causal or j <= i)
 *   s_j        = scale * <Q[b][h][i], K[b][h][j]>  if allowed(j), else -inf
 *   O[b][h][i] = sum_j softmax(s)_j * V[b][h][j]
 *   LSE[b][h][i] = ln sum_j exp(s_j)            (natural log)
 *   rows with no allowed key: O = 0, LSE = -inf
 *
 * Defined by "Writing Pallas Kernels for JAX: Stepping Outside the XLA Safety
 * Net": section "Designing the Block Specification" (Q of shape (batch,
 * seq_len, head_dim) handled in 128-token query blocks; a block mask fed per
 * (query block, key block) pair) and section "Writing the Kernel Logic: Load,
 * Compute, Store" (scores q.k * 1/sqrt(head_dim), masked scores set to -inf,
 * softmax over keys, product with V).  The softmax is exact over all live
 * keys of a row, computed blockwise the flash-attention way ("Pallas-Triton
 * kernels and kernel auto-tuning", section "Flash Attention": exact,
 * cache-friendly attention).  Dead blocks are never read: the grid walks only
 * the live (query block, key block) pairs, which is the point of the block
 * mask in "Writing the Kernel Logic" (only the small 128x128 block is ever
 * materialised).  The causal flag, LSE and the O = 0 / LSE = -inf rule for
 * fully masked rows are this library's definitions; the pages do not state
 * them.
 *
 * Conventions for every entry point:
 *  - Pointers named d_* and every tensor argument are DEVICE pointers (CUDA
 *    global memory on the current device); the caller owns them.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Every function returns a bsattn_status and never aborts the process.
 *    All argument checks run on the host before any launch; on a non-OK
 *    return nothing has been launched.
 *  - Layouts: Q, K, V, O are [B][H][S][D] row-major and contiguous; LSE is
 *    [B][H][S] fp32; the mask is uint8 [B][H][S/128][S/128], nonzero = live.
 *  - Supported: D in {64, 128}; S a positive multiple of 128 with S/128 <= 4096;
 *    B*H*S < 2^31; Q, K, V bf16; O bf16 (default) or fp32 (BSATTN_OUT_F32).
 *  - Arithmetic: S = Q K^T on the tensor core in bf16 with fp32 accumulation;
 *    the probabilities P and the product P V in bf16 at D = 128, in fp16 at
 *    D = 64 (V converted exactly from bf16; |V| above 65504, or a non-finite
 *    V, is reported as BSATTN_ERR_RANGE), fp32 accumulation; softmax in fp32.
 */
#ifndef BSATTN_H_
#define BSATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BSATTN_OK = 0,
  BSATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, plan mismatch */
  BSATTN_ERR_UNSUPPORTED = 2,  /* valid request outside the supported set (e.g. D=96) */
  BSATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  BSATTN_ERR_OOM = 4,          /* device or host allocation failed */
  BSATTN_ERR_TIMEOUT = 5,      /* a kernel gave up waiting (bounded wait ran out) */
  BSATTN_ERR_INTERNAL = 6,     /* a kernel detected an inconsistent state */
  BSATTN_ERR_SCRATCH_LIMIT = 7, /* problem too large for bsattn_fwd_noalloc's fixed scratch */
  BSATTN_ERR_RANGE = 8         /* an input value outside what the kernel's arithmetic holds:
                                  at D = 64 the forward pass multiplies P by V in fp16, so
                                  every V entry must be finite with |v| <= 65504; reported
                                  after the launch, by the status calls */
} bsattn_status;

/* Opaque plan: the per-query-tile list of live key blocks and the tile order. */
typedef struct bsattn_plan_s* bsattn_plan_t;

/* Plan flags. */
enum {
  BSATTN_CAUSAL = 1u,   /* also require key j <= query i (element level, inclusive) */
  BSATTN_OUT_F32 = 2u,  /* bsattn_fwd writes O as fp32 instead of bf16 */
  BSATTN_MASK_SHARED_HEADS = 4u, /* bsattn_plan only: d_mask is [B][1][S/128][S/128],
                                    one mask per batch entry for all its H heads */
  BSATTN_KEY_BLOCK_64 = 8u       /* bsattn_plan only: key blocks of 64 keys; d_mask is
                                    [B][H][S/128][S/64] (one entry per 128-query x
                                    64-key block); forward pass only */
};

/*
 * bsattn_plan -- build the plan for one block mask.
 *
 * The plan is the compressed-sparse-row list of live key blocks of every
 * query tile (row r = (b*H + h)*(S/128) + qb; col_idx ascending; under
 * BSATTN_CAUSAL only kb <= qb is kept) and a schedule: the non-empty tiles
 * in chunks of C = max(1, 768 / (S/128)) consecutive heads (b*H + h order),
 * most live blocks first inside a chunk (ties: head, then qb ascending),
 * except that a tile of chunk k > 0 with more live blocks than
 * (live blocks of chunk k) / (2 * number of SMs of the current device) is
 * listed in chunk k-1; and the list of empty tiles (head by head, qb
 * ascending).  Built on the device by kernels on `stream`.  This is the
 * only call that synchronises: it waits for `stream` once to learn the number
 * of live blocks before allocating.
 *
 *   d_mask     device uint8 [B][H][S/128][S/128] ([B][1][S/128][S/128] with
 *              BSATTN_MASK_SHARED_HEADS); read during the call only.
 *   B, H, S    sizes; S % 128 == 0.
 *   flags      BSATTN_CAUSAL | BSATTN_OUT_F32 | BSATTN_MASK_SHARED_HEADS.
 *   stream     cudaStream_t.
 *   out_plan   receives the handle; the library owns its device memory until
 *              bsattn_plan_free.  Unchanged on error.
 * Errors: INVALID_ARG (null, sizes), UNSUPPORTED (S/128 > 4096), OOM, CUDA.
 */
bsattn_status bsattn_plan(const uint8_t* d_mask, int B, int H, int S, unsigned flags,
                          void* stream, bsattn_plan_t* out_plan);

/* Device pointers to the plan's CSR (row_ptr: B*H*S/128 + 1 int32, col_idx:
   nnz int32) and its size; valid until bsattn_plan_free.  For tests/tools. */
bsattn_status bsattn_plan_csr(bsattn_plan_t plan, const int32_t** d_row_ptr,
                              const int32_t** d_col_idx, int64_t* nnz);

/* Device pointers to the plan's transposed list (col_ptr: B*H*S/128 + 1
   int32 indexed by key block (b*H + h)*nb + kb; row_idx: nnz int32, the
   ascending live query blocks of each key block) and its size; valid until
   bsattn_plan_free.  For tests/tools. */
bsattn_status bsattn_plan_csc(bsattn_plan_t plan, const int32_t** d_col_ptr,
                              const int32_t** d_row_idx, int64_t* nnz);

/* Device pointers to the schedule: non-empty tile ids in processing order
   (n_live int32) and empty tile ids (n_empty int32).  For tests/tools. */
bsattn_status bsattn_plan_schedule(bsattn_plan_t plan, const int32_t** d_tile_order,
                                   int64_t* n_live, const int32_t** d_empty_tiles,
                                   int64_t* n_empty);

/* Device pointer and size in bytes of the plan's fp16 copy of V (head_dim 64
   and e4m3 inputs, see bsattn_fwd and bsattn_fwd_fp8), or NULL and 0 while
   no forward call has made one; valid
   until the next forward call with the plan or bsattn_plan_free.  For
   tests/tools. */
bsattn_status bsattn_plan_v16(bsattn_plan_t plan, const void** d_v16, size_t* bytes);

/*
 * bsattn_fwd -- O, LSE = block-sparse attention(Q, K, V; plan's mask).
 *
 *   q, k, v    device bf16 [B][H][S][D], 16-byte aligned.
 *   plan       from bsattn_plan with the same B, H, S.
 *   out        device [B][H][S][D], bf16 (or fp32 with BSATTN_OUT_F32), 16-byte aligned
 *              (32-byte aligned: written with full-sector stores, slightly faster).
 *   lse        device fp32 [B][H][S], 16-byte aligned.
 *   D          64 or 128.
 *   scale      finite; multiplies q.k before masking (1/sqrt(D) in the pages).
 *   stream     cudaStream_t; the call is stream-ordered and never synchronises.
 * Uses the plan's small device workspace (tile counter, status word), so calls
 * with the same plan must not overlap on the GPU.  A kernel-side failure
 * (bounded wait ran out) is recorded in the plan and returned by
 * bsattn_plan_status.
 * At D = 64 P V runs in fp16 (V converts exactly for 2^-14 <= |v| <= 65504; a
 * V entry beyond 65504, or not finite, is reported as BSATTN_ERR_RANGE by
 * bsattn_plan_status).  When V has at least 16384 rows (B*Hkv*S) and the plan
 * has at least 4 live blocks per key block of V on average, the call first
 * converts V into an fp16 copy held by the plan (one extra kernel launch;
 * B*Hkv*S*64*2 bytes, allocated with cudaMallocAsync on `stream` by the first
 * call that needs it, or a larger one, and freed by bsattn_plan_free); it
 * allocates nothing while `stream` is being captured, and if the allocation
 * fails the forward kernel converts each V tile itself, as it does below
 * those sizes.
 * Errors: INVALID_ARG (null/misaligned, sizes differ from the plan, non-finite
 * scale), UNSUPPORTED (D), CUDA (launch failure).
 */
bsattn_status bsattn_fwd(const void* q, const void* k, const void* v, bsattn_plan_t plan,
                         void* out, float* lse, int B, int H, int S, int D, float scale,
                         void* stream);

/*
 * bsattn_bwd -- dQ, dK, dV: gradients of bsattn_fwd's O with respect to Q, K, V,
 * given the upstream gradient dO.  "Writing Pallas Kernels for JAX: Stepping
 * Outside the XLA Safety Net" (section "The Empathy of the Void") asks for
 * hand-written gradient definitions; these are the exact derivative of the
 * forward operation over the plan's live blocks:
 *   P = softmax of the scaled, masked scores (recomputed from lse),
 *   dS = P * (dO V^T - rowsum(dO * O)),
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 *
 *   q, k, v    device bf16 [B][H][S][D], the forward's inputs, 16-byte aligned.
 *   o, lse     the forward's outputs for the same plan: o bf16 (or fp32 when the
 *              plan has BSATTN_OUT_F32) [B][H][S][D], lse fp32 [B][H][S].
 *   dout       device bf16 [B][H][S][D]: the upstream gradient dO.
 *   plan       from bsattn_plan with the same B, H, S (its transposed list is used).
 *   dq, dk, dv device fp32 [B][H][S][D], 16-byte aligned, written in full (rows
 *              of query tiles with no live key block get dQ = 0, key blocks no
 *              query attends get dK = dV = 0).
 *   D, scale   as in bsattn_fwd (the same scale as the forward call).
 *   stream     cudaStream_t; stream-ordered, never synchronises.
 * Uses the plan's workspace (status word, a B*H*S fp32 scratch row term), so
 * calls with the same plan must not overlap on the GPU; a kernel-side failure
 * is returned by bsattn_plan_status.
 * Errors: INVALID_ARG (null/misaligned, sizes differ from the plan, non-finite
 * scale), UNSUPPORTED (D), CUDA (launch failure).
 */
bsattn_status bsattn_bwd(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, bsattn_plan_t plan, float* dq,
                         float* dk, float* dv, int B, int H, int S, int D, float scale,
                         void* stream);

/*
 * bsattn_bwd_gqa -- bsattn_bwd for grouped-query attention (as bsattn_fwd_gqa):
 * k, v, dk, dv are [B][Hkv][S][D]; dK and dV of a K/V head sum the gradients
 * of all H / Hkv query heads that attend with it.  H / Hkv <= 64.
 * Errors: as bsattn_bwd; INVALID_ARG when H % Hkv != 0, UNSUPPORTED when
 * H / Hkv > 64.
 */
bsattn_status bsattn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, bsattn_plan_t plan, float* dq,
                             float* dk, float* dv, int B, int H, int Hkv, int S, int D,
                             float scale, void* stream);

/*
 * bsattn_fwd_gqa -- bsattn_fwd with grouped-query attention: K and V have Hkv
 * heads and query head h of a batch entry attends with K/V head h / (H / Hkv)
 * (Hkv = 1: multi-query attention; Hkv = H: bsattn_fwd).  The result equals
 * bsattn_fwd on K and V with each head repeated H / Hkv times.
 *
 *   q, out, lse  as bsattn_fwd ([B][H][S][D] / [B][H][S]).
 *   k, v         device bf16 [B][Hkv][S][D], 16-byte aligned.
 *   Hkv          K/V heads, 1 <= Hkv, H % Hkv == 0.
 * Errors: as bsattn_fwd; INVALID_ARG also when H % Hkv != 0.
 */
bsattn_status bsattn_fwd_gqa(const void* q, const void* k, const void* v, bsattn_plan_t plan,
                             void* out, float* lse, int B, int H, int Hkv, int S, int D,
                             float scale, void* stream);

/*
 * bsattn_fwd_fp8 -- the forward pass on FP8 (e4m3) Q, K, V.
 *
 * "JAX Pallas and Blackwell", section "What the Tutorial Covers": Blackwell's
 * tensor cores take FP8 operands with fp32 accumulation.  Here S = Q K^T runs
 * on e4m3 operands (the OCP 8-bit format: sign, 4 exponent bits with bias 7,
 * 3 mantissa bits) with fp32 accumulation; V is converted to fp16 (exactly:
 * once per call into a copy, or tile by tile in shared memory, see below) and
 * P V runs in fp16, fp32 accumulation.
 * The result is the attention of bsattn_fwd on the decoded values:
 *
 *   O = v_scale * softmax(scale * Q K^T + mask) V,  LSE as bsattn_fwd.
 *
 * FP8 tensors usually carry scales (value = scale_t * decoded bits): pass
 * scale = softmax scale * q_scale * k_scale, and v_scale = V's scale.
 *
 *   q8, k8, v8 device e4m3 [B][H][S][D] (one byte per element), 16-byte aligned.
 *   plan       from bsattn_plan (any flags bsattn_fwd takes, 64-key blocks too).
 *   out, lse   as bsattn_fwd.
 *   D          128 (UNSUPPORTED otherwise).
 *   scale, v_scale  finite.
 * Errors: as bsattn_fwd; a NaN entry of V (e4m3 0x7F / 0xFF) is reported as
 * BSATTN_ERR_RANGE by the status calls.
 * V's fp16 conversion: as at D = 64 in bsattn_fwd (an fp16 copy of V held
 * by the plan, B*H*S*128*2 bytes, converted before the kernel when V has at
 * least 16384 rows and the plan at least 4 live blocks per key block of V;
 * otherwise the kernel converts each V tile after its load).
 */
bsattn_status bsattn_fwd_fp8(const void* q8, const void* k8, const void* v8, bsattn_plan_t plan,
                             void* out, float* lse, int B, int H, int S, int D, float scale,
                             float v_scale, void* stream);

/* Wait for `stream`, then report and clear the device-side status of the
   plan's kernels: OK, TIMEOUT, INTERNAL or RANGE (or CUDA if the wait
   failed). */
bsattn_status bsattn_plan_status(bsattn_plan_t plan, void* stream);

/* Release the plan (waits for the device first).  NULL is ignored. */
void bsattn_plan_free(bsattn_plan_t plan);

/* Static text for a status code. */
const char* bsattn_status_string(bsattn_status status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int bsattn_version(void);

/*
 * bsattn_fwd_noalloc -- the same forward pass for callers that cannot
 * allocate device memory.  No counterpart on the pages.
 *
 * bsattn_plan allocates its arrays with cudaMalloc.  Some callers cannot:
 * a host framework that owns all GPU memory through its own pool, a plug-in
 * that may not allocate once running, or a latency-critical loop that cannot
 * absorb cudaMalloc's device-wide synchronisation.  This call builds the plan
 * and runs the forward kernel with every piece of scratch (the plan's CSR and
 * schedule, the tile counter and the status word) inside one fixed device
 * array that is part of the library: 16 MiB, held by every GPU that loads the
 * library until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 *   q, k, v, out, lse, B, H, S, D, scale: as bsattn_fwd.
 *   d_mask     device uint8 [B][H][S/128][S/128], as bsattn_plan.
 *   flags      BSATTN_CAUSAL | BSATTN_OUT_F32.
 *   stream     cudaStream_t; the call synchronises it twice (to size the
 *              plan and to read the kernel's status) and returns the kernel's
 *              TIMEOUT / INTERNAL status directly.
 * Limit: with R = B*H*(S/128) query tiles and nb = S/128, the plan needs
 * about R*(nb + 4) + 2*B*H + 16 int32 words; more than 16 MiB / 4 words is
 * rejected with BSATTN_ERR_SCRATCH_LIMIT before anything is launched.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture begins.
 * All calls share the array and it keeps the last call's contents; each call
 * clears what must start at zero.  Calls that overlap on the GPU race on the
 * array, so issue them one after another.
 * Errors: as bsattn_plan and bsattn_fwd, plus SCRATCH_LIMIT.
 */
bsattn_status bsattn_fwd_noalloc(const void* q, const void* k, const void* v,
                                 const uint8_t* d_mask, void* out, float* lse, int B, int H,
                                 int S, int D, float scale, unsigned flags, void* stream);

/*
 * bsattn_selftest_wait_timeout -- checks that the library's bounded device
 * waits end on their own.  Launches one small kernel whose threads wait on a
 * barrier that nothing completes, with a limit of `timeout_ns` nanoseconds
 * (1e3 .. 5e9), and synchronises `stream`.  Returns BSATTN_ERR_TIMEOUT when the
 * kernel gave up and reported it as designed (the expected result), OK if the
 * barrier somehow completed, CUDA on a CUDA error.  Not part of the
 * attention path; no counterpart on the pages.
 */
bsattn_status bsattn_selftest_wait_timeout(int64_t timeout_ns, void* stream);

/*
 * Forward passes on HOST-resident tensors, with the transfers overlapped.
 *
 * Not on the pages: the forward pass above needs Q, K, V in device memory.
 * A pipeline owns device copies of the whole problem and cuts the flattened
 * (b, h) range into `pieces` contiguous parts, each with its own plan (built
 * at creation, from the corresponding slice of the mask).  bsattn_pipeline_run
 * enqueues, for every part, the host-to-device copy of its Q, K, V on one
 * stream, its forward kernel on a second and the device-to-host copy of its
 * O and LSE on a third, so one part's upload overlaps another part's kernel
 * and a third part's download.  Every run copies all inputs in and all
 * results out; results are identical to bsattn_fwd's (same kernel, same
 * tiles).  Copies are plain cudaMemcpyAsync calls; host buffers must be
 * pinned (page-locked) for the copies to overlap.
 *
 * bsattn_pipeline_create
 *   d_mask     device uint8 [B][H][S/128][S/128]; read during the call only.
 *   B, H, S, D sizes as for bsattn_plan / bsattn_fwd (D = 64 or 128).
 *   flags      BSATTN_CAUSAL | BSATTN_OUT_F32.
 *   pieces     number of parts, clamped to [1, B*H].
 *   stream     cudaStream_t for the plan kernels (synchronised once per part).
 *   out        receives the handle; the library owns the device buffers
 *              (Q, K, V, O, LSE of the whole problem), the plans, three
 *              streams and the events until bsattn_pipeline_free.
 * Errors: INVALID_ARG, UNSUPPORTED, OOM, CUDA (as bsattn_plan).
 *
 * bsattn_pipeline_run
 *   hq, hk, hv host bf16 [B][H][S][D]; hout host [B][H][S][D] bf16 (fp32 with
 *              BSATTN_OUT_F32); hlse host fp32 [B][H][S].  Read / written
 *              asynchronously: `stream` is made to wait for the run's last
 *              copy, so synchronise it before touching the buffers.
 *   scale      finite multiplier of q.k.
 *   Runs on one pipeline are ordered: a part's device buffers are reused
 *   only after the previous run is done with them.
 * Errors: INVALID_ARG (null pipeline or pointers, non-finite scale), CUDA.
 *
 * bsattn_pipeline_status -- waits for the pipeline's streams and reports the
 *   kernels' recorded status (TIMEOUT / INTERNAL) like bsattn_plan_status.
 * bsattn_pipeline_free -- waits, then releases everything; NULL is a no-op.
 */
typedef struct bsattn_pipeline_s* bsattn_pipeline_t;

bsattn_status bsattn_pipeline_create(const uint8_t* d_mask, int B, int H, int S, int D,
                                     unsigned flags, int pieces, void* stream,
                                     bsattn_pipeline_t* out);
bsattn_status bsattn_pipeline_run(bsattn_pipeline_t pipe, const void* hq, const void* hk,
                                  const void* hv, void* hout, float* hlse, float scale,
                                  void* stream);
bsattn_status bsattn_pipeline_status(bsattn_pipeline_t pipe);
void bsattn_pipeline_free(bsattn_pipeline_t pipe);

#ifdef __cplusplus
}
#endif

#endif /* BSATTN_H_ */
