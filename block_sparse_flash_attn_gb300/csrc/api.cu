// C ABI (include/bsattn.h): argument checks, plan ownership, TMA tensor-map
// encoding and kernel launches.  All checks run before anything is launched;
// no function aborts the process.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>

#include "bwd.h"
#include "internal.h"

using namespace bsattn;

struct bsattn_plan_s {
  uint32_t magic = 0;
  int B = 0, H = 0, S = 0, nb = 0;
  int kdiv = 1;  // key blocks of 128 / kdiv keys (BSATTN_KEY_BLOCK_64: 2)
  unsigned flags = 0;
  int device = 0;
  int64_t nnz = 0, n_live = 0, n_empty = 0;
  PlanDevice dev;
};

namespace bsattn {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

int device_sm_count(int dev) {
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

bsattn_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return BSATTN_OK;
  return e == cudaErrorMemoryAllocation ? BSATTN_ERR_OOM : BSATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The softmax works with a strictly positive multiplier sl = |scale| log2(e):
// a negative scale is folded into the S MMA (-Q K^T), and scale = 0 becomes
// sl = 1e-30, for which every exponent 2^(s*sl - m) of an allowed key is 1.0
// in fp32 (|s*sl| < 1e-26), i.e. exactly the uniform weights of scale 0.
void set_scale_params(FwdParams& p, float scale) {
  const double a = std::fabs((double)scale) * 1.4426950408889634074;
  p.scale_log2 = (scale == 0.0f) ? 1e-30f : (float)a;
  p.neg_scale = scale < 0.0f ? 1 : 0;
}

// 2-D view (rows = B*H*S, cols = D) of a bf16 tensor; box 64 columns x
// box_rows rows (128, or 64 for the halves of a tile of 64-key blocks; one
// 128-byte swizzle span per row), 128B swizzle.
bsattn_status encode_bf16_map(CUtensorMap* m, const void* ptr, int D, long long rows,
                              int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSATTN_OK : BSATTN_ERR_CUDA;
}

// 2-D view (rows = B*H*S, cols = D bytes) of an e4m3 tensor (uint8 elements);
// box D = 128 bytes x box_rows rows, 128B swizzle: the same 128-byte rows and
// swizzle as one 64-column box of a bf16 tile.
bsattn_status encode_e4m3_map(CUtensorMap* m, const void* ptr, int D, long long rows,
                              int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D};
  cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSATTN_OK : BSATTN_ERR_CUDA;
}

}  // namespace bsattn

namespace {

bool plan_ok(const bsattn_plan_s* p) { return p != nullptr && p->magic == kPlanMagic; }

void free_plan_memory(bsattn_plan_s* p) {
  cudaFree(p->dev.row_ptr);
  cudaFree(p->dev.col_idx);
  cudaFree(p->dev.tile_order);
  cudaFree(p->dev.empty_tiles);
  cudaFree(p->dev.work);
  cudaFree(p->dev.col_ptr);
  cudaFree(p->dev.row_idx);
  cudaFree(p->dev.kv_order);
  cudaFree(p->dev.dl);
  cudaFree(p->dev.v16);
  p->dev = PlanDevice{};
}

}  // namespace

namespace bsattn {

bsattn_status prepare_fwd(const void* q, const void* k, const void* v, bsattn_plan_t plan,
                          void* out, float* lse, int B, int H, int S, int D, float scale,
                          PreparedFwd* pf, int Hkv, bool in8, float v_scale, bool v16_ok,
                          cudaStream_t stream) {
  if (!plan_ok(plan) || !pf) return BSATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !lse) return BSATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return BSATTN_ERR_INVALID_ARG;
  if (B != plan->B || H != plan->H || S != plan->S) return BSATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return BSATTN_ERR_UNSUPPORTED;
  if (in8 && D != 128) return BSATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !std::isfinite(v_scale)) return BSATTN_ERR_INVALID_ARG;
  if (Hkv <= 0 || H % Hkv != 0) return BSATTN_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) return BSATTN_ERR_INVALID_ARG;
  if (!get_tensor_map_encoder()) return BSATTN_ERR_CUDA;

  const long long rows = (long long)B * H * S;
  const long long kv_rows = (long long)B * Hkv * S;
  bsattn_status rc;
  // K and V come in halves of 64 rows when the plan's key blocks have 64 keys
  const int kv_box = kBlock / plan->kdiv;
  auto encode = in8 ? encode_e4m3_map : encode_bf16_map;
  if ((rc = encode(&pf->tq, q, D, rows, kBlock)) != BSATTN_OK) return rc;
  if ((rc = encode(&pf->tk, k, D, kv_rows, kv_box)) != BSATTN_OK) return rc;

  // head_dim 64 and e4m3 inputs multiply P by V in fp16.  The kernel can
  // convert each V tile in shared memory after its load, once per (query
  // tile, key block) pair; when the key blocks are shared by several query
  // tiles on average and V is not tiny, one conversion pass over V before
  // the launch costs less (one read of V, one write of its fp16 copy).
  // Never allocated during stream capture; if the allocation fails the
  // kernel converts V itself.
  bool v_pre = false;
  const size_t v16_bytes = (size_t)kv_rows * D * 2;
  const long long kv_units = (long long)B * Hkv * plan->nb * plan->kdiv;  // key blocks of V
  if (v16_ok && (D == 64 || in8) && kv_rows >= kV16MinRows &&
      plan->nnz >= kV16MinReuse * kv_units) {
    if (plan->dev.v16_bytes >= v16_bytes) {
      v_pre = true;
    } else {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusActive;
      void* buf = nullptr;
      if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone &&
          cudaMallocAsync(&buf, v16_bytes, stream) == cudaSuccess) {
        if (plan->dev.v16) cudaFreeAsync(plan->dev.v16, stream);
        plan->dev.v16 = buf;
        plan->dev.v16_bytes = v16_bytes;
        v_pre = true;
      } else {
        (void)cudaGetLastError();  // the kernel converts V itself
      }
    }
  }
  // the fp16 copy is read like bf16 V (16-bit elements, 64-column boxes)
  if ((rc = v_pre ? encode_bf16_map(&pf->tv, plan->dev.v16, D, kv_rows, kv_box)
                  : encode(&pf->tv, v, D, kv_rows, kv_box)) != BSATTN_OK)
    return rc;
  pf->v_src = v_pre ? v : nullptr;
  pf->v16 = v_pre ? plan->dev.v16 : nullptr;
  pf->v16_elems = v_pre ? kv_rows * D : 0;

  FwdParams& prm = pf->prm;
  prm = FwdParams{};
  prm.row_ptr = plan->dev.row_ptr;
  prm.col_idx = plan->dev.col_idx;
  prm.tile_order = plan->dev.tile_order;
  prm.empty_tiles = plan->dev.empty_tiles;
  prm.out = out;
  prm.lse = lse;
  prm.counter = plan->dev.work + kWorkCounter;
  prm.done = plan->dev.work + kWorkDone;
  prm.status = plan->dev.work + kWorkStatus;
  prm.n_live = (int)plan->n_live;
  prm.n_empty = (int)plan->n_empty;
  prm.nb = plan->nb;
  prm.S = S;
  set_scale_params(prm, scale);
  prm.causal = (plan->flags & BSATTN_CAUSAL) ? 1 : 0;
  prm.timeout_ns = kDefaultWaitTimeoutNs;
  prm.H = H;
  prm.kv_group = H / Hkv;
  prm.kdiv = plan->kdiv;
  prm.v_scale = v_scale;
  prm.v_pre = v_pre ? 1 : 0;
  pf->D = D;
  pf->in8 = in8;
  pf->out_f32 = (plan->flags & BSATTN_OUT_F32) != 0;
  pf->grid = device_sm_count(dev);
  return BSATTN_OK;
}

cudaError_t launch_prepared(const PreparedFwd& pf, cudaStream_t stream) {
  if (pf.prm.v_pre) {
    const cudaError_t e =
        pf.in8 ? launch_v16_convert_e4m3(pf.v_src, pf.v16, pf.v16_elems, pf.prm.status, pf.grid,
                                         stream)
               : launch_v16_convert(pf.v_src, pf.v16, pf.v16_elems, pf.prm.status, pf.grid,
                                    stream);
    if (e != cudaSuccess) return e;
  }
  return launch_fwd(pf.D, pf.out_f32, pf.tq, pf.tk, pf.tv, pf.prm, pf.grid, stream, pf.in8);
}

}  // namespace bsattn

extern "C" {

int bsattn_version(void) { return 100; }

const char* bsattn_status_string(bsattn_status s) {
  switch (s) {
    case BSATTN_OK: return "ok";
    case BSATTN_ERR_INVALID_ARG: return "invalid argument";
    case BSATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case BSATTN_ERR_CUDA: return "CUDA error";
    case BSATTN_ERR_OOM: return "out of memory";
    case BSATTN_ERR_TIMEOUT: return "device wait timed out";
    case BSATTN_ERR_INTERNAL: return "internal error detected on device";
    case BSATTN_ERR_SCRATCH_LIMIT: return "problem exceeds the no-allocation scratch size";
    case BSATTN_ERR_RANGE: return "input value out of the supported range (D = 64: |V| <= 65504)";
  }
  return "unknown status";
}

bsattn_status bsattn_plan(const uint8_t* d_mask, int B, int H, int S, unsigned flags,
                          void* stream, bsattn_plan_t* out_plan) {
  if (!d_mask || !out_plan) return BSATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || S <= 0 || (S % kBlock) != 0) return BSATTN_ERR_INVALID_ARG;
  if (flags & ~(unsigned)(BSATTN_CAUSAL | BSATTN_OUT_F32 | BSATTN_MASK_SHARED_HEADS |
                          BSATTN_KEY_BLOCK_64))
    return BSATTN_ERR_INVALID_ARG;
  const int nb = S / kBlock;
  if (nb > kMaxBlocksPerRow) return BSATTN_ERR_UNSUPPORTED;
  if ((long long)B * H * S >= (1ll << 31)) return BSATTN_ERR_UNSUPPORTED;
  const int BH = B * H;
  const int rows = BH * nb;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  bsattn_plan_s* p = new (std::nothrow) bsattn_plan_s();
  if (!p) return BSATTN_ERR_OOM;
  p->B = B;
  p->H = H;
  p->S = S;
  p->nb = nb;
  p->flags = flags;
  p->kdiv = (flags & BSATTN_KEY_BLOCK_64) ? 2 : 1;
  cudaGetDevice(&p->device);
  const int causal = (flags & BSATTN_CAUSAL) ? 1 : 0;
  const int mdiv = (flags & BSATTN_MASK_SHARED_HEADS) ? H : 1;  // mask heads: H or 1
  const int kdiv = p->kdiv;

  int* tmp = nullptr;  // counts[rows] | live_per_head[BH] | live_off[BH+1] | totals (2 x int64)
  const size_t tmp_ints = (size_t)rows + BH + (BH + 1) + 1 + 4;
  long long h_tot[2] = {0, 0};
  auto fail = [&](bsattn_status s) {
    cudaFree(tmp);
    free_plan_memory(p);
    delete p;
    return s;
  };
  cudaError_t e;
  if ((e = cudaMalloc(&p->dev.row_ptr, sizeof(int) * ((size_t)rows + 1))) != cudaSuccess)
    return fail(from_cuda(e));
  if ((e = cudaMalloc(&p->dev.work, sizeof(int) * kWorkWords)) != cudaSuccess)
    return fail(from_cuda(e));
  if ((e = cudaMalloc(&tmp, sizeof(int) * tmp_ints)) != cudaSuccess) return fail(from_cuda(e));
  int* d_counts = tmp;
  int* d_live_off = tmp + rows + BH;
  // 8-byte aligned slot for the two int64 totals
  size_t tot_off = (size_t)rows + BH + BH + 1;
  tot_off = (tot_off + 1) & ~(size_t)1;
  int* d_totals = tmp + tot_off;
  if ((e = cudaMemsetAsync(p->dev.work, 0, sizeof(int) * kWorkWords, st)) != cudaSuccess)
    return fail(from_cuda(e));
  if ((e = plan_count_and_scan(d_mask, BH, nb, causal, d_counts, p->dev.row_ptr, d_live_off,
                               d_totals, st, mdiv, kdiv)) != cudaSuccess)
    return fail(from_cuda(e));
  if ((e = cudaMemcpyAsync(h_tot, d_totals, sizeof(h_tot), cudaMemcpyDeviceToHost, st)) !=
      cudaSuccess)
    return fail(from_cuda(e));
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(from_cuda(e));
  p->nnz = h_tot[0];
  p->n_live = h_tot[1];
  p->n_empty = (int64_t)rows - p->n_live;
  if (p->nnz < 0 || p->nnz >= (1ll << 31) || p->n_live < 0 || p->n_live > rows)
    return fail(BSATTN_ERR_UNSUPPORTED);
  if ((e = cudaMalloc(&p->dev.col_idx, sizeof(int) * (size_t)(p->nnz > 0 ? p->nnz : 1))) !=
      cudaSuccess)
    return fail(from_cuda(e));
  if ((e = cudaMalloc(&p->dev.tile_order,
                      sizeof(int) * (size_t)(p->n_live > 0 ? p->n_live : 1))) != cudaSuccess)
    return fail(from_cuda(e));
  if ((e = cudaMalloc(&p->dev.empty_tiles,
                      sizeof(int) * (size_t)(p->n_empty > 0 ? p->n_empty : 1))) != cudaSuccess)
    return fail(from_cuda(e));
  if ((e = plan_fill_and_order(d_mask, BH, nb, causal, p->dev.row_ptr, d_live_off,
                               p->dev.col_idx, p->dev.tile_order, p->dev.empty_tiles,
                               device_sm_count(p->device), st, mdiv, kdiv)) != cudaSuccess)
    return fail(from_cuda(e));
  // Transposed plan for the backward pass (same number of live blocks) and
  // its per-row scratch; d_counts is free again once the CSR is built.  The
  // backward pass takes 128-key blocks only, so plans of 64-key blocks have none.
  if (kdiv == 1) {
    if ((e = cudaMalloc(&p->dev.col_ptr, sizeof(int) * ((size_t)rows + 1))) != cudaSuccess)
      return fail(from_cuda(e));
    if ((e = cudaMalloc(&p->dev.row_idx, sizeof(int) * (size_t)(p->nnz > 0 ? p->nnz : 1))) !=
        cudaSuccess)
      return fail(from_cuda(e));
    if ((e = cudaMalloc(&p->dev.dl, sizeof(float) * (size_t)B * H * S)) != cudaSuccess)
      return fail(from_cuda(e));
    if ((e = cudaMalloc(&p->dev.kv_order, sizeof(int) * (size_t)rows)) != cudaSuccess)
      return fail(from_cuda(e));
    if ((e = plan_csc(d_mask, BH, nb, causal, d_counts, d_live_off, d_totals, p->dev.col_ptr,
                      p->dev.row_idx, p->dev.kv_order, device_sm_count(p->device), st, mdiv)) !=
        cudaSuccess)
      return fail(from_cuda(e));
  }
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(from_cuda(e));
  cudaFree(tmp);
  tmp = nullptr;
  p->magic = kPlanMagic;
  *out_plan = p;
  return BSATTN_OK;
}

bsattn_status bsattn_plan_csr(bsattn_plan_t plan, const int32_t** d_row_ptr,
                              const int32_t** d_col_idx, int64_t* nnz) {
  if (!plan_ok(plan) || !d_row_ptr || !d_col_idx || !nnz) return BSATTN_ERR_INVALID_ARG;
  *d_row_ptr = plan->dev.row_ptr;
  *d_col_idx = plan->dev.col_idx;
  *nnz = plan->nnz;
  return BSATTN_OK;
}

bsattn_status bsattn_plan_csc(bsattn_plan_t plan, const int32_t** d_col_ptr,
                              const int32_t** d_row_idx, int64_t* nnz) {
  if (!plan_ok(plan) || !d_col_ptr || !d_row_idx || !nnz) return BSATTN_ERR_INVALID_ARG;
  if (plan->kdiv != 1) return BSATTN_ERR_UNSUPPORTED;  // no transposed list for 64-key blocks
  *d_col_ptr = plan->dev.col_ptr;
  *d_row_idx = plan->dev.row_idx;
  *nnz = plan->nnz;
  return BSATTN_OK;
}

bsattn_status bsattn_plan_v16(bsattn_plan_t plan, const void** d_v16, size_t* bytes) {
  if (!plan_ok(plan) || !d_v16 || !bytes) return BSATTN_ERR_INVALID_ARG;
  *d_v16 = plan->dev.v16;
  *bytes = plan->dev.v16_bytes;
  return BSATTN_OK;
}

bsattn_status bsattn_plan_schedule(bsattn_plan_t plan, const int32_t** d_tile_order,
                                   int64_t* n_live, const int32_t** d_empty_tiles,
                                   int64_t* n_empty) {
  if (!plan_ok(plan) || !d_tile_order || !n_live || !d_empty_tiles || !n_empty)
    return BSATTN_ERR_INVALID_ARG;
  *d_tile_order = plan->dev.tile_order;
  *n_live = plan->n_live;
  *d_empty_tiles = plan->dev.empty_tiles;
  *n_empty = plan->n_empty;
  return BSATTN_OK;
}

bsattn_status bsattn_fwd(const void* q, const void* k, const void* v, bsattn_plan_t plan,
                         void* out, float* lse, int B, int H, int S, int D, float scale,
                         void* stream) {
  PreparedFwd pf;
  const bsattn_status rc = prepare_fwd(q, k, v, plan, out, lse, B, H, S, D, scale, &pf, H, false,
                                       1.0f, true, static_cast<cudaStream_t>(stream));
  if (rc != BSATTN_OK) return rc;
  return from_cuda(launch_prepared(pf, static_cast<cudaStream_t>(stream)));
}

bsattn_status bsattn_fwd_gqa(const void* q, const void* k, const void* v, bsattn_plan_t plan,
                             void* out, float* lse, int B, int H, int Hkv, int S, int D,
                             float scale, void* stream) {
  PreparedFwd pf;
  const bsattn_status rc = prepare_fwd(q, k, v, plan, out, lse, B, H, S, D, scale, &pf, Hkv, false,
                                       1.0f, true, static_cast<cudaStream_t>(stream));
  if (rc != BSATTN_OK) return rc;
  return from_cuda(launch_prepared(pf, static_cast<cudaStream_t>(stream)));
}

bsattn_status bsattn_fwd_fp8(const void* q8, const void* k8, const void* v8, bsattn_plan_t plan,
                             void* out, float* lse, int B, int H, int S, int D, float scale,
                             float v_scale, void* stream) {
  PreparedFwd pf;
  const bsattn_status rc =
      prepare_fwd(q8, k8, v8, plan, out, lse, B, H, S, D, scale, &pf, H, true, v_scale, true,
                  static_cast<cudaStream_t>(stream));
  if (rc != BSATTN_OK) return rc;
  return from_cuda(launch_prepared(pf, static_cast<cudaStream_t>(stream)));
}

bsattn_status bsattn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, bsattn_plan_t plan, float* dq,
                             float* dk, float* dv, int B, int H, int Hkv, int S, int D,
                             float scale, void* stream) {
  if (!plan_ok(plan)) return BSATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return BSATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return BSATTN_ERR_INVALID_ARG;
  if (B != plan->B || H != plan->H || S != plan->S) return BSATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return BSATTN_ERR_UNSUPPORTED;
  if (plan->kdiv != 1) return BSATTN_ERR_UNSUPPORTED;  // gradients over 128-key blocks only
  if (!std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;
  if (Hkv <= 0 || H % Hkv != 0) return BSATTN_ERR_INVALID_ARG;
  if (H / Hkv > 64) return BSATTN_ERR_UNSUPPORTED;  // query heads per K/V head walked by one CTA
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) return BSATTN_ERR_INVALID_ARG;
  if (!get_tensor_map_encoder()) return BSATTN_ERR_CUDA;
  const long long rows = (long long)B * H * S;
  const long long kv_rows = (long long)B * Hkv * S;
  // The backward kernels load tiles by halves: 64-row boxes.
  CUtensorMap tq, tk, tv, tdo;
  bsattn_status rc;
  if ((rc = encode_bf16_map(&tq, q, D, rows, 64)) != BSATTN_OK) return rc;
  if ((rc = encode_bf16_map(&tk, k, D, kv_rows, 64)) != BSATTN_OK) return rc;
  if ((rc = encode_bf16_map(&tv, v, D, kv_rows, 64)) != BSATTN_OK) return rc;
  if ((rc = encode_bf16_map(&tdo, dout, D, rows, 64)) != BSATTN_OK) return rc;
  BwdParams prm{};
  prm.col_ptr = plan->dev.col_ptr;
  prm.row_idx = plan->dev.row_idx;
  prm.row_ptr = plan->dev.row_ptr;
  prm.col_idx = plan->dev.col_idx;
  prm.lse = lse;
  prm.dl = plan->dev.dl;
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.status = plan->dev.work + kWorkStatus;
  prm.nb = plan->nb;
  prm.S = S;
  prm.causal = (plan->flags & BSATTN_CAUSAL) ? 1 : 0;
  prm.scale = scale;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634074);
  prm.timeout_ns = kDefaultWaitTimeoutNs;
  prm.H = H;
  prm.kv_group = H / Hkv;
  prm.tile_order = plan->dev.tile_order;
  prm.empty_tiles = plan->dev.empty_tiles;
  prm.kv_order = plan->dev.kv_order;
  prm.n_live = (int)plan->n_live;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bwd_prep(D, (plan->flags & BSATTN_OUT_F32) != 0, o, dout, plan->dev.dl,
                                  rows, st);
  if (e != cudaSuccess) return from_cuda(e);
  return from_cuda(launch_bwd(D, tq, tk, tv, tdo, prm, B * Hkv * plan->nb, B * H * plan->nb, st));
}

bsattn_status bsattn_bwd(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, bsattn_plan_t plan, float* dq,
                         float* dk, float* dv, int B, int H, int S, int D, float scale,
                         void* stream) {
  return bsattn_bwd_gqa(q, k, v, o, lse, dout, plan, dq, dk, dv, B, H, H, S, D, scale, stream);
}

bsattn_status bsattn_plan_status(bsattn_plan_t plan, void* stream) {
  if (!plan_ok(plan)) return BSATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return BSATTN_ERR_CUDA;
  int words[kWorkWords] = {0};
  if (cudaMemcpy(words, plan->dev.work, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BSATTN_ERR_CUDA;
  // Clear the status and rewind the scheduler so the plan is usable again.
  if (cudaMemset(plan->dev.work, 0, sizeof(words)) != cudaSuccess) return BSATTN_ERR_CUDA;
  const int s = words[kWorkStatus];
  if (s & kStatusInternal) return BSATTN_ERR_INTERNAL;
  if (s & kStatusTimeout) return BSATTN_ERR_TIMEOUT;
  if (s & kStatusRange) return BSATTN_ERR_RANGE;
  return BSATTN_OK;
}

void bsattn_plan_free(bsattn_plan_t plan) {
  if (!plan_ok(plan)) return;
  cudaDeviceSynchronize();
  free_plan_memory(plan);
  plan->magic = 0;
  delete plan;
}

bsattn_status bsattn_selftest_wait_timeout(int64_t timeout_ns, void* stream) {
  if (timeout_ns < 1000 || timeout_ns > 5000000000ll) return BSATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* d_status = nullptr;
  cudaError_t e = cudaMalloc(&d_status, sizeof(int));
  if (e != cudaSuccess) return from_cuda(e);
  int h = 0;
  bsattn_status rc = BSATTN_OK;
  if ((e = cudaMemsetAsync(d_status, 0, sizeof(int), st)) != cudaSuccess ||
      (e = launch_selftest_wait((unsigned long long)timeout_ns, d_status, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(&h, d_status, sizeof(int), cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess) {
    rc = BSATTN_ERR_CUDA;
  } else {
    rc = (h & kStatusTimeout) ? BSATTN_ERR_TIMEOUT : BSATTN_OK;
  }
  cudaFree(d_status);
  return rc;
}

}  // extern "C"
