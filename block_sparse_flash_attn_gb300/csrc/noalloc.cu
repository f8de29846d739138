// bsattn_fwd_noalloc: the forward pass for callers that cannot allocate GPU
// memory.
//
// bsattn_plan allocates the plan's arrays and a small workspace with
// cudaMalloc.  Some callers cannot do that.  Examples: a host framework that
// owns all device memory through its own pool, or a plug-in that may not
// allocate after start-up.  Another example is a latency-critical loop where
// cudaMalloc's implicit device-wide synchronisation is not acceptable.  This
// entry point builds the same plan and runs the same kernels.  The plan
// arrays and the forward kernel's scratch words (tile counter, finished-CTA
// count, status word) live in one file-scope device array of fixed size
// instead of allocated memory.  The caller still provides Q, K, V, the mask,
// O and LSE.
//
// The array is kNoAllocScratchBytes (16 MiB).  Every GPU that loads this
// library keeps it until the process exits.  Its device address is looked
// up once per device, on the first call made on that device, with that
// device current (cudaGetSymbolAddress).  That first call should come before
// any stream capture starts.  Every call shares the array, and the array
// keeps the previous call's contents: each call clears the words that must
// start at zero.  Calls whose work overlaps on the GPU race on the array;
// issue them one after another.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace bsattn {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
constexpr size_t kNoAllocWords = kNoAllocScratchBytes / sizeof(int);
constexpr int kMaxDevices = 64;

}  // namespace
}  // namespace bsattn

// The scratch itself.  Host code must not pass `g_noalloc_scratch` to a kernel:
// on the host the name is only a stand-in, not a device address.
static __device__ __align__(256) int g_noalloc_scratch[bsattn::kNoAllocWords];

namespace bsattn {
namespace {

std::mutex g_scratch_mu;
int* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
bsattn_status scratch_on_current_device(int** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BSATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return BSATTN_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_scratch_ptr[dev];
  return BSATTN_OK;
}

size_t align4(size_t words) { return (words + 3) & ~(size_t)3; }

// Word offsets of the plan inside the scratch array (every part 16-byte aligned).
struct Layout {
  size_t work, row_ptr, counts, live_off, totals, col_idx, tile_order, empty, end;
};

Layout layout_for(size_t BH, size_t nb) {
  const size_t rows = BH * nb;
  Layout L{};
  L.work = 0;
  L.row_ptr = align4(L.work + kWorkWords);
  L.counts = align4(L.row_ptr + rows + 1);        // counts[rows] then live_per_head[BH]
  L.live_off = align4(L.counts + rows + BH);
  L.totals = align4(L.live_off + BH + 1);         // two int64
  L.col_idx = align4(L.totals + 4);               // worst case: every block live
  L.tile_order = align4(L.col_idx + rows * nb);
  L.empty = align4(L.tile_order + rows);
  L.end = align4(L.empty + rows);
  return L;
}

}  // namespace
}  // namespace bsattn

using namespace bsattn;

extern "C" bsattn_status bsattn_fwd_noalloc(const void* q, const void* k, const void* v,
                                            const uint8_t* d_mask, void* out, float* lse, int B,
                                            int H, int S, int D, float scale, unsigned flags,
                                            void* stream) {
  if (!q || !k || !v || !d_mask || !out || !lse) return BSATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return BSATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || S <= 0 || (S % kBlock) != 0) return BSATTN_ERR_INVALID_ARG;
  if (flags & ~(unsigned)(BSATTN_CAUSAL | BSATTN_OUT_F32)) return BSATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return BSATTN_ERR_UNSUPPORTED;
  const int nb = S / kBlock;
  if (nb > kMaxBlocksPerRow) return BSATTN_ERR_UNSUPPORTED;
  if ((long long)B * H * S >= (1ll << 31)) return BSATTN_ERR_UNSUPPORTED;
  const int BH = B * H;
  const int rows = BH * nb;
  const Layout L = layout_for((size_t)BH, (size_t)nb);
  if (L.end > kNoAllocWords) return BSATTN_ERR_SCRATCH_LIMIT;
  if (!get_tensor_map_encoder()) return BSATTN_ERR_CUDA;

  int* scratch = nullptr;
  bsattn_status rc = scratch_on_current_device(&scratch);
  if (rc != BSATTN_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSATTN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int causal = (flags & BSATTN_CAUSAL) ? 1 : 0;

  int* work = scratch + L.work;
  int* row_ptr = scratch + L.row_ptr;
  int* counts = scratch + L.counts;
  int* live_off = scratch + L.live_off;
  int* totals = scratch + L.totals;
  int* col_idx = scratch + L.col_idx;
  int* tile_order = scratch + L.tile_order;
  int* empty = scratch + L.empty;

  // The tile counter, finished-CTA count and status word must start at zero.
  cudaError_t e = cudaMemsetAsync(work, 0, sizeof(int) * kWorkWords, st);
  if (e != cudaSuccess) return from_cuda(e);
  e = plan_count_and_scan(d_mask, BH, nb, causal, counts, row_ptr, live_off, totals, st);
  if (e != cudaSuccess) return from_cuda(e);
  long long h_tot[2] = {0, 0};
  if ((e = cudaMemcpyAsync(h_tot, totals, sizeof(h_tot), cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return from_cuda(e);
  const long long n_live = h_tot[1];
  if (h_tot[0] < 0 || h_tot[0] > (long long)rows * nb || n_live < 0 || n_live > rows)
    return BSATTN_ERR_INTERNAL;
  e = plan_fill_and_order(d_mask, BH, nb, causal, row_ptr, live_off, col_idx, tile_order, empty,
                          device_sm_count(dev), st);
  if (e != cudaSuccess) return from_cuda(e);

  const long long nrows = (long long)B * H * S;
  CUtensorMap tq, tk, tv;
  if ((rc = encode_bf16_map(&tq, q, D, nrows)) != BSATTN_OK) return rc;
  if ((rc = encode_bf16_map(&tk, k, D, nrows)) != BSATTN_OK) return rc;
  if ((rc = encode_bf16_map(&tv, v, D, nrows)) != BSATTN_OK) return rc;

  FwdParams prm{};
  prm.row_ptr = row_ptr;
  prm.col_idx = col_idx;
  prm.tile_order = tile_order;
  prm.empty_tiles = empty;
  prm.out = out;
  prm.lse = lse;
  prm.counter = work + kWorkCounter;
  prm.done = work + kWorkDone;
  prm.status = work + kWorkStatus;
  prm.n_live = (int)n_live;
  prm.n_empty = (int)(rows - n_live);
  prm.nb = nb;
  prm.S = S;
  set_scale_params(prm, scale);
  prm.causal = causal;
  prm.timeout_ns = kDefaultWaitTimeoutNs;
  e = launch_fwd(D, (flags & BSATTN_OUT_F32) != 0, tq, tk, tv, prm, device_sm_count(dev), st);
  if (e != cudaSuccess) return from_cuda(e);

  // Report what the kernel recorded (timeout / internal) before returning.
  int status = 0;
  if ((e = cudaMemcpyAsync(&status, work + kWorkStatus, sizeof(int), cudaMemcpyDeviceToHost,
                           st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return from_cuda(e);
  if (status & kStatusInternal) return BSATTN_ERR_INTERNAL;
  if (status & kStatusTimeout) return BSATTN_ERR_TIMEOUT;
  if (status & kStatusRange) return BSATTN_ERR_RANGE;
  return BSATTN_OK;
}
