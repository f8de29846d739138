// Plan kernels: block mask -> per-query-tile CSR of live key blocks, and the
// tile schedule used by the forward kernel.
//
// The block mask is the one of "Writing Pallas Kernels for JAX: Stepping
// Outside the XLA Safety Net" (section "Designing the Block Specification":
// one entry per (128-query block, 128-key block) pair).  Instead of a grid
// over every (query block, key block) pair (section "Deploying via JAX Pallas
// Call"), the forward kernel walks, for each query tile, only the list built
// here, so dead blocks cost nothing.
//
// Layout: row r = (b*H + h)*nb + qb; row_ptr[r]..row_ptr[r+1] index col_idx,
// which lists kb ascending with mask != 0 (and kb <= qb when causal).
// Schedule: non-empty tiles grouped by head in head order (so one head's K/V
// stay resident in L2 while its tiles run), inside a head sorted by live
// count descending then qb ascending (longest-processing-time first); empty
// tiles listed separately (the forward kernel writes O = 0, LSE = -inf there).
#include <cstdint>

#include "internal.h"

namespace bsattn {
namespace {

constexpr int kScanThreads = 1024;

__device__ __forceinline__ bool block_live(const uint8_t* mask_row, int kb, int qb, int causal) {
  return mask_row[kb] != 0 && (!causal || kb <= qb);
}

// One warp per CSR row: number of live key blocks.  Also counts, per head, the
// rows with at least one live block.
__global__ void count_kernel(const uint8_t* __restrict__ mask, int rows, int nb, int causal,
                             int* __restrict__ counts, int* __restrict__ live_per_head) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int qb = warp % nb;
  const uint8_t* mrow = mask + (size_t)warp * nb;
  int c = 0;
  for (int kb = lane; kb < nb; kb += 32) c += block_live(mrow, kb, qb, causal) ? 1 : 0;
  c = __reduce_add_sync(0xffffffffu, c);
  if (lane == 0) {
    counts[warp] = c;
    if (c > 0) atomicAdd(&live_per_head[warp / nb], 1);
  }
}

// Exclusive scan of in[0..n) into out[0..n], out[n] = total (one 1024-thread
// block, each thread owning a contiguous chunk).  Returns the 64-bit total.
__device__ long long block_exclusive_scan(const int* __restrict__ in, int* __restrict__ out,
                                          int n, long long* sh) {
  const int t = threadIdx.x;
  const int chunk = (n + kScanThreads - 1) / kScanThreads;
  const int lo = min(n, t * chunk), hi = min(n, lo + chunk);
  long long s = 0;
  for (int i = lo; i < hi; ++i) s += in[i];
  sh[t] = s;
  __syncthreads();
  // Hillis-Steele inclusive scan over the 1024 partial sums.
  for (int off = 1; off < kScanThreads; off <<= 1) {
    long long v = (t >= off) ? sh[t - off] : 0;
    __syncthreads();
    sh[t] += v;
    __syncthreads();
  }
  long long run = sh[t] - s;
  for (int i = lo; i < hi; ++i) {
    out[i] = (int)run;
    run += in[i];
  }
  const long long total = sh[kScanThreads - 1];
  if (t == 0) out[n] = (int)total;
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kScanThreads)
    scan_kernel(const int* __restrict__ counts, int rows, const int* __restrict__ live_per_head,
                int heads, int* __restrict__ row_ptr, int* __restrict__ live_off,
                long long* __restrict__ totals) {
  __shared__ long long sh[kScanThreads];
  const long long nnz = block_exclusive_scan(counts, row_ptr, rows, sh);
  const long long live = block_exclusive_scan(live_per_head, live_off, heads, sh);
  if (threadIdx.x == 0) {
    totals[0] = nnz;
    totals[1] = live;
  }
}

// One warp per CSR row: write the live kb in ascending order.
__global__ void fill_kernel(const uint8_t* __restrict__ mask, int rows, int nb, int causal,
                            const int* __restrict__ row_ptr, int* __restrict__ col_idx) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int qb = warp % nb;
  const uint8_t* mrow = mask + (size_t)warp * nb;
  int base = row_ptr[warp];
  for (int kb0 = 0; kb0 < nb; kb0 += 32) {
    const int kb = kb0 + lane;
    const bool live = kb < nb && block_live(mrow, kb, qb, causal);
    const unsigned bal = __ballot_sync(0xffffffffu, live);
    if (live) col_idx[base + __popc(bal & ((1u << lane) - 1u))] = kb;
    base += __popc(bal);
  }
}

// One block per head: sort the head's tiles by (live count desc, qb asc) with
// a shared-memory bitonic sort, then split into the live and empty lists.
__global__ void __launch_bounds__(1024)
    order_kernel(const int* __restrict__ row_ptr, const int* __restrict__ live_off, int nb,
                 int* __restrict__ tile_order, int* __restrict__ empty_tiles) {
  extern __shared__ uint32_t keys[];
  const int bh = blockIdx.x;
  int n2 = 1;
  while (n2 < nb) n2 <<= 1;
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    if (i < nb) {
      const int r = bh * nb + i;
      const uint32_t cnt = (uint32_t)(row_ptr[r + 1] - row_ptr[r]);
      keys[i] = (((uint32_t)nb - cnt) << 12) | (uint32_t)i;
    } else {
      keys[i] = 0xFFFFFFFFu;
    }
  }
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const uint32_t a = keys[i], b = keys[p];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const int live0 = live_off[bh];
  const int nlive = live_off[bh + 1] - live0;
  const int empty0 = bh * nb - live0;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    const int qb = (int)(keys[i] & 0xFFFu);
    const int tile = bh * nb + qb;
    if (i < nlive) tile_order[live0 + i] = tile;
    else empty_tiles[empty0 + (i - nlive)] = tile;
  }
}

}  // namespace

cudaError_t plan_count_and_scan(const uint8_t* d_mask, int BH, int nb, int causal, int* d_counts,
                                int* d_row_ptr, int* d_live_off, int* d_totals,
                                cudaStream_t stream) {
  const int rows = BH * nb;
  int* live_per_head = d_counts + rows;  // caller sized d_counts as rows + BH
  cudaError_t e = cudaMemsetAsync(live_per_head, 0, sizeof(int) * BH, stream);
  if (e != cudaSuccess) return e;
  const int warps_per_block = 8;
  const int grid = (rows + warps_per_block - 1) / warps_per_block;
  count_kernel<<<grid, 32 * warps_per_block, 0, stream>>>(d_mask, rows, nb, causal, d_counts,
                                                          live_per_head);
  scan_kernel<<<1, kScanThreads, 0, stream>>>(d_counts, rows, live_per_head, BH, d_row_ptr,
                                              d_live_off, reinterpret_cast<long long*>(d_totals));
  return cudaGetLastError();
}

cudaError_t plan_fill_and_order(const uint8_t* d_mask, int BH, int nb, int causal,
                                const int* d_row_ptr, const int* d_live_off, int* d_col_idx,
                                int* d_tile_order, int* d_empty_tiles, cudaStream_t stream) {
  const int rows = BH * nb;
  const int warps_per_block = 8;
  const int grid = (rows + warps_per_block - 1) / warps_per_block;
  fill_kernel<<<grid, 32 * warps_per_block, 0, stream>>>(d_mask, rows, nb, causal, d_row_ptr,
                                                         d_col_idx);
  int n2 = 1;
  while (n2 < nb) n2 <<= 1;
  order_kernel<<<BH, 1024, sizeof(uint32_t) * n2, stream>>>(d_row_ptr, d_live_off, nb,
                                                            d_tile_order, d_empty_tiles);
  return cudaGetLastError();
}

}  // namespace bsattn
