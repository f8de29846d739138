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
// which lists kb ascending with mask != 0 (and kb <= qb when causal).  The
// mask of head (b*H + h) is mask[(b*H + h) / mdiv]: mdiv = 1 for one mask per
// head, H for one mask per batch entry shared by its heads.
// Schedule: non-empty tiles in chunks of consecutive heads (so a chunk's K/V
// stay resident in L2 while its tiles run), inside a chunk sorted by live
// count descending (longest-processing-time first), with the few tiles that
// are long for their chunk moved one chunk earlier (see order_kernel); empty
// tiles listed separately (the forward kernel writes O = 0, LSE = -inf there).
// The transposed plan (col_ptr / row_idx: per key block, the ascending live
// query blocks) drives the backward kernel, one CTA per key block.
#include <cstdint>

#include "internal.h"

namespace bsattn {
namespace {

constexpr int kScanThreads = 1024;
// Key blocks of K/V per schedule chunk: 768 blocks of 128 keys x D=128 bf16
// K and V = 48 MB, well inside the 126 MB L2.
#ifndef BSATTN_SCHED_CHUNK_BLOCKS
#define BSATTN_SCHED_CHUNK_BLOCKS 768
#endif
constexpr int kChunkKeyBlocks = BSATTN_SCHED_CHUNK_BLOCKS;

// Key blocks are 128 / kdiv keys (kdiv = 1: 128, kdiv = 2: 64); a query
// block qb (128 queries) has kdiv * nb key blocks per mask row.  Under causal
// a key block is kept when its first key is <= the tile's last query, i.e.
// kb < (qb + 1) * kdiv.
__device__ __forceinline__ bool block_live(const uint8_t* mask_row, int kb, int qb, int causal,
                                           int kdiv) {
  return mask_row[kb] != 0 && (!causal || kb < (qb + 1) * kdiv);
}

// One warp per CSR row: number of live key blocks.  Also counts, per head, the
// rows with at least one live block.
__global__ void count_kernel(const uint8_t* __restrict__ mask, int rows, int nb, int kdiv,
                             int causal, int mdiv, int* __restrict__ counts,
                             int* __restrict__ live_per_head) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int qb = warp % nb;
  const int nbk = nb * kdiv;
  const uint8_t* mrow = mask + ((size_t)(warp / nb / mdiv) * nb + qb) * nbk;
  int c = 0;
  for (int kb = lane; kb < nbk; kb += 32) c += block_live(mrow, kb, qb, causal, kdiv) ? 1 : 0;
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
__global__ void fill_kernel(const uint8_t* __restrict__ mask, int rows, int nb, int kdiv,
                            int causal, int mdiv, const int* __restrict__ row_ptr,
                            int* __restrict__ col_idx) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int qb = warp % nb;
  const int nbk = nb * kdiv;
  const uint8_t* mrow = mask + ((size_t)(warp / nb / mdiv) * nb + qb) * nbk;
  int base = row_ptr[warp];
  for (int kb0 = 0; kb0 < nbk; kb0 += 32) {
    const int kb = kb0 + lane;
    const bool live = kb < nbk && block_live(mrow, kb, qb, causal, kdiv);
    const unsigned bal = __ballot_sync(0xffffffffu, live);
    if (live) col_idx[base + __popc(bal & ((1u << lane) - 1u))] = kb;
    base += __popc(bal);
  }
}

// One block per chunk of `kh` consecutive heads (the heads whose K/V fill
// about kChunkKeyBlocks key blocks, so that a chunk's K/V stay resident in L2
// while its tiles run).  The chunk's tiles are sorted by live count
// descending, ties by (head, qb) ascending (longest-processing-time first).
// A tile of chunk k > 0 whose count exceeds half of chunk k's blocks per SM
// (`nsm` SMs) is moved into chunk k-1: such a tile alone is about as long as
// the chunk's whole share per SM, and at the end of the schedule it would
// run long after every other SM has finished.  Chunk k's slice of tile_order
// therefore holds its own short enough tiles plus the long tiles of chunk
// k+1, and starts at (live tiles of chunks < k) + (tiles moved out of chunk
// k).  Empty tiles are listed head by head, qb ascending.  With kdiv = 2
// (64-key blocks, run in pairs) a tile's length is its pairs,
// ceil(live blocks / 2), and a chunk's blocks count in pairs likewise.
// With empty_rev > 0, empty tile number e is written to
// empty_tiles[empty_rev - 1 - e] instead of empty_tiles[e] (so that one array
// of empty_rev entries holds the live tiles in order followed by the empty ones).
__global__ void __launch_bounds__(1024)
    order_kernel(const int* __restrict__ row_ptr, const int* __restrict__ live_off, int BH, int nb,
                 int kdiv, int kh, int nsm, int* __restrict__ tile_order,
                 int* __restrict__ empty_tiles, int empty_rev) {
  extern __shared__ uint32_t keys[];
  __shared__ int n_in, n_moved;
  const int k = blockIdx.x;
  const int h0 = k * kh;
  const int h1 = min(BH, h0 + kh);  // own heads [h0, h1)
  const int h2 = min(BH, h1 + kh);  // next chunk's heads [h1, h2)
  // a count above thr is "long" in its chunk
  const long long thr_own =
      (long long)(row_ptr[h1 * nb] - row_ptr[h0 * nb]) / kdiv / (2ll * nsm);
  const long long thr_next =
      (h2 > h1) ? (long long)(row_ptr[h2 * nb] - row_ptr[h1 * nb]) / kdiv / (2ll * nsm)
                : (1ll << 40);
  const int own = (h1 - h0) * nb;
  const int pool = (h2 - h0) * nb;
  int n2 = 1;
  while (n2 < pool) n2 <<= 1;
  if (threadIdx.x == 0) {
    n_in = 0;
    n_moved = 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    uint32_t key = 0xFFFFFFFFu;
    if (i < pool) {
      const int r = h0 * nb + i;
      const int cnt = (row_ptr[r + 1] - row_ptr[r] + kdiv - 1) / kdiv;  // blocks, or pairs
      bool in;
      if (i < own) {
        const bool moved = k > 0 && cnt > thr_own;
        if (moved && cnt > 0) atomicAdd(&n_moved, 1);
        in = cnt > 0 && !moved;
      } else {
        in = cnt > 0 && cnt > thr_next;
      }
      if (in) {
        key = ((uint32_t)(nb - cnt) << 14) | (uint32_t)i;  // i < 2^14: pool <= 2 * 4096
        atomicAdd(&n_in, 1);
      }
    }
    keys[i] = key;
  }
  __syncthreads();
  for (int kk = 2; kk <= n2; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int p = i ^ j;
        if (p > i) {
          const uint32_t a = keys[i], b = keys[p];
          const bool up = (i & kk) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const int start = live_off[h0] + n_moved;
  for (int i = threadIdx.x; i < n_in; i += blockDim.x)
    tile_order[start + i] = h0 * nb + (int)(keys[i] & 0x3FFFu);
  // empty tiles: one warp per own head, qb ascending
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int h = h0 + warp; h < h1; h += blockDim.x >> 5) {
    int pos = h * nb - live_off[h];
    for (int q0 = 0; q0 < nb; q0 += 32) {
      const int qb = q0 + lane;
      const int r = h * nb + qb;
      const bool empty = qb < nb && row_ptr[r + 1] == row_ptr[r];
      const unsigned bal = __ballot_sync(0xffffffffu, empty);
      if (empty) {
        const int e = pos + __popc(bal & ((1u << lane) - 1u));
        empty_tiles[empty_rev > 0 ? empty_rev - 1 - e : e] = r;
      }
      pos += __popc(bal);
    }
  }
}

// Transposed plan, one warp per key block c = (b*H + h)*nb + kb: the query
// blocks qb with mask[b][h][qb][kb] != 0 (and qb >= kb when causal).
__device__ __forceinline__ bool col_live(const uint8_t* mask_bh, int nb, int qb, int kb,
                                         int causal) {
  return mask_bh[(size_t)qb * nb + kb] != 0 && (!causal || qb >= kb);
}

__global__ void csc_count_kernel(const uint8_t* __restrict__ mask, int cols, int nb, int causal,
                                 int mdiv, int* __restrict__ counts,
                                 int* __restrict__ live_per_head) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= cols) return;
  const int kb = warp % nb;
  const uint8_t* mbh = mask + (size_t)(warp / nb / mdiv) * nb * nb;
  int c = 0;
  for (int qb = lane; qb < nb; qb += 32) c += col_live(mbh, nb, qb, kb, causal) ? 1 : 0;
  c = __reduce_add_sync(0xffffffffu, c);
  if (lane == 0) {
    counts[warp] = c;
    if (c > 0) atomicAdd(&live_per_head[warp / nb], 1);
  }
}

__global__ void csc_fill_kernel(const uint8_t* __restrict__ mask, int cols, int nb, int causal,
                                int mdiv, const int* __restrict__ col_ptr,
                                int* __restrict__ row_idx) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= cols) return;
  const int kb = warp % nb;
  const uint8_t* mbh = mask + (size_t)(warp / nb / mdiv) * nb * nb;
  int pos = col_ptr[warp];
  for (int q0 = 0; q0 < nb; q0 += 32) {
    const int qb = q0 + lane;
    const bool live = qb < nb && col_live(mbh, nb, qb, kb, causal);
    const unsigned bal = __ballot_sync(0xffffffffu, live);
    if (live) row_idx[pos + __popc(bal & ((1u << lane) - 1u))] = qb;
    pos += __popc(bal);
  }
}

}  // namespace

cudaError_t plan_count_and_scan(const uint8_t* d_mask, int BH, int nb, int causal, int* d_counts,
                                int* d_row_ptr, int* d_live_off, int* d_totals,
                                cudaStream_t stream, int mdiv, int kdiv) {
  const int rows = BH * nb;
  int* live_per_head = d_counts + rows;  // caller sized d_counts as rows + BH
  cudaError_t e = cudaMemsetAsync(live_per_head, 0, sizeof(int) * BH, stream);
  if (e != cudaSuccess) return e;
  const int warps_per_block = 8;
  const int grid = (rows + warps_per_block - 1) / warps_per_block;
  count_kernel<<<grid, 32 * warps_per_block, 0, stream>>>(d_mask, rows, nb, kdiv, causal, mdiv,
                                                          d_counts, live_per_head);
  scan_kernel<<<1, kScanThreads, 0, stream>>>(d_counts, rows, live_per_head, BH, d_row_ptr,
                                              d_live_off, reinterpret_cast<long long*>(d_totals));
  return cudaGetLastError();
}

int schedule_chunk_heads(int nb) { return nb >= kChunkKeyBlocks ? 1 : kChunkKeyBlocks / nb; }

cudaError_t plan_fill_and_order(const uint8_t* d_mask, int BH, int nb, int causal,
                                const int* d_row_ptr, const int* d_live_off, int* d_col_idx,
                                int* d_tile_order, int* d_empty_tiles, int nsm,
                                cudaStream_t stream, int mdiv, int kdiv) {
  const int rows = BH * nb;
  const int warps_per_block = 8;
  const int grid = (rows + warps_per_block - 1) / warps_per_block;
  fill_kernel<<<grid, 32 * warps_per_block, 0, stream>>>(d_mask, rows, nb, kdiv, causal, mdiv,
                                                         d_row_ptr, d_col_idx);
  const int kh = schedule_chunk_heads(nb);
  const int chunks = (BH + kh - 1) / kh;
  int n2 = 1;
  while (n2 < 2 * kh * nb) n2 <<= 1;
  order_kernel<<<chunks, 1024, sizeof(uint32_t) * n2, stream>>>(
      d_row_ptr, d_live_off, BH, nb, kdiv, kh, nsm > 0 ? nsm : 1, d_tile_order, d_empty_tiles, 0);
  return cudaGetLastError();
}

cudaError_t plan_csc(const uint8_t* d_mask, int BH, int nb, int causal, int* d_counts,
                     int* d_live_off, int* d_totals, int* d_col_ptr, int* d_row_idx,
                     int* d_kv_order, int nsm, cudaStream_t stream, int mdiv) {
  const int cols = BH * nb;
  int* live_per_head = d_counts + cols;  // caller sized d_counts as cols + BH
  cudaError_t e = cudaMemsetAsync(live_per_head, 0, sizeof(int) * BH, stream);
  if (e != cudaSuccess) return e;
  const int warps_per_block = 8;
  const int grid = (cols + warps_per_block - 1) / warps_per_block;
  csc_count_kernel<<<grid, 32 * warps_per_block, 0, stream>>>(d_mask, cols, nb, causal, mdiv,
                                                              d_counts, live_per_head);
  scan_kernel<<<1, kScanThreads, 0, stream>>>(d_counts, cols, live_per_head, BH, d_col_ptr,
                                              d_live_off, reinterpret_cast<long long*>(d_totals));
  csc_fill_kernel<<<grid, 32 * warps_per_block, 0, stream>>>(d_mask, cols, nb, causal, mdiv,
                                                             d_col_ptr, d_row_idx);
  // the key tiles for the dK/dV kernel: the same longest-first order within
  // head chunks as the forward tiles, empty key tiles at the end
  const int kh = schedule_chunk_heads(nb);
  const int chunks = (BH + kh - 1) / kh;
  int n2 = 1;
  while (n2 < 2 * kh * nb) n2 <<= 1;
  order_kernel<<<chunks, 1024, sizeof(uint32_t) * n2, stream>>>(
      d_col_ptr, d_live_off, BH, nb, 1, kh, nsm > 0 ? nsm : 1, d_kv_order, d_kv_order, cols);
  return cudaGetLastError();
}

}  // namespace bsattn
