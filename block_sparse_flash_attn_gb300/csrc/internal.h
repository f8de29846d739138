// Internal declarations shared by the host API (api.cu), the plan kernels
// (plan.cu) and the forward kernel (fwd_sm103.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "bsattn.h"

namespace bsattn {

constexpr int kBlock = 128;           // query tile rows = key block rows = mask granularity
constexpr int kMaxBlocksPerRow = 4096;
constexpr uint32_t kPlanMagic = 0x42535041u;  // "BSPA"

// Status bits written by kernels into the caller's status word.
// kStatusRange: an input value the kernel's arithmetic cannot hold (see
// BSATTN_ERR_RANGE).
enum : int { kStatusTimeout = 1, kStatusInternal = 2, kStatusRange = 4 };

// Device workspace words owned by a plan.
enum : int { kWorkCounter = 0, kWorkStatus = 1, kWorkDone = 2, kWorkWords = 4 };

struct PlanDevice {
  int* row_ptr = nullptr;      // [R + 1]
  int* col_idx = nullptr;      // [nnz]
  int* tile_order = nullptr;   // [n_live] non-empty tiles, head-major, longest first
  int* empty_tiles = nullptr;  // [n_empty]
  int* work = nullptr;         // [kWorkWords] tile counter, status word
  // transposed plan: per key block c = (b*H + h)*nb + kb, the ascending live
  // query blocks row_idx[col_ptr[c] .. col_ptr[c+1])
  int* col_ptr = nullptr;      // [R + 1]
  int* row_idx = nullptr;      // [nnz]
  // key tiles in the dK/dV kernel's launch order: those with live query
  // blocks longest first (within head chunks, as tile_order), then the empty ones
  int* kv_order = nullptr;     // [R]
  float* dl = nullptr;         // [B*H*S] backward scratch: dO_i . O_i
  // head_dim-64 forward: an fp16 copy of V (allocated by the first forward
  // call that uses it, stream-ordered; grows when a call needs more)
  void* v16 = nullptr;
  size_t v16_bytes = 0;
};

// Everything the forward kernel needs besides the three tensor maps.
struct FwdParams {
  const int* row_ptr;
  const int* col_idx;
  const int* tile_order;
  const int* empty_tiles;
  void* out;
  float* lse;
  int* counter;  // tile counter, zero at launch; rewound by the last CTA
  int* done;     // CTAs finished
  int* status;
  int n_live;
  int n_empty;
  int nb;            // S / 128
  int S;
  float scale_log2;  // |scale| * log2(e) (> 0; a tiny positive value stands in for scale = 0)
  int neg_scale;     // scale < 0: the S MMA computes -Q K^T
  int causal;
  unsigned long long timeout_ns;
  // grouped-query attention: query head h of a batch entry reads K/V head
  // h / kv_group (H query heads, H / kv_group K/V heads); 1 = one K/V head per
  // query head
  int H = 1;
  int kv_group = 1;
  // multiplies O (the scale of e4m3 V; 1 for bf16 inputs)
  float v_scale = 1.0f;
  // key blocks of 128 / kdiv keys: 2 = 64-key blocks, which the kernel runs in
  // pairs (two consecutive entries of a tile's list fill one 128-key stage;
  // the K and V tensor maps then have 64-row boxes)
  int kdiv = 1;
  // P V in fp16 (head_dim 64, or e4m3 inputs): V's tensor map reads an fp16
  // copy of V written before the launch (v16_convert_kernel, or the e4m3
  // one), so the epilogue warps do not convert each V tile in shared memory
  int v_pre = 0;
};


constexpr unsigned long long kDefaultWaitTimeoutNs = 2000ull * 1000 * 1000;  // 2 s per wait

// api.cu helpers
void set_scale_params(FwdParams& p, float scale);
bool get_tensor_map_encoder();
int device_sm_count(int dev);
bool aligned16(const void* p);
bsattn_status from_cuda(cudaError_t e);
bsattn_status encode_bf16_map(CUtensorMap* m, const void* ptr, int D, long long rows,
                              int box_rows = kBlock);
bsattn_status encode_e4m3_map(CUtensorMap* m, const void* ptr, int D, long long rows,
                              int box_rows = kBlock);

// One forward launch with everything resolved: tensor maps, kernel
// parameters, grid.  prepare_fwd checks the arguments exactly as bsattn_fwd
// does; launch_prepared only launches.
struct PreparedFwd {
  CUtensorMap tq, tk, tv;
  FwdParams prm;
  int D = 0;
  bool out_f32 = false;
  bool in8 = false;
  int grid = 0;
  // prm.v_pre: convert v_src (bf16) into v16 (fp16, v16_elems values) first
  const void* v_src = nullptr;
  void* v16 = nullptr;
  long long v16_elems = 0;
};
// The V conversion pass (fp16 P V) runs when V has at least kV16MinRows rows
// (2 MiB; below, its launch costs more than it saves) and the plan has at
// least kV16MinReuse live blocks per key block of V on average (the kernel
// would otherwise convert each V tile that many times).
constexpr long long kV16MinRows = 16384;
constexpr long long kV16MinReuse = 4;
// Hkv: K/V heads (H % Hkv == 0; Hkv == H for plain multi-head attention).
// in8: q, k, v are e4m3 (D = 128); v_scale multiplies O.
// v16_ok: where P V runs in fp16 (head_dim 64, or e4m3 inputs) the call may
// give V an fp16 copy in the plan's scratch (allocated on `stream` when
// missing, never during stream capture), converted once per launch instead
// of once per query tile in the kernel.
bsattn_status prepare_fwd(const void* q, const void* k, const void* v, bsattn_plan_t plan,
                          void* out, float* lse, int B, int H, int S, int D, float scale,
                          PreparedFwd* pf, int Hkv, bool in8 = false, float v_scale = 1.0f,
                          bool v16_ok = false, cudaStream_t stream = nullptr);
cudaError_t launch_prepared(const PreparedFwd& pf, cudaStream_t stream);

// plan.cu
// mdiv: head (b*H + h) reads mask (b*H + h) / mdiv (1: a mask per head; H: one
// mask per batch entry shared by its heads)
// kdiv: key blocks of 128 / kdiv keys (1: 128-key blocks, the mask is
// [nb][nb] per head; 2: 64-key blocks, [nb][2 nb]); the CSR then lists 64-key
// blocks, and the schedule counts a tile's length in pairs of them.
cudaError_t plan_count_and_scan(const uint8_t* d_mask, int BH, int nb, int causal, int* d_counts,
                                int* d_row_ptr, int* d_live_off, int* d_totals,
                                cudaStream_t stream, int mdiv = 1, int kdiv = 1);
cudaError_t plan_fill_and_order(const uint8_t* d_mask, int BH, int nb, int causal,
                                const int* d_row_ptr, const int* d_live_off, int* d_col_idx,
                                int* d_tile_order, int* d_empty_tiles, int nsm,
                                cudaStream_t stream, int mdiv = 1, int kdiv = 1);
// Transposed plan (per key block, the ascending live query blocks); d_counts
// is scratch of R ints.
cudaError_t plan_csc(const uint8_t* d_mask, int BH, int nb, int causal, int* d_counts,
                     int* d_live_off, int* d_totals, int* d_col_ptr, int* d_row_idx,
                     int* d_kv_order, int nsm, cudaStream_t stream, int mdiv = 1);
// Heads per schedule chunk for S/128 = nb key blocks per head.
int schedule_chunk_heads(int nb);

// fwd_sm103.cu
// in8: Q, K, V are e4m3 (D = 128 only; the tensor maps are of uint8 elements)
// bf16 -> fp16 copy of V (n values, a multiple of 8, both pointers 16-byte
// aligned); a value fp16 cannot hold (|v| > 65504, inf, NaN) sets kStatusRange.
cudaError_t launch_v16_convert(const void* v, void* v16, long long n, int* status, int grid,
                               cudaStream_t stream);
// The same from e4m3 V (n a multiple of 16); an e4m3 NaN sets kStatusRange.
cudaError_t launch_v16_convert_e4m3(const void* v8, void* v16, long long n, int* status,
                                    int grid, cudaStream_t stream);
cudaError_t launch_fwd(int D, bool out_f32, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t stream,
                       bool in8 = false);
size_t fwd_smem_bytes(int D);
cudaError_t launch_selftest_wait(unsigned long long timeout_ns, int* d_status,
                                 cudaStream_t stream);


}  // namespace bsattn
