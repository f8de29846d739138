// Backward-pass declarations shared by the host API and the backward
// kernels (bwd_sm103.cu): kept apart from internal.h, whose contents the
// forward kernel depends on.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace bsattn {

// Everything the backward kernel needs besides its four tensor maps.
struct BwdParams {
  const int* col_ptr;  // transposed plan (dK, dV kernel)
  const int* row_idx;
  const int* row_ptr;  // forward plan (dQ kernel)
  const int* col_idx;
  const float* lse;  // natural-log LSE of the forward pass
  const float* dl;   // dO_i . O_i
  float* dq;
  float* dk;
  float* dv;
  int* status;
  int nb;
  int S;
  int causal;
  float scale;
  float scale_log2;  // scale * log2(e), signed
  unsigned long long timeout_ns;
  int H = 1;         // query heads; kv_group query heads share one K/V head
  int kv_group = 1;
  // launch orders: the dQ kernel's CTA i takes tile_order[i] (i < n_live),
  // then empty_tiles[i - n_live]; the dK/dV kernel's CTA i takes kv_order[i]
  // (kv_group == 1) or key tile i (grouped-query attention)
  const int* tile_order = nullptr;
  const int* empty_tiles = nullptr;
  const int* kv_order = nullptr;
  int n_live = 0;
};

// Dl = dO . O per row (row term of the gradients)
cudaError_t launch_bwd_prep(int D, bool o_f32, const void* o, const void* dout, float* dl,
                            long long rows, cudaStream_t stream);
// The backward pass: n_kv dK/dV CTAs (key tiles) and n_q dQ CTAs (query
// tiles) in one launch.
cudaError_t launch_bwd(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, int n_kv, int n_q,
                       cudaStream_t stream);

}  // namespace bsattn
