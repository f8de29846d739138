// bsattn_pipeline_*: forward passes on host-resident tensors, the transfers
// of one part of the (batch, head) range overlapping the kernel of another.
//
// Per part c of a run (three streams, events ordering them):
//   upload stream   waits until run-1's kernel of part c is done with the
//                   part's input buffers, copies its Q, K, V in, records in[c]
//   kernel stream   waits for in[c] and for run-1's download of part c (the
//                   output buffers), launches the prepared forward, records
//                   done[c]
//   download stream waits for done[c], copies O and LSE out, records out[c]
// The caller's stream first releases the upload stream (start event) and at
// the end waits for the download stream (end event).  Each part's launch is
// prepared at creation (tensor maps and kernel parameters over the
// pipeline's fixed device buffers), so a run only enqueues copies, event
// operations and launches.
#include <cmath>
#include <new>
#include <vector>

#include "internal.h"

namespace {

constexpr uint32_t kPipeMagic = 0x42535050u;  // "BSPP"

}  // namespace

struct bsattn_pipeline_s {
  uint32_t magic = 0;
  int B = 0, H = 0, S = 0, D = 0;
  unsigned flags = 0;
  int device = 0;
  size_t out_elem = 2;
  std::vector<int> edge;  // part c covers flattened heads [edge[c], edge[c+1])
  std::vector<bsattn_plan_t> plans;
  std::vector<bsattn::PreparedFwd> prep;
  void* dq = nullptr;
  void* dk = nullptr;
  void* dv = nullptr;
  void* dout = nullptr;
  float* dlse = nullptr;
  cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> ev_in, ev_done, ev_out;
  cudaEvent_t ev_start = nullptr, ev_end = nullptr;
};

namespace {

bool pipe_ok(const bsattn_pipeline_s* p) { return p != nullptr && p->magic == kPipeMagic; }

void release(bsattn_pipeline_s* p) {
  for (bsattn_plan_t pl : p->plans) bsattn_plan_free(pl);
  p->plans.clear();
  cudaFree(p->dq);
  cudaFree(p->dk);
  cudaFree(p->dv);
  cudaFree(p->dout);
  cudaFree(p->dlse);
  for (auto* v : {&p->ev_in, &p->ev_done, &p->ev_out})
    for (cudaEvent_t e : *v)
      if (e) cudaEventDestroy(e);
  if (p->ev_start) cudaEventDestroy(p->ev_start);
  if (p->ev_end) cudaEventDestroy(p->ev_end);
  for (cudaStream_t s : {p->s_in, p->s_run, p->s_out})
    if (s) cudaStreamDestroy(s);
}

}  // namespace

using namespace bsattn;

extern "C" bsattn_status bsattn_pipeline_create(const uint8_t* d_mask, int B, int H, int S, int D,
                                                unsigned flags, int pieces, void* stream,
                                                bsattn_pipeline_t* out) {
  if (!d_mask || !out) return BSATTN_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || S <= 0 || (S % kBlock) != 0) return BSATTN_ERR_INVALID_ARG;
  if (flags & ~(unsigned)(BSATTN_CAUSAL | BSATTN_OUT_F32)) return BSATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return BSATTN_ERR_UNSUPPORTED;
  if ((long long)B * H * S >= (1ll << 31)) return BSATTN_ERR_UNSUPPORTED;
  const int BH = B * H;
  const int nb = S / kBlock;
  if (nb > kMaxBlocksPerRow) return BSATTN_ERR_UNSUPPORTED;
  if (pieces < 1) pieces = 1;
  if (pieces > BH) pieces = BH;

  bsattn_pipeline_s* p = new (std::nothrow) bsattn_pipeline_s();
  if (!p) return BSATTN_ERR_OOM;
  auto fail = [&](bsattn_status s) {
    release(p);
    delete p;
    return s;
  };
  p->B = B;
  p->H = H;
  p->S = S;
  p->D = D;
  p->flags = flags;
  p->out_elem = (flags & BSATTN_OUT_F32) ? 4 : 2;
  if (cudaGetDevice(&p->device) != cudaSuccess) return fail(BSATTN_ERR_CUDA);

  const size_t rows = (size_t)BH * S;
  cudaError_t e;
  if ((e = cudaMalloc(&p->dq, rows * D * 2)) != cudaSuccess ||
      (e = cudaMalloc(&p->dk, rows * D * 2)) != cudaSuccess ||
      (e = cudaMalloc(&p->dv, rows * D * 2)) != cudaSuccess ||
      (e = cudaMalloc(&p->dout, rows * D * p->out_elem)) != cudaSuccess ||
      (e = cudaMalloc(&p->dlse, rows * sizeof(float))) != cudaSuccess)
    return fail(from_cuda(e));
  for (cudaStream_t* s : {&p->s_in, &p->s_run, &p->s_out})
    if ((e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking)) != cudaSuccess)
      return fail(from_cuda(e));
  for (auto* v : {&p->ev_in, &p->ev_done, &p->ev_out}) {
    v->assign(pieces, nullptr);
    for (cudaEvent_t& ev : *v)
      if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
        return fail(from_cuda(e));
  }
  if ((e = cudaEventCreateWithFlags(&p->ev_start, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreateWithFlags(&p->ev_end, cudaEventDisableTiming)) != cudaSuccess)
    return fail(from_cuda(e));

  p->edge.resize(pieces + 1);
  for (int c = 0; c <= pieces; ++c) p->edge[c] = (int)((long long)BH * c / pieces);
  p->prep.resize(pieces);
  for (int c = 0; c < pieces; ++c) {
    const int a = p->edge[c], h = p->edge[c + 1] - a;
    bsattn_plan_t pl = nullptr;
    bsattn_status rc = bsattn_plan(d_mask + (size_t)a * nb * nb, 1, h, S, flags, stream, &pl);
    if (rc != BSATTN_OK) return fail(rc);
    p->plans.push_back(pl);
    const size_t off = (size_t)a * S * D;
    rc = prepare_fwd(static_cast<const char*>(p->dq) + off * 2,
                     static_cast<const char*>(p->dk) + off * 2,
                     static_cast<const char*>(p->dv) + off * 2, pl,
                     static_cast<char*>(p->dout) + off * p->out_elem, p->dlse + (size_t)a * S, 1,
                     h, S, D, 1.0f, &p->prep[c], h, false, 1.0f, true,
                     static_cast<cudaStream_t>(stream));
    if (rc != BSATTN_OK) return fail(rc);
  }
  // the parts' fp16 V copies (head_dim 64) are allocated on `stream`; the
  // runs use them from the pipeline's own streams
  if ((e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return fail(from_cuda(e));
  p->magic = kPipeMagic;
  *out = p;
  return BSATTN_OK;
}

extern "C" bsattn_status bsattn_pipeline_run(bsattn_pipeline_t p, const void* hq, const void* hk,
                                             const void* hv, void* hout, float* hlse, float scale,
                                             void* stream) {
  if (!pipe_ok(p) || !hq || !hk || !hv || !hout || !hlse) return BSATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return BSATTN_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) return BSATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t S = p->S, D = p->D;
  cudaError_t e;
#define BSATTN_TRY(x) \
  if ((e = (x)) != cudaSuccess) return from_cuda(e)
  BSATTN_TRY(cudaEventRecord(p->ev_start, st));
  BSATTN_TRY(cudaStreamWaitEvent(p->s_in, p->ev_start, 0));
  const int pieces = (int)p->prep.size();
  for (int c = 0; c < pieces; ++c) {
    const size_t a = p->edge[c], h = p->edge[c + 1] - a;
    const size_t off = a * S * D, n = h * S * D;
    // inputs of part c (the previous run's kernel must be done with them)
    BSATTN_TRY(cudaStreamWaitEvent(p->s_in, p->ev_done[c], 0));
    BSATTN_TRY(cudaMemcpyAsync(static_cast<char*>(p->dq) + off * 2,
                               static_cast<const char*>(hq) + off * 2, n * 2,
                               cudaMemcpyHostToDevice, p->s_in));
    BSATTN_TRY(cudaMemcpyAsync(static_cast<char*>(p->dk) + off * 2,
                               static_cast<const char*>(hk) + off * 2, n * 2,
                               cudaMemcpyHostToDevice, p->s_in));
    BSATTN_TRY(cudaMemcpyAsync(static_cast<char*>(p->dv) + off * 2,
                               static_cast<const char*>(hv) + off * 2, n * 2,
                               cudaMemcpyHostToDevice, p->s_in));
    BSATTN_TRY(cudaEventRecord(p->ev_in[c], p->s_in));
    // kernel of part c (the previous run's download must be done with its outputs)
    BSATTN_TRY(cudaStreamWaitEvent(p->s_run, p->ev_in[c], 0));
    BSATTN_TRY(cudaStreamWaitEvent(p->s_run, p->ev_out[c], 0));
    set_scale_params(p->prep[c].prm, scale);
    BSATTN_TRY(launch_prepared(p->prep[c], p->s_run));
    BSATTN_TRY(cudaEventRecord(p->ev_done[c], p->s_run));
    // results of part c
    BSATTN_TRY(cudaStreamWaitEvent(p->s_out, p->ev_done[c], 0));
    BSATTN_TRY(cudaMemcpyAsync(static_cast<char*>(hout) + off * p->out_elem,
                               static_cast<const char*>(p->dout) + off * p->out_elem,
                               n * p->out_elem, cudaMemcpyDeviceToHost, p->s_out));
    BSATTN_TRY(cudaMemcpyAsync(hlse + a * S, p->dlse + a * S, h * S * sizeof(float),
                               cudaMemcpyDeviceToHost, p->s_out));
    BSATTN_TRY(cudaEventRecord(p->ev_out[c], p->s_out));
  }
  BSATTN_TRY(cudaEventRecord(p->ev_end, p->s_out));
  BSATTN_TRY(cudaStreamWaitEvent(st, p->ev_end, 0));
#undef BSATTN_TRY
  return BSATTN_OK;
}

extern "C" bsattn_status bsattn_pipeline_status(bsattn_pipeline_t p) {
  if (!pipe_ok(p)) return BSATTN_ERR_INVALID_ARG;
  for (cudaStream_t s : {p->s_in, p->s_run, p->s_out})
    if (cudaStreamSynchronize(s) != cudaSuccess) return BSATTN_ERR_CUDA;
  bsattn_status worst = BSATTN_OK;
  for (bsattn_plan_t pl : p->plans) {
    const bsattn_status rc = bsattn_plan_status(pl, p->s_run);
    if (rc != BSATTN_OK && worst == BSATTN_OK) worst = rc;
  }
  return worst;
}

extern "C" void bsattn_pipeline_free(bsattn_pipeline_t p) {
  if (!pipe_ok(p)) return;
  for (cudaStream_t s : {p->s_in, p->s_run, p->s_out}) cudaStreamSynchronize(s);
  release(p);
  p->magic = 0;
  delete p;
}
