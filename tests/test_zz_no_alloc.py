"""bsattn_fwd_noalloc: the forward pass for callers that cannot allocate GPU
memory (a framework that owns the device memory pool, a plug-in that may not
allocate once running, a loop that cannot absorb cudaMalloc's device-wide
synchronisation).  Its plan and scratch live in the library's fixed device
array, so it must give the same O and LSE as bsattn_plan + bsattn_fwd.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It builds the library itself
so it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import workloads
from _util import compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bs():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import block_sparse_flash_attn_gb300 as bs
    bs.load()
    return bs


def _case(seed, B, H, S, D, p, causal):
    rng = np.random.default_rng(seed)
    nb = S // 128
    mask = (rng.random((B, H, nb, nb)) < p).astype(np.uint8)
    mask[:, :, np.arange(nb), np.arange(nb)] = 1
    mask[0, 0, nb - 1] = 0  # one empty query tile
    q, k, v = workloads.custom(seed, B, H, S, D)
    return q, k, v, mask, causal


def _call_noalloc(bs, q, k, v, mask_d, causal, out_f32, scale):
    import torch
    lib = bs.load()
    B, H, S, D = q.shape
    out = torch.empty((B, H, S, D), dtype=torch.float32 if out_f32 else torch.bfloat16,
                      device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    flags = (bs.CAUSAL if causal else 0) | (bs.OUT_F32 if out_f32 else 0)
    vp = ctypes.c_void_p
    st = lib.bsattn_fwd_noalloc(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()),
                                vp(mask_d.data_ptr()), vp(out.data_ptr()), vp(lse.data_ptr()),
                                B, H, S, D, ctypes.c_float(scale), flags,
                                vp(torch.cuda.current_stream().cuda_stream))
    assert st == bs.OK, bs.status_string(st)
    return out, lse


def test_noalloc_matches_plan_and_fwd_on_two_calls(bs):
    import torch
    cases = [_case(501, 2, 4, 1024, 128, 0.4, True), _case(502, 1, 3, 512, 64, 0.6, False)]
    for i, (qb, kb, vb, mask, causal) in enumerate(cases):
        out_f32 = i == 0
        q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
        mask_d = torch.from_numpy(mask).cuda()
        scale = qb.shape[-1] ** -0.5
        # existing entry points
        p = bs.plan(mask_d, causal=causal, out_f32=out_f32)
        o_ref, l_ref = bs.fwd(q, k, v, p, scale)
        bs.plan_status(p)
        p.close()
        # the allocation-free entry point, through the C ABI
        o, l = _call_noalloc(bs, q, k, v, mask_d, causal, out_f32, scale)
        ok, rep = compare(o.float().cpu().numpy(), l.cpu().numpy(),
                          o_ref.float().cpu().numpy().astype(np.float64),
                          l_ref.cpu().numpy().astype(np.float64), out_bf16=not out_f32)
        assert ok, (i, rep)


def test_noalloc_rejects_problems_beyond_its_scratch(bs):
    import torch
    lib = bs.load()
    vp = ctypes.c_void_p
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    ptr = vp(buf.data_ptr())
    # 32 heads of S=65536 need about 8.4M words of plan, more than the 4M words available
    st = lib.bsattn_fwd_noalloc(ptr, ptr, ptr, ptr, ptr, ptr, 1, 32, 65536, 128,
                                ctypes.c_float(0.1), 0, vp(torch.cuda.current_stream().cuda_stream))
    assert st == bs.ERR_SCRATCH_LIMIT
