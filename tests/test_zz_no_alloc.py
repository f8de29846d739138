"""bsattn_fwd_noalloc: the forward pass for callers that cannot allocate GPU
memory (a framework that owns the device memory pool, a plug-in that may not
allocate once running, a loop that cannot absorb cudaMalloc's device-wide
synchronisation).  Its plan and scratch live in the library's fixed device
array; it must match the fp64 oracle at the forward tolerance, and give
the same O and LSE as bsattn_plan + bsattn_fwd.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It builds the library itself
so it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
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


def _outputs(q, out_f32):
    import torch
    B, H, S, D = q.shape
    out = torch.empty((B, H, S, D), dtype=torch.float32 if out_f32 else torch.bfloat16,
                      device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    return out, lse


def _call_noalloc(bs, q, k, v, mask_d, causal, scale, out, lse):
    import torch
    lib = bs.load()
    B, H, S, D = q.shape
    flags = (bs.CAUSAL if causal else 0) | (bs.OUT_F32 if out.dtype == torch.float32 else 0)
    vp = ctypes.c_void_p
    st = lib.bsattn_fwd_noalloc(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()),
                                vp(mask_d.data_ptr()), vp(out.data_ptr()), vp(lse.data_ptr()),
                                B, H, S, D, ctypes.c_float(scale), flags,
                                vp(torch.cuda.current_stream().cuda_stream))
    assert st == bs.OK, bs.status_string(st)


def test_noalloc_matches_oracle_and_plan_fwd_on_two_calls(bs):
    """Two calls in a row through the C ABI: each is checked against the fp64
    oracle and against bsattn_plan + bsattn_fwd, at the forward tolerance.
    The second call must also leave the device's free memory unchanged (it
    allocates nothing), and the Python wrapper must give the same result."""
    import torch
    cases = [_case(501, 2, 4, 1024, 128, 0.4, True), _case(502, 1, 3, 512, 64, 0.6, False)]
    for i, (qb, kb, vb, mask, causal) in enumerate(cases):
        out_f32 = i == 0
        q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
        mask_d = torch.from_numpy(mask).cuda()
        scale = qb.shape[-1] ** -0.5
        O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(scale), causal)
        # the existing entry points
        p = bs.plan(mask_d, causal=causal, out_f32=out_f32)
        o_pf, l_pf = bs.fwd(q, k, v, p, scale)
        bs.plan_status(p)
        p.close()
        o_pf = o_pf.float().cpu().numpy().astype(np.float64)
        l_pf = l_pf.cpu().numpy().astype(np.float64)
        out, lse = _outputs(q, out_f32)
        for call in range(2):
            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
            _call_noalloc(bs, q, k, v, mask_d, causal, scale, out, lse)
            torch.cuda.synchronize()
            if call == 1:  # after one warm call (lazy module loading is done)
                assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated"
            o = out.float().cpu().numpy()
            l = lse.cpu().numpy()
            ok, rep = compare(o, l, O_ref, L_ref, out_bf16=not out_f32)
            assert ok, ("oracle", i, call, rep)
            ok, rep = compare(o, l, o_pf, l_pf, out_bf16=not out_f32)
            assert ok, ("plan+fwd", i, call, rep)
        o_w, l_w = bs.fwd_noalloc(q, k, v, mask_d, causal=causal, scale=scale, out_f32=out_f32)
        torch.cuda.synchronize()
        assert torch.equal(o_w, out) and torch.equal(l_w, lse)


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
