"""GPU parity of grouped-query attention (K/V with fewer heads than Q) and of
plans built from one mask shared by the heads of a batch entry, against the
oracle (tolerances as in test_gpu_parity.py and test_gpu_bwd.py)."""
import numpy as np
import pytest

import oracle
import workloads
from _util import compare, to_dev
from test_gpu_bwd import _bf16_bits, _check

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


def _mask_iid(seed, B, H, nb, p, diag=False):
    rng = np.random.default_rng(seed)
    m = (rng.random((B, H, nb, nb)) < p).astype(np.uint8)
    if diag:
        m[:, :, np.arange(nb), np.arange(nb)] = 1
    return m


# the last case is large enough for the fp16 copy of V (B * Hkv * S = 16384
# rows, ~14 live blocks per key block of V): the copy has Hkv heads
@pytest.mark.parametrize("Hkv,D,causal,S", [(1, 128, True, 1024), (2, 64, False, 1024),
                                            (4, 128, False, 1024), (8, 64, True, 1024),
                                            (4, 64, False, 2048)])
def test_gqa_every_row(bs, Hkv, D, causal, S):
    import torch
    B, H = 2, 8
    qb = workloads.custom(500 + Hkv, B, H, S, D)[0]
    _, kb, vb = workloads.custom(600 + Hkv, B, Hkv, S, D)
    mask = _mask_iid(12 + Hkv, B, H, S // 128, 0.4, diag=True)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=causal, out_f32=True)
    o, lse = bs.fwd(to_dev(qb), to_dev(kb), to_dev(vb), p, D ** -0.5)
    bs.plan_status(p)
    assert bs.plan_v16_bytes(p) == (B * Hkv * S * D * 2 if S == 2048 else 0)
    p.close()
    O_ref, L_ref = oracle.attention_gqa(qb, kb, vb, mask, np.float32(D ** -0.5), causal)
    ok, rep = compare(o.cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref)
    assert ok, rep


def test_gqa_rejects_bad_group(bs):
    import torch
    q = torch.zeros((1, 6, 256, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 4, 256, 64), dtype=torch.bfloat16, device="cuda")
    p = bs.plan(torch.ones((1, 6, 2, 2), dtype=torch.uint8, device="cuda"))
    with pytest.raises(ValueError):
        bs.fwd(q, k, k, p)
    p.close()


def test_shared_mask_plan_fwd_bwd(bs):
    import torch
    B, H, S, D = 2, 6, 1024, 128
    causal, scale = True, 128 ** -0.5
    mask1 = _mask_iid(20, B, 1, S // 128, 0.4, diag=True)
    full = np.ascontiguousarray(np.broadcast_to(mask1, (B, H) + mask1.shape[2:]))
    p = bs.plan(torch.from_numpy(mask1).cuda(), causal=causal, heads=H)
    rp, ci = bs.plan_csr(p)
    cp, ri = bs.plan_csc(p)
    rp_ref, ci_ref = oracle.csr(full, causal)
    cp_ref, ri_ref = oracle.csc(full, causal)
    assert np.array_equal(rp.cpu().numpy(), rp_ref) and np.array_equal(ci.cpu().numpy(), ci_ref)
    assert np.array_equal(cp.cpu().numpy(), cp_ref) and np.array_equal(ri.cpu().numpy(), ri_ref)

    qb, kb, vb = workloads.custom(700, B, H, S, D)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    o, lse = bs.fwd(q, k, v, p, scale)
    bs.plan_status(p)
    O_ref, L_ref = oracle.attention_gqa(qb, kb, vb, mask1, np.float32(scale), causal)
    ok, rep = compare(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref, out_bf16=True)
    assert ok, rep

    gb = workloads.upstream_grad(701, B, H, S, D)
    o_in = to_dev(_bf16_bits(O_ref))
    lse_in = torch.from_numpy(L_ref.astype(np.float32)).cuda()
    dq, dk, dv = bs.bwd(q, k, v, o_in, lse_in, to_dev(gb), p, scale)
    bs.plan_status(p)
    p.close()
    ref, bound = oracle.attention_bwd(qb, kb, vb, gb, full, np.float32(scale), causal, bounds=True)
    for got, r, b, nm in zip((dq, dk, dv), ref, bound, ("dQ", "dK", "dV")):
        _check(got, r, b, f"shared mask {nm}")


@pytest.mark.parametrize("Hkv,D,causal", [(1, 128, True), (2, 64, False), (4, 128, False)])
def test_gqa_gradients(bs, Hkv, D, causal):
    """dQ, and dK, dV summed over each K/V head's group, against the oracle
    (O and LSE from the oracle, per-element bound as in test_gpu_bwd.py)."""
    import torch
    B, H, S = 1, 8, 1024
    scale = D ** -0.5
    qb = workloads.custom(800 + Hkv, B, H, S, D)[0]
    _, kb, vb = workloads.custom(900 + Hkv, B, Hkv, S, D)
    gb = workloads.upstream_grad(950 + Hkv, B, H, S, D)
    mask = _mask_iid(30 + Hkv, B, H, S // 128, 0.5, diag=True)
    O_ref, L_ref = oracle.attention_gqa(qb, kb, vb, mask, np.float32(scale), causal)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=causal)
    dq, dk, dv = bs.bwd(to_dev(qb), to_dev(kb), to_dev(vb), to_dev(_bf16_bits(O_ref)),
                        torch.from_numpy(L_ref.astype(np.float32)).cuda(), to_dev(gb), p, scale)
    bs.plan_status(p)
    p.close()
    assert dk.shape == (B, Hkv, S, D) and dv.shape == (B, Hkv, S, D)
    ref, bound = oracle.attention_bwd_gqa(qb, kb, vb, gb, mask, np.float32(scale), causal,
                                          bounds=True)
    for got, r, b, nm in zip((dq, dk, dv), ref, bound, ("dQ", "dK", "dV")):
        _check(got, r, b, f"gqa {Hkv} {nm}")
