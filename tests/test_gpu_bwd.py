"""GPU parity of the backward pass: the CUDA path (through the C ABI) against
the fp64 gradient oracle.

Tolerance: the per-element bound that oracle.attention_bwd(..., bounds=True)
derives from the kernel's arithmetic (bf16 rounding of P and dS, unit
roundoff 2^-8; the given O's rounding in dO.O; fp32 accumulation over every
live row or key; the error of recomputing P from the fp32 LSE with a
hardware exp2), with no extra factor.  The transposed plan must match the
oracle's bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads
from _util import to_dev

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


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _mask_iid(seed, B, H, nb, p, diag=False):
    rng = np.random.default_rng(seed)
    m = (rng.random((B, H, nb, nb)) < p).astype(np.uint8)
    if diag:
        m[:, :, np.arange(nb), np.arange(nb)] = 1
    return m


def _check(got, ref, bound, name):
    """Every element within the oracle's derived bound (no extra factor)."""
    got = got.detach().float().cpu().numpy().astype(np.float64)
    ok_rows = ~np.isnan(ref)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)[ok_rows]
    tol = bound[ok_rows]
    worst = float(np.max(err / tol))
    assert np.all(err <= tol), f"{name}: max err/bound {worst:.3g}, max err {err.max():.3g}"
    print(f"{name}: max err/bound {worst:.3f}")
    return worst


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_plan_csc_bit_exact(bs, wid):
    import torch
    w = workloads.WORKLOADS[wid]
    mask = workloads.make_mask(w)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=w.causal)
    cp, ri = bs.plan_csc(p)
    cp_ref, ri_ref = oracle.csc(mask, w.causal)
    assert np.array_equal(cp.cpu().numpy(), cp_ref)
    assert np.array_equal(ri.cpu().numpy(), ri_ref)
    p.close()


CASES = {
    # name: (B, H, S, D, mask builder, causal, scale, mult)
    "d128_sparse": (1, 2, 1024, 128, lambda: _mask_iid(1, 1, 2, 8, 0.4, diag=True), False, 128 ** -0.5, 1.0),
    "d128_causal": (1, 2, 1024, 128, lambda: _mask_iid(2, 1, 2, 8, 0.5, diag=True), True, 128 ** -0.5, 1.0),
    "d64_sparse": (2, 2, 1024, 64, lambda: _mask_iid(3, 2, 2, 8, 0.3), False, 0.125, 1.0),
    "d64_causal_dense": (1, 2, 1024, 64, lambda: np.ones((1, 2, 8, 8), np.uint8), True, 0.125, 1.0),
    "one_tile_d128": (1, 1, 128, 128, lambda: np.ones((1, 1, 1, 1), np.uint8), False, 128 ** -0.5, 1.0),
    "empty_rows_cols": (1, 2, 512, 128, lambda: np.array([[[[1, 0, 0, 1], [0, 0, 0, 0], [0, 1, 1, 0], [0, 0, 0, 0]],
                                                           [[0, 0, 0, 0], [1, 1, 1, 1], [0, 0, 0, 0], [0, 0, 0, 1]]]], np.uint8),
                        False, 0.09, 1.0),
    "all_dead": (1, 1, 256, 64, lambda: np.zeros((1, 1, 2, 2), np.uint8), False, 0.125, 1.0),
    "scale_negative": (1, 1, 512, 128, lambda: _mask_iid(4, 1, 1, 4, 0.6, diag=True), True, -0.2, 1.0),
    "scale_zero": (1, 1, 512, 64, lambda: _mask_iid(5, 1, 1, 4, 0.6, diag=True), False, 0.0, 1.0),
    "wide_logits_d64": (1, 2, 1024, 64, lambda: np.ones((1, 2, 8, 8), np.uint8), False, 0.125, 2.0),
    "long_column_d128": (1, 1, 4096, 128, lambda: _mask_iid(6, 1, 1, 32, 0.7, diag=True), True, 128 ** -0.5, 1.0),
}


def _inputs(name):
    B, H, S, D, mk, causal, scale, mult = CASES[name]
    qb, kb, vb = workloads.custom(300 + len(name), B, H, S, D, mult)
    gb = workloads.upstream_grad(400 + len(name), B, H, S, D)
    return B, H, S, D, mk(), causal, scale, qb, kb, vb, gb


@pytest.mark.parametrize("o_f32", [False, True], ids=["o_bf16", "o_f32"])
@pytest.mark.parametrize("name", list(CASES))
def test_bwd_small(bs, name, o_f32):
    """Every gradient element against the oracle; O and LSE given from the oracle."""
    import torch
    B, H, S, D, mask, causal, scale, qb, kb, vb, gb = _inputs(name)
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(scale), causal)
    if o_f32:
        o = torch.from_numpy(O_ref.astype(np.float32)).cuda()
    else:
        o = to_dev(_bf16_bits(O_ref))
    lse = torch.from_numpy(L_ref.astype(np.float32)).cuda()
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=causal, out_f32=o_f32)
    dq, dk, dv = bs.bwd(to_dev(qb), to_dev(kb), to_dev(vb), o, lse, to_dev(gb), p, scale)
    bs.plan_status(p)
    p.close()
    ref, bound = oracle.attention_bwd(qb, kb, vb, gb, mask, np.float32(scale), causal, bounds=True,
                                      o_bf16=not o_f32)
    for got, r, b, nm in zip((dq, dk, dv), ref, bound, ("dQ", "dK", "dV")):
        _check(got, r, b, f"{name} {nm}")


def test_bwd_through_forward(bs):
    """Forward kernel, then backward on its own O and LSE (normwise: the
    forward's own error enters through dO.O)."""
    import torch
    B, H, S, D, mask, causal, scale, qb, kb, vb, gb = _inputs("d128_causal")
    q, k, v, g = to_dev(qb), to_dev(kb), to_dev(vb), to_dev(gb)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=causal)
    o, lse = bs.fwd(q, k, v, p, scale)
    dq, dk, dv = bs.bwd(q, k, v, o, lse, g, p, scale)
    bs.plan_status(p)
    p.close()
    ref = oracle.attention_bwd(qb, kb, vb, gb, mask, np.float32(scale), causal)
    for got, r, nm in zip((dq, dk, dv), ref, ("dQ", "dK", "dV")):
        e = np.abs(got.cpu().numpy() - r)
        assert e.max() <= 0.02 * np.abs(r).max() and e.mean() <= 0.01 * np.abs(r).mean(), nm


def test_bwd_repeated_calls(bs):
    """Every gradient row is written once by one CTA in a fixed order: repeated
    calls give bit-identical dQ, dK and dV."""
    import torch
    B, H, S, D, mask, causal, scale, qb, kb, vb, gb = _inputs("d64_sparse")
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(scale), causal)
    o, lse = to_dev(_bf16_bits(O_ref)), torch.from_numpy(L_ref.astype(np.float32)).cuda()
    q, k, v, g = to_dev(qb), to_dev(kb), to_dev(vb), to_dev(gb)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=causal)
    first = bs.bwd(q, k, v, o, lse, g, p, scale)
    for _ in range(3):
        again = bs.bwd(q, k, v, o, lse, g, p, scale)
    bs.plan_status(p)
    p.close()
    for a, b in zip(first, again):
        assert torch.equal(a, b)


def test_bwd_full_size_causal_sampled_heads(bs):
    """The causal S=4096 D=128 workload at full size; two heads checked in full."""
    import torch
    w = workloads.WORKLOADS[2]
    qb, kb, vb = workloads.make_qkv(w)
    mask = workloads.make_mask(w)
    B, H, S, D = qb.shape
    gb = workloads.upstream_grad(w.data_seed, B, H, S, D)
    q, k, v, g = to_dev(qb), to_dev(kb), to_dev(vb), to_dev(gb)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=w.causal)
    o, lse = bs.fwd(q, k, v, p, w.scale)
    # oracle O and LSE for the checked heads replace the kernel's, so that the
    # per-element bound applies
    heads = [(0, 0), (B - 1, H - 1)]
    for b, h in heads:
        rows = (b * H + h) * S + np.arange(S, dtype=np.int64)
        O_h, L_h = oracle.attention(qb, kb, vb, mask, np.float32(w.scale), w.causal, rows=rows)
        o[b, h] = to_dev(_bf16_bits(O_h))
        lse[b, h] = torch.from_numpy(L_h.astype(np.float32)).cuda()
    dq, dk, dv = bs.bwd(q, k, v, o, lse, g, p, w.scale)
    bs.plan_status(p)
    p.close()
    ref, bound = oracle.attention_bwd(qb, kb, vb, gb, mask, np.float32(w.scale), w.causal,
                                      heads=heads, bounds=True)
    for got, r, b, nm in zip((dq, dk, dv), ref, bound, ("dQ", "dK", "dV")):
        _check(got, r, b, f"w2 {nm}")
