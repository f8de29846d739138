"""Pins of the backward oracle (CPU): what the mathematics fixes, independent
of the oracle's own formulas.

* central finite differences of the forward oracle (itself pinned in
  test_oracle_pins.py) on the scalar loss sum(dO * O);
* torch float64 autograd of dense attention (all-ones mask) and of causal
  attention (a library routine);
* closed forms: dO = 0 gives zero gradients; scale = 0 gives dQ = dK = 0 and
  dV_j = sum over rows i attending j of dO_i / (#keys row i attends);
* invariants: sum_j dK_j = 0 per head (the rows of dS sum to zero) and
  sum_j dV_j = sum over live rows of dO_i (the rows of P sum to one);
* the transposed plan against the forward CSR by enumeration;
* every planted mistake fails at least one of the above.
"""
import numpy as np
import pytest

import oracle
from oracle import backward as ob


def _rand(seed, shape, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _mask(seed, B, H, nb, p, diag=True):
    m = (np.random.default_rng(seed).random((B, H, nb, nb)) < p).astype(np.uint8)
    if diag:
        m[:, :, np.arange(nb), np.arange(nb)] = 1
    return m


# Small problems: (B, H, S, D, mask, causal, scale)
def _cases():
    return [
        (1, 1, 256, 8, _mask(1, 1, 1, 2, 0.5), False, 0.35),
        (1, 2, 256, 8, _mask(2, 1, 2, 2, 0.6), True, 0.35),
        (1, 1, 384, 4, np.array([[[[1, 0, 1], [0, 0, 0], [0, 1, 1]]]], np.uint8), False, 0.5),
        (1, 1, 256, 8, np.array([[[[0, 0], [1, 1]]]], np.uint8), True, -0.3),
    ]


def _fd_check(B, H, S, D, mask, causal, scale, seed=0, n_samples=12):
    """Gradients of L = sum(G * O) by central differences of the forward oracle."""
    q, k, v, G = (_rand(seed + i, (B, H, S, D)) for i in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, G, mask, scale, causal)
    rng = np.random.default_rng(seed + 99)
    h = 1e-5
    worst = 0.0
    for X, dX in ((q, dq), (k, dk), (v, dv)):
        for _ in range(n_samples):
            idx = tuple(int(rng.integers(0, n)) for n in X.shape)
            old = X[idx]
            X[idx] = old + h
            Op, _ = oracle.attention(q, k, v, mask, scale, causal)
            X[idx] = old - h
            Om, _ = oracle.attention(q, k, v, mask, scale, causal)
            X[idx] = old
            fd = (np.nansum(G * Op) - np.nansum(G * Om)) / (2 * h)
            worst = max(worst, abs(fd - dX[idx]) / (1.0 + abs(dX[idx])))
    return worst


@pytest.mark.parametrize("case", range(4))
def test_finite_differences(case):
    assert _fd_check(*_cases()[case]) < 1e-6


def _torch_grads(q, k, v, G, scale, causal):
    torch = pytest.importorskip("torch")
    t = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v)]
    o = torch.nn.functional.scaled_dot_product_attention(t[0], t[1], t[2], is_causal=causal,
                                                         scale=scale)
    (o * torch.tensor(G)).sum().backward()
    return [x.grad.numpy() for x in t]


@pytest.mark.parametrize("causal", [False, True])
def test_torch_autograd_dense(causal):
    B, H, S, D = 1, 2, 256, 16
    q, k, v, G = (_rand(10 + i, (B, H, S, D)) for i in range(4))
    mask = np.ones((B, H, 2, 2), np.uint8)
    ref = _torch_grads(q, k, v, G, 0.25, causal)
    got = oracle.attention_bwd(q, k, v, G, mask, 0.25, causal)
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b)) < 1e-10


def test_zero_upstream_gradient():
    B, H, S, D, mask, causal, scale = _cases()[1]
    q, k, v = (_rand(20 + i, (B, H, S, D)) for i in range(3))
    for g in oracle.attention_bwd(q, k, v, np.zeros_like(q), mask, scale, causal):
        assert np.all(g == 0.0)


def test_scale_zero_closed_form():
    B, H, S, D = 1, 1, 256, 8
    mask = np.array([[[[1, 0], [1, 1]]]], np.uint8)
    q, k, v, G = (_rand(30 + i, (B, H, S, D)) for i in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, G, mask, 0.0, True)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    allowed = np.repeat(np.repeat(mask[0, 0] != 0, 128, 0), 128, 1) & np.tril(np.ones((S, S), bool))
    n = allowed.sum(axis=1)
    expect = np.zeros((S, D))
    for j in range(S):
        rows = np.flatnonzero(allowed[:, j])
        expect[j] = (G[0, 0, rows] / n[rows, None]).sum(axis=0)
    assert np.max(np.abs(dv[0, 0] - expect)) < 1e-12


@pytest.mark.parametrize("case", range(4))
def test_sum_invariants(case):
    B, H, S, D, mask, causal, scale = _cases()[case]
    q, k, v, G = (_rand(40 + i, (B, H, S, D)) for i in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, G, mask, scale, causal)
    for b in range(B):
        for h in range(H):
            allowed = ob.allowed_matrix(mask[b, h], S, causal)
            live = allowed.any(axis=1)
            assert np.max(np.abs(dk[b, h].sum(axis=0))) < 1e-9 * (1 + np.abs(dk[b, h]).sum())
            assert np.allclose(dv[b, h].sum(axis=0), G[b, h][live].sum(axis=0), atol=1e-9)
            assert np.all(dq[b, h][~live] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_csc_is_the_transposed_csr(causal):
    mask = _mask(50, 2, 3, 6, 0.4, diag=False)
    rp, ci = oracle.csr(mask, causal)
    cp, ri = oracle.csc(mask, causal)
    B, H, nb, _ = mask.shape
    pairs_csr = {(t // nb, t % nb, int(c)) for t in range(B * H * nb) for c in ci[rp[t]:rp[t + 1]]}
    pairs_csc = {(t // nb, int(r), t % nb) for t in range(B * H * nb) for r in ri[cp[t]:cp[t + 1]]}
    assert pairs_csr == pairs_csc
    assert cp[-1] == rp[-1] == len(pairs_csr)
    for t in range(B * H * nb):  # ascending query blocks per key block
        assert np.all(np.diff(ri[cp[t]:cp[t + 1]]) > 0)


def _all_pins_pass():
    try:
        test_finite_differences(1)
        test_finite_differences(3)
        test_torch_autograd_dense(False)
        test_torch_autograd_dense(True)
        test_scale_zero_closed_form()
        for c in range(4):
            test_sum_invariants(c)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("m", sorted(ob.BWD_MUTATIONS))
def test_planted_mistakes_are_caught(m):
    ob.set_bwd_mutation(m)
    try:
        assert not _all_pins_pass(), f"mutation {m} ({ob.BWD_MUTATIONS[m]}) passed every pin"
    finally:
        ob.set_bwd_mutation(0)


@pytest.mark.parametrize("Hkv,causal", [(1, False), (2, True)])
def test_gqa_gradients_against_torch_autograd(Hkv, causal):
    """Grouped-query gradients against torch float64 autograd of SDPA with enable_gqa."""
    torch = pytest.importorskip("torch")
    B, H, S, D = 1, 4, 256, 8
    q, G = _rand(80, (B, H, S, D)), _rand(81, (B, H, S, D))
    k, v = _rand(82, (B, Hkv, S, D)), _rand(83, (B, Hkv, S, D))
    t = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v)]
    try:
        o = torch.nn.functional.scaled_dot_product_attention(t[0], t[1], t[2], is_causal=causal,
                                                             scale=0.3, enable_gqa=True)
    except TypeError:
        pytest.skip("torch without enable_gqa")
    (o * torch.tensor(G)).sum().backward()
    mask = np.ones((B, 1, S // 128, S // 128), np.uint8)
    got = oracle.attention_bwd_gqa(q, k, v, G, mask, 0.3, causal)
    for a, x in zip(got, t):
        assert np.max(np.abs(a - x.grad.numpy())) < 1e-10


def _bf16_round(x):
    """Round float32 values to bf16 (nearest, ties to even), returned as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("o_bf16", [True, False])
@pytest.mark.parametrize("case", range(4))
def test_error_bounds_cover_a_reduced_precision_emulation(case, o_bf16):
    """The per-element bounds hold for a numpy emulation of the error model
    they describe (fp32 products and sums, P from the fp32 LSE with a float32
    exp2, bf16-rounded P and dS as product operands, O given rounded), and
    are not vacuous: the worst element uses a sizeable part of its bound."""
    B, H, S, D, mask, causal, scale = _cases()[case]
    f32 = np.float32
    q, k, v, do = (_bf16_round(_rand(60 + case * 4 + i, (B, H, S, D))).astype(np.float64)
                   for i in range(4))
    O, L = oracle.attention(q, k, v, mask, scale, causal)
    (dq, dk, dv), bounds = ob.attention_bwd(q, k, v, do, mask, scale, causal, bounds=True,
                                            o_bf16=o_bf16)
    ratios = []
    for b in range(B):
        for h in range(H):
            allowed = ob.allowed_matrix(mask[b, h], S, causal)
            live = allowed.any(axis=1)
            qq, kk, vv, gg = (x[b, h].astype(f32) for x in (q, k, v, do))
            sl = f32(scale / np.log(2.0))
            l2 = np.where(live, L[b, h] / np.log(2.0), 0.0).astype(f32)
            s = qq @ kk.T
            p = np.where(allowed, np.exp2(s * sl - l2[:, None]), f32(0)).astype(f32)
            o_in = _bf16_round(O[b, h].astype(f32)) if o_bf16 else O[b, h].astype(f32)
            dl = (gg * o_in).sum(axis=1, dtype=f32)
            dp = gg @ vv.T
            ds = (p * (dp - dl[:, None])).astype(f32)
            pb, dsb = _bf16_round(p), _bf16_round(ds)
            got = (f32(scale) * (dsb @ kk), f32(scale) * (dsb.T @ qq), pb.T @ gg)
            for g, ref, bd in zip(got, (dq, dk, dv), bounds):
                err = np.abs(g.astype(np.float64) - ref[b, h])
                assert np.all(err <= bd[b, h])
                ratios.append(float(np.max(err / bd[b, h])))
    print("max err / bound", max(ratios))
    assert max(ratios) > 0.02, ratios
