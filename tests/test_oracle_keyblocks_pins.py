"""Pins of the oracle for 64-key blocks (CPU): a mask at 64-key granularity
that repeats a 128-key mask reduces to the pinned oracle.attention; brute
force with math.exp / math.fsum on tiny shapes; torch float64 SDPA with the
expanded boolean mask; rows with no allowed key; the CSR against the
element-level allowed pattern; planted mistakes."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import keyblocks as kbo


def _mask64(seed, B, H, nbq, p, causal_diag=False):
    rng = np.random.default_rng(seed)
    m = (rng.random((B, H, nbq, 2 * nbq)) < p).astype(np.uint8)
    if causal_diag:
        m[:, :, np.arange(nbq), 2 * np.arange(nbq)] = 1
    return m


def test_repeated_128_mask_equals_the_128_oracle():
    B, H, S, D = 1, 2, 512, 32
    q, k, v = workloads.custom(41, B, H, S, D)
    m128 = (np.random.default_rng(2).random((B, H, 4, 4)) < 0.5).astype(np.uint8)
    m64 = np.repeat(m128, 2, axis=3)
    for causal in (False, True):
        O1, L1 = oracle.attention(q, k, v, m128, 0.2, causal)
        O2, L2 = kbo.attention_kb(q, k, v, m64, 0.2, causal)
        assert np.allclose(O1, O2, rtol=1e-12, atol=1e-13)
        assert np.array_equal(np.isneginf(L1), np.isneginf(L2))
        fin = np.isfinite(L1)
        assert np.allclose(L1[fin], L2[fin], rtol=1e-12, atol=1e-12)


def test_brute_force_tiny():
    B, H, S, D = 1, 1, 256, 4
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((B, H, S, D)) for _ in range(3))
    mask = np.array([[[[1, 0, 0, 1], [0, 1, 0, 1]]]], np.uint8)
    O, L = kbo.attention_kb(q, k, v, mask, 0.7, causal=True)
    for i in (0, 5, 63, 64, 100, 127, 128, 191, 192, 200, 255):
        allowed = [j for j in range(S) if mask[0, 0, i // 128, j // 64] and j <= i]
        if not allowed:
            assert L[0, 0, i] == -math.inf and np.all(O[0, 0, i] == 0)
            continue
        s = [0.7 * math.fsum(q[0, 0, i, d] * k[0, 0, j, d] for d in range(D)) for j in allowed]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        l = math.fsum(w)
        for d in range(D):
            ref = math.fsum(wj * v[0, 0, j, d] for wj, j in zip(w, allowed)) / l
            assert abs(O[0, 0, i, d] - ref) <= 1e-12
        assert abs(L[0, 0, i] - (mx + math.log(l))) <= 1e-12


def test_rows_without_an_allowed_key():
    """Causal with only the second 64-key block of the diagonal live: rows
    0..63 of the query block have no allowed key."""
    B, H, S, D = 1, 1, 128, 8
    q, k, v = workloads.custom(7, B, H, S, D)
    mask = np.array([[[[0, 1]]]], np.uint8)
    O, L = kbo.attention_kb(q, k, v, mask, 0.3, causal=True)
    assert np.all(np.isneginf(L[0, 0, :64])) and np.all(O[0, 0, :64] == 0)
    assert np.all(np.isfinite(L[0, 0, 64:]))


@pytest.mark.parametrize("causal", [False, True])
def test_torch_sdpa_with_the_expanded_mask(causal):
    B, H, S, D = 2, 2, 384, 16
    q, k, v = workloads.custom(9, B, H, S, D)
    mask = _mask64(4, B, H, S // 128, 0.4, causal_diag=True)
    O, L = kbo.attention_kb(q, k, v, mask, 0.25, causal)
    qf, kf, vf = (torch.from_numpy(kbo._f64(x)) for x in (q, k, v))
    allowed = torch.from_numpy(np.repeat(np.repeat(mask, 128, axis=2), 64, axis=3).astype(bool))
    if causal:
        allowed &= torch.tril(torch.ones(S, S, dtype=torch.bool))
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=allowed,
                                                           scale=0.25)
    live = allowed.any(-1).numpy()
    assert np.allclose(O[live], ref.numpy()[live], rtol=1e-12, atol=1e-12)
    s = (0.25 * qf @ kf.transpose(-1, -2)).masked_fill(~allowed, float("-inf"))
    lse = torch.logsumexp(s, -1).numpy()
    assert np.allclose(L[live], lse[live], rtol=1e-12, atol=1e-12)
    assert np.all(np.isneginf(L[~live])) and np.all(O[~live] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_csr_against_the_allowed_elements(causal):
    B, H, nbq = 1, 2, 5
    S = nbq * 128
    mask = _mask64(11, B, H, nbq, 0.5)
    rp, ci = kbo.csr_kb(mask, causal)
    r = 0
    for b in range(B):
        for h in range(H):
            for qb in range(nbq):
                rows_i = qb * 128 + np.arange(128)
                a = kbo.allowed_rows(mask[b, h], rows_i, S, 64, causal)
                want = [kb for kb in range(2 * nbq) if a[:, kb * 64:(kb + 1) * 64].any()]
                assert list(ci[rp[r]:rp[r + 1]]) == want
                r += 1


@pytest.mark.parametrize("m", sorted(kbo.KB_MUTATIONS))
def test_planted_mistakes_are_caught(m):
    kbo.set_kb_mutation(m)
    try:
        failed = 0
        for t in (test_repeated_128_mask_equals_the_128_oracle, test_brute_force_tiny,
                  test_rows_without_an_allowed_key):
            try:
                t()
            except AssertionError:
                failed += 1
        for causal in (False, True):
            try:
                test_torch_sdpa_with_the_expanded_mask(causal)
            except AssertionError:
                failed += 1
        assert failed > 0, kbo.KB_MUTATIONS[m]
    finally:
        kbo.set_kb_mutation(0)
