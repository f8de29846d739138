"""Host-side accounting of bench.py (no GPU): the exact count of (query, key)
pairs that the metric's whole-block count stands beside."""
import numpy as np
import pytest

import bench


def _brute(mask, causal, key_block):
    nbq = mask.shape[-2]
    S = nbq * 128
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    total = 0
    for b in range(mask.shape[0]):
        for h in range(mask.shape[1]):
            a = mask[b, h][i // 128, j // key_block].astype(bool)
            if causal:
                a &= j <= i
            total += int(a.sum())
    return total


@pytest.mark.parametrize("key_block", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_allowed_pairs_matches_brute_force(key_block, causal):
    rng = np.random.default_rng(7)
    nbq = 4
    mask = (rng.random((2, 3, nbq, nbq * 128 // key_block)) < 0.6).astype(np.uint8)
    assert bench.allowed_pairs(mask, causal) == _brute(mask, causal, key_block)


def test_allowed_pairs_causal_workload():
    # lower-triangular 32 x 32 blocks: 496 full blocks and 32 diagonal ones of 128 * 129 / 2 pairs
    mask = np.tril(np.ones((1, 1, 32, 32), dtype=np.uint8))
    assert bench.allowed_pairs(mask, True) == 496 * 128 * 128 + 32 * (128 * 129 // 2)
    assert bench.live_blocks(mask, True) == 528
