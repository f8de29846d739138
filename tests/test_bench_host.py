"""Host-side accounting of bench.py (no GPU): the exact count of (query, key)
pairs that the metric's whole-block count stands beside, and the lookup of
measured DRAM traffic by kernel source hash."""
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


def test_traffic_table_applies_only_to_its_kernel_source(monkeypatch):
    """A line of the committed DRAM-traffic table gives read + write bytes
    while the kernel source hash equals the line's, and nothing (null in the
    bench line) under any other hash."""
    lines = [l.split() for l in open(bench.TRAFFIC_TABLE)
             if l.strip() and not l.startswith("#")]
    assert lines
    for key, out, sha, rd, wr in (l[:5] for l in lines):
        monkeypatch.setattr(bench, "kernel_source_sha16", lambda s=sha: s)
        assert bench.measured_traffic(key, out == "f32") == int(rd) + int(wr)
        monkeypatch.setattr(bench, "kernel_source_sha16", lambda: "0" * 16)
        assert bench.measured_traffic(key, out == "f32") is None
    # one capture: every line carries the same source hash
    assert len({l[2] for l in lines}) == 1
