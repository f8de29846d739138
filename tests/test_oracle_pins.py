"""Pins that tie the fp64 oracle to things other than itself.

Each pin is a plain function returning (ok, detail) so that
test_every_planted_mistake_is_caught can re-run all of them against an oracle
with a deliberate mistake planted (oracle.set_mutation) and show that every
such mistake trips at least one pin.

Pins used (the pages print no worked numeric example for attention):
  * hand-derived worked examples (tests/golden/worked_examples.json)
  * brute force: per-element softmax with Python's math.exp / math.fsum
  * library special cases: torch float64 scaled_dot_product_attention for the
    all-ones mask, the causal mask and an element-expanded block mask
  * closed forms: scale = 0 (mean of allowed V, LSE = ln #allowed), constant
    V, a single allowed key
  * invariants: joint K/V row permutation inside a live block, key shift
    K + 1 u^T (O unchanged, LSE + scale * q.u), diagonal-only mask equals
    independent 128-token attention per block
  * fully masked rows give O = 0, LSE = -inf
  * the CSR plan against a nested-loop enumeration and the popcount
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
TOL = 1e-10


def _f64(bits):
    return workloads.bf16_bits_to_f32(bits).astype(np.float64)


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    same_inf = (np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b)))
    if np.isnan(a).any() or np.isnan(b).any():
        return False, "nan"
    fin = ~same_inf
    if (np.isinf(a[fin]).any()) or (np.isinf(b[fin]).any()):
        return False, "inf mismatch"
    err = np.max(np.abs(a[fin] - b[fin])) if fin.any() else 0.0
    return bool(err <= tol), f"max err {err:.3e}"


def _dense_element_mask(mask, S, causal):
    """[B][H][S][S] bool expanded from the block mask (and the causal flag)."""
    m = np.repeat(np.repeat(mask.astype(bool), 128, axis=2), 128, axis=3)
    if causal:
        m = m & np.tril(np.ones((S, S), dtype=bool))[None, None]
    return m


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def _golden_tensor(spec, S, D):
    if spec.get("index"):
        return np.arange(S, dtype=np.float64).reshape(S, 1).repeat(D, axis=1)
    t = np.tile(np.asarray(spec["default"], dtype=np.float64), (S, 1))
    for r, val in spec["rows"].items():
        if val[0] == "ln":
            t[int(r)] = [math.log(val[1])] + list(val[2:])
        else:
            t[int(r)] = val
    return t


def pin_worked_examples():
    with open(GOLDEN) as f:
        ex = json.load(f)["examples"]
    for e in ex:
        S, D = e["S"], e["D"]
        q = _golden_tensor(e["q"], S, D)[None, None]
        k = _golden_tensor(e["k"], S, D)[None, None]
        v = _golden_tensor(e["v"], S, D)[None, None]
        mask = np.asarray(e["mask"], dtype=np.uint8)[None, None]
        rows = [x["row"] for x in e["expect"]]
        O, L = oracle.attention(q, k, v, mask, e["scale"], e["causal"], rows=rows)
        for i, x in enumerate(e["expect"]):
            lse = -math.inf if x["LSE"] == "-inf" else math.log(x["LSE"][1])
            ok, d = _close(O[i], x["O"], 1e-12)
            ok2, d2 = _close([L[i]], [lse], 1e-12)
            if not (ok and ok2):
                return False, f"{e['name']} row {x['row']}: O {d}, LSE {d2}"
    return True, "ok"


def _bruteforce(qf, kf, vf, mask, scale, causal):
    B, H, S, D = qf.shape
    O = np.zeros((B, H, S, D))
    L = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            qq, kk, vv = qf[b, h].tolist(), kf[b, h].tolist(), vf[b, h].tolist()
            for i in range(S):
                scores = []
                for j in range(S):
                    live = mask[b, h, i // 128, j // 128] != 0 and (not causal or j <= i)
                    if live:
                        scores.append((j, scale * math.fsum(a * c for a, c in zip(qq[i], kk[j]))))
                if not scores:
                    L[b, h, i] = -math.inf
                    continue
                mx = max(s for _, s in scores)
                ws = [(j, math.exp(s - mx)) for j, s in scores]
                l = math.fsum(w for _, w in ws)
                for d in range(D):
                    O[b, h, i, d] = math.fsum(w * vv[j][d] for j, w in ws) / l
                L[b, h, i] = mx + math.log(l)
    return O, L


def pin_bruteforce():
    S, D = 256, 4
    q, k, v = workloads.custom(7, 1, 2, S, D)
    mask = np.array([[[[1, 0], [1, 1]], [[0, 1], [0, 1]]]], dtype=np.uint8)  # asymmetric, per head
    for causal in (False, True):
        O, L = oracle.attention(q, k, v, mask, 0.4, causal)
        Ob, Lb = _bruteforce(_f64(q), _f64(k), _f64(v), mask, 0.4, causal)
        ok, d = _close(O, Ob, 1e-12)
        ok2, d2 = _close(L, Lb, 1e-12)
        if not (ok and ok2):
            return False, f"causal={causal}: O {d}, LSE {d2}"
    return True, "ok"


def _sdpa(qf, kf, vf, scale, dense_mask=None, is_causal=False):
    q, k, v = (torch.from_numpy(x) for x in (qf, kf, vf))
    am = None if dense_mask is None else torch.from_numpy(dense_mask)
    O = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=am,
                                                         is_causal=is_causal, scale=scale)
    scores = scale * (q @ k.transpose(-1, -2))
    if is_causal:
        S = q.shape[-2]
        scores = scores.masked_fill(~torch.ones(S, S, dtype=torch.bool).tril(), -math.inf)
    if am is not None:
        scores = scores.masked_fill(~am, -math.inf)
    return O.numpy(), torch.logsumexp(scores, dim=-1).numpy()


def pin_sdpa_dense():
    q, k, v = workloads.custom(11, 1, 2, 256, 16)
    mask = np.ones((1, 2, 2, 2), dtype=np.uint8)
    O, L = oracle.attention(q, k, v, mask, 0.3, False)
    Os, Ls = _sdpa(_f64(q), _f64(k), _f64(v), 0.3)
    ok, d = _close(O, Os, 1e-9)
    ok2, d2 = _close(L, Ls, 1e-9)
    return ok and ok2, f"O {d}, LSE {d2}"


def pin_sdpa_causal():
    q, k, v = workloads.custom(12, 2, 1, 384, 8)
    mask = np.broadcast_to(np.tril(np.ones((3, 3), dtype=np.uint8)), (2, 1, 3, 3)).copy()
    O, L = oracle.attention(q, k, v, mask, 0.25, True)
    Os, Ls = _sdpa(_f64(q), _f64(k), _f64(v), 0.25, is_causal=True)
    ok, d = _close(O, Os, 1e-9)
    ok2, d2 = _close(L, Ls, 1e-9)
    return ok and ok2, f"O {d}, LSE {d2}"


def pin_sdpa_block_mask():
    """Asymmetric block mask, no fully masked row: SDPA with the expanded boolean mask."""
    q, k, v = workloads.custom(13, 1, 2, 384, 8)
    mask = np.array([[[[0, 1, 0], [1, 1, 0], [0, 0, 1]],
                      [[1, 0, 1], [0, 0, 1], [1, 1, 0]]]], dtype=np.uint8)
    dm = _dense_element_mask(mask, 384, False)
    O, L = oracle.attention(q, k, v, mask, 0.5, False)
    Os, Ls = _sdpa(_f64(q), _f64(k), _f64(v), 0.5, dense_mask=dm)
    ok, d = _close(O, Os, 1e-9)
    ok2, d2 = _close(L, Ls, 1e-9)
    return ok and ok2, f"O {d}, LSE {d2}"


def pin_scale_zero():
    q, k, v = workloads.custom(14, 1, 2, 256, 8)
    mask = np.array([[[[1, 0], [1, 1]], [[0, 1], [1, 0]]]], dtype=np.uint8)
    vf = _f64(v)
    for causal in (False, True):
        O, L = oracle.attention(q, k, v, mask, 0.0, causal)
        dm = _dense_element_mask(mask, 256, causal)
        for h in range(2):
            for i in range(256):
                allowed = np.flatnonzero(dm[0, h, i])
                if allowed.size == 0:
                    continue
                ok, d = _close(O[0, h, i], vf[0, h, allowed].mean(axis=0), 1e-12)
                ok2, d2 = _close([L[0, h, i]], [math.log(allowed.size)], 1e-12)
                if not (ok and ok2):
                    return False, f"causal={causal} h={h} i={i}: {d} {d2}"
    return True, "ok"


def pin_constant_v():
    q, k, _ = workloads.custom(15, 1, 1, 256, 8)
    c = np.array([0.5, -1.25, 3.0, 0.0, 7.5, -2.0, 1.0, 0.125], dtype=np.float32)
    v = np.broadcast_to(c.view(np.uint32) >> 16, (1, 1, 256, 8)).astype(np.uint16).copy()
    mask = np.array([[[[1, 1], [0, 1]]]], dtype=np.uint8)
    O, _ = oracle.attention(q, k, v, mask, 0.7, True)
    return _close(O, np.broadcast_to(c.astype(np.float64), O.shape), 1e-12)


def pin_single_key():
    """Causal, block 0 live: query 0 sees key 0 only -> O_0 = v_0, LSE_0 = scale*q_0.k_0."""
    q, k, v = (_f64(x) for x in workloads.custom(16, 1, 3, 256, 8))
    mask = np.ones((1, 3, 2, 2), dtype=np.uint8)
    rows = [h * 256 for h in range(3)]
    O, L = oracle.attention(q, k, v, mask, 0.3, True, rows=rows)
    for h in range(3):
        ok, d = _close(O[h], v[0, h, 0], 1e-12)
        ok2, d2 = _close([L[h]], [0.3 * float(np.dot(q[0, h, 0], k[0, h, 0]))], 1e-12)
        if not (ok and ok2):
            return False, f"h={h}: {d} {d2}"
    return True, "ok"


def pin_permutation_invariance():
    q, k, v = (_f64(x) for x in workloads.custom(17, 1, 1, 384, 8))
    mask = np.array([[[[1, 0, 1], [1, 1, 0], [0, 1, 1]]]], dtype=np.uint8)
    O, L = oracle.attention(q, k, v, mask, 0.6, False)
    rng = np.random.default_rng(5)
    k2, v2 = k.copy(), v.copy()
    for blk in range(3):
        perm = blk * 128 + rng.permutation(128)
        k2[0, 0, blk * 128:(blk + 1) * 128] = k[0, 0, perm]
        v2[0, 0, blk * 128:(blk + 1) * 128] = v[0, 0, perm]
    O2, L2 = oracle.attention(q, k2, v2, mask, 0.6, False)
    ok, d = _close(O, O2, 1e-12)
    ok2, d2 = _close(L, L2, 1e-12)
    return ok and ok2, f"O {d}, LSE {d2}"


def pin_shift_invariance():
    q, k, v = (_f64(x) for x in workloads.custom(18, 1, 2, 256, 8))
    u = workloads.normal_f64(99, 1, (8,))
    mask = np.array([[[[1, 1], [0, 1]], [[1, 0], [1, 1]]]], dtype=np.uint8)
    for causal in (False, True):
        O, L = oracle.attention(q, k, v, mask, 0.45, causal)
        O2, L2 = oracle.attention(q, k + u, v, mask, 0.45, causal)
        ok, d = _close(O, O2, 1e-11)
        ok2, d2 = _close(L2, L + 0.45 * (q @ u), 1e-11)
        if not (ok and ok2):
            return False, f"causal={causal}: O {d}, LSE {d2}"
    return True, "ok"


def pin_diagonal_only():
    q, k, v = workloads.custom(19, 1, 2, 384, 16)
    mask = np.broadcast_to(np.eye(3, dtype=np.uint8), (1, 2, 3, 3)).copy()
    O, L = oracle.attention(q, k, v, mask, 0.25, False)
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    for blk in range(3):
        sl = slice(blk * 128, (blk + 1) * 128)
        Os, Ls = _sdpa(qf[:, :, sl], kf[:, :, sl], vf[:, :, sl], 0.25)
        ok, d = _close(O[:, :, sl], Os, 1e-9)
        ok2, d2 = _close(L[:, :, sl], Ls, 1e-9)
        if not (ok and ok2):
            return False, f"block {blk}: O {d}, LSE {d2}"
    return True, "ok"


def pin_fully_masked_rows():
    q, k, v = workloads.custom(20, 1, 2, 256, 8)
    mask = np.array([[[[0, 0], [1, 0]], [[0, 0], [0, 0]]]], dtype=np.uint8)
    O, L = oracle.attention(q, k, v, mask, 0.5, False)
    if np.isnan(O).any() or np.isnan(L).any():
        return False, "nan"
    dead = [(0, slice(0, 128)), (1, slice(0, 256))]
    for h, sl in dead:
        if not (np.all(O[0, h, sl] == 0.0) and np.all(np.isneginf(L[0, h, sl]))):
            return False, f"head {h} not O=0/LSE=-inf"
    live = L[0, 0, 128:]
    return bool(np.all(np.isfinite(live))), "live rows finite"


def pin_csr():
    rng = np.random.default_rng(3)
    for causal in (False, True):
        mask = (rng.random((2, 3, 7, 7)) < 0.4).astype(np.uint8)
        mask[0, 0, 2] = 0  # an empty row
        row_ptr, col_idx = oracle.csr(mask, causal)
        exp_ptr, exp_col = [0], []
        for b in range(2):
            for h in range(3):
                for qb in range(7):
                    for kb in range(7):
                        if mask[b, h, qb, kb] and (not causal or kb <= qb):
                            exp_col.append(kb)
                    exp_ptr.append(len(exp_col))
        m = mask.astype(bool)
        if causal:
            m = m & np.tril(np.ones((7, 7), dtype=bool))
        if row_ptr.tolist() != exp_ptr or col_idx.tolist() != exp_col:
            return False, f"causal={causal}: enumeration differs"
        if int(row_ptr[-1]) != int(m.sum()):
            return False, "nnz != popcount"
    return True, "ok"


PINS = [pin_worked_examples, pin_bruteforce, pin_sdpa_dense, pin_sdpa_causal,
        pin_sdpa_block_mask, pin_scale_zero, pin_constant_v, pin_single_key,
        pin_permutation_invariance, pin_shift_invariance, pin_diagonal_only,
        pin_fully_masked_rows, pin_csr]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(oracle_lib, gen, pin):
    oracle.set_mutation(0)
    ok, detail = pin()
    assert ok, detail


def test_every_planted_mistake_is_caught(oracle_lib, gen):
    """Each plausible mistake planted in the oracle makes at least one pin fail."""
    missed = []
    try:
        for m, what in oracle.MUTATIONS.items():
            oracle.set_mutation(m)
            failed = []
            for pin in PINS:
                try:
                    ok, _ = pin()
                except Exception:  # noqa: BLE001 - a crash also counts as caught
                    ok = False
                if not ok:
                    failed.append(pin.__name__)
            if not failed:
                missed.append(what)
    finally:
        oracle.set_mutation(0)
    assert not missed, f"mistakes no pin catches: {missed}"


def test_generator_matches_published_splitmix64(gen):
    """splitmix64 seeded with 0: the published first outputs."""
    got = workloads.splitmix64_raw(0, 3)
    assert [int(x) for x in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_generator_normal_moments(gen):
    x = workloads.bf16_bits_to_f32(workloads.normal_bf16(1, 1, (1 << 20,))).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    # bf16 round-to-nearest-even: every value is exactly representable as bf16
    assert np.all((x.astype(np.float32).view(np.uint32) & 0xFFFF) == 0)


def test_workload_masks(gen):
    w = workloads.WORKLOADS
    m3 = workloads.make_mask(w[3], B=1, H=2)
    assert m3.shape == (1, 2, 128, 128)
    assert np.all(m3.sum(axis=-1)[:, :, :2] == 128)     # global rows
    assert np.all(m3[:, :, :, :2] == 1)                 # global cols
    assert int(m3.sum()) == 2 * 2000                    # window + global + 3 random per row
    m1 = workloads.make_mask(w[1])
    assert np.all(np.diagonal(m1, axis1=2, axis2=3) == 1)
    m2 = workloads.make_mask(w[2], B=1, H=1)
    assert np.array_equal(m2[0, 0], np.tril(np.ones((32, 32), dtype=np.uint8)))


# ----------------------------------------------------------------------------
# grouped-query attention and a mask shared by the heads
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("Hkv,causal", [(1, False), (2, True), (4, False)])
def test_gqa_against_torch_sdpa(Hkv, causal):
    """torch float64 SDPA with enable_gqa (a library routine) for an all-ones mask."""
    torch = pytest.importorskip("torch")
    B, H, S, D = 1, 4, 256, 8
    rng = np.random.default_rng(60 + Hkv)
    q = rng.standard_normal((B, H, S, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    mask = np.ones((B, 1, S // 128, S // 128), np.uint8)
    O, _ = oracle.attention_gqa(q, k, v, mask, 0.3, causal)
    try:
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q), torch.tensor(k), torch.tensor(v), is_causal=causal, scale=0.3,
            enable_gqa=True).numpy()
    except TypeError:
        pytest.skip("torch without enable_gqa")
    assert np.max(np.abs(O - ref)) < 1e-12


def test_shared_mask_equals_per_head_copies():
    """A [B, 1, nb, nb] mask gives, for every head, the result of that head with the
    mask copied to it (checked head by head against single-head calls)."""
    B, H, S, D = 2, 3, 256, 8
    rng = np.random.default_rng(70)
    q, k, v = (rng.standard_normal((B, H, S, D)) for _ in range(3))
    mask = np.array([[[[1, 0], [1, 1]]], [[[0, 1], [1, 0]]]], np.uint8)  # [B=2, 1, 2, 2]
    O, L = oracle.attention_gqa(q, k, v, mask, 0.5, False)
    for b in range(B):
        for h in range(H):
            Oh, Lh = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                      mask[b:b + 1], 0.5, False)
            assert np.array_equal(O[b, h], Oh[0, 0]) and np.array_equal(L[b, h], Lh[0, 0],
                                                                        equal_nan=True)
