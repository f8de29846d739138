"""GPU parity of 64-key blocks (a plan built with key_block=64: one mask
entry per 128-query x 64-key block), through the C ABI, against the oracle
(oracle.attention_kb): the CSR bit for bit, the schedule, every row of the
forward pass in both output modes, and bit-identity with the 128-key path
when the mask repeats a 128-key mask (the kernel then runs the same pairs of
halves as whole blocks)."""
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


def _mask64(seed, B, H, nbq, p, diag=True):
    rng = np.random.default_rng(seed)
    m = (rng.random((B, H, nbq, 2 * nbq)) < p).astype(np.uint8)
    if diag:
        m[:, :, np.arange(nbq), 2 * np.arange(nbq)] = 1
    return m


def _expected_schedule(counts, BH, nb, nsm, kdiv=2):
    """The documented tile order with lengths counted in pairs of 64-key
    blocks: chunks of max(1, 768 // nb) heads, longest first inside a chunk
    (ties by tile id), tiles long for their chunk moved one chunk earlier."""
    kh = max(1, 768 // nb)
    c = counts.reshape(BH, nb)
    keys = []
    for h in range(BH):
        k = h // kh
        thr = int(c[k * kh:(k + 1) * kh].sum()) // kdiv // (2 * nsm)
        for qb in range(nb):
            n = -(-int(c[h, qb]) // kdiv)
            if n == 0:
                continue
            kk = k - 1 if (k > 0 and n > thr) else k
            keys.append((kk, -n, h * nb + qb))
    keys.sort()
    return np.asarray([t for _, _, t in keys], dtype=np.int64)


@pytest.mark.parametrize("causal", [False, True])
def test_plan_csr_and_schedule(bs, causal):
    import torch
    B, H, nbq = 2, 12, 40
    mask = _mask64(1, B, H, nbq, 0.3)
    mask[0, 3] = 0                 # a dead head
    mask[1, 2, 7] = 0              # an empty query tile
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=causal, key_block=64)
    rp, ci = bs.plan_csr(p)
    rp_ref, ci_ref = oracle.csr_kb(mask, causal)
    assert np.array_equal(rp.cpu().numpy(), rp_ref)
    assert np.array_equal(ci.cpu().numpy(), ci_ref)
    order, empty = (x.cpu().numpy() for x in bs.plan_schedule(p))
    counts = np.diff(rp_ref)
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    assert np.array_equal(order, _expected_schedule(counts, B * H, nbq, nsm))
    assert np.array_equal(empty, np.flatnonzero(counts == 0))
    p.close()


CASES = {
    # name: (B, H, S, D, mask builder, causal, scale, mult)
    "d128_sparse": (1, 3, 1024, 128, lambda: _mask64(2, 1, 3, 8, 0.35), False, 128 ** -0.5, 1.0),
    "d128_causal": (1, 3, 1024, 128, lambda: _mask64(3, 1, 3, 8, 0.45), True, 128 ** -0.5, 1.0),
    "d64_sparse": (2, 2, 1024, 64, lambda: _mask64(4, 2, 2, 8, 0.3, diag=False), False, 0.125, 1.0),
    "d64_causal_wide": (1, 2, 1024, 64, lambda: _mask64(5, 1, 2, 8, 0.6), True, 0.125, 2.0),
    # causal, only the second half of each diagonal live: rows 0..63 of every
    # query tile see no key at all (O = 0, LSE = -inf inside a live tile)
    "second_half_only": (1, 2, 512, 128,
                         lambda: np.tile(np.kron(np.eye(4, dtype=np.uint8), np.array([[0, 1]], np.uint8)),
                                         (1, 2, 1, 1)), True, 0.09, 1.0),
    # one live 64-key block per tile: every pair is an odd tail
    "odd_tails": (1, 2, 768, 64, lambda: np.eye(6, 12, k=3, dtype=np.uint8)[None, None].repeat(2, 1),
                  False, 0.125, 1.0),
    "all_dead": (1, 1, 256, 128, lambda: np.zeros((1, 1, 2, 4), np.uint8), False, 0.1, 1.0),
    "long_rows": (1, 1, 4096, 128, lambda: _mask64(6, 1, 1, 32, 0.8), True, 128 ** -0.5, 1.0),
}


@pytest.mark.parametrize("out_f32", [True, False], ids=["o_f32", "o_bf16"])
@pytest.mark.parametrize("name", list(CASES))
def test_small_every_row(bs, name, out_f32):
    import torch
    B, H, S, D, mk, causal, scale, mult = CASES[name]
    qb, kb, vb = workloads.custom(600 + len(name), B, H, S, D, mult)
    mask = mk()
    p = bs.plan(torch.from_numpy(np.ascontiguousarray(mask)).cuda(), causal=causal,
                out_f32=out_f32, key_block=64)
    o, lse = bs.fwd(to_dev(qb), to_dev(kb), to_dev(vb), p, scale)
    bs.plan_status(p)
    p.close()
    O_ref, L_ref = oracle.attention_kb(qb, kb, vb, mask, np.float32(scale), causal)
    ok, rep = compare(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref,
                      out_bf16=not out_f32)
    assert ok, rep


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_repeated_mask_bit_identical_to_128_key_blocks(bs, wid):
    """The five workloads' masks re-expressed at 64-key granularity (every
    128-key entry repeated): the same pairs of halves run as the 128-key
    blocks, so O and LSE are bit-identical (the 128-key path is checked
    against the oracle on every row)."""
    import torch
    w = workloads.WORKLOADS[wid]
    qb, kb, vb = workloads.make_qkv(w)
    mask = workloads.make_mask(w)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    p128 = bs.plan(torch.from_numpy(mask).cuda(), causal=w.causal)
    p64 = bs.plan(torch.from_numpy(np.repeat(mask, 2, axis=3)).cuda(), causal=w.causal,
                  key_block=64)
    o1, l1 = bs.fwd(q, k, v, p128, w.scale)
    o2, l2 = bs.fwd(q, k, v, p64, w.scale)
    bs.plan_status(p128)
    bs.plan_status(p64)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    p128.close()
    p64.close()


def test_full_size_fine_mask_every_row(bs):
    """A random mask drawn at 64-key granularity (10 % density, diagonal
    blocks live) at S = 16384, D = 128, every row against the oracle."""
    import torch
    B, H, S, D = 1, 4, 16384, 128
    nbq = S // 128
    rng = np.random.default_rng(21)
    mask = (rng.random((B, H, nbq, 2 * nbq)) < 0.1).astype(np.uint8)
    mask[:, :, np.arange(nbq), 2 * np.arange(nbq)] = 1
    qb, kb, vb = workloads.custom(22, B, H, S, D)
    p = bs.plan(torch.from_numpy(mask).cuda(), out_f32=True, key_block=64)
    o, lse = bs.fwd(to_dev(qb), to_dev(kb), to_dev(vb), p, D ** -0.5)
    bs.plan_status(p)
    p.close()
    o = o.reshape(-1, D).cpu().numpy()
    lse = lse.reshape(-1).cpu().numpy()
    for h in range(B * H):
        rows = np.arange(h * S, (h + 1) * S, dtype=np.int64)
        O_ref, L_ref = oracle.attention_kb(qb, kb, vb, mask, np.float32(D ** -0.5), False,
                                           rows=rows)
        ok, rep = compare(o[rows], lse[rows], O_ref, L_ref)
        assert ok, (h, rep)


def test_backward_rejects_64_key_blocks(bs):
    import torch
    B, H, S, D = 1, 1, 256, 64
    mask = torch.ones((B, H, 2, 4), dtype=torch.uint8, device="cuda")
    p = bs.plan(mask, key_block=64)
    x = torch.zeros((B, H, S, D), dtype=torch.bfloat16, device="cuda")
    o, lse = bs.fwd(x, x, x, p, 0.1)
    with pytest.raises(bs.BsattnError) as e:
        bs.bwd(x, x, x, o, lse, x, p, 0.1)
    assert e.value.status == bs.ERR_UNSUPPORTED
    with pytest.raises(bs.BsattnError):
        bs.plan_csc(p)
    bs.plan_status(p)
    p.close()
