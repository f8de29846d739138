"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Element-by-element comparison on seeded inputs at sizes the oracle finishes
in seconds (several tiles, rows of different lengths, empty tiles), and at
the five workloads' full sizes on every row, in the launch configuration
the bench times.  The plan's CSR must match the
oracle's bit for bit; the schedule must be a valid ordering.
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


def _run(bs, qb, kb, vb, mask, scale, causal, out_f32):
    import torch
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    p = bs.plan(torch.from_numpy(np.ascontiguousarray(mask)).cuda(), causal=causal, out_f32=out_f32)
    o, lse = bs.fwd(q, k, v, p, scale)
    bs.plan_status(p)
    return o.float().cpu().numpy(), lse.cpu().numpy(), p


# ----------------------------------------------------------------------------
# device-side timeout path
# ----------------------------------------------------------------------------

def test_bounded_wait_times_out(bs):
    """A wait on a barrier nothing completes ends by its limit and reports it."""
    assert bs.selftest_wait_timeout(2_000_000) == bs.ERR_TIMEOUT
    assert bs.selftest_wait_timeout(200_000) == bs.ERR_TIMEOUT


# ----------------------------------------------------------------------------
# plan: CSR bit-exact, schedule valid
# ----------------------------------------------------------------------------

def _check_plan(bs, mask, causal):
    import torch
    p = bs.plan(torch.from_numpy(np.ascontiguousarray(mask)).cuda(), causal=causal)
    rp, ci = bs.plan_csr(p)
    rp_ref, ci_ref = oracle.csr(mask, causal)
    assert np.array_equal(rp.cpu().numpy(), rp_ref)
    assert np.array_equal(ci.cpu().numpy(), ci_ref)
    order, empty = (x.cpu().numpy() for x in bs.plan_schedule(p))
    counts = np.diff(rp_ref)
    B, H, nb, _ = mask.shape
    live = np.flatnonzero(counts > 0)
    assert np.array_equal(np.sort(order), live)
    assert np.array_equal(np.sort(empty), np.flatnonzero(counts == 0))
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    assert np.array_equal(order, _expected_schedule(counts, B * H, nb, nsm))
    assert np.array_equal(empty, np.flatnonzero(counts == 0)), "empty tiles head by head, qb asc"
    p.close()


def _expected_schedule(counts, BH, nb, nsm):
    """The documented tile order, restated with plain loops: chunks of
    max(1, 768 // nb) heads, longest first inside a chunk (ties by tile id),
    tiles long for their chunk (count > chunk blocks // (2 * nsm)) moved one
    chunk earlier."""
    kh = max(1, 768 // nb)
    c = counts.reshape(BH, nb)
    keys = []
    for h in range(BH):
        k = h // kh
        thr = int(c[k * kh:(k + 1) * kh].sum()) // (2 * nsm)
        for qb in range(nb):
            n = int(c[h, qb])
            if n == 0:
                continue
            kk = k - 1 if (k > 0 and n > thr) else k
            keys.append((kk, -n, h * nb + qb))
    keys.sort()
    return np.asarray([t for _, _, t in keys], dtype=np.int64)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_plan_csr_bit_exact(bs, wid):
    w = workloads.WORKLOADS[wid]
    _check_plan(bs, workloads.make_mask(w), w.causal)


def test_plan_edge_masks(bs):
    rng = np.random.default_rng(0)
    m = (rng.random((2, 3, 9, 9)) < 0.3).astype(np.uint8)
    m[0, 1] = 0                       # a fully dead head
    m[1, 2, 4] = 0                    # one empty row
    for causal in (False, True):
        _check_plan(bs, m, causal)
    _check_plan(bs, np.zeros((1, 1, 1, 1), np.uint8), False)
    _check_plan(bs, np.ones((1, 1, 1, 1), np.uint8), True)


# ----------------------------------------------------------------------------
# small cases, every row compared
# ----------------------------------------------------------------------------

def _mask_iid(seed, B, H, nb, p, diag=False):
    rng = np.random.default_rng(seed)
    m = (rng.random((B, H, nb, nb)) < p).astype(np.uint8)
    if diag:
        m[:, :, np.arange(nb), np.arange(nb)] = 1
    return m


CASES = {
    # name: (B, H, S, D, mask builder, causal, scale, mult)
    "w1": (1, 2, 512, 64, lambda: workloads.make_mask(workloads.WORKLOADS[1]), False, 0.125, 1.0),
    "s1024_d128_causal": (1, 2, 1024, 128, lambda: _mask_iid(1, 1, 2, 8, 0.4, diag=True), True, 128 ** -0.5, 1.0),
    "s1024_d64_sparse": (1, 2, 1024, 64, lambda: _mask_iid(2, 1, 2, 8, 0.3), False, 0.125, 1.0),
    "one_tile_d128": (1, 1, 128, 128, lambda: np.ones((1, 1, 1, 1), np.uint8), False, 128 ** -0.5, 1.0),
    "one_tile_d64_causal": (2, 1, 128, 64, lambda: np.ones((2, 1, 1, 1), np.uint8), True, 0.125, 1.0),
    "all_dead": (1, 2, 256, 128, lambda: np.zeros((1, 2, 2, 2), np.uint8), False, 0.1, 1.0),
    "empty_rows": (1, 2, 512, 128, lambda: np.array([[[[1, 0, 0, 1], [0, 0, 0, 0], [0, 1, 1, 0], [0, 0, 0, 0]],
                                                      [[0, 0, 0, 0], [1, 1, 1, 1], [0, 0, 0, 0], [0, 0, 0, 1]]]], np.uint8),
                   False, 0.09, 1.0),
    "one_block_per_row": (1, 2, 1024, 64, lambda: np.eye(8, dtype=np.uint8)[np.random.default_rng(3).permutation(8)][None, None].repeat(2, 1), False, 0.125, 1.0),
    "causal_dead_diag": (1, 1, 512, 128, lambda: np.tril(np.ones((4, 4), np.uint8), -1)[None, None], True, 0.09, 1.0),
    "scale_zero": (1, 1, 512, 128, lambda: _mask_iid(4, 1, 1, 4, 0.6, diag=True), True, 0.0, 1.0),
    "scale_tiny": (1, 1, 512, 64, lambda: _mask_iid(5, 1, 1, 4, 0.6, diag=True), False, 1e-6, 1.0),
    "scale_large": (1, 1, 512, 64, lambda: _mask_iid(6, 1, 1, 4, 0.6, diag=True), False, 2.0, 1.0),
    "scale_negative": (1, 1, 512, 128, lambda: _mask_iid(7, 1, 1, 4, 0.6, diag=True), True, -0.2, 1.0),
    "wide_logits_d64": (1, 2, 1024, 64, lambda: np.ones((1, 2, 8, 8), np.uint8), False, 0.125, 2.0),
    "many_tiles": (4, 16, 1024, 128, lambda: _mask_iid(8, 4, 16, 8, 0.35, diag=True), False, 128 ** -0.5, 1.0),
    "many_tiles_causal_d64": (2, 16, 2048, 64, lambda: _mask_iid(9, 2, 16, 16, 0.5, diag=True), True, 0.125, 1.0),
}


@pytest.mark.parametrize("out_f32", [True, False], ids=["o_f32", "o_bf16"])
@pytest.mark.parametrize("name", list(CASES))
def test_small_every_row(bs, name, out_f32):
    B, H, S, D, mk, causal, scale, mult = CASES[name]
    qb, kb, vb = workloads.custom(100 + len(name), B, H, S, D, mult)
    mask = mk()
    o, lse, p = _run(bs, qb, kb, vb, mask, scale, causal, out_f32)
    p.close()
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(scale), causal)
    ok, rep = compare(o, lse, O_ref, L_ref, out_bf16=not out_f32)
    assert ok, rep


def test_repeated_calls_same_plan(bs):
    """The plan's workspace (tile counter) rewinds itself between launches."""
    import torch
    B, H, S, D = 2, 8, 1024, 128
    qb, kb, vb = workloads.custom(77, B, H, S, D)
    mask = _mask_iid(10, B, H, 8, 0.5, diag=True)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    p = bs.plan(torch.from_numpy(mask).cuda(), out_f32=True)
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(D ** -0.5), False)
    for _ in range(5):
        o, lse = bs.fwd(q, k, v, p, D ** -0.5)
    bs.plan_status(p)
    ok, rep = compare(o.cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref)
    assert ok, rep
    p.close()


@pytest.mark.parametrize("out_f32", [True, False], ids=["o_f32", "o_bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_output_only_16_byte_aligned(bs, D, out_f32):
    """An output buffer that is 16- but not 32-byte aligned (a view into a
    larger allocation) gets the same values as an aligned one, and nothing
    around it is written."""
    import torch
    B, H, S = 1, 4, 512
    qb, kb, vb = workloads.custom(91 + D, B, H, S, D)
    mask = _mask_iid(11, B, H, S // 128, 0.5, diag=True)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=True, out_f32=out_f32)
    o_al, l_al = bs.fwd(q, k, v, p, D ** -0.5)
    odt = torch.float32 if out_f32 else torch.bfloat16
    n = B * H * S * D
    pad = 16 // odt.itemsize + 32 // odt.itemsize  # 16-byte offset, then a guard band
    raw = torch.full((n + 2 * pad,), -7.0, dtype=odt, device="cuda")
    off = 16 // odt.itemsize
    base = raw.data_ptr() % 32
    if base != 0:  # make raw[off:] sit 16 bytes past a 32-byte boundary
        off += (32 - base) // odt.itemsize
    out = raw[off:off + n].view(B, H, S, D)
    assert out.data_ptr() % 32 == 16
    o_un, l_un = bs.fwd(q, k, v, p, D ** -0.5, out=out)
    bs.plan_status(p)
    assert torch.equal(o_un, o_al) and torch.equal(l_un, l_al)
    assert bool((raw[:off] == -7.0).all()) and bool((raw[off + n:] == -7.0).all())
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(D ** -0.5), True)
    ok, rep = compare(o_un.float().cpu().numpy(), l_un.cpu().numpy(), O_ref, L_ref,
                      out_bf16=not out_f32)
    assert ok, rep
    p.close()


# ----------------------------------------------------------------------------
# full-size workloads, every row
# ----------------------------------------------------------------------------

# Rows per oracle call at full size: bounds the host memory of one chunk of
# the fp64 reference (rows x D x 8 bytes) to about 256 MB.
_CHUNK_BYTES = 256 << 20


@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_full_size_every_row(bs, wid):
    """The workload at full size, in the launch configuration the bench times,
    both output modes; every row of O and LSE against the oracle, element by
    element, whole heads at a time."""
    import torch
    w = workloads.WORKLOADS[wid]
    qb, kb, vb = workloads.make_qkv(w)
    mask = workloads.make_mask(w)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    mask_d = torch.from_numpy(mask).cuda()
    B, H, S, D = qb.shape
    results = {}
    for out_f32 in (False, True):
        p = bs.plan(mask_d, causal=w.causal, out_f32=out_f32)
        o, lse = bs.fwd(q, k, v, p, w.scale)
        bs.plan_status(p)
        p.close()
        results[out_f32] = (o.reshape(-1, D).float().cpu().numpy(), lse.reshape(-1).cpu().numpy())
        del o, lse
    del q, k, v
    torch.cuda.empty_cache()
    heads = max(1, _CHUNK_BYTES // (S * D * 8))
    worst = {False: {}, True: {}}
    for h0 in range(0, B * H, heads):
        rows = np.arange(h0 * S, min(B * H, h0 + heads) * S, dtype=np.int64)
        O_ref, L_ref = oracle.attention(qb, kb, vb, mask, w.scale, w.causal, rows=rows)
        for out_f32, (o, lse) in results.items():
            ok, rep = compare(o[rows], lse[rows], O_ref, L_ref, out_bf16=not out_f32)
            assert ok, (wid, out_f32, h0, rep)
            for key in ("max_dO", "mean_dO", "max_dLSE"):
                worst[out_f32][key] = max(worst[out_f32].get(key, 0.0), rep[key])
    print(f"workload {wid} every row: bf16 O {worst[False]}, fp32 O {worst[True]}")


# ----------------------------------------------------------------------------
# argument checks with a real plan (nothing is launched on error)
# ----------------------------------------------------------------------------

def test_fwd_argument_errors(bs):
    import torch
    lib = bs.load()
    mask = torch.ones((1, 1, 2, 2), dtype=torch.uint8, device="cuda")
    p = bs.plan(mask)
    buf = torch.zeros(1 * 1 * 256 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(256, dtype=torch.float32, device="cuda")
    ptr = buf.data_ptr()
    vp = ctypes.c_void_p
    st = vp(torch.cuda.current_stream().cuda_stream)

    def call(q=ptr, k=ptr, v=ptr, out=ptr, l=lse.data_ptr(), B=1, H=1, S=256, D=128, scale=0.1):
        return lib.bsattn_fwd(vp(q), vp(k), vp(v), p.handle, vp(out), vp(l), B, H, S, D,
                              ctypes.c_float(scale), st)

    assert call(q=ptr + 2) == bs.ERR_INVALID_ARG            # misaligned
    assert call(out=0) == bs.ERR_INVALID_ARG                # null
    assert call(S=512) == bs.ERR_INVALID_ARG                # differs from the plan
    assert call(H=2) == bs.ERR_INVALID_ARG
    assert call(D=96) == bs.ERR_UNSUPPORTED
    assert call(scale=float("inf")) == bs.ERR_INVALID_ARG
    assert call(scale=float("nan")) == bs.ERR_INVALID_ARG
    assert lib.bsattn_fwd(vp(ptr), vp(ptr), vp(ptr), vp(0), vp(ptr), vp(lse.data_ptr()), 1, 1, 256,
                          128, ctypes.c_float(0.1), st) == bs.ERR_INVALID_ARG  # no plan
    bs.plan_status(p)
    p.close()


# ----------------------------------------------------------------------------
# host-buffer path: same kernel per piece, so bit-identical to the device path
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("wid,chunks", [(1, 2), (2, 3), (5, 4)])
def test_host_pipeline_matches_device_path(bs, wid, chunks):
    import torch
    w = workloads.WORKLOADS[wid]
    qb, kb, vb = workloads.make_qkv(w)
    mask = workloads.make_mask(w)
    mask_d = torch.from_numpy(mask).cuda()
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    p = bs.plan(mask_d, causal=w.causal)
    o_ref, l_ref = bs.fwd(q, k, v, p, w.scale)
    bs.plan_status(p)
    p.close()
    host = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory()
    hq, hk, hv = host(qb), host(kb), host(vb)
    ho = torch.empty(o_ref.shape, dtype=o_ref.dtype).pin_memory()
    hl = torch.empty(l_ref.shape, dtype=l_ref.dtype).pin_memory()
    pipe = bs.HostPipeline(mask_d, w.D, causal=w.causal, chunks=chunks)
    for _ in range(2):  # the second call reuses the device buffers
        ho.zero_()
        pipe.run(hq, hk, hv, ho, hl, w.scale)
        torch.cuda.current_stream().synchronize()
        pipe.status()
        assert torch.equal(ho, o_ref.cpu())
        assert torch.equal(hl, l_ref.cpu())
    pipe.close()


# ----------------------------------------------------------------------------
# the largest supported sequence (S/128 = 4096 key blocks per row), sampled rows
# ----------------------------------------------------------------------------

def test_max_blocks_per_row_sampled(bs):
    import torch
    B, H, S, D = 1, 1, 4096 * 128, 128
    nb = S // 128
    rng = np.random.default_rng(11)
    mask = np.zeros((B, H, nb, nb), np.uint8)
    mask[0, 0, np.arange(nb), np.arange(nb)] = 1                       # diagonal
    mask[0, 0, np.arange(nb)[:, None], rng.integers(0, nb, (nb, 2))] = 1  # two random blocks per row
    mask[0, 0, 5, :] = 1                                                 # one row with every block live
    qb, kb, vb = workloads.custom(211, B, H, S, D, 1.0)
    scale = D ** -0.5
    o, lse, p = _run(bs, qb, kb, vb, mask, scale, False, True)
    p.close()
    rows = np.unique(np.concatenate([5 * 128 + np.arange(128),            # the dense tile
                                     rng.integers(0, S, 96)])).astype(np.int64)
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(scale), False, rows=rows)
    ok, rep = compare(o.reshape(-1, D)[rows], lse.reshape(-1)[rows], O_ref, L_ref, out_bf16=False)
    assert ok, rep


# ----------------------------------------------------------------------------
# a later key block whose scores far exceed the first block's (the softmax
# must abandon its running reference for that block and rescale)
# ----------------------------------------------------------------------------

def _bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("D", [64, 128])
def test_scores_jump_in_a_later_block(bs, D):
    B, H, S = 1, 2, 768
    qb, kb, vb = workloads.custom(313, B, H, S, D, 1.0)
    q = np.abs(_bf16_float(qb))                 # positive queries
    k = _bf16_float(kb)
    k[:, :, 384:512, :] = np.abs(k[:, :, 384:512, :]) * 6.0    # block 3: scores far above block 0
    k[:, :, 640:, :] = np.abs(k[:, :, 640:, :]) * 12.0         # block 5: far above block 3
    qb, kb = _bf16_bits(q), _bf16_bits(k)
    mask = np.ones((B, H, S // 128, S // 128), np.uint8)
    scale = D ** -0.5
    for out_f32 in (True, False):
        o, lse, p = _run(bs, qb, kb, vb, mask, scale, False, out_f32)
        p.close()
        O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(scale), False)
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
        ok, rep = compare(o, lse, O_ref, L_ref, out_bf16=not out_f32)
        assert ok, (out_f32, rep)


# ----------------------------------------------------------------------------
# D = 64 multiplies P by V in fp16: a V entry beyond fp16's range is reported
# ----------------------------------------------------------------------------

# (D, B, H, S): at D = 64 the small size converts V in the kernel, the large
# one through the plan's fp16 copy of V (16 heads x 2048 rows, ~5 live blocks
# per key block)
@pytest.mark.parametrize("D,B,H,S", [(64, 1, 2, 512), (64, 1, 16, 2048), (128, 1, 2, 512)])
def test_v_beyond_fp16_range(bs, D, B, H, S):
    import torch
    qb, kb, vb = workloads.custom(417 + D, B, H, S, D)
    mask = _mask_iid(12, B, H, S // 128, 0.6, diag=True)
    v = _bf16_float(vb)
    v_big = v.copy()
    v_big[0, 1, S - 212, 7] = 70000.0     # rounds to a bf16 above 65504
    v_edge = v.copy()
    v_edge[0, 1, S - 212, 7] = 65280.0    # the largest bf16 below 65504: exact in fp16
    p = bs.plan(torch.from_numpy(mask).cuda(), out_f32=True)
    q, k = to_dev(qb), to_dev(kb)
    o, _ = bs.fwd(q, k, to_dev(_bf16_bits(v_edge)), p, D ** -0.5)
    bs.plan_status(p)
    assert bool(torch.isfinite(o).all())
    assert (bs.plan_v16_bytes(p) > 0) == (D == 64 and H * S >= 16384)
    o, _ = bs.fwd(q, k, to_dev(_bf16_bits(v_big)), p, D ** -0.5)
    if D == 64:
        with pytest.raises(bs.BsattnError) as e:
            bs.plan_status(p)
        assert e.value.status == bs.ERR_RANGE
    else:
        bs.plan_status(p)
        assert bool(torch.isfinite(o).all())
    # the status was cleared: the plan works again
    o, lse = bs.fwd(q, k, to_dev(vb), p, D ** -0.5)
    bs.plan_status(p)
    p.close()
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(D ** -0.5), False)
    ok, rep = compare(o.cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref)
    assert ok, rep


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_v16_copy_matches_in_kernel_conversion(bs, causal):
    """At head_dim 64 a plan whose key blocks serve several query tiles gets an
    fp16 copy of V before the launch, and the kernel reads it instead of
    converting each V tile in shared memory.  Both give the same fp16 values,
    so O and LSE must agree bit for bit with the in-kernel conversion (which
    bsattn_fwd_noalloc always uses), and every row with the oracle."""
    import torch
    B, H, S, D = 1, 16, 2048, 64
    qb, kb, vb = workloads.custom(611 + causal, B, H, S, D)
    mask = _mask_iid(13, B, H, S // 128, 0.6, diag=True)
    mask_d = torch.from_numpy(mask).cuda()
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    p = bs.plan(mask_d, causal=causal)
    assert bs.plan_v16_bytes(p) == 0
    o, lse = bs.fwd(q, k, v, p, 0.125)
    bs.plan_status(p)
    assert bs.plan_v16_bytes(p) == B * H * S * D * 2
    o2, lse2 = bs.fwd(q, k, v, p, 0.125)  # the copy is reused
    bs.plan_status(p)
    p.close()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    o3, lse3 = bs.fwd_noalloc(q, k, v, mask_d, causal=causal, scale=0.125)
    torch.cuda.synchronize()
    assert torch.equal(o, o3) and torch.equal(lse, lse3)
    O_ref, L_ref = oracle.attention(qb, kb, vb, mask, np.float32(0.125), causal)
    ok, rep = compare(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref, out_bf16=True)
    assert ok, rep
