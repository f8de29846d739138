"""GPU parity of the forward pass on FP8 (e4m3) inputs, through the C ABI,
against the fp64 oracle on the decoded inputs (oracle.attention_fp8): every
row, both output modes, the tolerances of the bf16 path (the kernel's S
products of e4m3 values are exact in fp32, and P V runs in fp16)."""
import numpy as np
import pytest

import oracle
import workloads
from _util import compare

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


def _dev8(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits)).cuda().view(torch.float8_e4m3fn)


def _inputs(seed, B, H, S, D, mult=1.0):
    return tuple(workloads.normal_e4m3(seed, st, (B, H, S, D), mult)
                 for st in (workloads.STREAM_Q, workloads.STREAM_K, workloads.STREAM_V))


def _mask_iid(seed, B, H, nb, p, diag=True, kdiv=1):
    rng = np.random.default_rng(seed)
    m = (rng.random((B, H, nb, kdiv * nb)) < p).astype(np.uint8)
    if diag:
        m[:, :, np.arange(nb), kdiv * np.arange(nb)] = 1
    return m


CASES = {
    # name: (B, H, S, mask builder, causal, scale, v_scale, mult, key_block)
    "sparse": (1, 3, 1024, lambda: _mask_iid(1, 1, 3, 8, 0.4), False, 128 ** -0.5, 1.0, 1.0, 128),
    "causal": (2, 2, 1024, lambda: _mask_iid(2, 2, 2, 8, 0.5), True, 128 ** -0.5, 1.0, 1.0, 128),
    "scaled": (1, 2, 512, lambda: np.ones((1, 2, 4, 4), np.uint8), True, 0.05, 0.25, 4.0, 128),
    "negative_scale": (1, 2, 512, lambda: _mask_iid(3, 1, 2, 4, 0.6), False, -0.1, 2.0, 1.0, 128),
    "empty_rows": (1, 2, 512, lambda: np.array([[[[1, 0, 0, 1], [0, 0, 0, 0], [0, 1, 1, 0], [0, 0, 0, 0]],
                                                [[0, 0, 0, 0], [1, 1, 1, 1], [0, 0, 0, 0], [0, 0, 0, 1]]]],
                                              np.uint8), False, 0.09, 1.0, 1.0, 128),
    "key_block_64": (1, 2, 1024, lambda: _mask_iid(4, 1, 2, 8, 0.3, kdiv=2), True, 128 ** -0.5, 1.0,
                     1.0, 64),
    "long_rows": (1, 1, 4096, lambda: _mask_iid(5, 1, 1, 32, 0.8), False, 128 ** -0.5, 1.0, 1.0, 128),
}


@pytest.mark.parametrize("out_f32", [True, False], ids=["o_f32", "o_bf16"])
@pytest.mark.parametrize("name", list(CASES))
def test_small_every_row(bs, name, out_f32):
    import torch
    B, H, S, mk, causal, scale, v_scale, mult, kblk = CASES[name]
    D = 128
    q8, k8, v8 = _inputs(700 + len(name), B, H, S, D, mult)
    mask = mk()
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=causal, out_f32=out_f32, key_block=kblk)
    o, lse = bs.fwd_fp8(_dev8(q8), _dev8(k8), _dev8(v8), p, scale, v_scale)
    bs.plan_status(p)
    p.close()
    if kblk == 128:
        O_ref, L_ref = oracle.attention_fp8(q8, k8, v8, mask, np.float32(scale), causal,
                                            v_scale=v_scale)
    else:
        q, k, v = (oracle.decode_e4m3(x) for x in (q8, k8, v8))
        O_ref, L_ref = oracle.attention_kb(q, k, v, mask, np.float32(scale), causal)
        O_ref = O_ref * v_scale
    ok, rep = compare(o.float().cpu().numpy(), lse.cpu().numpy(), O_ref, L_ref,
                      out_bf16=not out_f32)
    assert ok, rep


@pytest.mark.parametrize("wid", [2, 3])
def test_full_size_every_row(bs, wid):
    """The causal S = 4096 and BigBird S = 16384 workloads (D = 128) with
    e4m3 inputs drawn from the same normal streams, every row."""
    import torch
    w = workloads.WORKLOADS[wid]
    q8, k8, v8 = _inputs(w.data_seed, w.B, w.H, w.S, w.D)
    mask = workloads.make_mask(w)
    p = bs.plan(torch.from_numpy(mask).cuda(), causal=w.causal, out_f32=True)
    o, lse = bs.fwd_fp8(_dev8(q8), _dev8(k8), _dev8(v8), p, w.scale)
    bs.plan_status(p)
    p.close()
    o = o.reshape(-1, w.D).cpu().numpy()
    lse = lse.reshape(-1).cpu().numpy()
    heads = max(1, (256 << 20) // (w.S * w.D * 8))
    for h0 in range(0, w.B * w.H, heads):
        rows = np.arange(h0 * w.S, min(w.B * w.H, h0 + heads) * w.S, dtype=np.int64)
        O_ref, L_ref = oracle.attention_fp8(q8, k8, v8, mask, w.scale, w.causal, rows=rows)
        ok, rep = compare(o[rows], lse[rows], O_ref, L_ref)
        assert ok, (h0, rep)


# (B, H, S): V converted tile by tile in the kernel, and through the plan's
# fp16 copy of V (16 heads x 2048 rows, 16 live blocks per key block)
@pytest.mark.parametrize("B,H,S", [(1, 1, 256), (1, 16, 2048)])
def test_nan_in_v_is_reported_and_d64_unsupported(bs, B, H, S):
    import torch
    D = 128
    q8, k8, v8 = _inputs(9, B, H, S, D)
    v8 = v8.copy()
    v8[0, 0, 200, 3] = 0x7F  # e4m3 NaN
    nb = S // 128
    p = bs.plan(torch.ones((B, H, nb, nb), dtype=torch.uint8, device="cuda"))
    bs.fwd_fp8(_dev8(q8), _dev8(k8), _dev8(v8), p, 0.1)
    with pytest.raises(bs.BsattnError) as e:
        bs.plan_status(p)
    assert e.value.status == bs.ERR_RANGE
    assert (bs.plan_v16_bytes(p) > 0) == (B * H * S >= 16384)
    x = torch.zeros((B, H, S, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(bs.BsattnError) as e:
        bs.fwd_fp8(x, x, x, p, 0.1)
    assert e.value.status == bs.ERR_UNSUPPORTED
    p.close()
