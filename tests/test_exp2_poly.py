"""CPU checks of the forward kernel's exponential on the FMA pipes (the part
of the softmax's 2^x that does not use the MUFU unit): its constants are read
from the kernel source, the algorithm is restated here in float32 numpy and
compared with the exact 2^x, and the coefficients are re-derived by the same
published method (least maximum relative error on [-1/2, 1/2], Lawson's
iteration) to show they are that fit."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "block_sparse_flash_attn_gb300", "csrc", "fwd_sm103.cu")


def _constants():
    text = open(SRC).read()
    c = [float(re.search(rf"kExp2C{i} = ([0-9.eE+-]+)f", text).group(1)) for i in range(4)]
    magic = float(re.search(r"kRoundMagic = ([0-9.]+)f", text).group(1))
    return np.array(c, dtype=np.float32), np.float32(magic)


def _fma32(a, b, c):
    """fp32 fused multiply-add: exact product and sum in float64, one rounding."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def _exp2_poly(x):
    """The kernel's algorithm, step by step, in float32."""
    c, magic = _constants()
    x = np.minimum(np.maximum(x.astype(np.float32), np.float32(-126.0)), np.float32(126.0))
    t = (x + magic).astype(np.float32)              # magic + round(x)
    nf = (t - magic).astype(np.float32)             # round(x)
    f = _fma32(nf, np.float32(-1.0), x)             # x - round(x)
    p = _fma32(np.full_like(f, c[3]), f, np.full_like(f, c[2]))
    p = _fma32(p, f, np.full_like(f, c[1]))
    p = _fma32(p, f, np.full_like(f, c[0]))
    bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_relative_error_over_the_normal_range():
    x = np.linspace(-125.0, 126.0, 2_000_001, dtype=np.float64).astype(np.float32)
    y = _exp2_poly(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    assert np.all(np.isfinite(y)) and rel.max() <= 1e-4, rel.max()


def test_clamped_ends_and_masked_scores():
    lo = _exp2_poly(np.array([-126.5, -200.0, -1e30, -np.inf], dtype=np.float32))
    assert np.all(lo >= 0) and np.all(lo <= 2.0 ** -125)
    hi = _exp2_poly(np.array([126.5, 200.0, 1e30, np.inf], dtype=np.float32))
    assert np.all(np.isfinite(hi)) and np.all(hi >= 2.0 ** 125)  # a block-sum test sees them


def test_integers_and_half_integers():
    x = np.arange(-120, 121, dtype=np.float32)
    assert np.allclose(_exp2_poly(x), np.exp2(x.astype(np.float64)), rtol=1e-4, atol=0)
    x = x + np.float32(0.5)
    assert np.allclose(_exp2_poly(x), np.exp2(x.astype(np.float64)), rtol=1e-4, atol=0)


def _lawson_fit(deg, iters=30):
    n = 4000
    x = np.cos(np.pi * (np.arange(n) + 0.5) / n) * 0.5
    A = np.vander(x, deg + 1, increasing=True) / np.exp2(x)[:, None]
    w = np.ones(n)
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], sw, rcond=None)
        e = np.abs(A @ c - 1.0)
        w = w * e
        w /= w.sum()
    return c


def test_coefficients_are_the_minimax_cubic():
    c_src, _ = _constants()
    c_fit = _lawson_fit(3)
    assert np.allclose(c_src, c_fit, rtol=1e-5, atol=1e-7), (c_src, c_fit)
    x = np.linspace(-0.5, 0.5, 200001)
    err = np.abs(np.polyval(c_src[::-1].astype(np.float64), x) / np.exp2(x) - 1).max()
    assert err <= 7.6e-5, err
