"""ORACLE -- test infrastructure, not product code.

Block-sparse attention on FP8 (e4m3) inputs, in fp64: the inputs are decoded
exactly to their real values and the fp64 definition of ``oracle.attention``
is applied to them; O is then multiplied by the caller's V scale.  Only the
tests and the bench's reference leg may use this module; it shares nothing
with the CUDA path.

"JAX Pallas and Blackwell" (section "What the Tutorial Covers") names FP8
operands with fp32 accumulation as a precision the Blackwell tensor cores
take.  The pages do not fix an FP8 format; the one taken is e4m3 as the OCP
8-bit floating-point specification ("OFP8 Formats for Deep Learning",
Micikevicius et al., 2022) defines it, the format GB300's tensor cores read:

    bits  s eeee mmm   (sign, 4 exponent bits with bias 7, 3 mantissa bits)
    e = 0            value = (-1)^s * (m / 8) * 2^-6            (subnormal)
    0 < e < 15       value = (-1)^s * (1 + m / 8) * 2^(e - 7)
    e = 15, m < 7    value = (-1)^s * (1 + m / 8) * 2^8         (up to 448)
    e = 15, m = 7    NaN   (no infinities)

FP8 tensors carry scales in practice: the value a caller means is
scale_t * value(bits).  Here the scales of Q and K are folded into the
softmax scale by the caller (scale * q_scale * k_scale), and V's scale
multiplies O (attention is linear in V).

Pinned by tests/test_oracle_fp8_pins.py (format table values, every code
against torch's float8_e4m3fn, the round trip of the input encoder, torch
float64 SDPA on decoded inputs, linearity in the V scale).
"""
from __future__ import annotations

import numpy as np

_mutation = 0
FP8_MUTATIONS = {1: "exponent bias 8 instead of 7", 2: "subnormals decoded as normals",
                 3: "V scale not applied"}


def set_fp8_mutation(m: int) -> None:
    """Plant mistake number m (0 = none).  Tests only."""
    global _mutation
    _mutation = int(m)


def decode_e4m3(bits) -> np.ndarray:
    """e4m3 bit patterns (uint8) -> float64, exactly, per the format above."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    bias = 8 if _mutation == 1 else 7
    normal = s * (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - bias)
    sub = s * (m / 8.0) * 2.0 ** (1 - bias)
    val = normal if _mutation == 2 else np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((b & 7) == 7), np.nan, val)


def attention_fp8(q8, k8, v8, mask, scale: float, causal: bool = False, rows=None,
                  v_scale: float = 1.0):
    """Exact block-sparse attention (oracle.attention, fp64) on e4m3 inputs
    q8, k8, v8 (uint8 bit patterns [B][H][S][D]), O multiplied by v_scale.
    Returns (O, LSE) shaped as oracle.attention returns them."""
    from . import attention
    q, k, v = (np.ascontiguousarray(decode_e4m3(x)) for x in (q8, k8, v8))
    O, L = attention(q, k, v, mask, scale, causal, rows=rows)
    if _mutation != 3:
        O = O * float(v_scale)
    return O, L
