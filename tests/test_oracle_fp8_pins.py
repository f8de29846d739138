"""Pins of the FP8 (e4m3) oracle (CPU): the decode against the format's own
table values and against torch's float8_e4m3fn (a library routine), the
input encoder's round trip, attention on decoded inputs against torch
float64 SDPA, linearity in the V scale, and planted mistakes."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import fp8


def test_decode_table_values():
    """Values the format definition fixes: zero, the smallest subnormal
    (2^-9), the smallest normal (2^-6), one, the largest finite (448), signs,
    and the NaN codes."""
    got = fp8.decode_e4m3(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x7E, 0xFE, 0xB8],
                                   np.uint8))
    assert list(got) == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.5, 448.0, -448.0, -1.0]
    assert np.isnan(fp8.decode_e4m3(np.array([0x7F, 0xFF], np.uint8))).all()


def test_decode_every_code_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.decode_e4m3(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_encoder_round_trip_and_rounding():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], np.uint8)
    vals = fp8.decode_e4m3(codes)
    assert np.array_equal(workloads.e4m3_bits(vals), codes)
    # ties go to the even code: 1 + 1/16 lies between 1 (0x38) and 1.125 (0x39)
    assert workloads.e4m3_bits(np.array([1.0625, 1.1875]))[0] == 0x38
    assert workloads.e4m3_bits(np.array([1.1875]))[0] == 0x3A   # between 0x39 and 0x3A -> even
    assert workloads.e4m3_bits(np.array([1e4, -1e4])).tolist() == [0x7E, 0xFE]  # saturates


def _case(seed, B=1, H=2, S=256, D=16, mult=1.0):
    q8, k8, v8 = (workloads.normal_e4m3(seed, s, (B, H, S, D), mult) for s in (1, 2, 3))
    return q8, k8, v8


def test_dense_attention_equals_torch_sdpa_on_decoded_inputs():
    q8, k8, v8 = _case(5, mult=2.0)
    B, H, S, D = q8.shape
    mask = np.ones((B, H, S // 128, S // 128), np.uint8)
    O, L = fp8.attention_fp8(q8, k8, v8, mask, 0.25, causal=True)
    q, k, v = (torch.from_numpy(fp8.decode_e4m3(x)) for x in (q8, k8, v8))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.25)
    assert np.allclose(O, ref.numpy(), rtol=1e-12, atol=1e-12)
    s = 0.25 * (q @ k.transpose(-1, -2))
    s = s.masked_fill(torch.triu(torch.ones(S, S, dtype=torch.bool), 1), float("-inf"))
    assert np.allclose(L, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)


def test_v_scale_is_linear():
    q8, k8, v8 = _case(6)
    mask = np.array([[[[1, 0], [1, 1]], [[0, 1], [1, 0]]]], np.uint8)
    O1, L1 = fp8.attention_fp8(q8, k8, v8, mask, 0.3)
    O2, L2 = fp8.attention_fp8(q8, k8, v8, mask, 0.3, v_scale=0.125)
    assert np.array_equal(L1, L2)
    assert np.allclose(O2, 0.125 * O1, rtol=0, atol=1e-15)


@pytest.mark.parametrize("m", sorted(fp8.FP8_MUTATIONS))
def test_planted_mistakes_are_caught(m):
    fp8.set_fp8_mutation(m)
    try:
        failed = 0
        for t in (test_decode_table_values, test_decode_every_code_against_torch,
                  test_dense_attention_equals_torch_sdpa_on_decoded_inputs, test_v_scale_is_linear):
            try:
                t()
            except AssertionError:
                failed += 1
        assert failed > 0, fp8.FP8_MUTATIONS[m]
    finally:
        fp8.set_fp8_mutation(0)
