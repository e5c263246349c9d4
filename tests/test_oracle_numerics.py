"""Pins of the oracle's number formats: bf16 rounding and the int4 code."""

import numpy as np
import pytest
import torch

import oracle
from golden_io import lines, table


def test_bf16_round_hand_values():
    for a, b in lines("bf16_round.txt"):
        got = oracle.bf16_round(np.array([float(a)]))[0]
        assert got == float(b), (a, got, b)
    assert np.signbit(oracle.bf16_round(np.array([-0.0]))[0])


def test_bf16_round_matches_library_on_fp32_inputs():
    # For inputs exactly representable in fp32, rounding fp64 -> bf16 is the
    # library's fp32 -> bf16 round-to-nearest-even (no double rounding).
    g = torch.Generator().manual_seed(1)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 8)
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(x.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)


def test_bf16_round_overflow_and_subnormal():
    big = (2.0 - 2.0 ** -8) * 2.0 ** 127          # halfway above bf16 max
    assert np.isinf(oracle.bf16_round(np.array([big * 1.0000001]))[0])
    tiny = 3 * 2.0 ** -134                          # 1.5 subnormal ulps -> 2 ulps
    assert oracle.bf16_round(np.array([tiny]))[0] == 2 * 2.0 ** -133


def test_bf16_bits_roundtrip():
    vals = np.array([1.0, -2.5, 3.140625, 0.0, 65536.0])
    np.testing.assert_array_equal(oracle.from_bf16_bits(oracle.bf16_bits(vals)), vals)
    assert oracle.bf16_bits(np.array([1.0]))[0] == 0x3F80


def test_int4_dequant_hand_values():
    for byte, scale, lo, hi in lines("int4_dequant.txt"):
        packed = np.array([[int(byte, 16)]], dtype=np.uint8)
        scales = np.array([[float(scale)]], dtype=np.float16)
        w = oracle.dequant_w4(packed, scales, K=2, g=2)
        assert w[0, 0] == float(lo) and w[0, 1] == float(hi), (byte, w)


def test_int4_dequant_exhaustive_codes():
    # Every code 0..15 in both nibble positions, several scales, against a
    # table written out independently of the oracle's unpacking.
    codes = np.arange(16)
    expected_q = [-8, -7, -6, -5, -4, -3, -2, -1, 0, 1, 2, 3, 4, 5, 6, 7]
    for scale in (1.0, 0.0078125, 0.5, 3.0, 0.000244140625):
        for lo in codes:
            for hi in codes:
                packed = np.array([[lo | (hi << 4)]], dtype=np.uint8)
                w = oracle.dequant_w4(packed, np.array([[scale]], np.float16), K=2, g=2)
                assert w[0, 0] == expected_q[lo] * scale
                assert w[0, 1] == expected_q[hi] * scale


def test_int4_group_scale_indexing():
    # Group g of row n uses scales[n, k // g]: rows and groups carry distinct
    # scales, all codes are +1 (u = 9), so each weight equals its scale.
    N, K, g = 3, 8, 4
    packed = np.full((N, K // 2), 0x99, dtype=np.uint8)
    scales = np.array([[1, 2], [4, 8], [16, 32]], dtype=np.float16)
    w = oracle.dequant_w4(packed, scales, K, g)
    expect = np.array([[1] * 4 + [2] * 4, [4] * 4 + [8] * 4, [16] * 4 + [32] * 4], float)
    np.testing.assert_array_equal(w, expect)


def test_quantize_hand_values():
    t = table("int4_quantize.txt")
    w = np.array([[float(v) for v in t["weights"]]], dtype=np.float32)
    packed, scales = oracle.quantize_w4(w, int(t["group"][0]))
    assert scales.view(np.uint16)[0, 0] == int(t["scale_bits"][0], 16)
    assert list(packed[0]) == [int(b, 16) for b in t["bytes"]]


def test_quantize_dequant_roundtrip():
    # Codes in [-7, 7] with a +-7 in every group and an fp16 scale s: the group
    # absmax is 7s, so re-encoding recovers exactly the same codes and scales.
    rng = np.random.default_rng(3)
    N, K, g = 16, 128, 32
    q = rng.integers(-7, 8, size=(N, K))
    q[:, ::g] = rng.choice([-7, 7], size=(N, K // g))
    scales = rng.uniform(1e-3, 1.0, size=(N, K // g)).astype(np.float16)
    packed = oracle.pack_int4((q + 8).astype(np.uint8))
    w = oracle.dequant_w4(packed, scales, K, g).astype(np.float32)
    p2, s2 = oracle.quantize_w4(w, g)
    np.testing.assert_array_equal(s2, scales)
    np.testing.assert_array_equal(p2, packed)


def test_quantize_error_bound_and_zero_group():
    rng = np.random.default_rng(4)
    N, K, g = 32, 256, 64
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[3, 64:128] = 0.0
    packed, scales = oracle.quantize_w4(w, g)
    deq = oracle.dequant_w4(packed, scales, K, g)
    s = np.repeat(scales.astype(np.float64), g, axis=1)
    # |w - deq| <= s/2 unless the fp16 scale rounded down far enough that the
    # absmax element clamps at 7 (then the error is below s/2 + 7s*2^-11).
    assert np.all(np.abs(w - deq) <= s * (0.5 + 7 * 2.0 ** -11) + 1e-12)
    assert scales[3, 1] == 0 and np.all(deq[3, 64:128] == 0)
    u = oracle.unpack_int4(packed, K)
    assert u.min() >= 1   # symmetric code never uses -8 on its own data


def test_pack_unpack_inverse():
    rng = np.random.default_rng(5)
    u = rng.integers(0, 16, size=(7, 40)).astype(np.uint8)
    np.testing.assert_array_equal(oracle.unpack_int4(oracle.pack_int4(u), 40), u)
