"""Number formats of the W4A16 path: bf16 activations, packed int4 weights.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[Batched serving, §1 Contribution and §3 Results] keeps every linear weight
as packed 4-bit codes and computes with 16-bit activations (W4A16).
[KV-slot isolation, follow-up update] has the batched and single-stream
dense projections dequantize the same way, so dequantization is a fixed
function of the stored codes and scales.  The pages print neither the
code nor the packing, so these readings are taken:

* int4 code: symmetric per-group quantization.  For a group of g consecutive
  input features of one output row, s = fp16(absmax / 7) with the division in
  fp32, q = clamp(rint_half_even(w / fp32(s)), -8, 7), stored offset-binary
  u = q + 8.  An all-zero group has s = 0 and q = 0.  Dequantized value
  w = (u - 8) * s, which is exact in fp32 and fp64.
* packing: row-major [N][K/2] bytes along K; element 2j sits in the low
  nibble of byte j, element 2j+1 in the high nibble.  Scales are fp16 [N][K/g].
* bf16: round to nearest, ties to even, from the exact (fp64) value.
"""

import numpy as np

_BF16_MIN_NORMAL = 2.0 ** -126
_BF16_SUBNORMAL_ULP = 2.0 ** -133


def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value (ties to even).

    Returns float64 arrays whose values are exactly representable in bf16.
    bf16 has fp32's exponent range and 8 significant bits, so a normal fp64
    value keeps the top 7 of its 52 stored mantissa bits; the 45 dropped bits
    decide the rounding.  Values below bf16's smallest normal are rounded to a
    multiple of its smallest subnormal.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    tiny = finite & (np.abs(x) < _BF16_MIN_NORMAL)
    normal = finite & ~tiny
    bits = x[normal].view(np.uint64)
    drop = np.uint64(45)
    keep_lsb = (bits >> drop) & np.uint64(1)
    bits = bits + (np.uint64((1 << 44) - 1) + keep_lsb)
    bits = bits & ~np.uint64((1 << 45) - 1)
    r = bits.view(np.float64)
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, r), r)
    out[normal] = r
    out[tiny] = np.round(x[tiny] / _BF16_SUBNORMAL_ULP) * _BF16_SUBNORMAL_ULP
    out[~finite] = x[~finite]
    return out


def bf16_bits(x):
    """uint16 bit patterns of values that are already bf16-representable."""
    r = bf16_round(x)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def from_bf16_bits(b):
    """float64 values of uint16 bf16 bit patterns."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def unpack_int4(packed, K):
    """Offset-binary codes u in [0, 15], shape [N][K], from [N][K/2] bytes."""
    packed = np.asarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    u = np.empty((N, K), dtype=np.uint8)
    u[:, 0::2] = packed & 0x0F
    u[:, 1::2] = packed >> 4
    return u


def pack_int4(u):
    """Inverse of ``unpack_int4``: [N][K] codes in [0, 15] -> [N][K/2] bytes."""
    u = np.asarray(u, dtype=np.uint8)
    assert u.shape[1] % 2 == 0 and int(u.max(initial=0)) <= 15
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def dequant_w4(packed, scales, K, g):
    """Dequantized weights (float64 [N][K]): w[n, k] = (u - 8) * s[n, k // g]."""
    u = unpack_int4(packed, K).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    N = u.shape[0]
    assert s.shape == (N, K // g)
    return ((u - 8.0).reshape(N, K // g, g) * s[:, :, None]).reshape(N, K)


def quantize_w4(w, g):
    """Symmetric per-group int4 quantization of fp32 weights [N][K].

    Returns (packed uint8 [N][K/2], scales float16 [N][K/g]).  Every decision
    (scale, rounding of each code) is taken in fp32, the precision of the
    stored weights, so a GPU encoder doing the same fp32 operations produces
    identical bytes.
    """
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % g == 0 and g % 2 == 0
    wg = w.reshape(N, K // g, g)
    absmax = np.abs(wg).max(axis=2)
    s16 = (absmax / np.float32(7.0)).astype(np.float32).astype(np.float16)
    sf = s16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (wg / sf[:, :, None]).astype(np.float32)
    ratio = np.where(sf[:, :, None] > 0, ratio, np.float32(0.0))
    ratio = np.where(np.isfinite(ratio), ratio, np.float32(0.0))
    q = np.clip(np.rint(ratio), -8, 7).astype(np.int16)
    u = (q + 8).astype(np.uint8).reshape(N, K)
    return pack_int4(u), s16
