"""bfloat16 <-> float64 conversions written from the format's definition.

TEST INFRASTRUCTURE (see the package docstring). The kernel stores bf16 with
round-to-nearest-even ([W] "Caveats worth knowing": the kernel is bf16 only).

bfloat16 is the upper 16 bits of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits (bias 127), 7 fraction bits. Normal numbers are (-1)^s * 2^(e-127) *
(1 + f/128); e == 0 encodes zero and subnormals (-1)^s * 2^-126 * f/128;
e == 255 encodes infinities and NaN.
"""

import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
BF16_MIN_NORMAL_EXP = -126
BF16_FRAC_BITS = 7


def decode(bits):
    """uint16 bf16 bit patterns -> float64 values, from the fields."""
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    exp = (b >> 7) & 0xFF
    frac = (b & 0x7F).astype(np.float64)
    with np.errstate(over="ignore"):
        normal = sign * np.ldexp(1.0 + frac / 128.0, (exp - 127).astype(np.int32))
    sub = sign * np.ldexp(frac / 128.0, -126)
    special = np.where(frac == 0, sign * np.inf, np.nan)
    out = np.where(exp == 0, sub, np.where(exp == 255, special, normal))
    return out.astype(np.float64)


def ulp(x):
    """Spacing of bf16 numbers at |x| (x in float64): 2^(max(floor(log2|x|), -126) - 7).

    For x == 0 this is the subnormal spacing 2^-133.
    """
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(x)  # x = m * 2^e with 0.5 <= m < 1, so floor(log2 x) = e - 1
    e = np.where(x == 0, BF16_MIN_NORMAL_EXP + 1, e)
    return np.ldexp(1.0, (np.maximum(e - 1, BF16_MIN_NORMAL_EXP) - BF16_FRAC_BITS).astype(np.int32))


def round_rne(x):
    """Round float64 values to the nearest bf16 value, ties to even, once.

    The scaled value x / ulp(x) is exact (a power-of-two scaling); np.rint
    rounds half to even, which at the integer grid of the significand is the
    IEEE tie rule. Results above the largest finite bf16 become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    u = ulp(x)
    with np.errstate(over="ignore", invalid="ignore"):
        v = np.rint(x / u) * u
        v = np.where(np.abs(v) > BF16_MAX, np.copysign(np.inf, x), v)
    return np.where(np.isnan(x), np.nan, v)


def encode_rne(x):
    """float64 (or float32) values -> uint16 bf16 bits, round to nearest even.

    After round_rne the value is exactly representable in bf16, hence in
    binary32; its binary32 encoding's upper half is the bf16 encoding.
    """
    v = round_rne(np.asarray(x, dtype=np.float64)).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)
