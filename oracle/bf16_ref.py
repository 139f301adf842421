"""bfloat16 conversions written out from the format's definition (oracle, test
infrastructure only).

bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
bits and 7 stored mantissa bits, i.e. 8 significant bits for normal numbers and
a subnormal quantum of 2**-133. Rounding is round-to-nearest, ties-to-even.

The rounding here starts from a float64 value and rounds it ONCE to bfloat16
(the exact value of a rotated key or of an output, computed in float64, is
rounded straight to bf16; no intermediate float32 rounding).
"""

import numpy as np

_BF16_MAX_EXP = 128          # |x| >= 2**128 after rounding overflows to inf


def bf16_bits_to_f64(bits):
    """bf16 bit patterns (uint16 / int16 array) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x):
    """Round float64 values to the nearest bf16 value (ties to even).

    Returns float64 arrays holding bf16-representable values (inf on
    overflow, NaN propagated).
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)                       # x = m * 2**e, 0.5 <= |m| < 1
        q_exp = np.maximum(e - 8, -133)          # 8 significant bits, subnormal floor
        scaled = np.ldexp(x, -q_exp)
        r = np.round(scaled)                     # numpy rounds half to even
        out = np.ldexp(r, q_exp)
        out = np.where(np.abs(out) >= 2.0 ** _BF16_MAX_EXP,
                       np.copysign(np.inf, x), out)
        out = np.where(np.isnan(x), np.nan, out)
        out = np.where(np.isinf(x), x, out)
    return out


def f64_to_bf16_bits(x):
    """float64 values -> bf16 bit patterns (uint16), round-to-nearest-even."""
    r = round_to_bf16(x).astype(np.float32)      # exact: r is bf16-representable
    bits = (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(r)
    if np.any(nan):
        bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits
