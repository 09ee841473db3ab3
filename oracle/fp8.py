"""Number formats used by the oracle: FP8 e4m3 (OCP "E4M3FN") and bfloat16.

TEST INFRASTRUCTURE ONLY: this package is the slow reference that the CUDA
path is checked against. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it; the product path never does.

PTPC quantisation ("Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD
MI300X Series", section 2.1.1 and Figure 3) stores activations and weights as
FP8. The pages name FP8 but not the bit layout; the layer uses e4m3 as the
OCP 8-bit floating point specification defines it:

* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
* exponent field 0 holds subnormals m * 2**-9 (m = 0..7);
* exponent field 15 with mantissa 7 is NaN; there is no infinity;
* the largest finite magnitude is 1.75 * 2**8 = 448.

Encoding rounds to nearest, ties to even, and saturates: every finite input
whose magnitude rounds above 448 (and +-inf) becomes +-448.

Everything here is exact: inputs are fp32 values, which fp64 holds exactly, and
all steps are scalings by powers of two and integer rounding.
"""

import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6       # smallest normal exponent of e4m3
_SUBNORMAL_QUANTUM = 2.0 ** -9


def _decode_formula(codes):
    """Value of each e4m3 code from its bit fields (fp64)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp_field = (c >> 3) & 0xF
    mant = (c & 0x7).astype(np.float64)
    normal = (1.0 + mant / 8.0) * np.ldexp(1.0, exp_field - 7)
    subnormal = mant * _SUBNORMAL_QUANTUM
    val = np.where(exp_field == 0, subnormal, normal)
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


_DECODE_TABLE = _decode_formula(np.arange(256))


def e4m3_decode(codes):
    """Map e4m3 byte codes to their values (fp64). NaN codes give NaN.

    A lookup in the 256-entry table of the bit-field formula above."""
    return _DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


_CHUNK = 1 << 16


def e4m3_encode(values):
    """Round fp32 values to e4m3 codes: nearest, ties to even, saturating.

    `values` is converted to fp32 first (the quantiser's inputs are fp32 on
    both sides of the parity check), then handled exactly in fp64, in chunks
    that stay in cache.
    """
    v32 = np.asarray(values, dtype=np.float32)
    flat = v32.reshape(-1)
    out = np.empty(flat.size, dtype=np.uint8)
    for i in range(0, flat.size, _CHUNK):
        out[i:i + _CHUNK] = _encode_chunk(flat[i:i + _CHUNK])
    return out.reshape(v32.shape)


def _encode_chunk(v32):
    v = v32.astype(np.float64)
    sign_bit = np.signbit(v).astype(np.uint8) << 7
    a = np.abs(v)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # Saturation: every magnitude at or beyond 448 (including inf) maps to
    # 448, the largest finite value.
    a = np.minimum(a, E4M3_MAX)

    # Exponent e with 2**e <= a < 2**(e+1); frexp is exact.
    _, ex = np.frexp(a)
    e = ex.astype(np.int64) - 1
    # Below the smallest normal the spacing is fixed at 2**-9.
    e = np.maximum(e, _MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, e - 3)          # spacing of e4m3 values at exponent e
    n = np.rint(a / quantum)                # round half to even, exact
    # n counts quanta: for a normal number n is in [8, 16]; n == 16 carries
    # into the next binade. For subnormals n is in [0, 8]; n == 8 is the
    # smallest normal, which the general formula below also produces.
    carry = n >= 16
    n = np.where(carry, n / 2, n)
    e = np.where(carry, e + 1, e)
    is_sub = n < 8                          # only possible when e == -6
    exp_field = np.where(is_sub, 0, e + 7)
    mant = np.where(is_sub, n, n - 8).astype(np.int64)
    code = (exp_field.astype(np.int64) << 3) | mant
    code = code.astype(np.uint8) | sign_bit
    code = np.where(nan, np.uint8(0x7F), code)
    return code.astype(np.uint8)


def bf16_round(values):
    """Round fp64 values to the nearest bfloat16 (ties to even).

    Returns fp32 numbers that hold the bf16 values exactly. bfloat16 has 8
    significant bits and the fp32 exponent range.
    """
    v = np.asarray(values, dtype=np.float64)
    _, ex = np.frexp(v)                       # v = f * 2**ex, 0.5 <= |f| < 1
    e = np.maximum(ex.astype(np.int64) - 1, -126)
    quantum = np.ldexp(1.0, e - 7)
    r = np.rint(v / quantum) * quantum
    return r.astype(np.float32)


def bf16_bits(values_fp32):
    """The 16-bit patterns of fp32 numbers that hold bf16 values exactly."""
    u = np.asarray(values_fp32, dtype=np.float32).view(np.uint32)
    return (u >> 16).astype(np.uint16)


def bf16_from_bits(bits):
    """fp32 numbers for 16-bit bfloat16 patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
