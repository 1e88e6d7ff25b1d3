"""Number formats used by the decode step, written from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

* BF16: IEEE-754 binary32 truncated to 8 significant bits (1 implicit + 7
  stored), same exponent range as binary32; rounding is round-to-nearest-even
  (the cache write and the q output of the fused prologue store BF16 values;
  page "vLLM and Tencent Hunyuan upstream two HPC backends for NVIDIA Hopper",
  section "Why does dynamic scheduling matter for attention?", last paragraph:
  the backend supports BF16 and FP8).
* FP8 E4M3 as defined by the OCP "OFP8 Formats for Deep Learning" v1.0: 1 sign,
  4 exponent (bias 7), 3 mantissa bits; no infinities; S.1111.111 is NaN; the
  largest finite magnitude is S.1111.110 = 448; subnormals 2^-6 * m/8.  The
  encoder rounds to nearest, ties to even, and saturates to +-448 (page "[vllm]
  Introducing the HPC-Ops attention backend", introduction: the backend targets
  FP8 (E4M3) models).

Everything here works on float64 NumPy arrays, elementwise, with no blocking.
"""

import numpy as np

# ---------------------------------------------------------------- BF16 -----

_BF16_MANT_BITS = 8            # significant bits including the implicit one
_BF16_MIN_EXP = -126           # smallest normal exponent (as binary32)
_BF16_SUBNORMAL_ULP = 2.0 ** (_BF16_MIN_EXP - (_BF16_MANT_BITS - 1))  # 2^-133


def bf16_round(x):
    """Round float64 values to the nearest BF16 value, ties to even.

    For finite nonzero x with |x| in [2^(E-1), 2^E) the BF16 spacing is
    2^(E-8); below the normal range the spacing is fixed at 2^-133.  x / ulp is
    exact in float64 (division by a power of two), ``np.rint`` rounds half to
    even, and values that round past the largest finite BF16 become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    _, e = np.frexp(xf)                      # |xf| = m * 2^e, m in [0.5, 1)
    ulp = np.ldexp(1.0, e - _BF16_MANT_BITS)
    ulp = np.maximum(ulp, _BF16_SUBNORMAL_ULP)
    r = np.rint(xf / ulp) * ulp
    max_finite = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > max_finite, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def bf16_bits(x):
    """BF16 bit patterns (uint16) of float64 values that are already BF16."""
    x = np.asarray(x, dtype=np.float64)
    f32 = x.astype(np.float32)               # exact: BF16 is a subset of binary32
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(bits):
    """float64 values of BF16 bit patterns (uint16)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):          # NaN payloads pass through
        return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- E4M3 -----

E4M3_MAX = 448.0
_E4M3_BIAS = 7
_E4M3_MIN_NORMAL_EXP = 1 - _E4M3_BIAS      # -6
_E4M3_SUBNORMAL_STEP = 2.0 ** (_E4M3_MIN_NORMAL_EXP - 3)   # 2^-9


def _e4m3_value(c):
    """float64 value of each E4M3 code in the int64 array c, from the fields:
    sign S, exponent E (bias 7) and mantissa M; E = 0 is subnormal
    (M/8 * 2^-6), otherwise (1 + M/8) * 2^(E-7); S.1111.111 is NaN."""
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = np.ldexp(1.0 + m / 8.0, e - _E4M3_BIAS)
    sub = np.ldexp(m / 8.0, _E4M3_MIN_NORMAL_EXP)
    val = sign * np.where(e == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


# the value of every one of the 256 codes, each formed once by _e4m3_value
_E4M3_VALUES = _e4m3_value(np.arange(256, dtype=np.int64))


def e4m3_decode(codes):
    """float64 values of E4M3 codes (uint8); S.1111.111 decodes to NaN.
    Each code's value is the field formula of ``_e4m3_value``, looked up."""
    return _E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x):
    """E4M3 codes (uint8) of float64 values: round to nearest even, saturate.

    |x| >= 448 encodes as 448 (S.1111.110); NaN encodes as S.1111.111.  Below
    2^-6 the grid is uniform with step 2^-9 (subnormals); above, a binade
    [2^E, 2^(E+1)) has 8 values with step 2^(E-3).  A value that rounds up to
    the next binade becomes that binade's first code.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    code = np.zeros(a.shape, dtype=np.int64)

    sub = a < 2.0 ** _E4M3_MIN_NORMAL_EXP
    # subnormal range: q in 0..8; q == 8 is the smallest normal, code 0x08
    code[sub] = np.rint(a[sub] / _E4M3_SUBNORMAL_STEP).astype(np.int64)

    nrm = ~sub
    an = a[nrm]
    _, e2 = np.frexp(an)                     # an = m * 2^e2, m in [0.5, 1)
    E = e2 - 1                               # an in [2^E, 2^(E+1))
    q = np.rint(an / np.ldexp(1.0, E - 3)).astype(np.int64)   # in 8..16
    up = q == 16
    E = np.where(up, E + 1, E)
    q = np.where(up, 8, q)
    code[nrm] = ((E + _E4M3_BIAS) << 3) | (q - 8)

    code = np.minimum(code, 0x7E)            # saturation guard (448)
    code = np.where(nan, 0x7F, code) | sign
    return code.astype(np.uint8)


def e4m3_step(value):
    """Spacing of the E4M3 grid at |value| (float64), for 1-code tolerances."""
    a = np.abs(np.asarray(value, dtype=np.float64))
    _, e2 = np.frexp(np.maximum(a, 2.0 ** _E4M3_MIN_NORMAL_EXP))
    return np.ldexp(1.0, (e2 - 1) - 3)
