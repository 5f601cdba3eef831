"""FP8 E4M3 codec for the latent KV cache (oracle; test infrastructure only).

[CF] "Smaller, faster, safer: running Kimi and GLM at scale", section
"Quantizing the KV cache": the KV cache is kept in 8-bit floating point of the
e4m3 kind instead of BF16, which halves its size; the attention kernel converts
the stored values back as it reads them.

The page names the format only as "FP8, e4m3". We read it as the OCP E4M3
variant that GPUs implement (often written ``e4m3fn``):

* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
* exponent field 0 encodes subnormals ``(-1)^s * m/8 * 2^-6`` (step 2^-9);
* there is no infinity; the largest finite magnitude is ``1.75 * 2^8 = 448``
  (code 0x7E); codes 0x7F and 0xFF are NaN.

Encoding (the write side is not described on the page; the readings are ours):

* the value stored for a real ``x`` under a per-tensor scale ``s`` is
  ``x / s`` rounded to the nearest e4m3 value, ties to the even code;
* magnitudes above 448 saturate to +-448 (no overflow to NaN);
* the rounding is of the exact real quotient ``x / s``. Here the quotient is
  formed in float64: for ``x`` a bfloat16 (8 significant bits) and ``s`` a
  float32 (24 bits), a float64 quotient can only land exactly on an e4m3
  rounding midpoint when the real quotient is that midpoint (the gap from a
  29-bit product to an 8-bit numerator cannot be below 2^-53 relative unless
  it is zero), so rounding the float64 quotient equals rounding the real one;
* NaN input gives a NaN code (0x7F, or 0xFF for negative sign); -0 keeps its
  sign bit.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9


def code_value(code: int) -> float:
    """Value of one e4m3 code, written straight from the format definition."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** -6
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


# 256-entry decode table built from the definition above.
DECODE_TABLE = np.array([code_value(c) for c in range(256)], dtype=np.float64)


def decode(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) -> float64 values, by table lookup."""
    codes = np.asarray(codes, dtype=np.uint8)
    return DECODE_TABLE[codes]


def _magnitude_code(v: np.ndarray) -> np.ndarray:
    """Code (without sign) of non-negative values that are exact e4m3 values."""
    out = np.zeros(v.shape, dtype=np.uint8)
    sub = v < E4M3_MIN_NORMAL
    out[sub] = np.rint(v[sub] / E4M3_SUBNORMAL_STEP).astype(np.uint8)
    nrm = ~sub
    if np.any(nrm):
        mant, exp = np.frexp(v[nrm])          # v = mant * 2^exp, mant in [0.5, 1)
        e = exp - 1                            # v = (2*mant) * 2^e, 2*mant in [1, 2)
        m = np.rint((2.0 * mant - 1.0) * 8.0)  # exact: v sits on the grid
        out[nrm] = (((e + 7) << 3) + m).astype(np.uint8)
    return out


def round_to_e4m3(q: np.ndarray) -> np.ndarray:
    """Round float64 values to the e4m3 grid: nearest, ties to even, saturate.

    Returns float64 values that are exactly representable in e4m3 (NaN stays
    NaN). The grid spacing in the binade [2^e, 2^(e+1)) is 2^(e-3) for
    e >= -6 and 2^-9 below 2^-6 (subnormals).
    """
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    out = np.empty_like(a)
    nan = np.isnan(a)
    sat = (~nan) & (a > E4M3_MAX)
    small = (~nan) & (~sat) & (a < E4M3_MIN_NORMAL)
    norm = (~nan) & (~sat) & (~small)
    out[nan] = np.nan
    out[sat] = E4M3_MAX
    # Subnormal range: multiples of 2^-9; np.rint rounds half to even.
    out[small] = np.rint(a[small] / E4M3_SUBNORMAL_STEP) * E4M3_SUBNORMAL_STEP
    if np.any(norm):
        _, exp = np.frexp(a[norm])
        quantum = np.ldexp(1.0, exp - 1 - 3)   # 2^(e-3) with e = floor(log2 a)
        out[norm] = np.rint(a[norm] / quantum) * quantum
    # Rounding up from just below 448 cannot exceed 448 (448 is on the grid),
    # so no second saturation is needed.
    return np.copysign(out, q)


def encode(x: np.ndarray, kv_scale: float) -> np.ndarray:
    """Quantise real values to e4m3 codes: code = e4m3_rne_sat(x / kv_scale).

    ``x`` holds exact values (e.g. bfloat16 inputs widened to float64);
    ``kv_scale`` is the per-tensor float32 scale. Returns uint8 codes.
    """
    x = np.asarray(x, dtype=np.float64)
    q = x / np.float64(np.float32(kv_scale))
    r = round_to_e4m3(q)
    nan = np.isnan(r)
    mag = np.where(nan, 0.0, np.abs(r))
    codes = _magnitude_code(mag)
    codes[nan] = 0x7F
    sign = np.signbit(r)
    codes = codes | np.where(sign, 0x80, 0).astype(np.uint8)
    return codes.astype(np.uint8)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):     # NaN patterns widen to NaN
        return b.view(np.float32).astype(np.float64)
