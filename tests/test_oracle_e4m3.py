"""Pins for the oracle's e4m3 codec (CPU).

The codec follows "Smaller, faster, safer: running Kimi and GLM at scale",
section "Quantizing the KV cache" (cache stored as FP8 e4m3). What pins it,
independently of the oracle's own code:

* closed-form code values of the format (max 448, smallest normal 2^-6,
  smallest subnormal 2^-9, NaN codes);
* torch's float8_e4m3fn -> float32 conversion (a library routine) on all 256
  codes;
* brute force: for every bfloat16 input and several awkward scales, the exact
  nearest finite e4m3 value to the real quotient x/s, compared with rational
  arithmetic, ties to the even code;
* torch's float32 -> float8_e4m3fn cast where x/s is exact in float32 and in
  range.
"""

import bisect
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import e4m3


def test_closed_form_codes():
    assert e4m3.code_value(0x7E) == 448.0
    assert e4m3.code_value(0xFE) == -448.0
    assert e4m3.code_value(0x08) == 2.0 ** -6
    assert e4m3.code_value(0x07) == 7 * 2.0 ** -9
    assert e4m3.code_value(0x01) == 2.0 ** -9
    assert e4m3.code_value(0x38) == 1.0
    assert e4m3.code_value(0x00) == 0.0
    v = e4m3.code_value(0x80)
    assert v == 0.0 and np.signbit(v)
    assert np.isnan(e4m3.code_value(0x7F)) and np.isnan(e4m3.code_value(0xFF))
    finite = [c for c in range(256) if not np.isnan(e4m3.code_value(c))]
    assert len(finite) == 254


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    ours = e4m3.decode(np.arange(256, dtype=np.uint8))
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    assert np.array_equal(ref[~both_nan], ours[~both_nan])


def _all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = e4m3.bf16_bits_to_f64(bits)
    keep = np.isfinite(vals)
    return bits[keep], vals[keep]


_POS_VALUES = sorted({Fraction(e4m3.code_value(c)) for c in range(0x7F)})
_POS_CODE = {Fraction(e4m3.code_value(c)): c for c in range(0x7F)}


def _brute_force_code(x: float, s: float) -> int:
    """Nearest finite e4m3 value to the exact quotient x/s; ties to even code."""
    q = Fraction(x) / Fraction(s)
    neg = q < 0 or (q == 0 and np.signbit(x))
    a = abs(q)
    i = bisect.bisect_left(_POS_VALUES, a)
    cands = [_POS_VALUES[k] for k in (i - 1, i) if 0 <= k < len(_POS_VALUES)]
    best = min(abs(a - c) for c in cands)
    tied = [c for c in cands if abs(a - c) == best]
    if len(tied) == 2:
        tied = [c for c in tied if _POS_CODE[c] % 2 == 0]
    code = _POS_CODE[tied[0]]
    return code | (0x80 if neg else 0)


@pytest.mark.parametrize("scale", [1.0, float(np.float32(4.0 / 448.0)),
                                   float(np.float32(0.0123456)), float(np.float32(3.0e-5))])
def test_encode_all_bf16_inputs_brute_force(scale):
    bits, vals = _all_bf16_values()
    # every 3rd bf16 input keeps the suite quick while covering every binade
    sel = slice(0, None, 3) if scale != 1.0 else slice(None)
    vals = vals[sel]
    ours = e4m3.encode(vals, scale)
    ref = np.array([_brute_force_code(float(v), scale) for v in vals], dtype=np.uint8)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(vals[i], scale, hex(ours[i]), hex(ref[i])) for i in bad[:5]]


def test_encode_exact_midpoints_go_to_even():
    # midpoints between neighbouring codes, built as exact rationals
    for c in range(0x00, 0x7E):
        lo, hi = Fraction(e4m3.code_value(c)), Fraction(e4m3.code_value(c + 1))
        mid = (lo + hi) / 2
        got = int(e4m3.encode(np.array([float(mid)]), 1.0)[0])
        assert got == (c if c % 2 == 0 else c + 1)
        # just above / below the midpoint
        assert int(e4m3.encode(np.array([np.nextafter(float(mid), np.inf)]), 1.0)[0]) == c + 1
        assert int(e4m3.encode(np.array([np.nextafter(float(mid), -np.inf)]), 1.0)[0]) == c


def test_round_trip_and_monotone():
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    for s in (1.0, 0.5, 2.0 ** -7):
        vals = e4m3.decode(finite) * s
        assert np.array_equal(e4m3.encode(vals, s), finite)
    xs = np.linspace(-500, 500, 20001)
    dec = e4m3.decode(e4m3.encode(xs, 1.0))
    assert np.all(np.diff(dec) >= 0)


def test_saturation_and_specials():
    codes = e4m3.encode(np.array([448.0, 464.0, 479.0, 480.0, 1e30, -1e30, -500.0]), 1.0)
    assert list(codes) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    codes = e4m3.encode(np.array([np.nan, -np.nan, 0.0, -0.0, -1e-30, 2.0 ** -10]), 1.0)
    assert codes[0] in (0x7F, 0xFF) and codes[1] in (0x7F, 0xFF)
    assert list(codes[2:]) == [0x00, 0x80, 0x80, 0x00]   # 2^-10 ties to 0 (even)


def test_encode_matches_torch_cast_in_range():
    bits, vals = _all_bf16_values()
    for s in (1.0, 0.25, 8.0):
        q = vals / s                      # exact: power-of-two scale
        keep = np.abs(q) <= 448.0
        ref = torch.from_numpy(q[keep].astype(np.float32)).to(torch.float8_e4m3fn)
        ref = ref.view(torch.uint8).numpy()
        ours = e4m3.encode(vals[keep], s)
        assert np.array_equal(ours, ref)
