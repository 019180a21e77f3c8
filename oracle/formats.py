"""Number formats used by the oracle: OCP FP8 e4m3 (the "fn" variant), bfloat16, fp32 rounding.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this package; only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

Everything here is written from the format definitions, not from any GPU code:

* e4m3 ("fn", as used by the FP8 datapath of the ZYFA pages): 1 sign bit, 4 exponent bits with bias 7,
  3 mantissa bits.  Normal value ``2^(E-7) * (1 + M/8)``, subnormal (E = 0) value ``M * 2^-9``, the
  all-ones pattern S.1111.111 is NaN, there is no infinity, the largest finite magnitude is 448
  (code 0x7E).  The pages rely on one property of this encoding: read as an integer, the code of a
  positive normal number grows by 8 for every doubling (spbcomputers.ru ZYFA article, section
  "Три приёма", Lean P bullet; captivela ZYFA article, section "Tiga Trik").
* bfloat16: the upper 16 bits of an IEEE binary32, rounded to nearest, ties to even.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e4m3_decode_fields(codes) -> np.ndarray:
    """Decode e4m3 bit patterns (uint8) to float64 values, straight from the field definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = m * 2.0 ** -9
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


# All 256 patterns decoded once by the field definition; decoding is then a table lookup.
_E4M3_TABLE = _e4m3_decode_fields(np.arange(256, dtype=np.uint8))


def e4m3_decode(codes) -> np.ndarray:
    """Decode e4m3 bit patterns (uint8) to float64 values."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


# The 127 non-negative finite values, in code order 0x00..0x7E.  Codes are monotone in value, so
# this table is sorted; rounding below picks from it.
_E4M3_POS = e4m3_decode(np.arange(0, 127, dtype=np.uint8))


def e4m3_encode_rne_satfinite(x) -> np.ndarray:
    """Round float values to the nearest e4m3 code, ties to the even code, saturating to +-448.

    "Nearest" is taken over the finite e4m3 values by direct comparison of distances, so the
    rounding is exact for any float64 input.  NaN inputs map to the NaN code 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    a_sat = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, a_sat, side="left")          # first table value >= a
    hi = np.clip(hi, 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    vhi = _E4M3_POS[hi]
    vlo = _E4M3_POS[lo]
    dhi = vhi - a_sat
    dlo = a_sat - vlo
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(a_sat == vhi, hi, code)                        # exact hits
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def fl32(x) -> np.ndarray:
    """Round to the nearest binary32 (ties to even) and return the value as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """Round binary32 values to bfloat16, nearest-even, returned as float64.

    The input is first rounded to binary32 (the GPU rounds fp32 registers).  The rounding adds
    0x7FFF plus the lowest kept bit to the 32-bit pattern and truncates the low half: the textbook
    round-half-to-even on the bit pattern, valid for all finite inputs below the overflow point.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = rounded.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isnan(f), np.nan, out)


def bf16_bits_to_float(bits) -> np.ndarray:
    """Interpret uint16 bfloat16 bit patterns as float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
