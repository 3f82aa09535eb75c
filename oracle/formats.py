"""Number formats used by the KV pools (oracle; test infrastructure only).

bf16: IEEE binary32 with the low 16 bits dropped (1 sign, 8 exponent, 7
mantissa bits).  fp32 -> bf16 is round-to-nearest-even on the 16 dropped bits.

e4m3 ("e4m3fn", OCP 8-bit floating point): 1 sign, 4 exponent (bias 7), 3
mantissa bits; no infinities; S.1111.111 is NaN, so the largest finite
magnitude is 1.75 * 2^8 = 448; exponent field 0 encodes subnormals m/8 * 2^-6.
[PR1012] "Description": the sliding family's K/V are stored as e4m3 at scale
1.0, i.e. the stored code is the e4m3 rounding of the value itself.  Rounding
is to nearest, ties to even, and saturating ("satfinite"): anything whose
rounding would exceed 448 in magnitude becomes +-448.

Everything here is written from those definitions with integer bit operations
on NumPy arrays; no cast routine of any library is used.
"""

import numpy as np

E4M3_MAX = 448.0


def bf16_bits_to_f32(u16):
    """bf16 bit patterns (uint16 array) -> exact float32 values."""
    u16 = np.asarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(u16):
    return bf16_bits_to_f32(u16).astype(np.float64)


def f32_to_bf16_bits(x32):
    """float32 -> bf16 bits, round to nearest, ties to even.

    The kept 16 bits are incremented when the dropped 16 bits exceed half an
    ulp (0x8000), or equal it and the kept value is odd.  NaN maps to a quiet
    NaN; the synthetic inputs contain none.
    """
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    keep = u >> np.uint64(16)
    dropped = u & np.uint64(0xFFFF)
    up = (dropped > 0x8000) | ((dropped == 0x8000) & ((keep & np.uint64(1)) == 1))
    out = (keep + up.astype(np.uint64)).astype(np.uint16)
    nan = np.isnan(x32)
    if nan.any():
        out = np.where(nan, np.uint16(0x7FC0) | (keep.astype(np.uint16) & np.uint16(0x8000)), out)
    return out


def e4m3_to_f64(b):
    """e4m3 codes (uint8 array) -> float64 values; NaN code -> nan."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def _rne_shift(sig, shift):
    """Round the non-negative integers sig / 2^shift to nearest, ties to even."""
    sig = np.asarray(sig).astype(np.uint64)
    shift = np.clip(np.asarray(shift), 0, 63).astype(np.uint64)
    q = sig >> shift
    rem = sig - (q << shift)
    one = np.uint64(1)
    half = np.left_shift(one, np.maximum(shift, one) - one)   # 2^(shift-1)
    up = (shift >= one) & ((rem > half) | ((rem == half) & ((q & one) == one)))
    return (q + up.astype(np.uint64)).astype(np.int64)


def f32_to_e4m3(x32):
    """float32 -> e4m3 code, round to nearest even, saturating to +-448.

    Work on the binary32 fields (sign s, biased exponent E, mantissa M):
      * value = 1.M * 2^(E-127) for E >= 1, 0.M * 2^-126 for E == 0.
      * If the unbiased exponent e >= -6 the target is an e4m3 normal of the
        same binade: keep 4 significant bits (1 + 3 mantissa), i.e. round the
        24-bit significand by 20 bits.  A carry out of 16 moves to the next
        binade.  A result above 1.75 * 2^8 saturates to 448.
      * Otherwise the target grid is the subnormal step 2^-9: round
        significand * 2^(e-23) / 2^-9 to an integer q in [0, 8]; q == 8 is the
        smallest normal, whose code is exactly 0x08.
    """
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.int64)
    sign = (u >> 31) & 1
    E = (u >> 23) & 0xFF
    M = u & 0x7FFFFF
    sig = np.where(E == 0, M, M | (1 << 23))
    e = np.where(E == 0, -126, E - 127)

    # normal branch
    qn = _rne_shift(sig, np.full_like(sig, 20))
    en = np.where(qn == 16, e + 1, e)
    qn = np.where(qn == 16, 8, qn)
    code_n = ((en + 7) << 3) | (qn - 8)
    sat = (en > 8) | ((en == 8) & (qn > 14))
    code_n = np.where(sat, 0x7E, code_n)

    # subnormal branch: q = round(sig * 2^(e - 23 + 9)) = round(sig >> (14 - e))
    qs = _rne_shift(sig, (14 - e))
    code_s = qs  # 0..8; 8 is the smallest normal 0x08

    code = np.where(e >= -6, code_n, code_s)
    code = np.where(E == 0xFF, 0x7E, code)  # +-inf saturates (satfinite)
    code = np.where(np.isnan(x32), 0x7F, code)
    return ((sign << 7) | code).astype(np.uint8)


def bf16_bits_to_e4m3(u16):
    """bf16 -> e4m3 with a single rounding from the exact bf16 value."""
    return f32_to_e4m3(bf16_bits_to_f32(u16))
