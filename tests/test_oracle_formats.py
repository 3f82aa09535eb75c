"""Pins for the oracle's bf16 / e4m3 conversions (CPU only).

The oracle converts by integer bit operations written from the format
definitions.  These tests check it against things that are not itself:
  * a nearest-value search over the finite codes (ties to the even code),
  * torch's float8_e4m3fn / bfloat16 casts (a library routine) in range,
  * fixed points of the OCP 8-bit floating point definition (golden file).
"""

import json
import os

import numpy as np
import pytest
import torch

from oracle import formats

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _e4m3_magnitudes():
    """Values of the 127 finite non-negative codes 0x00..0x7E, from torch (library)."""
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _search_e4m3(x64):
    """Nearest finite e4m3 code by search; ties -> even code; beyond 448 -> 448."""
    mags = _e4m3_magnitudes()                # strictly increasing
    a = np.abs(x64)
    idx = np.clip(np.searchsorted(mags, a), 1, len(mags) - 1)
    lo, hi = idx - 1, idx
    dlo, dhi = a - mags[lo], mags[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= mags[-1], len(mags) - 1, pick)
    sign = np.signbit(x64).astype(np.int64)
    return ((sign << 7) | pick).astype(np.uint8)


def test_e4m3_decode_matches_library_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = formats.e4m3_to_f64(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])
    assert nan.sum() == 2          # S.1111.111 only: e4m3fn has no infinities


def test_e4m3_golden_points():
    with open(os.path.join(GOLD, "e4m3_points.json")) as f:
        g = json.load(f)
    for code_hex, val in g["decode"].items():
        v = formats.e4m3_to_f64(np.array([int(code_hex, 16)], np.uint8))[0]
        if val == "nan":
            assert np.isnan(v)
        else:
            assert v == float(val), code_hex
    for val, code_hex in g["encode"]:
        c = formats.f32_to_e4m3(np.array([float(val)], np.float32))[0]
        assert c == int(code_hex, 16), (val, hex(c), code_hex)


def test_bf16_to_e4m3_exhaustive_against_search():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x32 = formats.bf16_bits_to_f32(bits)
    fin = np.isfinite(x32)
    got = formats.bf16_bits_to_e4m3(bits[fin])
    want = _search_e4m3(x32[fin].astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(int(bits[fin][i])), hex(int(got[i])), hex(int(want[i]))) for i in bad[:8]]


@pytest.mark.parametrize("seed", [0, 1])
def test_f32_to_e4m3_random_against_search(seed):
    g = np.random.Generator(np.random.PCG64(seed))
    n = 5_000_000
    # log-uniform magnitudes across the whole e4m3 range and beyond, random signs
    mag = np.exp2(g.uniform(-14.0, 10.0, n)).astype(np.float32)
    x = np.where(g.random(n) < 0.5, -mag, mag).astype(np.float32)
    # plus exact midpoints between neighbouring codes (the tie cases)
    mags = _e4m3_magnitudes()
    mids = ((mags[:-1] + mags[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0, 448.0, 464.0, 1e30, -1e30])])
    got = formats.f32_to_e4m3(x)
    want = _search_e4m3(x.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), hex(int(got[i])), hex(int(want[i]))) for i in bad[:8]]


def test_f32_to_e4m3_in_range_matches_library():
    g = np.random.Generator(np.random.PCG64(7))
    x = g.normal(0, 40, 2_000_000).astype(np.float32)
    x = x[np.abs(x) <= 448]
    got = formats.f32_to_e4m3(x)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, lib)


def test_f32_to_bf16_matches_library_and_search():
    g = np.random.Generator(np.random.PCG64(3))
    raw = g.integers(0, 2 ** 32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    x = raw.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3e38)]
    got = formats.f32_to_bf16_bits(x)
    lib = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, lib)
    # search: the two bf16 neighbours of x, nearest wins, ties to even
    sub = x[:200_000].astype(np.float64)
    t = (x[:200_000].view(np.uint32) >> 16).astype(np.uint16)
    lo = formats.bf16_bits_to_f64(t)
    hi = formats.bf16_bits_to_f64((t + 1).astype(np.uint16))
    dlo, dhi = np.abs(sub - lo), np.abs(hi - sub)
    want = np.where(dlo < dhi, t, np.where(dhi < dlo, t + 1, np.where(t % 2 == 0, t, t + 1))).astype(np.uint16)
    assert np.array_equal(got[:200_000], want)


def test_bf16_roundtrip_exact():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = formats.bf16_bits_to_f32(bits)
    fin = np.isfinite(x)
    assert np.array_equal(formats.f32_to_bf16_bits(x[fin]), bits[fin])
