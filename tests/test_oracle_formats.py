"""Pins of the oracle's number formats against the pages and library routines.

E2M1 and E4M3 are pinned by (a) the value set the pages print, (b) brute-force
nearest-value search and (c) the independent casts of ml_dtypes and torch.
"""
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden


def test_e2m1_value_set_matches_pages():
    # "nvfp4-kv-cache-memory-wall" section 2; tencent article, technical breakdown
    expected = [float(v) for v in read_golden("e2m1_values.txt")[0]]
    got = [oracle.e2m1_value(c) for c in range(16)]
    assert sorted(set(got)) == sorted(set(expected))
    # 8 magnitudes, each with both signs; -0 is code 8 (sign bit set)
    assert [abs(v) for v in got[:8]] == [abs(v) for v in got[8:]]
    assert all(math.copysign(1.0, v) < 0 for v in got[8:])
    assert max(got) == 6.0 and min(got) == -6.0


def test_e2m1_codes_follow_bit_fields():
    # 1 sign, 2 exponent, 1 mantissa bit (tencent article, technical breakdown):
    # for normal codes, value doubles with each exponent step
    for m in (0, 1):
        vals = [oracle.e2m1_value((e << 1) | m) for e in range(1, 4)]
        assert vals[1] == 2 * vals[0] and vals[2] == 2 * vals[1]
    # values increase with the code over the non-negative half
    mags = [oracle.e2m1_value(c) for c in range(8)]
    assert mags == sorted(mags) and len(set(mags)) == 8


def _e2m1_brute(y):
    """All codes at minimal distance from y (|y| clipped to the finite range)."""
    mag = min(abs(y), 6.0)
    d = [abs(mag - oracle.e2m1_value(c)) for c in range(8)]
    best = min(d)
    return [c for c in range(8) if d[c] == best]


def test_e2m1_encode_brute_force_and_ties_to_even():
    rng = np.random.default_rng(1)
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    ys = list(rng.uniform(-8, 8, 4000).astype(np.float32))
    for m in mids + [0.0, 0.5, 1, 1.5, 2, 3, 4, 6]:
        f = np.float32(m)
        for k in range(-3, 4):
            v = f
            step = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
            for _ in range(abs(k)):
                v = np.nextafter(v, step)
            ys += [v, -v]
    for y in ys:
        code = oracle.e2m1_encode(y)
        cands = _e2m1_brute(float(y))
        assert (code & 7) in cands, (y, code, cands)
        if len(cands) > 1:  # exact midpoint: the even code (mantissa bit 0)
            assert (code & 1) == 0, (y, code)
        assert (code >> 3) == (1 if np.signbit(y) else 0)
    # saturation
    assert oracle.e2m1_encode(7.0) == 7 and oracle.e2m1_encode(-1e30) == 15


def test_e2m1_encode_matches_ml_dtypes():
    mld = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(2)
    ys = np.concatenate([rng.uniform(-6, 6, 20000), rng.normal(0, 0.3, 20000),
                         np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])]).astype(np.float32)
    ys = np.concatenate([ys, -ys])
    ref = ys.astype(mld.float4_e2m1fn).astype(np.float64)
    got = np.array([oracle.e2m1_value(oracle.e2m1_encode(y)) for y in ys])
    np.testing.assert_array_equal(got, ref)
    # signed zeros agree too
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_e4m3_table():
    vals = [oracle.e4m3_value(c) for c in range(256)]
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    pos = vals[:0x7F]
    assert pos == sorted(pos) and len(set(pos)) == 127
    assert vals[0x80] == 0.0 and math.copysign(1.0, vals[0x80]) < 0


def test_e4m3_decode_matches_libraries():
    import torch

    codes = np.arange(256, dtype=np.uint8)
    ref_t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    np.testing.assert_array_equal(got, ref_t)
    mld = pytest.importorskip("ml_dtypes")
    ref_m = codes.view(mld.float8_e4m3fn).astype(np.float64)
    np.testing.assert_array_equal(got, ref_m)


def test_e4m3_encode_nearest_ties_even_saturating():
    mld = pytest.importorskip("ml_dtypes")
    vals = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    zs = []
    for m in list(mids) + list(vals):
        f = np.float32(m)
        zs += [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(0))]
    rng = np.random.default_rng(3)
    zs += list((2.0 ** rng.uniform(-12, 9, 20000)).astype(np.float32))
    zs = np.array(zs, np.float32)
    got = np.array([oracle.e4m3_encode(z) for z in zs], np.uint8)
    # brute force: minimal distance; on a tie the even code
    for z, c in zip(zs[:3000], got[:3000]):
        d = np.abs(vals - float(z))
        best = np.flatnonzero(d == d.min())
        assert c in best
        if len(best) > 1:
            assert c % 2 == 0
    # library cast (values within range; ml_dtypes rounds to nearest even)
    inrange = zs <= 448
    ref = zs[inrange].astype(mld.float8_e4m3fn).view(np.uint8)
    np.testing.assert_array_equal(got[inrange], ref)
    # saturation at 448 for anything larger, sign kept
    for z in (448.0, 449.0, 464.0, 500.0, 1e30, float("inf")):
        assert oracle.e4m3_encode(z) == 0x7E
        assert oracle.e4m3_encode(-z) == 0xFE
    # the subnormal/zero boundary: 2^-10 ties to 0, 1.5 * 2^-10 rounds up to 2^-9
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(1.5 * 2.0 ** -10) == 0x01


def test_bf16_widening():
    import torch

    rng = np.random.default_rng(4)
    x = rng.normal(0, 10, 1000).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle.lib().nvfp4_oracle_bf16_to_float(int(b)) for b in bits], np.float32)
    np.testing.assert_array_equal(got, ref)
