"""Pins for the oracle's FP4 (E2M1) and E4M3 codec."""
import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values_match_the_standard_table():
    g = read_golden("e2m1_values.txt")
    for k, v in g.items():
        got = oracle.e2m1_value(int(k, 16))
        assert got == float(v) and np.signbit(got) == np.signbit(float(v)), k


def test_e4m3_values_match_torch_float8():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for b in range(256):
        got = oracle.e4m3_value(b)
        if np.isnan(ref[b]):
            assert np.isnan(got), b
        else:
            assert got == ref[b] and np.signbit(got) == np.signbit(ref[b]), b
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(1) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.uniform(0, 460, 3000), np.exp(rng.uniform(np.log(1e-4), np.log(448), 3000)),
        [0.0, 2.0 ** -10, 2.0 ** -10 * 1.0001, 2.0 ** -9 * 1.5, 432.0, 447.0, 460.0, 463.9],
    ]).astype(np.float32)
    # every midpoint between neighbouring finite values (ties go to the even code)
    pos = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals, ref):
        assert oracle.e4m3_encode(v) == r, v


def test_e4m3_encode_saturates():
    for v in [464.0, 480.0, 1e4, 3.0e38]:
        assert oracle.e4m3_encode(v) == 0x7E


def test_e2m1_round_trip_and_ties():
    for s in [1.0, 0.75, 2.0 ** -9, 448.0]:
        for c in range(16):
            v = oracle.e2m1_value(c) * s
            want = 0 if c == 8 else c          # -0 is written as +0
            assert oracle.e2m1_encode(np.float32(v), s) == want, (c, s)
        # midpoints between neighbouring magnitudes go to the even code
        for m in range(7):
            mid = (GRID[m] + GRID[m + 1]) / 2 * s
            even = m if m % 2 == 0 else m + 1
            assert oracle.e2m1_encode(np.float32(mid), s) == even
            assert oracle.e2m1_encode(np.float32(-mid), s) == (even | 8 if even else 0)
        # saturation above 6s
        assert oracle.e2m1_encode(np.float32(7 * s), s) == 7
        assert oracle.e2m1_encode(np.float32(-1e30), s) == 15


def test_e2m1_nearest_value_brute_force():
    rng = np.random.default_rng(1)
    for _ in range(3000):
        s = float(oracle.e4m3_value(int(rng.integers(1, 0x7F))))
        x = np.float32(rng.normal() * s * 3)
        c = oracle.e2m1_encode(x, s)
        got = oracle.e2m1_value(c) * s
        # no grid point is strictly nearer
        best = min(abs(g * s * np.sign(x) - float(x)) for g in GRID)
        assert abs(got - float(x)) == pytest.approx(best, abs=0, rel=0)


def test_quantize_rows_exact_groups_and_scale_rule():
    rng = np.random.default_rng(2)
    # a group made of grid values times a scale that is an E4M3 value, with
    # amax = 6 * scale, quantises to exactly those codes and that scale byte
    for _ in range(200):
        sb = int(rng.integers(1, 0x7F))
        s = oracle.e4m3_value(sb)
        codes = rng.integers(0, 16, 16)
        codes[rng.integers(0, 16)] = 7
        x = np.array([oracle.e2m1_value(c) * s for c in codes], np.float32)
        c2, s2 = oracle.quantize_rows(x[None, :])
        assert s2[0, 0] == sb
        dec = oracle.dequant_rows(c2, s2)[0]
        assert np.array_equal(dec, x.astype(np.float64))
    # the scale byte is E4M3(float32(amax / 6)) as torch rounds it
    x = rng.normal(size=(500, 64)).astype(np.float32) * np.exp(rng.uniform(-6, 6, (500, 1))).astype(np.float32)
    _, sc = oracle.quantize_rows(x)
    amax = np.abs(x.reshape(500, 4, 16)).max(-1)
    ref = torch.from_numpy((amax / np.float32(6.0)).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(sc, ref)


def test_quantize_error_bound_and_zero_scale():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(300, 128)).astype(np.float32)
    c, s = oracle.quantize_rows(x)
    dq = oracle.dequant_rows(c, s)
    sv = np.array([[oracle.e4m3_value(b) for b in row] for row in s]).repeat(16, axis=1)
    # nearest-grid rounding: error at most half the widest gap (2*s) = s,
    # plus the part of |x| above 6*s that saturates
    over = np.maximum(np.abs(x) - 6 * sv, 0)
    assert np.all(np.abs(dq - x) <= sv + over + 1e-30)
    # a group whose amax/6 rounds to E4M3 zero gets all-zero codes
    tiny = np.full((1, 16), 2.0 ** -13, np.float32)
    c, s = oracle.quantize_rows(tiny)
    assert s[0, 0] == 0 and not c.any()
