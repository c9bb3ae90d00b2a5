"""Pins for the oracle's float8_e4m3fn codec and bf16 rounding.

The codec is checked against things other than itself: the code points fixed
by the OCP E4M3 definition and torch.finfo (tests/golden/e4m3_points.txt),
torch's own float8_e4m3fn conversion (an independent implementation), the
round-trip and tie-to-even properties, and the saturation rule.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_points():
    pts = []
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()[:2]
            pts.append((int(code, 16), float(val)))
    return pts


def test_decode_golden_points(oracle_mod):
    tab = oracle_mod.e4m3_table()
    for code, val in _golden_points():
        if math.isnan(val):
            assert math.isnan(tab[code]), hex(code)
        else:
            assert tab[code] == val, (hex(code), tab[code], val)
            assert math.copysign(1.0, tab[code]) == math.copysign(1.0, val)


def test_decode_table_matches_torch(oracle_mod):
    tab = oracle_mod.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_o, nan_r = np.isnan(tab), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert nan_o.sum() == 2  # 0x7F and 0xFF only
    assert (tab[~nan_o] == ref[~nan_r]).all()
    assert np.nanmax(tab) == 448.0 and np.nanmin(tab) == -448.0


def test_decode_table_matches_ml_dtypes(oracle_mod):
    ml = pytest.importorskip("ml_dtypes")
    tab = oracle_mod.e4m3_table()
    ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    assert ((tab == ref) | (np.isnan(tab) & np.isnan(ref))).all()


def test_encode_roundtrip_all_codes(oracle_mod):
    tab = oracle_mod.e4m3_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = tab[codes].astype(np.float32)
    assert (oracle_mod.e4m3_encode(vals) == codes).all()


def test_encode_midpoints_tie_to_even(oracle_mod):
    tab = oracle_mod.e4m3_table()
    for sign in (1.0, -1.0):
        sbit = 0 if sign > 0 else 0x80
        for c in range(0, 126):
            lo, hi = tab[c], tab[c + 1]
            mid = np.float32((lo + hi) / 2)        # 5 significant bits: exact in fp32
            assert float(mid) == (lo + hi) / 2
            even = c if c % 2 == 0 else c + 1
            x = np.array([sign * mid,
                          sign * np.nextafter(mid, np.float32(np.inf)),
                          sign * np.nextafter(mid, np.float32(-np.inf))], dtype=np.float32)
            got = oracle_mod.e4m3_encode(x)
            assert got[0] == (even | sbit), (c, sign)
            assert got[1] == ((c + 1) | sbit), (c, sign)
            assert got[2] == (c | sbit), (c, sign)


def test_encode_specials_and_saturation(oracle_mod):
    cases = [
        (0.0, 0x00), (-0.0, 0x80), (448.0, 0x7E), (-448.0, 0xFE),
        (448.5, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (479.0, 0x7E), (480.0, 0x7E),
        (1e30, 0x7E), (-1e30, 0xFE), (float("inf"), 0x7E), (float("-inf"), 0xFE),
        (float("nan"), 0x7F),
        (2.0 ** -10, 0x00),                 # tie between 0 and 2^-9 -> even (0)
        (-(2.0 ** -10), 0x80),              # negative underflow keeps the sign
        (2.0 ** -10 * 1.0000001, 0x01),
        (-(2.0 ** -11), 0x80), (1e-30, 0x00),
        (3 * 2.0 ** -10, 0x02),             # tie between 1 and 2 (x 2^-9) -> even (2)
        (240.0, 0x77), (248.0, 0x78),       # 248: tie between 240 (odd) and 256 (even)
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    got = oracle_mod.e4m3_encode(x)
    for (v, want), g in zip(cases, got):
        assert g == want, (v, hex(g), hex(want))


def test_encode_matches_torch_on_a_dense_grid(oracle_mod):
    """Every 37th fp32 bit pattern with |x| < 464 (where torch's cast, which maps
    overflow to NaN instead of saturating, is defined the same way)."""
    lim = np.float32(464.0).view(np.uint32)
    bits = np.arange(0, int(lim), 37, dtype=np.uint32)
    for sign in (0, 0x80000000):
        x = (bits | np.uint32(sign)).view(np.float32)
        got = oracle_mod.e4m3_encode(x)
        ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_encode_monotone(oracle_mod):
    x = np.linspace(-500, 500, 200001, dtype=np.float32)
    tab = oracle_mod.e4m3_table()
    v = tab[oracle_mod.e4m3_encode(x)]
    assert (np.diff(v) >= 0).all()


# ------------------------------------------------------------------ bf16 ---

def test_bf16_matches_torch_for_fp32_inputs(oracle_mod):
    g = np.random.default_rng(1)
    bits = g.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3.3e38)]
    got = oracle_mod.bf16_from_f64(x.astype(np.float64))
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_bf16_rounds_directly_from_double(oracle_mod):
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7 (bf16 0x3F80, 0x3F81)
    mid = 1.0 + 2.0 ** -8
    cases = [
        (mid, 0x3F80),                      # tie -> even mantissa
        (mid + 2.0 ** -40, 0x3F81),         # above the tie: an fp32 detour would tie
        (mid - 2.0 ** -40, 0x3F80),
        (1.0 + 3 * 2.0 ** -8, 0x3F82),      # tie between 0x3F81 and 0x3F82 -> even
        (-(mid + 2.0 ** -40), 0xBF81),
        (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000), (1.5 * 2.0 ** -133, 0x0002),
        (2.0 ** -126, 0x0080), (0.0, 0x0000), (-0.0, 0x8000),
        (float("inf"), 0x7F80), (3.5e38, 0x7F80),
    ]
    got = oracle_mod.bf16_from_f64(np.array([c[0] for c in cases]))
    for (v, want), g in zip(cases, got):
        assert g == want, (v, hex(g), hex(want))
