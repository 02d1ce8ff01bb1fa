"""Pins of the oracle's element and scale formats (CPU only).

The oracle's E2M1 and E4M3 encoders are checked against things other than
themselves:
  * torch's float8_e4m3fn conversion (a library routine) for E4M3 decode and
    round-to-nearest-even encode;
  * a generic binary-minifloat rounder written here with numpy's frexp/rint
    (rint rounds half to even), itself first checked against torch's E4M3
    cast, then applied with E2M1's parameters (1 mantissa bit, minimum
    exponent 0, largest magnitude 6);
  * exact rational arithmetic (fractions) near every rounding midpoint;
  * round trips of every representable value and the tie cases the format's
    round-half-to-even rule fixes.
Format facts: "NVFP4-KV-Cache auf der NVIDIA RTX PRO 6000 Blackwell Server
Edition", section "Bytes pro Token" (E2M1 = 1 sign, 2 exponent, 1 mantissa bit;
one E4M3 scale per 16 values).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def minifloat_round(y, man_bits, emin, maxval):
    """Nearest value of a binary float format (ties to even), saturating."""
    y = np.asarray(y, np.float32).astype(np.float64)
    a = np.abs(y)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    E = np.maximum(ex - 1, emin)
    quantum = np.ldexp(1.0, (E - man_bits).astype(np.int64))
    r = np.rint(a / quantum) * quantum
    r = np.minimum(r, maxval)
    return np.copysign(r, y)


def e4m3_ref_torch(y):
    t = torch.from_numpy(np.asarray(y, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def structured_fp32(lo_exp, hi_exp, seed=0, n_random=1 << 20):
    """fp32 values of every exponent in [lo_exp, hi_exp] with mantissas near
    the grid midpoints of low-precision formats, plus random ones."""
    rng = np.random.default_rng(seed)
    mants = []
    for top in range(16):                      # top 4 mantissa bits
        base = top << 19
        for low in (0, 1, 2, (1 << 18) - 1, 1 << 18, (1 << 18) + 1, (1 << 19) - 1):
            mants.append(base + low)
    mants = np.array(sorted(set(mants)), np.uint32)
    exps = np.arange(lo_exp + 127, hi_exp + 128, dtype=np.uint32)
    bits = (exps[:, None] << 23) | mants[None, :]
    vals = bits.reshape(-1).view(np.float32)
    rnd = rng.uniform(2.0 ** lo_exp, 2.0 ** (hi_exp + 1), size=n_random).astype(np.float32)
    allv = np.concatenate([vals, rnd, np.float32([0.0])])
    return np.concatenate([allv, -allv])


# --- the reference rounder itself is checked against a library routine -----

def test_minifloat_rounder_matches_torch_e4m3():
    y = structured_fp32(-12, 8)
    y = y[np.abs(y) <= 448]
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = minifloat_round(y, 3, -6, 448.0)
    np.testing.assert_array_equal(got, want)


# --- E4M3 -------------------------------------------------------------------

def test_e4m3_decode_table_matches_torch():
    mine = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.isnan(mine[nan]).all()
    np.testing.assert_array_equal(mine[~nan], ref[~nan])
    # signed zero: 0x80 decodes to -0
    assert np.signbit(mine[0x80]) and mine[0x80] == 0.0


def test_e4m3_encode_matches_torch_in_range():
    y = structured_fp32(-14, 8, seed=1)
    y = y[np.abs(y) <= 448]
    np.testing.assert_array_equal(oracle.e4m3_encode(y), e4m3_ref_torch(y))


def test_e4m3_encode_saturates():
    y = np.float32([448, 449, 463.99, 464, 479, 480, 1e6, 3.4e38])
    assert (oracle.e4m3_encode(y) == 0x7E).all()
    assert (oracle.e4m3_encode(-y) == 0xFE).all()


def test_e4m3_round_trip_every_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = oracle.e4m3_value(c)
        assert oracle.e4m3_encode(np.float32(v))[0] == c, hex(c)


def test_e4m3_exact_rational_near_midpoints():
    """Every midpoint between neighbouring E4M3 magnitudes, and fp32 values a
    few ulps either side, rounded with exact rationals (half to even)."""
    vals = [Fraction(oracle.e4m3_value(c)) for c in range(0x7F)]
    ys, want = [], []
    for c in range(0x7E):
        mid = (vals[c] + vals[c + 1]) / 2
        f = np.float32(float(mid))
        assert Fraction(float(f)) == mid
        for k in range(-3, 4):
            y = np.nextafter(f, np.float32(np.inf) if k > 0 else np.float32(0)) if k else f
            for _ in range(abs(k) - 1):
                y = np.nextafter(y, np.float32(np.inf) if k > 0 else np.float32(0))
            fy = Fraction(float(y))
            dlo, dhi = fy - vals[c], vals[c + 1] - fy
            if dlo < dhi:
                w = c
            elif dhi < dlo:
                w = c + 1
            else:
                w = c if c % 2 == 0 else c + 1
            ys.append(y)
            want.append(w)
    np.testing.assert_array_equal(oracle.e4m3_encode(np.float32(ys)), np.uint8(want))


# --- E2M1 -------------------------------------------------------------------

def test_e2m1_decode_table_structure():
    t = oracle.e2m1_table()
    grid = np.unique(np.abs(minifloat_round(np.linspace(0, 8, 100001), 1, 0, 6.0)))
    # the eight magnitudes are exactly the E2M1 grid, increasing with the code
    np.testing.assert_array_equal(t[:8], grid)
    assert (np.diff(t[:8]) > 0).all()
    # bit 3 is the sign, the low three bits the magnitude
    np.testing.assert_array_equal(t[8:], -t[:8])
    assert np.signbit(t[8]) and t[8] == 0.0
    # exponent field (bits 2..1) zero <=> subnormal magnitudes {0, 0.5}
    assert list(t[:2]) == [0.0, 0.5]
    assert t[7] == 6.0


def test_e2m1_encode_matches_minifloat_rounder():
    y = structured_fp32(-30, 10, seed=2)
    want_vals = minifloat_round(y, 1, 0, 6.0)
    t = oracle.e2m1_table()
    got_vals = t[oracle.e2m1_encode(y)]
    np.testing.assert_array_equal(got_vals, want_vals)
    # the sign bit follows the input's sign, zeros included
    codes = oracle.e2m1_encode(y)
    np.testing.assert_array_equal((codes >> 3) & 1, np.signbit(y).astype(np.uint8))


def test_e2m1_encode_sparse_sweep_of_all_bit_patterns():
    bits = np.arange(0, 1 << 32, 4093, dtype=np.uint64).astype(np.uint32)
    y = bits.view(np.float32)
    y = y[np.isfinite(y)]
    t = oracle.e2m1_table()
    np.testing.assert_array_equal(t[oracle.e2m1_encode(y)], minifloat_round(y, 1, 0, 6.0))


@pytest.mark.parametrize("y,code", [
    (0.0, 0x0), (-0.0, 0x8), (0.25, 0x0), (0.2500001, 0x1), (0.75, 0x2), (0.7499999, 0x1),
    (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6), (5.0000005, 0x7),
    (6.0, 0x7), (7.0, 0x7), (1e30, 0x7), (-0.1, 0x8), (-0.3, 0x9), (-6.5, 0xF),
])
def test_e2m1_tie_and_saturation_cases(y, code):
    assert oracle.e2m1_encode(np.float32(y))[0] == code


def test_e2m1_round_trip_every_code():
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert oracle.e2m1_encode(np.float32(v))[0] == c


def test_e2m1_encode_monotone():
    y = np.sort(structured_fp32(-8, 4, seed=3, n_random=1 << 16))
    v = oracle.e2m1_table()[oracle.e2m1_encode(y)]
    assert (np.diff(v) >= 0).all()
