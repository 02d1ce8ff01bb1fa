"""Pins of the oracle's NVFP4 block quantiser, cache write and storage sizes (CPU).

Block rule (reading of "NVFP4-KV-Cache auf der NVIDIA RTX PRO 6000 Blackwell
Server Edition", section "Bytes pro Token", and "SGLang stores KV cache in 4
bits" (LMSYS summary), Interpretation / Perspective): one E4M3 scale per 16
values, scale = E4M3(amax / 6), element = E2M1(x / scale), global scale 1.0.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "storage_figures.txt")


def load_golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split()
            vals[k] = float(v)
    return vals


def unpack(packed):
    packed = np.asarray(packed, np.uint8)
    return np.stack([packed & 15, packed >> 4], -1).reshape(*packed.shape[:-1], -1)


def brute_force_block(x):
    """Independent brute force for many blocks at once: x float32 [N][16].

    The scale is the E4M3 code (scanning all 127 finite non-negative codes)
    nearest to fl32(amax/6), tie to the even code; each element code is the
    E2M1 code (scanning all 16) nearest to fl32(x/s) with ties to the even
    code and the sign taken from the quotient.  Distances use float64, which
    is exact for these operands near ties.
    """
    x = np.asarray(x, np.float32)
    e4 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    e2 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    amax = np.abs(x).max(1)
    s32 = (amax / np.float32(6.0)).astype(np.float32).astype(np.float64)
    d = np.abs(s32[:, None] - e4[None, :])
    best = d.min(1, keepdims=True)
    cand = d == best
    # prefer even codes among tied candidates (at most two candidates tie)
    even = cand & (np.arange(127)[None, :] % 2 == 0)
    S = np.where(even.any(1), even.argmax(1), cand.argmax(1))
    S = np.where(s32 >= 448.0, 126, S)
    s = e4[S].astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (x / s[:, None]).astype(np.float32)
    a = np.abs(y).astype(np.float64)
    d2 = np.abs(a[..., None] - e2)
    best2 = d2.min(-1, keepdims=True)
    cand2 = d2 == best2
    even2 = cand2 & (np.arange(8) % 2 == 0)
    mag = np.where(even2.any(-1), even2.argmax(-1), cand2.argmax(-1))
    mag = np.where(a > 6.0, 7, mag)
    codes = (mag | (np.signbit(y).astype(np.int64) << 3)).astype(np.uint8)
    codes = np.where((s == 0)[:, None], 0, codes).astype(np.uint8)
    return codes, S.astype(np.uint8)


def oracle_blocks(x):
    x = np.asarray(x, np.float32)
    codes, scales = [], []
    for row in x:
        p, s = oracle.quantize_block16(row)
        codes.append(unpack(p))
        scales.append(s)
    return np.array(codes, np.uint8), np.array(scales, np.uint8)


def oracle_blocks_fast(x):
    """Many blocks [N][16] through the oracle's cache writer (rows of 8 blocks)."""
    x = np.asarray(x, np.float32).reshape(-1, 16)
    n = x.shape[0]
    x = np.pad(x, ((0, (-n) % 8), (0, 0))).reshape(-1, 1, 128)
    T = x.shape[0]
    data = np.zeros((T, 1, 1, 64), np.uint8)
    scale = np.zeros((T, 1, 1, 8), np.uint8)
    oracle.quantize_append(x, np.arange(T, dtype=np.int32), data, scale, page_size=1)
    return unpack(data.reshape(-1, 8))[:n], scale.reshape(-1)[:n]


def test_packing_order_low_nibble_is_even_element():
    # block with distinct codes 0..7 then 8..15 at scale 1 (one element at 6)
    vals = np.float32([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
    packed, S = oracle.quantize_block16(vals)
    assert oracle.e4m3_value(S) == 1.0
    assert list(packed) == [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]


def test_round_trip_every_normal_scale_and_code():
    """x = v_i * s with one element at +-6 s quantises back to (v_i, S)."""
    rng = np.random.default_rng(0)
    t = oracle.e2m1_table()
    for S in range(0x08, 0x7F):                # normal E4M3 scales
        s = oracle.e4m3_value(S)
        codes = rng.integers(0, 16, size=16).astype(np.uint8)
        codes[rng.integers(16)] = 7 | (8 if rng.integers(2) else 0)
        x = (t[codes] * s).astype(np.float32)
        p, got_S = oracle.quantize_block16(x)
        assert got_S == S
        want = codes.copy()
        # -0 * s quantises to code 8 (sign kept); +0 to 0
        np.testing.assert_array_equal(unpack(p), want)


def test_amax_element_gets_magnitude_six_for_normal_scales():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((4000, 16)) * np.exp2(rng.uniform(-5, 7, (4000, 1)))).astype(np.float32)
    codes, S = oracle_blocks_fast(x)
    normal = S >= 0x08
    arg = np.abs(x).argmax(1)
    mags = codes[np.arange(len(x)), arg] & 7
    assert normal.mean() > 0.9
    assert (mags[normal] == 7).all()


def test_error_bound_half_gap():
    """|x - dequant(x)| <= half the local E2M1 gap times s (no saturation)."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2000, 16)).astype(np.float32) * 3
    codes, S = oracle_blocks_fast(x)
    s = oracle.e4m3_table()[S][:, None]
    xh = oracle.e2m1_table()[codes] * s
    a = np.abs(x) / s
    gap = np.select([a < 2, a < 4], [0.5, 1.0], 2.0)
    sat = a > 6
    err = np.abs(x - xh)
    assert (err[~sat] <= gap[~sat] / 2 * s.repeat(16, 1)[~sat] * (1 + 1e-6)).all()


def test_zero_block_and_underflowing_scale():
    p, S = oracle.quantize_block16(np.zeros(16, np.float32))
    assert S == 0 and (p == 0).all()
    x = np.zeros(16, np.float32)
    x[3] = -1e-4                                # amax/6 < 2^-10 -> scale 0
    p, S = oracle.quantize_block16(x)
    assert S == 0 and (p == 0).all()
    x[3] = -2.0 ** -7                           # amax/6 rounds to 2^-9
    p, S = oracle.quantize_block16(x)
    assert S == 0x01
    assert unpack(p)[3] == 0xE                 # -2^-7 / 2^-9 = -4 (coarse subnormal scale)


def test_scale_rounding_on_fp32_quotient_agrees_with_exact_rational():
    """E4M3(fl32(amax/6)) equals round-half-even of the exact amax/6 for amax
    at and around 6 x every E4M3 midpoint."""
    e4 = [Fraction(oracle.e4m3_value(c)) for c in range(0x7F)]
    amaxes = []
    for c in range(0x7E):
        mid6 = np.float32(float((e4[c] + e4[c + 1]) / 2 * 6))
        v = mid6
        amaxes.append(v)
        up, dn = v, v
        for _ in range(3):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(0))
            amaxes += [up, dn]
    amaxes = np.float32(amaxes)
    blocks = np.zeros((len(amaxes), 16), np.float32)
    blocks[:, 5] = amaxes
    _, got = oracle_blocks_fast(blocks)
    for a, S in zip(amaxes, got):
        q = Fraction(float(a)) / 6
        if q >= 448:
            want = 0x7E
        else:
            hi = next(i for i in range(0x7F) if e4[i] > q)
            lo = hi - 1
            dlo, dhi = q - e4[lo], e4[hi] - q
            want = lo if dlo < dhi else hi if dhi < dlo else (lo if lo % 2 == 0 else hi)
        assert S == want, (a, S, want)


@pytest.mark.parametrize("values", [
    (0.0, 1.0, -2.9),
    (0.75, -1.25, 5.0),
    (0.1, 0.3, -0.55),
    (1.0, 3.0, -6.0),
])
def test_exhaustive_three_value_blocks(values):
    """All 3^8 patterns of 8 positions (mirrored into the other 8, negated)
    over a 3-value set, at 25 binary exponents: oracle == brute force."""
    vals = np.float32(values)
    idx = np.indices((3,) * 8).reshape(8, -1).T
    half = vals[idx]
    base = np.concatenate([half, -half[:, ::-1]], 1)
    xs = [base * np.float32(2.0 ** e) for e in range(-14, 11)]
    x = np.concatenate(xs, 0).astype(np.float32)
    codes_o, S_o = oracle_blocks_fast(x)
    codes_b, S_b = brute_force_block(x)
    np.testing.assert_array_equal(S_o, S_b)
    np.testing.assert_array_equal(codes_o, codes_b)


def test_random_blocks_match_brute_force_and_single_block_api():
    rng = np.random.default_rng(5)
    x = (rng.standard_t(3, (8192, 16)) * np.exp2(rng.uniform(-12, 10, (8192, 1)))).astype(np.float32)
    codes_o, S_o = oracle_blocks_fast(x)
    codes_b, S_b = brute_force_block(x)
    np.testing.assert_array_equal(S_o, S_b)
    np.testing.assert_array_equal(codes_o, codes_b)
    c1, s1 = oracle_blocks(x[:64])
    np.testing.assert_array_equal(c1, codes_b[:64])
    np.testing.assert_array_equal(s1, S_b[:64])


def test_append_scatters_rows_to_slots():
    """quantize_append writes token t, head h to page slot//P, offset slot%P."""
    rng = np.random.default_rng(6)
    T, Hkv, d, P, pages = 37, 3, 128, 16, 9
    x = rng.standard_normal((T, Hkv, d)).astype(np.float32)
    slots = rng.permutation(pages * P)[:T].astype(np.int32)
    slots[4] = -1                               # negative slot: skipped
    data = np.zeros((pages, Hkv, P, d // 2), np.uint8)
    scale = np.zeros((pages, Hkv, P, d // 16), np.uint8)
    oracle.quantize_append(x, slots, data, scale, page_size=P)
    for t in range(T):
        if slots[t] < 0:
            continue
        pg, off = divmod(int(slots[t]), P)
        for h in range(Hkv):
            for blk in range(8):
                p, s = oracle.quantize_block16(x[t, h, 16 * blk:16 * blk + 16])
                assert (data[pg, h, off, 8 * blk:8 * blk + 8] == p).all()
                assert scale[pg, h, off, blk] == s
    written = np.zeros((pages * P,), bool)
    written[slots[slots >= 0]] = True
    untouched = ~written.reshape(pages, P)
    assert (data.transpose(0, 2, 1, 3)[untouched] == 0).all()


def test_dequant_rows_is_value_times_scale():
    rng = np.random.default_rng(7)
    data = rng.integers(0, 256, (50, 64), dtype=np.uint8)
    scale = rng.integers(0, 0x7F, (50, 8), dtype=np.uint8)
    out = oracle.dequant_rows(data, scale)
    e4 = torch.from_numpy(scale).view(torch.float8_e4m3fn).double().numpy()
    codes = unpack(data)
    e2 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    want = e2[codes] * np.repeat(e4, 16, 1)
    np.testing.assert_array_equal(out, want.astype(np.float32))


def test_storage_sizes_match_printed_figures():
    g = load_golden()
    assert oracle.nvfp4_bytes(int(g["block_values"])) == g["block_packed_bytes"] + g["block_scale_bytes"]
    assert oracle.fp8_bytes(int(g["block_values"])) == g["fp8_block_bytes"]
    ratio = oracle.nvfp4_bytes(16 * 1000) / oracle.fp8_bytes(16 * 1000)
    assert ratio == g["ratio_nvfp4_to_fp8"]
    assert round(1 / ratio, 2) == g["capacity_gain_approx"]
    vpt = 2 * int(g["llama_layers"]) * int(g["llama_kv_heads"]) * int(g["llama_head_dim"])
    assert vpt == g["llama_values_per_token"]
    gib = 2.0 ** 30
    fp8_8k = oracle.fp8_bytes(vpt * 8192) / gib
    nv_8k = oracle.nvfp4_bytes(vpt * 8192) / gib
    assert fp8_8k == g["session_8k_fp8_gib"]
    assert round(nv_8k, 2) == g["session_8k_nvfp4_gib_rounded"]
    assert oracle.fp8_bytes(vpt * 131072) / gib == g["ctx128k_fp8_gib"]
    assert oracle.nvfp4_bytes(vpt * 131072) / gib == g["ctx128k_nvfp4_gib"]
    free = g["budget_gib"] - g["weights_fp8_gib"]
    assert int(free // fp8_8k) == g["sessions_fp8"]
    assert int(free // nv_8k) == g["sessions_nvfp4"]
