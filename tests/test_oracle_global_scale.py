"""Pins of the oracle's tensor (global) scale G (CPU only).

"NVFP4-KV-Cache auf der NVIDIA RTX PRO 6000 Blackwell Server Edition", "Bytes
pro Token": an FP32 tensor scale sits above the E4M3 block scales; "SGLang
stores KV cache in 4 bits" (LMSYS summary), Perspective: it is left at 1.0,
and calibrating it is the next step.  Reading: a cached value is
G * E4M3 scale * E2M1 code, so the block procedure runs on y = fl32(x / G);
decode attends over G * s * e; the prefix workspace holds
E4M3_RNE_sat(fl32(G * s * e)).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_oracle_attention import dequant_independent
from test_oracle_quant import brute_force_block, unpack

SCALES = [0.37, 3.1, 2.0 ** -7, 1.0 / 3.0]


@pytest.mark.parametrize("g", SCALES)
def test_blocks_match_brute_force_on_the_scaled_values(g):
    """Block codes and scale of x at tensor scale G equal the independent brute
    force applied to fl32(x / G)."""
    rng = np.random.default_rng(int(g * 1e6) % 1000)
    x = (rng.standard_t(3, (4096, 16)) * rng.uniform(0.01, 50, (4096, 1))).astype(np.float32)
    gs = np.float32(g)
    codes_ref, S_ref = brute_force_block((x / gs).astype(np.float32))
    for n in range(0, 4096, 97):
        packed, S = oracle.quantize_block16(x[n], global_scale=g)
        assert S == S_ref[n]
        np.testing.assert_array_equal(unpack(packed), codes_ref[n])


@pytest.mark.parametrize("g", SCALES)
def test_dequantised_values_stay_within_the_half_gap(g):
    """|x - G s e| <= G s (the largest E2M1 half gap, between 4 and 6, is one
    scale unit) plus the rounding of x / G: a G applied the wrong way round or
    twice breaks this."""
    rng = np.random.default_rng(5)
    T, Hkv = 64, 2
    # x / G spans the E4M3 scale range without saturating
    x = (rng.standard_normal((T, Hkv, 128)) * 7 * g).astype(np.float32)
    data = np.zeros((4, Hkv, 16, 64), np.uint8)
    scale = np.zeros((4, Hkv, 16, 8), np.uint8)
    oracle.quantize_append(x, np.arange(T, dtype=np.int32), data, scale, global_scale=g)
    deq = oracle.dequant_rows(data, scale, global_scale=g)          # [pages][Hkv][16][128]
    deq = deq.transpose(0, 2, 1, 3).reshape(-1, Hkv, 128)[:T]
    s = torch.from_numpy(scale.copy()).view(torch.float8_e4m3fn).double().numpy()
    s = np.repeat(s.transpose(0, 2, 1, 3).reshape(-1, Hkv, 8)[:T], 16, -1)
    bound = np.float64(np.float32(g)) * s * 1.0 + np.abs(x) * 2.0 ** -22
    assert (np.abs(x.astype(np.float64) - deq) <= bound).all()
    assert np.abs(x - deq).max() > 0


@pytest.mark.parametrize("g", [0.37, 3.1])
def test_decode_with_global_scale_matches_torch(g):
    """Attention over G-scaled values: torch float64 softmax and matmul on rows
    dequantised independently (nibbles x torch's E4M3 decode) times G."""
    w = workloads.custom(3, 8, 2, (40, 1, 77), seed=21)
    bt, num_pages = workloads.block_table(w, spare_pages=2)
    pools = {n: np.zeros((num_pages, 2, 16, 64 if n.endswith("d") else 8), np.uint8)
             for n in ("kd", "ks", "vd", "vs")}
    for b in range(w.batch):
        L = w.seq_lens[b]
        sm = workloads.slot_mapping(w, bt, b, 0, L)
        oracle.quantize_append(workloads.kv_rows(w, "k", b, 0, L).numpy() * 5, sm, pools["kd"], pools["ks"],
                               global_scale=g)
        oracle.quantize_append(workloads.kv_rows(w, "v", b, 0, L).numpy(), sm, pools["vd"], pools["vs"],
                               global_scale=g)
    q = workloads.query(w).float().numpy()
    got = oracle.paged_decode(pools["kd"], pools["ks"], pools["vd"], pools["vs"], q, bt,
                              np.int32(w.seq_lens), global_scale=g)
    K = dequant_independent(pools["kd"], pools["ks"]) * np.float64(np.float32(g))
    V = dequant_independent(pools["vd"], pools["vs"]) * np.float64(np.float32(g))
    for b in range(w.batch):
        L = w.seq_lens[b]
        pages = bt[b, :(L + 15) // 16]
        for i in range(w.num_q_heads):
            h = i // w.group
            Kb = torch.from_numpy(K[pages, h].reshape(-1, 128)[:L])
            Vb = torch.from_numpy(V[pages, h].reshape(-1, 128)[:L])
            p = torch.softmax(Kb @ torch.from_numpy(q[b, i].astype(np.float64)) / np.sqrt(128), 0)
            np.testing.assert_allclose(got[b, i], (p @ Vb).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("g", [0.37, 3.1])
def test_prefix_with_global_scale(g):
    """Every (E2M1 code, E4M3 scale) pair at tensor scale G: torch's float8
    cast of fl32(G s e), saturated at 448."""
    cc, ss = np.meshgrid(np.arange(16, dtype=np.uint8), np.arange(0x7F, dtype=np.uint8), indexing="ij")
    cc, ss = cc.ravel(), ss.ravel()
    n = cc.size
    data = np.zeros((n, 1, 1, 64), np.uint8)
    scale = np.zeros((n, 1, 1, 8), np.uint8)
    data[:, 0, 0, 0] = cc
    scale[:, 0, 0, 0] = ss
    bt = np.arange(n, dtype=np.int32)[None, :]
    out = oracle.dequant_prefix_fp8(data, scale, bt, np.int32([n]), np.int32([0, n]), global_scale=g)
    got = out[:, 0, 0]
    e2 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    prod = e2[cc] * torch.from_numpy(ss.copy()).view(torch.float8_e4m3fn).double().numpy()
    v32 = (prod * np.float64(np.float32(g))).astype(np.float32)
    small = np.abs(v32) <= 448
    ref = torch.from_numpy(v32[small]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got[small], ref)
    np.testing.assert_array_equal(got[~small], np.where(v32[~small] > 0, 0x7E, 0xFE))


# --- per-head factors ------------------------------------------------------------
#
# Reading (the pages name one FP32 tensor scale and its calibration as the next
# step; a per-head refinement is this library's): kv head h of K (or V) uses
# G_h = fl32(G * g_h), with g_h its per-head factor.

HEADS = np.float32([0.5, 3.0, 1.0 / 7.0, 1.0])


def eff(g, factors):
    return (np.float32(g) * np.asarray(factors, np.float32)).astype(np.float32)


def test_per_head_blocks_match_brute_force():
    """Each head's blocks equal the brute force applied to fl32(x / G_h)."""
    rng = np.random.default_rng(8)
    T, Hkv = 37, 4
    x = (rng.standard_t(3, (T, Hkv, 128)) * rng.uniform(0.05, 20, (T, Hkv, 1))).astype(np.float32)
    data = np.zeros((4, Hkv, 16, 64), np.uint8)
    scale = np.zeros((4, Hkv, 16, 8), np.uint8)
    oracle.quantize_append(x, np.arange(T, dtype=np.int32), data, scale, global_scale=0.37, head_scales=HEADS)
    G = eff(0.37, HEADS)
    for h in range(Hkv):
        y = (x[:, h, :] / G[h]).astype(np.float32).reshape(-1, 16)
        codes_ref, S_ref = brute_force_block(y)
        got_codes = unpack(data[:, h].reshape(-1, 64)[:T].reshape(-1, 8))
        got_S = scale[:, h].reshape(-1, 8)[:T].reshape(-1)
        np.testing.assert_array_equal(got_S, S_ref)
        np.testing.assert_array_equal(got_codes, codes_ref)


def test_unit_head_factors_change_nothing():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((20, 4, 128)).astype(np.float32)
    pools = [np.zeros((2, 4, 16, n), np.uint8) for n in (64, 8, 64, 8)]
    oracle.quantize_append(x, np.arange(20, dtype=np.int32), pools[0], pools[1], global_scale=0.37)
    oracle.quantize_append(x, np.arange(20, dtype=np.int32), pools[2], pools[3], global_scale=0.37,
                           head_scales=np.ones(4, np.float32))
    np.testing.assert_array_equal(pools[0], pools[2])
    np.testing.assert_array_equal(pools[1], pools[3])


def test_decode_with_per_head_scales_matches_torch():
    """Attention with K of head h scaled by Gk_h and V by Gv_h: torch float64
    on rows dequantised independently and multiplied by those scales."""
    w = workloads.custom(2, 8, 4, (50, 33), seed=31)
    bt, num_pages = workloads.block_table(w, spare_pages=1)
    hk, hv = HEADS, HEADS[::-1].copy()
    pools = {n: np.zeros((num_pages, 4, 16, 64 if n.endswith("d") else 8), np.uint8) for n in ("kd", "ks", "vd", "vs")}
    for b in range(w.batch):
        L = w.seq_lens[b]
        sm = workloads.slot_mapping(w, bt, b, 0, L)
        oracle.quantize_append(workloads.kv_rows(w, "k", b, 0, L).numpy() * 4, sm, pools["kd"], pools["ks"],
                               global_scale=1.5, head_scales=hk)
        oracle.quantize_append(workloads.kv_rows(w, "v", b, 0, L).numpy(), sm, pools["vd"], pools["vs"],
                               global_scale=1.5, head_scales=hv)
    q = workloads.query(w).float().numpy()
    got = oracle.paged_decode(pools["kd"], pools["ks"], pools["vd"], pools["vs"], q, bt, np.int32(w.seq_lens),
                              global_scale=1.5, head_scales=np.stack([hk, hv]))
    K = dequant_independent(pools["kd"], pools["ks"]) * eff(1.5, hk).astype(np.float64)[None, :, None, None]
    V = dequant_independent(pools["vd"], pools["vs"]) * eff(1.5, hv).astype(np.float64)[None, :, None, None]
    for b in range(w.batch):
        L = w.seq_lens[b]
        pages = bt[b, :(L + 15) // 16]
        for i in range(w.num_q_heads):
            h = i // w.group
            Kb = torch.from_numpy(K[pages, h].reshape(-1, 128)[:L])
            Vb = torch.from_numpy(V[pages, h].reshape(-1, 128)[:L])
            p = torch.softmax(Kb @ torch.from_numpy(q[b, i].astype(np.float64)) / np.sqrt(128), 0)
            np.testing.assert_allclose(got[b, i], (p @ Vb).numpy(), rtol=1e-12, atol=1e-12)


def test_prefix_with_per_head_scales():
    """Every (code, scale) pair in each head at that head's scale: torch's
    float8 cast of fl32(G_h s e), saturated at 448."""
    cc, ss = np.meshgrid(np.arange(16, dtype=np.uint8), np.arange(0x7F, dtype=np.uint8), indexing="ij")
    cc, ss = cc.ravel(), ss.ravel()
    n, Hkv = cc.size, 4
    data = np.zeros((n, Hkv, 1, 64), np.uint8)
    scale = np.zeros((n, Hkv, 1, 8), np.uint8)
    data[:, :, 0, 0] = cc[:, None]
    scale[:, :, 0, 0] = ss[:, None]
    bt = np.arange(n, dtype=np.int32)[None, :]
    out = oracle.dequant_prefix_fp8(data, scale, bt, np.int32([n]), np.int32([0, n]), global_scale=0.37,
                                    head_scales=HEADS)
    e2 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    prod = e2[cc] * torch.from_numpy(ss.copy()).view(torch.float8_e4m3fn).double().numpy()
    G = eff(0.37, HEADS)
    for h in range(Hkv):
        v32 = (prod * np.float64(G[h])).astype(np.float32)
        small = np.abs(v32) <= 448
        got = out[:, h, 0]
        ref = torch.from_numpy(v32[small]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(got[small], ref)
        np.testing.assert_array_equal(got[~small], np.where(v32[~small] > 0, 0x7E, 0xFE))
