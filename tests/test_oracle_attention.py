"""Pins of the oracle's paged decode, prefix dequant and FP8 paths (CPU only).

Decode attention ("SGLang stores KV cache in 4 bits" (LMSYS summary),
Interpretation: the decode kernel dequantises inside attention): for query
head i of sequence b and kv head h = i // g, o = softmax(q . k_j / sqrt(d)) V
over the L_b cached tokens gathered through the page table.  Checked against
closed forms, library routines (torch float64 softmax/matmul on tensors
dequantised independently here) and metamorphic relations.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

E2 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def dequant_independent(data, scale):
    """NVFP4 rows -> float64 using numpy nibbles and torch's E4M3 decode."""
    codes = np.stack([data & 15, data >> 4], -1).reshape(*data.shape[:-1], -1)
    s = torch.from_numpy(np.ascontiguousarray(scale)).view(torch.float8_e4m3fn).double().numpy()
    return E2[codes] * np.repeat(s, 16, -1)


def build_cache(w, rng_seed=0, spare=3):
    bt, num_pages = workloads.block_table(w, spare_pages=spare)
    Hkv, P, d = w.num_kv_heads, w.page_size, w.head_dim
    pools = {n: np.zeros((num_pages, Hkv, P, d // 2 if "data" in n else d // 16), np.uint8)
             for n in ("k_data", "k_scale", "v_data", "v_scale")}
    for b in range(w.batch):
        L = w.seq_lens[b]
        if L == 0:
            continue
        sm = workloads.slot_mapping(w, bt, b, 0, L)
        k = workloads.kv_rows(w, "k", b, 0, L).numpy()
        v = workloads.kv_rows(w, "v", b, 0, L).numpy()
        oracle.quantize_append(k, sm, pools["k_data"], pools["k_scale"], P)
        oracle.quantize_append(v, sm, pools["v_data"], pools["v_scale"], P)
    return pools, bt


def torch_reference(pools, bt, w, q):
    """float64 softmax attention per (b, i) with torch library routines."""
    K = dequant_independent(pools["k_data"], pools["k_scale"])   # [pages][Hkv][P][d]
    V = dequant_independent(pools["v_data"], pools["v_scale"])
    g = w.group
    out = np.zeros((w.batch, w.num_q_heads, w.head_dim))
    for b in range(w.batch):
        L = w.seq_lens[b]
        if L == 0:
            continue
        pages = bt[b, :(L + w.page_size - 1) // w.page_size]
        for i in range(w.num_q_heads):
            h = i // g
            Kb = torch.from_numpy(K[pages, h].reshape(-1, w.head_dim)[:L])
            Vb = torch.from_numpy(V[pages, h].reshape(-1, w.head_dim)[:L])
            qi = torch.from_numpy(q[b, i].astype(np.float64))
            p = torch.softmax(Kb @ qi / np.sqrt(w.head_dim), 0)
            out[b, i] = (p @ Vb).numpy()
    return out


def run_oracle(pools, bt, w, q):
    return oracle.paged_decode(pools["k_data"], pools["k_scale"], pools["v_data"],
                               pools["v_scale"], q, bt, np.int32(w.seq_lens))


@pytest.mark.parametrize("lens", [(256, 256), (1, 17, 40), (5, 0, 33)])
def test_decode_matches_torch_float64(lens):
    w = workloads.custom(len(lens), 6, 2, lens, seed=11)
    pools, bt = build_cache(w)
    q = workloads.query(w).float().numpy()
    got = run_oracle(pools, bt, w, q)
    want = torch_reference(pools, bt, w, q)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_tiny_workload_matches_torch_float64():
    w = workloads.make("tiny")
    pools, bt = build_cache(w, spare=0)
    q = workloads.query(w).float().numpy()
    np.testing.assert_allclose(run_oracle(pools, bt, w, q), torch_reference(pools, bt, w, q),
                               rtol=1e-12, atol=1e-12)


def test_equal_keys_give_mean_of_values():
    w = workloads.custom(1, 4, 1, (45,), seed=3)
    pools, bt = build_cache(w)
    pools["k_data"][:] = pools["k_data"][0:1, :, 0:1]          # every key row identical
    pools["k_scale"][:] = pools["k_scale"][0:1, :, 0:1]
    q = workloads.query(w).float().numpy()
    got = run_oracle(pools, bt, w, q)
    V = dequant_independent(pools["v_data"], pools["v_scale"])
    pages = bt[0, :3]
    mean = V[pages, 0].reshape(-1, 128)[:45].mean(0)
    for i in range(4):
        np.testing.assert_allclose(got[0, i], mean, rtol=1e-13, atol=1e-13)


def test_single_token_returns_its_value_row():
    w = workloads.custom(2, 4, 2, (1, 1), seed=4)
    pools, bt = build_cache(w)
    q = workloads.query(w).float().numpy()
    got = run_oracle(pools, bt, w, q)
    V = dequant_independent(pools["v_data"], pools["v_scale"])
    for b in range(2):
        for i in range(4):
            np.testing.assert_array_equal(got[b, i], V[bt[b, 0], i // 2, 0])


def test_gqa_head_mapping():
    """Query head i reads kv head i // g: equals a g=1 problem on that head."""
    w = workloads.custom(1, 8, 2, (70,), seed=5)
    pools, bt = build_cache(w)
    q = workloads.query(w).float().numpy()
    got = run_oracle(pools, bt, w, q)
    for i in range(8):
        h = i // 4
        single = {k: np.ascontiguousarray(v[:, h:h + 1]) for k, v in pools.items()}
        one = oracle.paged_decode(single["k_data"], single["k_scale"], single["v_data"],
                                  single["v_scale"], q[:, i:i + 1], bt, np.int32([70]))
        np.testing.assert_array_equal(got[0, i], one[0, 0])


def test_page_permutation_is_invisible():
    """Moving pages to other physical slots and updating the table changes nothing."""
    w = workloads.custom(2, 4, 2, (50, 33), seed=6)
    pools, bt = build_cache(w, spare=4)
    q = workloads.query(w).float().numpy()
    base = run_oracle(pools, bt, w, q)
    rng = np.random.default_rng(0)
    perm = rng.permutation(pools["k_data"].shape[0])
    moved = {k: np.empty_like(v) for k, v in pools.items()}
    for k in pools:
        moved[k][perm] = pools[k]
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    np.testing.assert_array_equal(run_oracle(moved, bt2, w, q), base)


def test_softmax_shift_invariance_and_scale():
    """Adding a constant to every score leaves o unchanged; sm_scale=0 gives mean V."""
    w = workloads.custom(1, 2, 1, (30,), seed=8)
    pools, bt = build_cache(w)
    q = workloads.query(w).float().numpy()
    flat = oracle.paged_decode(pools["k_data"], pools["k_scale"], pools["v_data"],
                               pools["v_scale"], q, bt, np.int32([30]), sm_scale=0.0)
    V = dequant_independent(pools["v_data"], pools["v_scale"])
    mean = V[bt[0, :2], 0].reshape(-1, 128)[:30].mean(0)
    np.testing.assert_allclose(flat[0, 0], mean, rtol=1e-13, atol=1e-13)


def test_empty_sequence_gives_zeros():
    w = workloads.custom(2, 2, 1, (0, 20), seed=9)
    pools, bt = build_cache(w)
    q = workloads.query(w).float().numpy()
    got = run_oracle(pools, bt, w, q)
    assert (got[0] == 0).all() and np.abs(got[1]).sum() > 0


def test_table_entries_past_a_sequence_are_never_read():
    """Only the first ceil(L_b / 16) block-table entries of a sequence take part:
    rewriting the rest (padding -1 or any page id) changes neither the decode
    nor the prefix dequant."""
    w = workloads.custom(5, 16, 4, (0, 1, 15, 17, 1000), seed=4)
    pools, bt = build_cache(w)
    q = workloads.query(w).float().numpy()
    bt_pad = bt.copy()
    for b, n in enumerate(w.pages_per_seq):
        bt_pad[b, n:] = -1
    bt_other = bt.copy()
    for b, n in enumerate(w.pages_per_seq):
        bt_other[b, n:] = (np.arange(bt.shape[1] - n) * 7 + b) % bt.max()
    a = run_oracle(pools, bt_pad, w, q)
    c = run_oracle(pools, bt_other, w, q)
    assert np.array_equal(a, c) and (a[0] == 0).all() and np.isfinite(a).all()
    lens = np.int32(w.seq_lens)
    ip = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32)
    for n in ("k", "v"):
        x = oracle.dequant_prefix_fp8(pools[n + "_data"], pools[n + "_scale"], bt_pad, lens, ip,
                                      out_rows=int(lens.sum()))
        y = oracle.dequant_prefix_fp8(pools[n + "_data"], pools[n + "_scale"], bt_other, lens, ip,
                                      out_rows=int(lens.sum()))
        assert np.array_equal(x, y)


# --- extend path: prefix -> FP8 workspace ------------------------------------

def test_prefix_value_map_exhaustive():
    """Every (E2M1 code, E4M3 scale) pair: E4M3_RNE_sat(value x scale), checked
    against torch's float8 cast (a library routine) below 448 and saturation
    above."""
    cc, ss = np.meshgrid(np.arange(16, dtype=np.uint8), np.arange(0x7F, dtype=np.uint8),
                         indexing="ij")
    cc, ss = cc.ravel(), ss.ravel()
    n = cc.size
    # each (code, scale) pair is element 0 of its own cached row
    data = np.zeros((n, 1, 1, 64), np.uint8)
    scale = np.zeros((n, 1, 1, 8), np.uint8)
    data[:, 0, 0, 0] = cc
    scale[:, 0, 0, 0] = ss
    bt = np.arange(n, dtype=np.int32)[None, :]
    out = oracle.dequant_prefix_fp8(data, scale, bt, np.int32([n]), np.int32([0, n]))
    got = out[:, 0, 0]
    prod = E2[cc] * torch.from_numpy(ss.copy()).view(torch.float8_e4m3fn).double().numpy()
    small = np.abs(prod) <= 448
    ref = torch.from_numpy(prod[small].astype(np.float32)).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(got[small], ref.view(torch.uint8).numpy())
    big = ~small
    assert big.any()
    np.testing.assert_array_equal(got[big], np.where(prod[big] > 0, 0x7E, 0xFE))


def test_prefix_layout_follows_indptr():
    w = workloads.custom(3, 4, 2, (40, 0, 19), seed=12)
    pools, bt = build_cache(w)
    indptr = np.int32([5, 45, 45, 64])       # rows start at 5; seq 1 empty
    out = oracle.dequant_prefix_fp8(pools["k_data"], pools["k_scale"], bt,
                                    np.int32(w.seq_lens), indptr, out_rows=70)
    K = dequant_independent(pools["k_data"], pools["k_scale"])
    assert (out[:5] == 0).all() and (out[64:] == 0).all()
    for b in (0, 2):
        L = w.seq_lens[b]
        pages = bt[b, :(L + 15) // 16]
        for h in range(2):
            vals = K[pages, h].reshape(-1, 128)[:L]
            ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn)
            ref = ref.view(torch.uint8).numpy()
            ok = np.abs(vals) <= 448
            got = out[indptr[b]:indptr[b] + L, h]
            np.testing.assert_array_equal(got[ok], ref[ok])


# --- FP8 comparison cache ------------------------------------------------------

def test_fp8_append_and_decode():
    w = workloads.custom(2, 4, 2, (37, 64), seed=13)
    bt, num_pages = workloads.block_table(w, spare_pages=2)
    kc = np.zeros((num_pages, 2, 16, 128), np.uint8)
    vc = np.zeros_like(kc)
    for b in range(2):
        L = w.seq_lens[b]
        sm = workloads.slot_mapping(w, bt, b, 0, L)
        k = workloads.kv_rows(w, "k", b, 0, L).numpy()
        v = workloads.kv_rows(w, "v", b, 0, L).numpy()
        oracle.fp8_quantize_append(k, sm, kc)
        oracle.fp8_quantize_append(v, sm, vc)
        ref = torch.from_numpy(k).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        j = np.arange(L)
        np.testing.assert_array_equal(kc[bt[b, j // 16], :, j % 16], ref)
    q = workloads.query(w).float().numpy()
    got = oracle.fp8_paged_decode(kc, vc, q, bt, np.int32(w.seq_lens))
    K = torch.from_numpy(kc).view(torch.float8_e4m3fn).double()
    V = torch.from_numpy(vc).view(torch.float8_e4m3fn).double()
    for b in range(2):
        L = w.seq_lens[b]
        pages = torch.from_numpy(bt[b, :(L + 15) // 16].astype(np.int64))
        for i in range(4):
            Kb = K[pages, i // 2].reshape(-1, 128)[:L]
            Vb = V[pages, i // 2].reshape(-1, 128)[:L]
            p = torch.softmax(Kb @ torch.from_numpy(q[b, i]).double() / np.sqrt(128), 0)
            np.testing.assert_allclose(got[b, i], (p @ Vb).numpy(), rtol=1e-12, atol=1e-12)
