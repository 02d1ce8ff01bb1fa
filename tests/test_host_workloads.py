"""The decode workloads' input recipe, checked on the CPU: sizes and lengths,
page tables, slot arithmetic, chunked regeneration and the value
distributions each workload is described with."""
import numpy as np
import pytest
import torch

import workloads as W


@pytest.mark.parametrize("name,batches,hq,hkv,lo,hi", [
    ("tiny", (2,), 8, 2, 256, 256),
    ("llama70b", (12, 21), 64, 8, 8192, 8192),
    ("ctx32k", (44, 70), 48, 8, 24576, 32768),
    ("ctx160k", (10, 15), 48, 8, 163840, 163840),
    ("ctx1m", (1, 2), 48, 8, 1048576, 1048576),
])
def test_workload_geometry(name, batches, hq, hkv, lo, hi):
    for B in batches:
        w = W.make(name, batch=B)
        assert (w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size) == (B, hq, hkv, 128, 16)
        assert len(w.seq_lens) == B
        assert all(lo <= L <= hi for L in w.seq_lens)
        assert w.pages_per_seq == [(L + 15) // 16 for L in w.seq_lens]
        assert w.num_pages == sum(w.pages_per_seq)


def test_ctx32k_lengths_are_ragged_and_seeded():
    a = W.make("ctx32k", batch=70)
    b = W.make("ctx32k", batch=70)
    assert a.seq_lens == b.seq_lens
    assert len(set(a.seq_lens)) > 50          # uniform over 8,193 lengths: almost all distinct


@pytest.mark.parametrize("spare", [0, 5])
def test_block_table_is_a_partial_permutation(spare):
    w = W.make("ctx32k", batch=6, seq_len=300)
    bt, num_pages = W.block_table(w, pad_value=-1, spare_pages=spare)
    assert bt.shape == (6, w.max_pages) and bt.dtype == np.int32
    assert num_pages == w.num_pages + spare
    used = []
    for b, n in enumerate(w.pages_per_seq):
        used.extend(bt[b, :n].tolist())
        assert (bt[b, n:] == -1).all()
    assert len(used) == len(set(used)) == w.num_pages
    assert all(0 <= p < num_pages for p in used)
    # shuffled: not the identity hand-out
    assert used != list(range(w.num_pages))


def test_slot_mapping_is_page_times_size_plus_offset():
    w = W.make("tiny")
    bt, _ = W.block_table(w)
    s = W.slot_mapping(w, bt, 1, 10, 60)
    for t, slot in zip(range(10, 60), s):
        assert slot == bt[1, t // 16] * 16 + t % 16


def test_rows_regenerate_identically_across_chunk_boundaries():
    w = W.make("ctx160k", batch=1, seq_len=3 * W.CHUNK)
    whole = W.kv_rows(w, "k", 0, 0, 3 * W.CHUNK)
    a = W.kv_rows(w, "k", 0, W.CHUNK - 7, W.CHUNK + 9)
    assert torch.equal(a, whole[W.CHUNK - 7:W.CHUNK + 9])
    assert torch.equal(W.kv_rows(w, "k", 0, 5, 6), whole[5:6])
    # K and V differ, and so do two sequences
    w2 = W.make("ctx160k", batch=2, seq_len=W.CHUNK)
    assert not torch.equal(W.kv_rows(w2, "k", 0, 0, 64), W.kv_rows(w2, "v", 0, 0, 64))
    assert not torch.equal(W.kv_rows(w2, "k", 0, 0, 64), W.kv_rows(w2, "k", 1, 0, 64))


def _std_by_channel(x):
    return x.double().std(dim=0)               # [Hkv][d]


def test_normal_rows_are_standard_normal():
    w = W.make("ctx160k", batch=1, seq_len=W.CHUNK)
    x = W.kv_rows(w, "v", 0, 0, W.CHUNK)
    assert x.dtype == torch.float32 and x.shape == (W.CHUNK, 8, 128)
    assert abs(x.double().mean().item()) < 0.01
    assert abs(x.double().std().item() - 1.0) < 0.01


def test_llama_outlier_channels_are_ten_times_wider_and_shared_by_k_and_v():
    w = W.make("llama70b", batch=1, seq_len=W.CHUNK)
    sk = _std_by_channel(W.kv_rows(w, "k", 0, 0, W.CHUNK))
    sv = _std_by_channel(W.kv_rows(w, "v", 0, 0, W.CHUNK))
    for s in (sk, sv):
        wide = s > 5.0
        assert (wide.sum(dim=1) == 4).all()                    # 4 of 128 channels per kv head
        assert ((s[wide] - 10.0).abs() < 0.5).all()
        assert ((s[~wide] - 1.0).abs() < 0.1).all()
    assert torch.equal(sk > 5.0, sv > 5.0)                     # the same channels for K and V
    # different kv heads pick their channels independently
    picks = {tuple(torch.nonzero(sk[h] > 5.0).flatten().tolist()) for h in range(8)}
    assert len(picks) > 1


def test_ctx32k_head_factors_are_uniform_half_to_four_per_tensor_and_head():
    w = W.make("ctx32k", batch=1, seq_len=W.CHUNK)
    stds = []
    n = w.seq_lens[0]
    for which in ("k", "v"):
        x = W.kv_rows(w, which, 0, 0, n)
        s = x.double().std(dim=(0, 2))                                 # one factor per kv head
        stds.append(s)
        assert ((s > 0.5 * 0.97) & (s < 4.0 * 1.03)).all()
    assert not torch.allclose(stds[0], stds[1])                        # K and V drawn separately


def test_ctx1m_heavy_tailed_channels():
    w = W.make("ctx1m", batch=1, seq_len=W.CHUNK)
    x = W.kv_rows(w, "k", 0, 0, W.CHUNK).double()
    # excess kurtosis per channel: 0 for a normal, large for Student-t(3)
    c = x - x.mean(dim=0)
    kurt = (c ** 4).mean(dim=0) / (c ** 2).mean(dim=0) ** 2 - 3.0
    heavy = kurt > 2.0
    assert (heavy.sum(dim=1) == 4).all()                               # 4 of 128 per kv head
    assert (kurt[~heavy].abs() < 0.5).all()
    # t(3) has variance 3 (its sample variance scatters widely: no fourth moment)
    var = x.var(dim=0)[heavy]
    assert (var > 1.5).all() and 2.0 < var.median().item() < 4.5


def test_queries_are_bf16_standard_normal():
    w = W.make("llama70b", batch=21)
    q = W.query(w)
    assert q.dtype == torch.bfloat16 and q.shape == (21, 64, 128)
    qf = q.double()
    assert abs(qf.mean().item()) < 0.02 and abs(qf.std().item() - 1.0) < 0.02
    assert torch.equal(q, W.query(w))
