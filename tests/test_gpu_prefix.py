"""GPU parity of the extend path (dequant_prefix_fp8): bit-exact against the
oracle ("SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation:
the cached prefix is dequantised into one FP8 workspace)."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import workloads
from gpu_util import Built, oracle_full

pytestmark = pytest.mark.gpu


def run(b: Built, prefix_lens, indptr, rows):
    pl = torch.tensor(prefix_lens, dtype=torch.int32, device="cuda")
    ip = torch.tensor(indptr, dtype=torch.int32, device="cuda")
    kf = torch.full((rows, b.w.num_kv_heads, 128), 0xAB, dtype=torch.uint8, device="cuda")
    vf = torch.full_like(kf, 0xAB)
    nv.nvfp4kv_dequant_prefix_fp8(b.cache, b.bt_d, pl, ip, kf, vf, dev_status=b.status)
    torch.cuda.synchronize()
    return kf.cpu().numpy(), vf.cpu().numpy()


def expected(b: Built, prefix_lens, indptr, rows):
    _, pools = oracle_full(b)
    g = b.global_scale
    hs = b.head_scales
    k = oracle.dequant_prefix_fp8(pools[0], pools[1], b.bt, np.int32(prefix_lens), np.int32(indptr), rows,
                                  global_scale=g, head_scales=None if hs is None else hs[0])
    v = oracle.dequant_prefix_fp8(pools[2], pools[3], b.bt, np.int32(prefix_lens), np.int32(indptr), rows,
                                  global_scale=g, head_scales=None if hs is None else hs[1])
    return k, v


@pytest.mark.parametrize("g,hs", [(0.37, None), (3.1, None), (0.37, [[0.5, 3.0], [2.0, 0.125]])])
def test_prefix_with_tensor_scale(g, hs):
    """Workspace values E4M3(fl32(G_h s e)) for a tensor scale G != 1, and with
    per-head factors (G_h = fl32(G * factor) per kv head of K and V)."""
    w = workloads.custom(2, 8, 2, (301, 40), seed=29)
    b = Built(w, fp8=False, global_scale=g, head_scales=hs)
    lens = list(w.seq_lens)
    indptr = [3, 3 + lens[0]]
    rows = 3 + sum(lens) + 2
    got = run(b, lens, indptr, rows)
    want = expected(b, lens, indptr, rows)
    for gv, wv in zip(got, want):
        for s, L in zip(indptr, lens):
            np.testing.assert_array_equal(gv[s:s + L], wv[s:s + L])
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("name", ["tiny", "llama70b", "ctx32k", "ctx1m"])
def test_prefix_bit_exact(name):
    w = workloads.make(name, batch=2, seq_len=700) if name != "tiny" else workloads.make("tiny")
    b = Built(w, fp8=False)
    lens = list(w.seq_lens)
    lens[0] = max(0, lens[0] - 13)                      # a ragged prefix
    indptr = [5, 5 + lens[0]]
    rows = 5 + sum(lens) + 3
    got = run(b, lens, indptr, rows)
    want = expected(b, lens, indptr, rows)
    for g_, w_ in zip(got, want):
        written = np.zeros(rows, bool)
        for s, L in zip(indptr, lens):
            written[s:s + L] = True
        np.testing.assert_array_equal(g_[written], w_[written])
        assert (g_[~written] == 0xAB).all()               # nothing else touched
    assert int(b.status.item()) == 0


def test_prefix_many_units_per_cta():
    """More (sequence, page, kv head) units than CTAs, ragged lengths: each CTA
    steps through several units whose page and sequence digits carry."""
    lens = (3000, 17, 2999, 0, 1600)
    w = workloads.custom(len(lens), 16, 8, lens, seed=33)
    b = Built(w, fp8=False)
    plens = [max(0, L - 5) for L in lens]
    indptr = list(np.concatenate([[2], 2 + np.cumsum(plens)[:-1]]))
    rows = 2 + sum(plens) + 1
    got = run(b, plens, indptr, rows)
    want = expected(b, plens, indptr, rows)
    for g_, w_ in zip(got, want):
        for s, L in zip(indptr, plens):
            np.testing.assert_array_equal(g_[s:s + L], w_[s:s + L])
    assert int(b.status.item()) == 0


def test_prefix_160k_sampled():
    """One 160K-token prefix (the long-context extend workload) checked on
    sampled token ranges."""
    w = workloads.make("ctx160k", batch=1)
    b = Built(w, fp8=False, in_dtype=torch.bfloat16)
    L = w.seq_lens[0]
    kf, vf = run(b, [L], [0], L)
    rng = np.random.default_rng(0)
    for t0 in [0, L - 100] + list(rng.integers(0, L - 100, 3)):
        t1 = t0 + 100
        for which, got in (("k", kf), ("v", vf)):
            rows = workloads.kv_rows(w, which, 0, t0, t1, device="cuda").to(torch.bfloat16).float().cpu().numpy()
            data = np.zeros((100, w.num_kv_heads, 1, 64), np.uint8)
            sc = np.zeros((100, w.num_kv_heads, 1, 8), np.uint8)
            oracle.quantize_append(rows, np.arange(100, dtype=np.int32), data, sc, page_size=1)
            want = oracle.dequant_prefix_fp8(data, sc, np.arange(100, dtype=np.int32)[None, :],
                                             np.int32([100]), np.int32([0]), 100)
            np.testing.assert_array_equal(got[t0:t1], want)
