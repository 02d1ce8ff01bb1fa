"""GPU parity of the paged decode (NVFP4 and the FP8 comparison kernel) against
the oracle, elementwise within |d| <= 2e-3 + 1e-2 |ref|.

Decode: "SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation --
the decode path dequantises inside the attention kernel."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import workloads
from gpu_util import DEV, Built, assert_close, oracle_full, oracle_single_head

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fp8", [False, True])
def test_tiny_workload_all_outputs(fp8):
    b = Built(workloads.make("tiny"), spare_pages=0)
    want, _ = oracle_full(b, fp8=fp8)
    assert_close(b.decode(torch.float32, fp8=fp8), want, "fp32 out")
    assert_close(b.decode(torch.bfloat16, fp8=fp8), want, "bf16 out")
    assert int(b.status.item()) == 0


GEOMS = [
    # (Hq, Hkv, lengths)
    (8, 8, (1, 15, 16, 17)),
    (16, 8, (33, 0, 100)),
    (12, 4, (250, 1, 64)),
    (16, 4, (513, 77)),
    (48, 8, (300, 129, 16)),
    (64, 8, (200, 5)),
    (24, 3, (47, 1000)),
]


@pytest.mark.parametrize("hq,hkv,lens", GEOMS)
@pytest.mark.parametrize("num_workers", [0, 1, 7])
def test_geometries_and_worker_counts(hq, hkv, lens, num_workers):
    w = workloads.custom(len(lens), hq, hkv, lens, seed=hq * 31 + hkv)
    b = Built(w, garbage=True)
    want, _ = oracle_full(b)
    got = b.decode(torch.float32, num_workers=num_workers)
    assert_close(got, want, f"nvfp4 workers={num_workers}")
    got8 = b.decode(torch.float32, num_workers=num_workers, fp8=True)
    want8, _ = oracle_full(b, fp8=True)
    assert_close(got8, want8, f"fp8 workers={num_workers}")
    assert int(b.status.item()) == 0


def test_worker_count_invariance():
    """The split changes the result only through rounding: P is rounded to
    fp16 against a running maximum that depends on where a split starts.

    Tolerance: each weight p_j is rounded to fp16 (relative error e_j with
    |e_j| <= 2^-11) in both runs, so an output o = sum_j p_j v_j / sum_j p_j
    moves by sum_j p_j e_j (v_j - o) / sum_j p_j to first order.  With all
    errors of one sign that is 2^-11 times the weighted mean of |v_j - o|
    (about 0.8 for N(0,1) values), so two runs differ by at most ~8e-4; the
    rounding errors of independent weights mostly cancel, leaving a spread
    of about that bound divided by the square root of the effective number
    of keys (1e-4 or less for the 37- to 2000-token sequences here).  Hence
    atol 5e-4, plus rtol 5e-3 for the summation order of the fp32 sums."""
    w = workloads.custom(3, 32, 4, (2000, 37, 900), seed=3)
    b = Built(w)
    ref = b.decode(torch.float32, num_workers=1)
    for nw in (2, 5, 64, 333, 0):
        np.testing.assert_allclose(b.decode(torch.float32, num_workers=nw), ref, rtol=5e-3, atol=5e-4)


@pytest.mark.parametrize("g", [0.37, 3.1])
def test_tensor_scale(g):
    """Decode over a cache with tensor scale G (values G * s * e): the query
    scale and the normaliser carry G."""
    w = workloads.custom(3, 16, 4, (300, 17, 1000), seed=23)
    b = Built(w, fp8=False, global_scale=g, garbage=True)
    want, _ = oracle_full(b)
    assert_close(b.decode(torch.float32), want, f"nvfp4 G={g}")
    assert_close(b.decode(torch.float32, num_workers=7), want, f"nvfp4 G={g} 7 workers")
    assert int(b.status.item()) == 0


PER_HEAD = [[0.5, 3.0, 1.0 / 7.0, 1.0], [2.0, 0.3, 1.0, 9.5]]     # [K, V][kv head]


def test_per_head_scales():
    """Decode over a cache whose kv heads carry their own K and V tensor
    scales: each head's query scale and normaliser carry them (owned and split
    segments, several worker counts)."""
    w = workloads.custom(3, 16, 4, (300, 17, 1000), seed=27)
    b = Built(w, fp8=False, global_scale=0.37, head_scales=PER_HEAD, garbage=True)
    want, _ = oracle_full(b)
    for nw in (0, 7, 333):
        assert_close(b.decode(torch.float32, num_workers=nw), want, f"per-head scales, {nw} workers")
    assert int(b.status.item()) == 0


def test_more_workers_than_page_heads():
    """One long sequence among many short ones: the automatic worker count,
    bounded by the largest batch the block table allows, and an explicit one
    both exceed the number of page-heads, so the split must leave no worker
    between two contributors of a segment without a range."""
    lens = (3000,) + tuple(range(1, 24))
    w = workloads.custom(len(lens), 16, 4, lens, seed=11)
    b = Built(w, garbage=True)
    want, _ = oracle_full(b)
    want8, _ = oracle_full(b, fp8=True)
    for nw in (0, 2000):
        assert_close(b.decode(torch.float32, num_workers=nw), want, f"nvfp4 workers={nw}")
        assert_close(b.decode(torch.float32, num_workers=nw, fp8=True), want8, f"fp8 workers={nw}")
    assert int(b.status.item()) == 0


def test_bad_page_and_length_are_reported_not_faulted():
    w = workloads.custom(2, 8, 2, (40, 40), seed=5)
    b = Built(w)
    bt = b.bt.copy()
    bt[1, 1] = b.num_pages + 7
    b.bt_d = torch.from_numpy(bt).to("cuda")
    out = b.decode(torch.float32)
    assert int(b.status.item()) & nv.DEV_BAD_PAGE
    assert np.isfinite(out[0]).all()
    b.status.zero_()
    b.bt_d = torch.from_numpy(b.bt).to("cuda")
    b.sl_d = torch.tensor([40, 10 ** 6], dtype=torch.int32, device="cuda")
    b.decode(torch.float32)
    assert int(b.status.item()) & nv.DEV_BAD_LEN
    # the same word through the C call that reads it
    assert nv.read_device_status(b.status) == int(b.status.item())
    b.status.zero_()
    assert nv.read_device_status(b.status) == 0


@pytest.mark.parametrize("name,batch", [("llama70b", 12), ("llama70b", 21)])
def test_llama70b_layer_sampled(name, batch):
    """Full-size Llama-3.3-70B-shaped layer (Hq=64, Hkv=8, 8192 tokens), as
    the bench launches it; oracle on sampled (sequence, kv head) pairs."""
    w = workloads.make(name, batch=batch)
    b = Built(w, spare_pages=0)
    got = b.decode(torch.bfloat16)
    got8 = b.decode(torch.bfloat16, fp8=True)
    rng = np.random.default_rng(batch)
    for seq, h in [(0, 0), (batch - 1, 7)] + [tuple(x) for x in rng.integers([0, 0], [batch, 8], (2, 2))]:
        g = w.group
        want = oracle_single_head(b, seq, h)
        assert_close(got[seq, h * g:(h + 1) * g], want, f"nvfp4 seq {seq} kv head {h}")
        want8 = oracle_single_head(b, seq, h, fp8=True)
        assert_close(got8[seq, h * g:(h + 1) * g], want8, f"fp8 seq {seq} kv head {h}")
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("name,batch,fp8", [("ctx32k", 44, True), ("ctx160k", 10, False), ("ctx1m", 1, True),
                                            ("ctx32k", 70, False), ("ctx160k", 15, False), ("ctx1m", 2, False)])
def test_long_context_sampled(name, batch, fp8):
    """Each long-context workload at both batch sizes the bench reports (the
    FP8-capacity and the NVFP4-capacity batch), as the bench launches it;
    oracle on sampled (sequence, kv head) pairs."""
    w = workloads.make(name, batch=batch)
    b = Built(w, spare_pages=0, fp8=fp8)
    got = b.decode(torch.bfloat16)
    got8 = b.decode(torch.bfloat16, fp8=True) if b.fp8 is not None else None
    for seq, h in [(0, 3), (batch - 1, 6)]:
        g = w.group
        assert_close(got[seq, h * g:(h + 1) * g], oracle_single_head(b, seq, h), f"{name} seq {seq} h {h}")
        if got8 is not None:
            assert_close(got8[seq, h * g:(h + 1) * g], oracle_single_head(b, seq, h, fp8=True),
                         f"{name} fp8 seq {seq} h {h}")
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("lens", [(37, 16, 1, 300, 0), (8192, 8191, 8177)])
def test_append_decode_equals_append_then_decode(fp8, lens, g=1.0, hs=None):
    """The fused step writes exactly the bytes quantize_append would and then
    decodes exactly as paged_decode does."""
    w = workloads.custom(len(lens), 32, 4, lens, seed=21)
    full = Built(w, global_scale=g, head_scales=hs)     # all tokens appended by quantize_append
    cache = (nv.FP8Cache.allocate(full.num_pages, w.num_kv_heads, device="cuda") if fp8 else
             nv.NVFP4Cache.allocate(full.num_pages, w.num_kv_heads, device="cuda", global_scale=g, head_scales=hs))
    app = nv.fp8kv_quantize_append if fp8 else nv.nvfp4kv_quantize_append
    k_new = torch.zeros((w.batch, w.num_kv_heads, 128), dtype=torch.float32, device="cuda")
    v_new = torch.zeros_like(k_new)
    for b, L in enumerate(w.seq_lens):
        if L == 0:
            continue
        if L > 1:
            sm = torch.from_numpy(workloads.slot_mapping(w, full.bt, b, 0, L - 1)).cuda()
            app(cache, workloads.kv_rows(w, "k", b, 0, L - 1, device="cuda"),
                workloads.kv_rows(w, "v", b, 0, L - 1, device="cuda"), sm)
        k_new[b] = workloads.kv_rows(w, "k", b, L - 1, L, device="cuda")[0]
        v_new[b] = workloads.kv_rows(w, "v", b, L - 1, L, device="cuda")[0]
    out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = nv.new_workspace(device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = nv.fp8kv_append_paged_decode if fp8 else nv.nvfp4kv_append_paged_decode
    step(cache, k_new, v_new, full.q, full.bt_d, full.sl_d, out, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_pool = (full.fp8 if fp8 else full.cache).pool
    np.testing.assert_array_equal(cache.pool.cpu().numpy(), ref_pool.cpu().numpy())
    np.testing.assert_array_equal(out.cpu().numpy(), full.decode(torch.float32, fp8=fp8))
    want, _ = oracle_full(full, fp8=fp8)
    assert_close(out.cpu().numpy(), want, "fused append + decode")


@pytest.mark.parametrize("name,batch", [("llama70b", 12), ("ctx160k", 15), ("ctx1m", 2)])
def test_fused_step_full_size_sampled(name, batch):
    """The step the bench times -- append_paged_decode at the full workload
    size with the automatic worker count: the cache holds seq_len - 1 tokens,
    the call writes token seq_len - 1 of every sequence and attends over all of
    them.  The written pool equals quantize_append's byte for byte, and sampled
    (sequence, kv head) outputs equal the oracle's decode over all tokens."""
    w = workloads.make(name, batch=batch)
    full = Built(w, spare_pages=0, fp8=False)            # every token through quantize_append
    cache = nv.NVFP4Cache.allocate(full.num_pages, w.num_kv_heads, device=DEV)
    k_new = torch.zeros((w.batch, w.num_kv_heads, 128), dtype=torch.bfloat16, device=DEV)
    v_new = torch.zeros_like(k_new)
    for b_, L in enumerate(w.seq_lens):
        for t0 in range(0, L - 1, workloads.CHUNK):
            t1 = min(L - 1, t0 + workloads.CHUNK)
            sm = torch.from_numpy(workloads.slot_mapping(w, full.bt, b_, t0, t1)).to(DEV)
            nv.nvfp4kv_quantize_append(cache, workloads.kv_rows(w, "k", b_, t0, t1, device=DEV),
                                       workloads.kv_rows(w, "v", b_, t0, t1, device=DEV), sm)
        k_new[b_] = workloads.kv_rows(w, "k", b_, L - 1, L, device=DEV)[0].to(torch.bfloat16)
        v_new[b_] = workloads.kv_rows(w, "v", b_, L - 1, L, device=DEV)[0].to(torch.bfloat16)
    # the bf16 rows are what both sides quantise: rebuild the reference's last token from them
    for b_, L in enumerate(w.seq_lens):
        sm = torch.from_numpy(workloads.slot_mapping(w, full.bt, b_, L - 1, L)).to(DEV)
        nv.nvfp4kv_quantize_append(full.cache, k_new[b_:b_ + 1].contiguous(), v_new[b_:b_ + 1].contiguous(), sm)
        full.rows[(b_, "last")] = (k_new[b_:b_ + 1].float().cpu().numpy(), v_new[b_:b_ + 1].float().cpu().numpy())
    out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = nv.new_workspace(device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    nv.nvfp4kv_append_paged_decode(cache, k_new, v_new, full.q, full.bt_d, full.sl_d, out, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(cache.pool, full.cache.pool), "fused write differs from quantize_append"
    got = out.float().cpu().numpy()
    g = w.group
    rng = np.random.default_rng(batch + 5)
    for seq, h in [(0, 0), (batch - 1, w.num_kv_heads - 1)] + [tuple(x) for x in rng.integers(
            [0, 0], [batch, w.num_kv_heads], (2, 2))]:
        L = w.seq_lens[seq]
        k = np.concatenate([full.rows_of(seq, "k", h)[:L - 1], full.rows[(seq, "last")][0][:, h:h + 1]], 0)
        v = np.concatenate([full.rows_of(seq, "v", h)[:L - 1], full.rows[(seq, "last")][1][:, h:h + 1]], 0)
        npg = (L + 15) // 16
        pools = [np.zeros((npg, 1, 16, s_), np.uint8) for s_ in (64, 8, 64, 8)]
        sm = np.arange(L, dtype=np.int32)
        oracle.quantize_append(k, sm, pools[0], pools[1])
        oracle.quantize_append(v, sm, pools[2], pools[3])
        q = full.q[seq:seq + 1, h * g:(h + 1) * g].float().cpu().numpy()
        want = oracle.paged_decode(*pools, q, np.arange(npg, dtype=np.int32)[None, :], np.int32([L]))[0]
        assert_close(got[seq, h * g:(h + 1) * g], want, f"{name} fused step seq {seq} kv head {h}")


def test_append_decode_with_tensor_scale():
    test_append_decode_equals_append_then_decode(False, (40, 1, 300), g=0.37)


def test_append_decode_with_per_head_scales():
    test_append_decode_equals_append_then_decode(False, (40, 1, 300), g=0.37, hs=PER_HEAD)


def test_multi_query_per_head_scales():
    """Multi-query decode (q_len 3, group 4) with per-head K and V scales."""
    w = workloads.custom(2, 16, 4, (129, 700), seed=41)
    b = Built(w, fp8=False, global_scale=1.5, head_scales=PER_HEAD)
    q_len = 3
    rng = np.random.default_rng(8)
    q = torch.from_numpy(rng.standard_normal((w.batch, q_len, 16, 128)).astype(np.float32)).to(torch.bfloat16)
    _, pools = oracle_full(b)
    ref = np.zeros((w.batch, q_len, 16, 128))
    for t in range(q_len):
        lt = np.maximum(np.int32(w.seq_lens) - q_len + t + 1, 0).astype(np.int32)
        ref[:, t] = oracle.paged_decode(*pools, q[:, t].float().numpy(), b.bt, lt, global_scale=1.5,
                                        head_scales=PER_HEAD)
    out = torch.full((w.batch, q_len, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = nv.new_workspace(device="cuda")
    nv.nvfp4kv_paged_decode_multi(b.cache, q.cuda(), b.bt_d, b.sl_d, out, ws, dev_status=b.status)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, "multi-query, per-head scales")
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("hq,hkv,q_len,lens", [
    (64, 8, 2, (300, 17, 1000)),      # group 8: two row groups per kv head
    (16, 4, 2, (129, 64)),            # group 4: both tokens in one row group
    (48, 8, 3, (500, 3, 2)),          # group 6, 18 rows; a sequence shorter than q_len
    (8, 8, 8, (40, 1000)),            # group 1, 8 tokens
])
def test_multi_query_decode(hq, hkv, q_len, lens):
    """Several query tokens per sequence at its last q_len positions, causal:
    token t attends over the first L - q_len + t + 1 tokens, i.e. the oracle's
    single-token decode at that length."""
    w = workloads.custom(len(lens), hq, hkv, lens, seed=31 + q_len)
    b = Built(w, fp8=False, garbage=True)
    rng = np.random.default_rng(7)
    q = torch.from_numpy(rng.standard_normal((w.batch, q_len, hq, 128)).astype(np.float32)).to(torch.bfloat16)
    want, pools = oracle_full(b)
    ref = np.zeros((w.batch, q_len, hq, 128))
    for t in range(q_len):
        lt = np.maximum(np.int32(w.seq_lens) - q_len + t + 1, 0).astype(np.int32)
        ref[:, t] = oracle.paged_decode(*pools, q[:, t].float().numpy(), b.bt, lt)
    for nw in (0, 7):
        out = torch.full((w.batch, q_len, hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        ws = nv.new_workspace(nw, device="cuda")
        ws.fill_(0xFF)
        nv.nvfp4kv_paged_decode_multi(b.cache, q.cuda(), b.bt_d, b.sl_d, out, ws, num_workers=nw,
                                      dev_status=b.status)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref, f"multi-query q_len={q_len} workers={nw}")
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("where", ["start", "middle", "end"])
@pytest.mark.parametrize("fp8", [False, True])
def test_score_spread_across_a_split_segment(where, fp8):
    """Keys whose scores stand ~370 (log2 units) above the others, in one
    stretch of each long segment: the split-KV partials of one segment then
    carry maxima hundreds apart, and the merge must weight them by the
    log-sum-exp rule without overflow or loss (workers 0, 1 and 3 put the
    stretch at the start, middle or end of a worker's range, or in a segment
    one worker covers).  The result is the oracle's softmax, which is all but
    entirely that stretch's mean of V."""
    lens = (3000, 4100)
    hq, hkv = 16, 2
    rng = np.random.default_rng(11)
    nb = len(lens)
    bt = np.full((nb, max((L + 15) // 16 for L in lens)), -1, np.int32)
    perm = rng.permutation(sum((L + 15) // 16 for L in lens)).astype(np.int32)
    off = 0
    for i, L in enumerate(lens):
        n = (L + 15) // 16
        bt[i, :n] = perm[off:off + n]
        off += n
    num_pages = off
    q = torch.ones((nb, hq, 128), dtype=torch.bfloat16)
    sm_scale = 0.5
    if fp8:
        cache = nv.FP8Cache.allocate(num_pages, hkv, device=DEV)
        kc = np.zeros((num_pages, hkv, 16, 128), np.uint8)
        vc = np.zeros_like(kc)
    else:
        cache = nv.NVFP4Cache.allocate(num_pages, hkv, device=DEV)
        pools = [np.zeros((num_pages, hkv, 16, s), np.uint8) for s in (64, 8, 64, 8)]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for i, L in enumerate(lens):
        k = rng.standard_normal((L, hkv, 128)).astype(np.float32)
        v = rng.standard_normal((L, hkv, 128)).astype(np.float32)
        a = {"start": 20, "middle": L // 2, "end": L - 200}[where]
        k[a:a + 100] = 4.0
        sm = (bt[i, np.arange(L) // 16].astype(np.int64) * 16 + np.arange(L) % 16).astype(np.int32)
        args = (torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV), torch.from_numpy(sm).to(DEV), status)
        if fp8:
            nv.fp8kv_quantize_append(cache, *args)
            oracle.fp8_quantize_append(k, sm, kc)
            oracle.fp8_quantize_append(v, sm, vc)
        else:
            nv.nvfp4kv_quantize_append(cache, *args)
            oracle.quantize_append(k, sm, pools[0], pools[1])
            oracle.quantize_append(v, sm, pools[2], pools[3])
    sl = np.int32(lens)
    if fp8:
        want = oracle.fp8_paged_decode(kc, vc, q.float().numpy(), bt, sl, sm_scale=sm_scale)
    else:
        want = oracle.paged_decode(*pools, q.float().numpy(), bt, sl, sm_scale=sm_scale)
    fn = nv.fp8kv_paged_decode if fp8 else nv.nvfp4kv_paged_decode
    for nw in (0, 1, 3):
        out = torch.full((nb, hq, 128), float("nan"), dtype=torch.float32, device=DEV)
        ws = nv.new_workspace(nw, device=DEV)
        ws.fill_(0xFF)
        fn(cache, q.to(DEV), torch.from_numpy(bt).to(DEV), torch.from_numpy(sl).to(DEV), out, ws,
           sm_scale=sm_scale, num_workers=nw, dev_status=status)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), want, f"score spread at the {where}, workers={nw}")
    assert int(status.item()) == 0
