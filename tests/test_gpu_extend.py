"""GPU parity of the extend attention against the oracle.

"SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation: the
extend path attends each chunk token over its sequence's FP8 prefix workspace
and the chunk up to itself.  Inputs come from workloads.extend_inputs; the
oracle runs in fp64 on the same bytes.
"""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import workloads
from gpu_util import DEV, assert_close

pytestmark = pytest.mark.gpu


def to_dev(x):
    return {k: v.to(DEV) for k, v in x.items()}


def oracle_out(e, x):
    return oracle.extend_attention(x["q"].float().numpy(), x["q_indptr"].numpy(), x["k_prefix"].numpy(),
                                   x["v_prefix"].numpy(), x["kv_indptr"].numpy(), x["prefix_lens"].numpy(),
                                   x["k_chunk"].float().numpy(), x["v_chunk"].float().numpy())


def run(e, xd, out_dtype=torch.float32, max_q_len=None, status=None, out=None):
    if out is None:
        out = torch.full((e.q_rows, e.num_q_heads, e.head_dim), float("nan"), dtype=out_dtype, device=DEV)
    nv.nvfp4kv_extend_attention_fp8(xd["q"], xd["q_indptr"], xd["k_prefix"], xd["v_prefix"], xd["kv_indptr"],
                                    xd["prefix_lens"], xd["k_chunk"], xd["v_chunk"], out,
                                    max_q_len=max(e.chunk_lens) if max_q_len is None else max_q_len,
                                    dev_status=status)
    torch.cuda.synchronize()
    return out


CASES = [
    # (prefix_lens, chunk_lens, Hq, Hkv): ragged prefixes across 64-key tiles,
    # chunks across 128-row tiles, groups 1, 3, 6 and 8
    ((0, 61, 200, 1000), (130, 1, 77, 64), 48, 8),
    ((64, 65), (128, 129), 8, 8),
    ((300,), (257,), 24, 8),
    ((0,), (300,), 8, 1),
    ((5, 0, 127), (0, 16, 40), 16, 2),
]


@pytest.mark.parametrize("prefix_lens,chunk_lens,hq,hkv", CASES)
def test_extend_matches_oracle(prefix_lens, chunk_lens, hq, hkv):
    e = workloads.extend_custom(prefix_lens, chunk_lens, hq, hkv, seed=len(prefix_lens) + hq)
    x = workloads.extend_inputs(e)
    want = oracle_out(e, x)
    got = run(e, to_dev(x)).cpu().numpy()
    assert_close(got, want, "extend fp32 out")


def test_extend_bf16_output():
    e = workloads.extend_make("ext_small")
    x = workloads.extend_inputs(e)
    want = oracle_out(e, x)
    got = run(e, to_dev(x), out_dtype=torch.bfloat16).float().cpu().numpy()
    assert_close(got, want, "extend bf16 out")


def test_extend_leaves_rows_outside_the_chunks_untouched():
    """Rows before q_indptr[0] and from q_indptr[batch] on keep their contents."""
    e = workloads.extend_custom((40, 70), (20, 30), 16, 2, seed=5)
    x = workloads.extend_inputs(e)
    want = oracle_out(e, x)
    xd = to_dev(x)
    lead, tail = 5, 4
    pad = lambda t: torch.cat([torch.zeros((lead,) + t.shape[1:], dtype=t.dtype, device=DEV), t,
                               torch.zeros((tail,) + t.shape[1:], dtype=t.dtype, device=DEV)])
    for k in ("q", "k_chunk", "v_chunk"):
        xd[k] = pad(xd[k])
    xd["q_indptr"] = xd["q_indptr"] + lead
    out = torch.full((lead + e.q_rows + tail, 16, 128), 7.0, device=DEV)
    run(e, xd, out=out)
    got = out.cpu().numpy()
    assert (got[:lead] == 7.0).all() and (got[lead + e.q_rows:] == 7.0).all()
    assert_close(got[lead:lead + e.q_rows], want, "extend with offset rows")


def test_extend_device_checks():
    """A chunk range outside q_rows, longer than max_q_len, or prefix rows
    outside the workspace sets NVFP4KV_DEV_BAD_LEN; that sequence writes
    nothing while the others are computed."""
    e = workloads.extend_custom((30, 50), (10, 12), 8, 2, seed=9)
    x = workloads.extend_inputs(e)
    want = oracle_out(e, x)
    for bad in ("q_end", "too_long", "prefix"):
        xd = to_dev(x)
        max_q_len = 12
        if bad == "q_end":
            xd["q_indptr"] = torch.tensor([0, 10, e.q_rows + 1], dtype=torch.int32, device=DEV)
        elif bad == "too_long":
            max_q_len = 11
        else:
            xd["prefix_lens"] = torch.tensor([30, e.prefix_rows], dtype=torch.int32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        out = torch.full((e.q_rows, 8, 128), 5.0, device=DEV)
        run(e, xd, max_q_len=max_q_len, status=status, out=out)
        assert status.item() == nv.DEV_BAD_LEN, bad
        got = out.cpu().numpy()
        assert (got[10:] == 5.0).all(), bad
        assert_close(got[:10], want[:10], f"extend good sequence next to a bad one ({bad})")


def test_extend_empty_inputs():
    e = workloads.extend_custom((4,), (0,), 8, 2, seed=1)
    x = to_dev(workloads.extend_inputs(e))
    out = torch.zeros((0, 8, 128), device=DEV)
    nv.nvfp4kv_extend_attention_fp8(x["q"], x["q_indptr"], x["k_prefix"], x["v_prefix"], x["kv_indptr"],
                                    x["prefix_lens"], x["k_chunk"], x["v_chunk"], out, max_q_len=0)
    torch.cuda.synchronize()


def test_extend_full_size_sampled_tokens():
    """The 160K workload in the launch configuration the bench times.  Chunk
    K/V are drawn as E4M3 codes (held in bf16, exactly), so the oracle can
    take chunk token t alone: its keys are the prefix rows followed by the
    codes of chunk tokens 0 .. t-1, then token t itself."""
    e = workloads.extend_make("ext160k")
    xd = to_dev(workloads.extend_inputs(e, device=DEV))
    gen = torch.Generator(device=DEV)
    gen.manual_seed(1234)
    kc = workloads.e4m3_codes((e.q_rows, e.num_kv_heads, 128), gen, DEV)
    vc = workloads.e4m3_codes((e.q_rows, e.num_kv_heads, 128), gen, DEV)
    xd["k_chunk"] = kc.view(torch.float8_e4m3fn).to(torch.bfloat16)
    xd["v_chunk"] = vc.view(torch.float8_e4m3fn).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(e, xd, out_dtype=torch.bfloat16, status=status)
    assert status.item() == 0
    P, p0 = e.prefix_lens[0], int(e.kv_indptr()[0])
    kp = xd["k_prefix"][p0:p0 + P].cpu().numpy()
    vp = xd["v_prefix"][p0:p0 + P].cpu().numpy()
    kcn, vcn = kc.cpu().numpy(), vc.cpu().numpy()
    q = xd["q"].float().cpu().numpy()
    got = out.float().cpu().numpy()
    for t in (0, 63, 64, 4097, 8191):
        k_pre = np.concatenate([kp, kcn[:t]])
        v_pre = np.concatenate([vp, vcn[:t]])
        kt = torch.from_numpy(kcn[t:t + 1]).view(torch.float8_e4m3fn).float().numpy()
        vt = torch.from_numpy(vcn[t:t + 1]).view(torch.float8_e4m3fn).float().numpy()
        want = oracle.extend_attention(q[t:t + 1], np.int32([0, 1]), k_pre, v_pre, np.int32([0]),
                                       np.int32([P + t]), kt, vt)
        assert_close(got[t:t + 1], want, f"ext160k token {t}")


# --- extend fused with the NVFP4 append of the chunk --------------------------

from layout import nvfp4_planes  # noqa: E402


def chunk_slots(e, seed, odd_shift=False):
    """Slots of each sequence's chunk tokens (positions P .. P + C - 1 of the
    sequence) on shuffled pages; odd_shift moves every position up by one."""
    rng = np.random.default_rng(seed)
    ends = [P + C + 1 for P, C in zip(e.prefix_lens, e.chunk_lens)]
    pages = [(n + 15) // 16 for n in ends]
    perm = rng.permutation(sum(pages) + 2).astype(np.int32)
    slots, k = [], 0
    for b, (P, C) in enumerate(zip(e.prefix_lens, e.chunk_lens)):
        table = perm[k:k + pages[b]]
        k += pages[b]
        pos = np.arange(P, P + C) + (1 if odd_shift else 0)
        slots.append(table[pos // 16] * 16 + pos % 16)
    return np.concatenate(slots).astype(np.int32), len(perm)


def run_fused(e, x, slots, num_pages, global_scale=1.0, status=None, head_scales=None):
    xd = to_dev(x)
    cache = nv.NVFP4Cache.allocate(num_pages, e.num_kv_heads, device=DEV, global_scale=global_scale,
                                   head_scales=head_scales)
    out = torch.full((e.q_rows, e.num_q_heads, 128), float("nan"), device=DEV)
    nv.nvfp4kv_extend_attention_fp8_append(cache, torch.from_numpy(slots).to(DEV), xd["q"], xd["q_indptr"],
                                           xd["k_prefix"], xd["v_prefix"], xd["kv_indptr"], xd["prefix_lens"],
                                           xd["k_chunk"], xd["v_chunk"], out, max_q_len=max(e.chunk_lens),
                                           dev_status=status)
    torch.cuda.synchronize()
    return out.cpu().numpy(), list(nvfp4_planes(cache.pool.cpu().numpy()))


def oracle_planes(e, x, slots, num_pages, global_scale=1.0, head_scales=None):
    pools = [np.zeros((num_pages, e.num_kv_heads, 16, n), np.uint8) for n in (64, 8, 64, 8)]
    hk = None if head_scales is None else head_scales[0]
    hv = None if head_scales is None else head_scales[1]
    oracle.quantize_append(x["k_chunk"].float().numpy(), slots, pools[0], pools[1], global_scale=global_scale,
                           head_scales=hk)
    oracle.quantize_append(x["v_chunk"].float().numpy(), slots, pools[2], pools[3], global_scale=global_scale,
                           head_scales=hv)
    return pools


@pytest.mark.parametrize("prefix_lens,chunk_lens,hq,hkv,odd", [
    ((0, 61, 200, 1000), (130, 1, 77, 64), 48, 8, False),
    ((64, 65), (128, 129), 8, 8, True),                 # pairs broken: atomic nibble merge
    ((0,), (300,), 8, 1, False),
    ((5, 0, 127), (0, 16, 40), 16, 2, True),
])
def test_fused_append_matches_oracle(prefix_lens, chunk_lens, hq, hkv, odd):
    """Attention as the oracle's extend; cache bytes as the oracle's
    quantize_append of the chunk rows, bit for bit."""
    e = workloads.extend_custom(prefix_lens, chunk_lens, hq, hkv, seed=3 * len(prefix_lens) + hq)
    x = workloads.extend_inputs(e)
    slots, num_pages = chunk_slots(e, seed=hq, odd_shift=odd)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, planes = run_fused(e, x, slots, num_pages, status=status)
    assert status.item() == 0
    assert_close(got, oracle_out(e, x), "fused extend out")
    for g_, w_ in zip(planes, oracle_planes(e, x, slots, num_pages)):
        np.testing.assert_array_equal(g_, w_)


def test_fused_append_tensor_scale_and_skipped_slots():
    """Tensor scale G = 0.37; slot -1 skips a token; a slot past the pool is
    skipped and reported."""
    e = workloads.extend_custom((33, 7), (90, 70), 24, 8, seed=77)
    x = workloads.extend_inputs(e)
    slots, num_pages = chunk_slots(e, seed=5)
    slots[[3, 4, 100]] = -1
    bad = slots.copy()
    bad[50] = num_pages * 16 + 3
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, planes = run_fused(e, x, bad, num_pages, global_scale=0.37, status=status)
    assert status.item() == nv.DEV_BAD_SLOT
    slots[50] = -1
    assert_close(got, oracle_out(e, x), "fused extend out, G = 0.37")
    for g_, w_ in zip(planes, oracle_planes(e, x, slots, num_pages, global_scale=0.37)):
        np.testing.assert_array_equal(g_, w_)


def test_fused_append_per_head_scales():
    """The chunk written at per-head tensor scales fl32(G * factor): bit-exact
    with the oracle's quantize_append at the same scales."""
    e = workloads.extend_custom((33, 70), (90, 41), 16, 4, seed=78)
    x = workloads.extend_inputs(e)
    slots, num_pages = chunk_slots(e, seed=6)
    hs = [[0.5, 3.0, 1.0 / 7.0, 1.0], [2.0, 0.3, 1.0, 9.5]]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, planes = run_fused(e, x, slots, num_pages, global_scale=0.37, status=status, head_scales=hs)
    assert status.item() == 0
    assert_close(got, oracle_out(e, x), "fused extend out, per-head scales")
    for g_, w_ in zip(planes, oracle_planes(e, x, slots, num_pages, global_scale=0.37, head_scales=hs)):
        np.testing.assert_array_equal(g_, w_)


@pytest.mark.parametrize("fused", [False, True])
def test_bf16_chunk_behind_long_prefix(fused):
    """A bf16 chunk behind FP8 prefixes of at least eight times its rows runs
    on the E4M3-key kernel, its key tiles split into two E4M3 terms under a
    power-of-two scale per tile.  Keys of magnitudes 1e-3 .. 1e3 (past E4M3's
    448 and below its normal range; q scaled down to keep the scores
    moderate), one sequence with no prefix among long ones, chunks across
    64-key tiles: attention against the oracle, cache bytes bit for bit."""
    e = workloads.extend_custom((3000, 0, 2500), (130, 70, 65), 48, 8, seed=91)
    assert e.prefix_rows >= 8 * e.q_rows
    x = workloads.extend_inputs(e)
    rng = np.random.default_rng(92)
    f = torch.from_numpy(10.0 ** rng.uniform(-3, 3, (e.q_rows, e.num_kv_heads, 1))).float()
    x["k_chunk"] = (x["k_chunk"].float() * f).to(torch.bfloat16)
    x["q"] = (x["q"].float() * 0.01).to(torch.bfloat16)
    want = oracle_out(e, x)
    if not fused:
        got = run(e, to_dev(x)).cpu().numpy()
        assert_close(got, want, "bf16 chunk behind a long prefix")
        return
    slots, num_pages = chunk_slots(e, seed=93)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, planes = run_fused(e, x, slots, num_pages, status=status)
    assert status.item() == 0
    assert_close(got, want, "fused bf16 chunk behind a long prefix")
    for g_, w_ in zip(planes, oracle_planes(e, x, slots, num_pages)):
        np.testing.assert_array_equal(g_, w_)
