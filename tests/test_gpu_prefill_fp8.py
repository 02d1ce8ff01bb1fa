"""GPU parity of prefill on FP8 keys and values against the oracle.

"SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation: initial
prefill attends directly on the current prompt's FP8 keys and values while the
same data is quantised into the NVFP4 cache.  The chunk's K/V arrive as E4M3
bytes; attention reads them exactly, and the fused write quantises the values
they stand for.  Attention within |d| <= 2e-3 + 1e-2 |ref| of the oracle's
fp64 extend over the same bytes; cache bytes equal to the oracle's
quantize_append of the decoded values, bit for bit.  The E4M3 bytes are
decoded for the oracle's quantize_append by torch's float8_e4m3fn cast.
"""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import workloads
from gpu_util import DEV, assert_close
from layout import nvfp4_planes

pytestmark = pytest.mark.gpu


def inputs(e):
    return workloads.extend_inputs(e, chunk="e4m3")


def to_dev(x):
    return {k: v.to(DEV) for k, v in x.items()}


def decoded(codes: torch.Tensor) -> np.ndarray:
    return codes.cpu().view(torch.float8_e4m3fn).float().numpy()


def oracle_out(x):
    return oracle.extend_attention(x["q"].float().numpy(), x["q_indptr"].numpy(), x["k_prefix"].numpy(),
                                   x["v_prefix"].numpy(), x["kv_indptr"].numpy(), x["prefix_lens"].numpy(),
                                   x["k_chunk"].numpy(), x["v_chunk"].numpy())


def slots_for(e, seed, odd_shift=False):
    """Slots of each sequence's chunk tokens (positions P .. P + C - 1) on
    shuffled pages; odd_shift moves every position up by one."""
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


def oracle_planes(e, x, slots, num_pages, global_scale=1.0, head_scales=None):
    pools = [np.zeros((num_pages, e.num_kv_heads, 16, n), np.uint8) for n in (64, 8, 64, 8)]
    hk = None if head_scales is None else head_scales[0]
    hv = None if head_scales is None else head_scales[1]
    oracle.quantize_append(decoded(x["k_chunk"]), slots, pools[0], pools[1], global_scale=global_scale,
                           head_scales=hk)
    oracle.quantize_append(decoded(x["v_chunk"]), slots, pools[2], pools[3], global_scale=global_scale,
                           head_scales=hv)
    return pools


CASES = [
    # (prefix_lens, chunk_lens, Hq, Hkv): initial prefill (no prefix) first,
    # then extends; chunks across 64-key and 128-row tiles, groups 1..8
    ((0,), (300,), 48, 8),
    ((0, 0, 0), (1, 64, 129), 16, 2),
    ((0,), (257,), 8, 1),
    ((0, 61, 200, 1000), (130, 1, 77, 64), 48, 8),
    ((5, 0, 127), (0, 16, 40), 24, 8),
]


@pytest.mark.parametrize("prefix_lens,chunk_lens,hq,hkv", CASES)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_chunk_attention_matches_oracle(prefix_lens, chunk_lens, hq, hkv, out_dtype):
    e = workloads.extend_custom(prefix_lens, chunk_lens, hq, hkv, seed=11 * len(prefix_lens) + hq)
    x = inputs(e)
    xd = to_dev(x)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((e.q_rows, hq, 128), float("nan"), dtype=out_dtype, device=DEV)
    nv.nvfp4kv_extend_attention_fp8(xd["q"], xd["q_indptr"], xd["k_prefix"], xd["v_prefix"], xd["kv_indptr"],
                                    xd["prefix_lens"], xd["k_chunk"], xd["v_chunk"], out,
                                    max_q_len=max(chunk_lens), dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert_close(out.float().cpu().numpy(), oracle_out(x), f"FP8-chunk attention, {out_dtype}")


def run_fused(e, x, slots, num_pages, global_scale=1.0, head_scales=None, status=None):
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


@pytest.mark.parametrize("prefix_lens,chunk_lens,hq,hkv,odd", [
    ((0,), (300,), 48, 8, False),                # initial prefill
    ((0, 0), (128, 129), 8, 8, True),            # token pairs broken: atomic nibble merge
    ((0, 61, 200, 1000), (130, 1, 77, 64), 48, 8, False),
    ((5, 0, 127), (0, 16, 40), 16, 2, True),
])
def test_fp8_chunk_fused_write_matches_oracle(prefix_lens, chunk_lens, hq, hkv, odd):
    e = workloads.extend_custom(prefix_lens, chunk_lens, hq, hkv, seed=5 * len(prefix_lens) + hq)
    x = inputs(e)
    slots, num_pages = slots_for(e, seed=hq, odd_shift=odd)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, planes = run_fused(e, x, slots, num_pages, status=status)
    assert status.item() == 0
    assert_close(got, oracle_out(x), "fused FP8-chunk prefill out")
    for name, g_, w_ in zip(("k data", "k scale", "v data", "v scale"), planes,
                            oracle_planes(e, x, slots, num_pages)):
        np.testing.assert_array_equal(g_, w_, err_msg=name)


def test_fp8_chunk_fused_write_scales_and_skipped_slots():
    """Tensor scale G = 0.37 with per-head factors; slot -1 skips a token; a
    slot past the pool is skipped and reported."""
    e = workloads.extend_custom((0, 7), (90, 70), 16, 4, seed=77)
    x = inputs(e)
    slots, num_pages = slots_for(e, seed=5)
    slots[[3, 4, 100]] = -1
    bad = slots.copy()
    bad[50] = num_pages * 16 + 3
    hs = [[0.5, 3.0, 1.0 / 7.0, 1.0], [2.0, 0.3, 1.0, 9.5]]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got, planes = run_fused(e, x, bad, num_pages, global_scale=0.37, head_scales=hs, status=status)
    assert status.item() == nv.DEV_BAD_SLOT
    slots[50] = -1
    assert_close(got, oracle_out(x), "fused FP8-chunk prefill out, scaled cache")
    for g_, w_ in zip(planes, oracle_planes(e, x, slots, num_pages, global_scale=0.37, head_scales=hs)):
        np.testing.assert_array_equal(g_, w_)


def test_fp8_chunk_equals_bf16_chunk_of_the_same_values():
    """E4M3 values held exactly in bf16 give the same cache bytes through the
    bf16 path: the two chunk modes read one set of values.  The attention runs
    on different kernels (E4M3 keys on kind::f8f6f4 with Q in two E4M3
    terms; bf16 keys on kind::f16 with Q in f16), so both outputs are held to
    the oracle's rather than to each other bit for bit."""
    e = workloads.extend_custom((0, 33), (100, 45), 24, 8, seed=3)
    x = inputs(e)
    slots, num_pages = slots_for(e, seed=3)
    got8, planes8 = run_fused(e, x, slots, num_pages)
    xb = dict(x)
    xb["k_chunk"] = x["k_chunk"].view(torch.float8_e4m3fn).to(torch.bfloat16)
    xb["v_chunk"] = x["v_chunk"].view(torch.float8_e4m3fn).to(torch.bfloat16)
    gotb, planesb = run_fused(e, xb, slots, num_pages)
    want = oracle_out(x)
    assert_close(got8, want, "E4M3 chunk")
    assert_close(gotb, want, "the same values as a bf16 chunk")
    for a, b in zip(planes8, planesb):
        np.testing.assert_array_equal(a, b)


def test_initial_prefill_8k_sampled_tokens():
    """Initial prefill of one 8,192-token prompt (48 query heads, 8 kv heads)
    on FP8 K/V with the NVFP4 write fused, as the bench launches it: sampled
    tokens against the oracle (token t sees chunk tokens 0 .. t, given to the
    oracle as tokens 0 .. t-1 in the FP8 workspace and token t as the chunk),
    every cache byte against the oracle's quantize_append."""
    e = workloads.extend_make("prefill8k")
    x = workloads.extend_inputs(e, device=DEV, chunk="e4m3")
    C = e.chunk_lens[0]
    cache = nv.NVFP4Cache.allocate(C // 16 + 1, e.num_kv_heads, device=DEV)
    slots = torch.arange(C, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty((C, e.num_q_heads, 128), dtype=torch.bfloat16, device=DEV)
    nv.nvfp4kv_extend_attention_fp8_append(cache, slots, x["q"], x["q_indptr"], x["k_prefix"], x["v_prefix"],
                                           x["kv_indptr"], x["prefix_lens"], x["k_chunk"], x["v_chunk"], out,
                                           max_q_len=C, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kc, vc = x["k_chunk"].cpu().numpy(), x["v_chunk"].cpu().numpy()
    q = x["q"].float().cpu().numpy()
    got = out.float().cpu().numpy()
    for t in (0, 1, 63, 64, 4097, 8191):
        want = oracle.extend_attention(q[t:t + 1], np.int32([0, 1]), kc[:t], vc[:t], np.int32([0]),
                                       np.int32([t]), kc[t:t + 1], vc[t:t + 1])
        assert_close(got[t:t + 1], want, f"prefill8k token {t}")
    pools = [np.zeros((C // 16 + 1, e.num_kv_heads, 16, n), np.uint8) for n in (64, 8, 64, 8)]
    sl = np.arange(C, dtype=np.int32)
    oracle.quantize_append(decoded(x["k_chunk"]), sl, pools[0], pools[1])
    oracle.quantize_append(decoded(x["v_chunk"]), sl, pools[2], pools[3])
    for g_, w_ in zip(nvfp4_planes(cache.pool.cpu().numpy()), pools):
        np.testing.assert_array_equal(g_, w_)
