"""GPU parity of the write side (quantize_append, NVFP4 and FP8): bit-exact
against the oracle ("SGLang stores KV cache in 4 bits" (LMSYS summary),
Interpretation: new K/V are quantised into the NVFP4 cache)."""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import workloads
from layout import fp8_planes, nvfp4_planes

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_gpu(x_k, x_v, slots, num_pages, hkv, fp8=False, global_scale=1.0, head_scales=None):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sm = torch.from_numpy(np.asarray(slots, np.int32)).to(DEV)
    if fp8:
        c = nv.FP8Cache.allocate(num_pages, hkv, device=DEV)
        nv.fp8kv_quantize_append(c, x_k.to(DEV), x_v.to(DEV), sm, status)
        torch.cuda.synchronize()
        return list(fp8_planes(c.pool.cpu().numpy())), int(status.item())
    c = nv.NVFP4Cache.allocate(num_pages, hkv, device=DEV, global_scale=global_scale, head_scales=head_scales)
    nv.nvfp4kv_quantize_append(c, x_k.to(DEV), x_v.to(DEV), sm, status)
    torch.cuda.synchronize()
    return list(nvfp4_planes(c.pool.cpu().numpy())), int(status.item())


def run_oracle(x_k, x_v, slots, num_pages, hkv, fp8=False, global_scale=1.0, head_scales=None):
    kf = x_k.float().numpy()
    vf = x_v.float().numpy()
    slots = np.asarray(slots, np.int32)
    if fp8:
        kc = np.zeros((num_pages, hkv, 16, 128), np.uint8)
        vc = np.zeros_like(kc)
        oracle.fp8_quantize_append(kf, slots, kc)
        oracle.fp8_quantize_append(vf, slots, vc)
        return [kc, vc]
    pools = [np.zeros((num_pages, hkv, 16, s), np.uint8) for s in (64, 8, 64, 8)]
    hk = None if head_scales is None else head_scales[0]
    hv = None if head_scales is None else head_scales[1]
    oracle.quantize_append(kf, slots, pools[0], pools[1], global_scale=global_scale, head_scales=hk)
    oracle.quantize_append(vf, slots, pools[2], pools[3], global_scale=global_scale, head_scales=hv)
    return pools


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fp8", [False, True])
def test_tiny_workload_bit_exact(dtype, fp8):
    w = workloads.make("tiny")
    bt, num_pages = workloads.block_table(w, spare_pages=2)
    ks, vs, slots = [], [], []
    for b in range(w.batch):
        L = w.seq_lens[b]
        ks.append(workloads.kv_rows(w, "k", b, 0, L))
        vs.append(workloads.kv_rows(w, "v", b, 0, L))
        slots.append(workloads.slot_mapping(w, bt, b, 0, L))
    k = torch.cat(ks).to(dtype)
    v = torch.cat(vs).to(dtype)
    slots = np.concatenate(slots)
    got, st = run_gpu(k, v, slots, num_pages, w.num_kv_heads, fp8)
    want = run_oracle(k, v, slots, num_pages, w.num_kv_heads, fp8)
    assert st == 0
    for g_, w_ in zip(got, want):
        np.testing.assert_array_equal(g_, w_)


@pytest.mark.parametrize("name", ["llama70b", "ctx32k", "ctx1m"])
def test_distributions_bit_exact(name):
    """Outlier channels, per-head scales, Student-t tails: 3000 tokens."""
    w = workloads.make(name, batch=1, seq_len=3000)
    L = w.seq_lens[0]
    bt, num_pages = workloads.block_table(w)
    k = workloads.kv_rows(w, "k", 0, 0, L)
    v = workloads.kv_rows(w, "v", 0, 0, L)
    slots = workloads.slot_mapping(w, bt, 0, 0, L)
    for fp8 in (False, True):
        got, st = run_gpu(k, v, slots, num_pages, w.num_kv_heads, fp8)
        want = run_oracle(k, v, slots, num_pages, w.num_kv_heads, fp8)
        assert st == 0
        for g_, w_ in zip(got, want):
            np.testing.assert_array_equal(g_, w_)


def test_v_nibble_pairs_written_by_separate_calls():
    """The two tokens of a V token pair share bytes; writing them in separate
    calls, in either order and over stale bytes, gives the oracle's result."""
    rng = np.random.default_rng(3)
    T, hkv, pages = 32, 2, 2
    k = torch.from_numpy(rng.standard_normal((T, hkv, 128)).astype(np.float32))
    v = torch.from_numpy(rng.standard_normal((T, hkv, 128)).astype(np.float32))
    slots = np.arange(T, dtype=np.int32)
    for fp8 in (False, True):
        c = (nv.FP8Cache if fp8 else nv.NVFP4Cache).allocate(pages, hkv, device=DEV)
        c.pool.fill_(0xA5)
        order = [1, 0, 3, 2] + list(range(4, T))           # odd token first for the first pairs
        for t in order:
            app = nv.fp8kv_quantize_append if fp8 else nv.nvfp4kv_quantize_append
            app(c, k[t:t + 1].to(DEV), v[t:t + 1].to(DEV), torch.from_numpy(slots[t:t + 1]).to(DEV))
        torch.cuda.synchronize()
        got = (fp8_planes if fp8 else nvfp4_planes)(c.pool.cpu().numpy())
        want = run_oracle(k, v, slots, pages, hkv, fp8)
        for g_, w_ in zip(got, want):
            np.testing.assert_array_equal(g_, w_)


@pytest.mark.parametrize("fp8", [False, True])
def test_odd_first_slot_and_broken_pairs(fp8):
    """Slots that start odd, jump, skip a token, swap a pair's order and run
    backwards, so that tokens taken in input order both do and do not form
    the record's token pairs."""
    slots = (list(range(5, 25)) + [-1] + list(range(41, 51)) + [60, 62, 61, 63] + [3, 2]
             + list(range(80, 87)))
    T, hkv, pages = len(slots), 2, 6
    rng = np.random.default_rng(11)
    k = torch.from_numpy(rng.standard_normal((T, hkv, 128)).astype(np.float32))
    v = torch.from_numpy((rng.standard_normal((T, hkv, 128)) * 3).astype(np.float32))
    got, st = run_gpu(k, v, slots, pages, hkv, fp8=fp8)
    want = run_oracle(k, v, slots, pages, hkv, fp8=fp8)
    assert st == 0
    for g_, w_ in zip(got, want):
        np.testing.assert_array_equal(g_, w_)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("g", [0.37, 3.1, 2.0 ** -7])
def test_tensor_scale_bit_exact(g, dtype):
    """Blocks taken of fl32(x / G) for a tensor scale G != 1 (calibration, the
    LMSYS summary's Perspective): codes and scales equal the oracle's."""
    rng = np.random.default_rng(17)
    T, hkv, pages = 100, 2, 9
    k = torch.from_numpy((rng.standard_t(3, (T, hkv, 128)) * 4 * g).astype(np.float32)).to(dtype)
    v = torch.from_numpy((rng.standard_normal((T, hkv, 128)) * g).astype(np.float32)).to(dtype)
    slots = list(rng.permutation(pages * 16)[:T])
    got, st = run_gpu(k, v, slots, pages, hkv, global_scale=g)
    want = run_oracle(k, v, slots, pages, hkv, global_scale=g)
    assert st == 0
    for g_, w_ in zip(got, want):
        np.testing.assert_array_equal(g_, w_)


HEAD_FACTORS = [[0.5, 3.0, 1.0 / 7.0, 1.0], [2.0, 0.3, 1.0, 9.5]]     # [K, V][kv head]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_per_head_scales_bit_exact(dtype):
    """Kv head h of K (V) quantised at fl32(G * factor): codes and scales equal
    the oracle's."""
    rng = np.random.default_rng(19)
    T, hkv, pages = 90, 4, 8
    k = torch.from_numpy((rng.standard_t(3, (T, hkv, 128)) * 3).astype(np.float32)).to(dtype)
    v = torch.from_numpy(rng.standard_normal((T, hkv, 128)).astype(np.float32)).to(dtype)
    slots = list(rng.permutation(pages * 16)[:T])
    got, st = run_gpu(k, v, slots, pages, hkv, global_scale=0.37, head_scales=HEAD_FACTORS)
    want = run_oracle(k, v, slots, pages, hkv, global_scale=0.37, head_scales=HEAD_FACTORS)
    assert st == 0
    for g_, w_ in zip(got, want):
        np.testing.assert_array_equal(g_, w_)


def test_skipped_and_out_of_range_slots():
    rng = np.random.default_rng(0)
    T, hkv, pages = 40, 2, 4
    k = torch.from_numpy(rng.standard_normal((T, hkv, 128)).astype(np.float32))
    v = torch.from_numpy(rng.standard_normal((T, hkv, 128)).astype(np.float32))
    slots = rng.permutation(pages * 16)[:T].astype(np.int32)
    slots[3] = -1
    slots[7] = -5
    good = slots.copy()
    slots[11] = pages * 16 + 3            # out of range: skipped and reported
    good[11] = -1
    got, st = run_gpu(k, v, slots, pages, hkv)
    want = run_oracle(k, v, good, pages, hkv)
    assert st == nv.DEV_BAD_SLOT
    for g_, w_ in zip(got, want):
        np.testing.assert_array_equal(g_, w_)


def _blocks_to_gpu_codes(blocks, global_scale=1.0):
    """Quantise float32 blocks [N][16] (N multiple of 8) as rows of one kv head;
    returns the K codes and scales (K rows of a record are in natural order)."""
    n = blocks.shape[0]
    T = n // 8
    pages = (T + 15) // 16
    x = torch.from_numpy(blocks.reshape(T, 1, 128)).to(DEV)
    c = nv.NVFP4Cache.allocate(pages, 1, device=DEV, global_scale=global_scale)
    sm = torch.arange(T, dtype=torch.int32, device=DEV)
    nv.nvfp4kv_quantize_append(c, x, x, sm)
    rec = c.pool.reshape(-1, nv.NVFP4_RECORD_BYTES)                   # one kv head: page = record
    data = rec[:, :1024].reshape(-1, 64)[:T].reshape(n, 8)
    scale = rec[:, 2048:2176].reshape(-1, 8)[:T].reshape(n)
    codes = torch.stack([data & 15, data >> 4], -1).reshape(n, 16)
    return codes, scale


def test_every_element_value_at_unit_scale():
    """Every finite fp32 with |x| <= 6 (about 2.2e9 values) is quantised at
    block scale 1 (each block holds 15 test values and one 6.0) and compared
    with the oracle's E2M1 encoder, value by value."""
    six = np.float32(6.0)
    lim = int(np.float32(6.0).view(np.uint32))           # all non-negative patterns <= 6.0
    step = 15 * 8 * (1 << 18)                            # values per chunk (multiple of 15*8)
    total_checked = 0
    for sign in (0, 0x80000000):
        for start in range(0, lim + 1, step):
            stop = min(lim + 1, start + step)
            bits = np.arange(start, stop, dtype=np.uint64).astype(np.uint32) | np.uint32(sign)
            vals = bits.view(np.float32)
            pad = (-len(vals)) % (15 * 8)
            vals_p = np.concatenate([vals, np.zeros(pad, np.float32)])
            blocks = np.empty((len(vals_p) // 15, 16), np.float32)
            blocks[:, :15] = vals_p.reshape(-1, 15)
            blocks[:, 15] = six
            codes, scale = _blocks_to_gpu_codes(blocks)
            assert bool((scale == 0x38).all())            # E4M3(1.0)
            got = codes[:, :15].reshape(-1)[:len(vals)].cpu().numpy()
            want = oracle.e2m1_encode(vals)
            np.testing.assert_array_equal(got, want)
            total_checked += len(vals)
    assert total_checked == 2 * (lim + 1)


def test_element_rounding_for_every_scale_mantissa():
    """Each code is decided on the IEEE quotient fl32(x / s), which the kernel
    forms without a division instruction.  An E4M3 scale has one of eight
    mantissas (s = 1 + m/8 up to a power of two, which scales every quotient
    exactly).  For each, every fp32 x with 1/8 <= x/s <= 6 (and the negatives
    for one of them) is quantised in blocks of 15 test values plus one 6s,
    and every code is compared with the oracle's encoder of the quotient."""
    step = 15 * 8 * (1 << 18)
    for m in range(8):
        s = np.float32(1 + m / 8)
        anchor = np.float32(s * np.float32(6.0))
        lo = int(np.float32(s * np.float32(0.125)).view(np.uint32))
        hi = int(anchor.view(np.uint32))
        for sign in ((0, 0x80000000) if m == 5 else (0,)):
            for start in range(lo, hi + 1, step):
                stop = min(hi + 1, start + step)
                bits = np.arange(start, stop, dtype=np.uint64).astype(np.uint32) | np.uint32(sign)
                vals = bits.view(np.float32)
                pad = (-len(vals)) % (15 * 8)
                vals_p = np.concatenate([vals, np.zeros(pad, np.float32)])
                blocks = np.empty((len(vals_p) // 15, 16), np.float32)
                blocks[:, :15] = vals_p.reshape(-1, 15)
                blocks[:, 15] = anchor
                codes, scale = _blocks_to_gpu_codes(blocks)
                assert bool((scale == 0x38 + m).all())
                got = codes[:, :15].reshape(-1)[:len(vals)].cpu().numpy()
                want = oracle.e2m1_encode((vals / s).astype(np.float32))
                np.testing.assert_array_equal(got, want)


def test_block_scale_sweep():
    """amax over every fp32 exponent from 2^-14 to 2^12 with the mantissa
    patterns next to every E4M3 rounding boundary, plus random amax: scale
    byte and all codes against the oracle's block quantiser."""
    mant = []
    for hi in range(1 << 16):
        for lo in (0, 1, 0x3F, 0x40, 0x41, 0x7F):
            mant.append((hi << 7) | lo)
    mant = np.array(mant, np.uint32)
    exps = np.arange(127 - 14, 127 + 13, dtype=np.uint32)
    amax = ((exps[:, None] << 23) | mant[None, :]).reshape(-1).view(np.float32)
    rng = np.random.default_rng(1)
    amax = np.concatenate([amax, np.exp2(rng.uniform(-20, 13, 1 << 20)).astype(np.float32)])
    n = len(amax) - len(amax) % 8
    amax = amax[:n]
    frac = rng.uniform(-1, 1, (n, 16)).astype(np.float32)
    blocks = (frac * amax[:, None]).astype(np.float32)
    blocks[np.arange(n), rng.integers(0, 16, n)] = amax * np.where(rng.integers(0, 2, n) == 1, 1, -1)
    for lo in range(0, n, 1 << 22):
        hi = min(n, lo + (1 << 22))
        codes, scale = _blocks_to_gpu_codes(blocks[lo:hi])
        x = blocks[lo:hi].reshape(-1, 1, 128)
        T = x.shape[0]
        data = np.zeros((T, 1, 1, 64), np.uint8)
        sc = np.zeros((T, 1, 1, 8), np.uint8)
        oracle.quantize_append(x, np.arange(T, dtype=np.int32), data, sc, page_size=1)
        np.testing.assert_array_equal(scale.cpu().numpy(), sc.reshape(-1))
        want = np.stack([data & 15, data >> 4], -1).reshape(hi - lo, 16)
        np.testing.assert_array_equal(codes.cpu().numpy(), want)


def _offsets(x0: np.ndarray, k: int) -> np.ndarray:
    """x0 moved by k units in the last place (away from zero for k > 0)."""
    bits = x0.astype(np.float32).view(np.int32)
    return (bits + np.int32(k)).view(np.float32)


def _oracle_codes(blocks, global_scale):
    T = blocks.shape[0] // 8
    data = np.zeros((T, 1, 1, 64), np.uint8)
    sc = np.zeros((T, 1, 1, 8), np.uint8)
    oracle.quantize_append(blocks.reshape(T, 1, 128), np.arange(T, dtype=np.int32), data, sc, page_size=1,
                           global_scale=global_scale)
    return np.stack([data & 15, data >> 4], -1).reshape(-1, 16), sc.reshape(-1)


TENSOR_SCALES = ([0.37, 3.1, 2.0 ** -7, 1.5, 3.0, 6.0, 448.0, 1.0 / 3.0,
                  float(np.uint32(0x3F800001).view(np.float32)),      # 1 + 2^-23
                  float(np.uint32(0x3F7FFFFF).view(np.float32)),      # 1 - 2^-24
                  float(np.uint32(0x3FFFFFFF).view(np.float32)),      # 2 - 2^-23
                  float(np.uint32(0x3FAAAAAB).view(np.float32)),      # RN(4/3)
                  1.3 * 2.0 ** -31, 1.7 * 2.0 ** 31,                  # near the ends of [2^-32, 2^32]
                  1.37 * 2.0 ** -33, 1.37 * 2.0 ** 33]                # outside it: the IEEE division
                 + [float(np.float32(g)) for g in np.exp2(np.random.default_rng(23).uniform(-30, 30, 24))])


@pytest.mark.parametrize("g", TENSOR_SCALES)
def test_tensor_scale_quotients_at_decision_boundaries(g):
    """The block procedure runs on fl32(x / G), which the kernel forms from
    RN(1/G) and correction steps rather than a division.  Values are placed
    within three ulps of x / G = b for every E2M1 rounding boundary b (block
    scale 1 from a sixth value 6 G), and block maxima within three ulps of
    x / G = 6 m for E4M3 midpoints m (the scale byte decided by one ulp),
    plus random full-mantissa values, values below 2^-80 next to larger ones
    and alone, and values of 2^64 and more: every scale byte and code equals
    the oracle's, which divides in IEEE fp32."""
    g32 = np.float32(g)
    rng = np.random.default_rng(int(g32.view(np.uint32)))
    blocks = []
    # element boundaries at block scale 1
    bounds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float64)
    base = np.concatenate([bounds, -bounds]) * np.float64(g32)
    vals = np.concatenate([_offsets(base.astype(np.float32), k) for k in range(-3, 4)])
    vals = np.concatenate([vals, np.zeros((-len(vals)) % 15, np.float32)])
    b = np.empty((len(vals) // 15, 16), np.float32)
    b[:, :15] = vals.reshape(-1, 15)
    b[:, 15] = np.float32(6.0 * np.float64(g32))
    blocks.append(b)
    # block maxima next to E4M3 midpoints (scale mantissas 1 + (2j+1)/16, three binades)
    mids = np.array([(1 + (2 * j + 1) / 16) * 2.0 ** e for e in (-3, 0, 3) for j in range(8)])
    amax = np.concatenate([_offsets((6 * mids * np.float64(g32)).astype(np.float32), k) for k in range(-3, 4)])
    b = (rng.uniform(-1, 1, (len(amax), 16)) * amax[:, None]).astype(np.float32)
    b[:, 0] = amax
    blocks.append(b)
    # random values with full mantissas, from 2^-12 G to 2^9 G
    b = (np.exp2(rng.uniform(-12, 9, (4096, 16))) * rng.choice([-1.0, 1.0], (4096, 16)) *
         np.float64(g32)).astype(np.float32)
    blocks.append(b)
    # tiny values (|x| < 2^-80), beside a value of 4 G and alone; huge values
    tiny = (rng.uniform(0.5, 1, (64, 16)) * 2.0 ** -90 * rng.choice([-1.0, 1.0], (64, 16))).astype(np.float32)
    mixed = tiny.copy()
    mixed[:, 7] = np.float32(4.0 * np.float64(g32))
    huge = (rng.uniform(-1, 1, (64, 16)) * 2.0 ** 70).astype(np.float32)
    blocks += [tiny, mixed, huge]
    blocks = np.concatenate(blocks)
    blocks = np.concatenate([blocks, np.zeros(((-len(blocks)) % 8, 16), np.float32)])
    codes, scale = _blocks_to_gpu_codes(blocks, global_scale=float(g32))
    want_codes, want_scale = _oracle_codes(blocks, float(g32))
    np.testing.assert_array_equal(scale.cpu().numpy(), want_scale)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_codes)


@pytest.mark.parametrize("hkv", [1, 3, 5, 8, 16, 17, 24, 32, 33, 40])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_kv_head_counts_and_ragged_token_counts(hkv, dtype):
    """kv head counts from 1 to 40 (powers of two and not), token counts from
    1 to several CTAs' worth, first slots even and odd, consecutive and
    shuffled slots: every byte against the oracle."""
    rng = np.random.default_rng(100 + hkv)
    for T, odd, shuffled in ((1, False, False), (2, True, False), (15, False, True), (33, True, False),
                             (100, False, False), (257, True, True)):
        pages = (T + 2) // 16 + 2
        if shuffled:
            slots = rng.permutation(pages * 16)[:T].astype(np.int32)
            if odd and slots[0] % 2 == 0:                  # put an odd slot first
                j = int(np.flatnonzero(slots % 2 == 1)[0])
                slots[[0, j]] = slots[[j, 0]]
        else:
            slots = np.arange(T, dtype=np.int32) + (1 if odd else 0)
        k = torch.from_numpy((rng.standard_normal((T, hkv, 128)) * 2).astype(np.float32)).to(dtype)
        v = torch.from_numpy(rng.standard_t(4, (T, hkv, 128)).astype(np.float32)).to(dtype)
        got, st = run_gpu(k, v, slots, pages, hkv)
        want = run_oracle(k, v, slots, pages, hkv)
        assert st == 0
        for name, g_, w_ in zip(("k data", "k scale", "v data", "v scale"), got, want):
            np.testing.assert_array_equal(g_, w_, err_msg=f"{name}, T={T}, hkv={hkv}")


@pytest.mark.parametrize("first", [0, 1])
def test_prefill_chunk_8k_tokens_8_heads(first):
    """The benchmarked size: 8,192 bf16 tokens of 8 kv heads into a cache of
    shuffled pages (the long-context workload's block table), starting on an
    even and on an odd slot; every byte against the oracle."""
    w = workloads.make("ctx160k", batch=1)
    bt, num_pages = workloads.block_table(w)
    T = 8192
    sm = workloads.slot_mapping(w, bt, 0, first, first + T)
    k = workloads.kv_rows(w, "k", 0, 0, T).to(torch.bfloat16)
    v = workloads.kv_rows(w, "v", 0, 0, T).to(torch.bfloat16)
    used = np.unique(sm // 16)
    got, st = run_gpu(k, v, sm, num_pages, w.num_kv_heads)
    want = run_oracle(k, v, sm, num_pages, w.num_kv_heads)
    assert st == 0
    for name, g_, w_ in zip(("k data", "k scale", "v data", "v scale"), got, want):
        np.testing.assert_array_equal(g_[used], w_[used], err_msg=name)
