"""Pins of the oracle's extend attention (CPU only).

"SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation: the
extend path dequantises the cached prefix into one FP8 workspace and attends
over it plus the new chunk.  Chunk token i of a sequence sees every prefix
token and chunk tokens 0 .. i.  Checked against torch's float64 attention
(with its causal scaled-dot-product routine where the prefix is empty) on
values decoded here independently.
"""
import numpy as np
import pytest
import torch

import oracle


def make_case(prefix_lens, chunk_lens, hq, hkv, seed):
    rng = np.random.default_rng(seed)
    B = len(prefix_lens)
    q_indptr = np.concatenate([[0], np.cumsum(chunk_lens)]).astype(np.int32)
    kv_indptr = np.concatenate([[3], 3 + np.cumsum(prefix_lens)[:-1]]).astype(np.int32)
    rows_q = int(q_indptr[-1])
    rows_kv = int(3 + sum(prefix_lens) + 2)
    q = rng.standard_normal((rows_q, hq, 128)).astype(np.float32)
    kc = rng.standard_normal((rows_q, hkv, 128)).astype(np.float32)
    vc = rng.standard_normal((rows_q, hkv, 128)).astype(np.float32)
    # prefix: E4M3 codes of normal values (finite codes only)
    raw = torch.from_numpy(rng.standard_normal((rows_kv, hkv, 128)).astype(np.float32) * 2)
    kp = raw.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    vp = torch.from_numpy(rng.standard_normal((rows_kv, hkv, 128)).astype(np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return q, q_indptr, kp, vp, kv_indptr, np.int32(prefix_lens), kc, vc


def torch_reference(q, q_indptr, kp, vp, kv_indptr, prefix_lens, kc, vc, hq, hkv):
    g = hq // hkv
    K8 = torch.from_numpy(kp).view(torch.float8_e4m3fn).double()
    V8 = torch.from_numpy(vp).view(torch.float8_e4m3fn).double()
    out = np.zeros(q.shape)
    for b in range(len(prefix_lens)):
        c0, c1 = q_indptr[b], q_indptr[b + 1]
        P, p0 = int(prefix_lens[b]), int(kv_indptr[b])
        for h in range(hq):
            kv = h // g
            K = torch.cat([K8[p0:p0 + P, kv], torch.from_numpy(kc[c0:c1, kv]).double()])
            V = torch.cat([V8[p0:p0 + P, kv], torch.from_numpy(vc[c0:c1, kv]).double()])
            Q = torch.from_numpy(q[c0:c1, h]).double()
            s = Q @ K.T / np.sqrt(128)
            C = c1 - c0
            mask = torch.ones(C, P + C, dtype=torch.bool)
            mask[:, P:] = torch.tril(torch.ones(C, C, dtype=torch.bool))
            s = s.masked_fill(~mask, float("-inf"))
            out[c0:c1, h] = (torch.softmax(s, -1) @ V).numpy()
    return out


@pytest.mark.parametrize("prefix_lens,chunk_lens,hq,hkv", [
    ((37, 0, 100), (5, 9, 1), 4, 2),
    ((64,), (64,), 8, 8),
    ((1, 300), (17, 40), 6, 1),
])
def test_extend_matches_torch(prefix_lens, chunk_lens, hq, hkv):
    case = make_case(prefix_lens, chunk_lens, hq, hkv, seed=len(prefix_lens) * 7 + hq)
    got = oracle.extend_attention(*case)
    want = torch_reference(*case, hq, hkv)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_empty_prefix_is_causal_self_attention():
    """No prefix: torch's causal scaled-dot-product attention in float64."""
    q, qi, kp, vp, ki, pl, kc, vc = make_case((0,), (33,), 2, 2, seed=3)
    got = oracle.extend_attention(q, qi, kp, vp, ki, pl, kc, vc)
    Q = torch.from_numpy(q).double().permute(1, 0, 2)
    K = torch.from_numpy(kc).double().permute(1, 0, 2)
    V = torch.from_numpy(vc).double().permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True).permute(1, 0, 2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_equal_keys_give_mean_of_visible_values():
    """All keys equal: token i averages the prefix values and chunk values 0..i."""
    q, qi, kp, vp, ki, pl, kc, vc = make_case((10,), (6,), 1, 1, seed=4)
    kp[:] = 0x38                                      # E4M3 1.0 everywhere
    kc[:] = 1.0
    got = oracle.extend_attention(q, qi, kp, vp, ki, pl, kc, vc)
    Vp = torch.from_numpy(vp).view(torch.float8_e4m3fn).double().numpy()[3:13, 0]
    for i in range(6):
        vis = np.concatenate([Vp, vc[:i + 1, 0].astype(np.float64)])
        np.testing.assert_allclose(got[i, 0], vis.mean(0), rtol=1e-12, atol=1e-12)


# --- the chunk in FP8 ---------------------------------------------------------
# "SGLang stores KV cache in 4 bits" (LMSYS summary), Interpretation: initial
# prefill attends on the prompt's FP8 keys and values.  The oracle takes the
# chunk as E4M3 bytes and decodes them itself; the pins decode them with torch's
# float8_e4m3fn instead.

def e4m3_chunk(kc, vc, scale=1.5):
    to8 = lambda x: torch.from_numpy(x * scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()  # noqa: E731
    return to8(kc), to8(vc)


def decoded(codes):
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()


@pytest.mark.parametrize("prefix_lens,chunk_lens,hq,hkv", [
    ((0, 0), (40, 7), 8, 2),          # initial prefill: no prefix at all
    ((37, 0, 100), (5, 9, 1), 4, 2),
    ((1, 300), (17, 40), 6, 1),
])
def test_e4m3_chunk_matches_torch(prefix_lens, chunk_lens, hq, hkv):
    q, qi, kp, vp, ki, pl, kc, vc = make_case(prefix_lens, chunk_lens, hq, hkv, seed=hq + 17)
    kc8, vc8 = e4m3_chunk(kc, vc)
    got = oracle.extend_attention(q, qi, kp, vp, ki, pl, kc8, vc8)
    want = torch_reference(q, qi, kp, vp, ki, pl, decoded(kc8), decoded(vc8), hq, hkv)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_e4m3_chunk_initial_prefill_is_causal_sdpa():
    """No prefix, chunk in FP8: torch's causal scaled-dot-product attention in
    float64 over the torch-decoded E4M3 keys and values."""
    q, qi, kp, vp, ki, pl, kc, vc = make_case((0,), (50,), 4, 2, seed=8)
    kc8, vc8 = e4m3_chunk(kc, vc, scale=3.0)
    got = oracle.extend_attention(q, qi, kp, vp, ki, pl, kc8, vc8)
    Q = torch.from_numpy(q).double().permute(1, 0, 2)
    K = torch.from_numpy(decoded(kc8)).double().repeat_interleave(2, 1).permute(1, 0, 2)
    V = torch.from_numpy(decoded(vc8)).double().repeat_interleave(2, 1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True).permute(1, 0, 2)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_e4m3_chunk_byte_order_matters():
    """A transposed channel order in the chunk's bytes changes the result (the
    pins above would notice a decode that reads the wrong byte)."""
    q, qi, kp, vp, ki, pl, kc, vc = make_case((0,), (9,), 2, 2, seed=12)
    kc8, vc8 = e4m3_chunk(kc, vc)
    a = oracle.extend_attention(q, qi, kp, vp, ki, pl, kc8, vc8)
    b = oracle.extend_attention(q, qi, kp, vp, ki, pl, kc8[:, :, ::-1].copy(), vc8)
    assert np.abs(a - b).max() > 1e-3
