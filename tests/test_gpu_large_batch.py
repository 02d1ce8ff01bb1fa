"""Decode at the batch sizes where the per-sequence offset table spans several
passes of the CTA (257 sequences and up, to the largest batch one call takes,
NVFP4KV_MAX_BATCH = 8,192): NVFP4 and FP8 decode, the fused append + decode
step, multi-query decode and the static-scratch entry point, every output
against the oracle within |d| <= 2e-3 + 1e-2 |ref|.

The pages' gain is more requests resident and decoded together ("SGLang stores
KV cache in 4 bits", Interpretation: 44 -> 70 requests at 32K, 10 -> 15 at
160K), so one call must be right for every batch it accepts.  Lengths are
short and ragged (0 to 39 tokens, some sequences empty) so the oracle finishes
in seconds.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import test_gpu_decode as tgd
import workloads
from gpu_util import Built, assert_close, oracle_full

pytestmark = pytest.mark.gpu

# 256 sequences fill one pass of the 512-thread decode CTA's offset scan;
# 257 and 300 take a second, partial pass; 513 and more take three or more.
BATCHES = [257, 300, 513, 1024, 4096]


def ragged(batch, seed, hi=40):
    return np.random.default_rng(seed).integers(0, hi, size=batch)


@pytest.mark.parametrize("batch", BATCHES)
def test_large_batch_decode(batch):
    w = workloads.custom(batch, 16, 4, ragged(batch, batch), seed=batch)
    b = Built(w, spare_pages=5, garbage=True)
    want, _ = oracle_full(b)
    want8, _ = oracle_full(b, fp8=True)
    for nw in (0, 333):
        assert_close(b.decode(torch.float32, num_workers=nw), want, f"nvfp4 batch {batch} workers {nw}")
        assert_close(b.decode(torch.float32, num_workers=nw, fp8=True), want8, f"fp8 batch {batch} workers {nw}")
    assert_close(b.decode(torch.bfloat16), want, f"nvfp4 bf16 out, batch {batch}")
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("batch", [300, 1024])
def test_large_batch_fused_append_decode(fp8, batch):
    """The fused step writes the bytes quantize_append would and decodes as
    paged_decode does, at a batch that needs several offset-scan passes."""
    lens = tuple(int(x) for x in ragged(batch, 7 * batch))
    tgd.test_append_decode_equals_append_then_decode(fp8, lens)


@pytest.mark.parametrize("batch,q_len", [(300, 2), (1024, 3)])
def test_large_batch_multi_query(batch, q_len):
    hq, hkv = 16, 4
    w = workloads.custom(batch, hq, hkv, ragged(batch, 3 * batch), seed=batch + 1)
    b = Built(w, fp8=False, garbage=True)
    rng = np.random.default_rng(batch)
    q = torch.from_numpy(rng.standard_normal((batch, q_len, hq, 128)).astype(np.float32)).to(torch.bfloat16)
    _, pools = oracle_full(b)
    ref = np.zeros((batch, q_len, hq, 128))
    for t in range(q_len):
        lt = np.maximum(np.int32(w.seq_lens) - q_len + t + 1, 0).astype(np.int32)
        ref[:, t] = oracle.paged_decode(*pools, q[:, t].float().numpy(), b.bt, lt)
    out = torch.full((batch, q_len, hq, 128), float("nan"), dtype=torch.float32, device="cuda")
    ws = nv.new_workspace(device="cuda")
    ws.fill_(0xFF)
    nv.nvfp4kv_paged_decode_multi(b.cache, q.cuda(), b.bt_d, b.sl_d, out, ws, dev_status=b.status)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, f"multi-query batch {batch} q_len {q_len}")
    assert int(b.status.item()) == 0


@pytest.mark.parametrize("batch", [513, 4096])
def test_large_batch_static_scratch(batch):
    w = workloads.custom(batch, 16, 4, ragged(batch, 5 * batch), seed=batch + 2)
    b = Built(w, fp8=False, garbage=True)
    want, _ = oracle_full(b)
    for nw in (0, nv.STATIC_SCRATCH_MAX_WORKERS):
        out = torch.full((batch, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
        st = nv.load().nvfp4kv_paged_decode_static_scratch(
            b.cache.c, b.q.data_ptr(), batch, 16, b.bt_d.data_ptr(), b.bt_d.shape[1], b.sl_d.data_ptr(),
            1.0 / math.sqrt(128), out.data_ptr(), nv.F32, nw, b.status.data_ptr(),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == nv.OK
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), want, f"static scratch batch {batch} workers {nw}")
    assert int(b.status.item()) == 0


def test_maximum_batch():
    """NVFP4KV_MAX_BATCH sequences: the offset table fills the decode's shared
    memory and the merge grid is 8,192 x 2 x 4 CTAs."""
    lens = np.random.default_rng(11).integers(0, 40, size=8192)
    w = workloads.custom(8192, 8, 2, lens, seed=11)
    b = Built(w, spare_pages=0)
    want, _ = oracle_full(b)
    assert_close(b.decode(torch.float32), want, "nvfp4, batch 8192")
    want8, _ = oracle_full(b, fp8=True)
    assert_close(b.decode(torch.float32, fp8=True), want8, "fp8, batch 8192")
    assert int(b.status.item()) == 0
