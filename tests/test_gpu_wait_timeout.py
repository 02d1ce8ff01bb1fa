"""Failure detection on the GPU without a fault: every bounded wait runs out.

Each kernel that waits (for its staged page records, or for another part of
its CTA) gives up after the process-wide poll limit, sets NVFP4KV_DEV_TIMEOUT
in the device status word, lets the copies and tensor-core operations it has
already started finish, and returns.  With the limit at 0 every such wait
gives up at once, deterministically: the calls must still return normally,
report the timeout, and leave the context usable -- the same calls at the
default limit right after give the oracle's results.
"""
import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import workloads
from gpu_util import DEV, Built, assert_close, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture
def run_out():
    """Call it once the inputs are built: from then on every wait gives up at
    once; the previous limit comes back after the test."""
    prev = nv.nvfp4kv_set_wait_limit(nv.WAIT_LIMIT_DEFAULT)
    try:
        yield lambda: nv.nvfp4kv_set_wait_limit(0)
    finally:
        nv.nvfp4kv_set_wait_limit(prev)


def run_decodes(b, status):
    w = b.w
    outs = []
    for fp8 in (False, True):
        out = torch.full((w.batch, w.num_q_heads, 128), float("nan"), device=DEV)
        ws = nv.new_workspace(device=DEV)
        fn = nv.fp8kv_paged_decode if fp8 else nv.nvfp4kv_paged_decode
        fn(b.fp8 if fp8 else b.cache, b.q, b.bt_d, b.sl_d, out, ws, dev_status=status)
        outs.append(out)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


def test_decode_wait_runs_out_then_recovers(run_out):
    w = workloads.custom(3, 16, 4, (300, 17, 1000), seed=61)
    b = Built(w)
    run_out()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_decodes(b, status)
    assert nv.read_device_status(status) == nv.DEV_TIMEOUT
    nv.nvfp4kv_set_wait_limit(nv.WAIT_LIMIT_DEFAULT)
    status.zero_()
    got, got8 = run_decodes(b, status)
    assert nv.read_device_status(status) == 0
    assert_close(got, oracle_full(b)[0], "nvfp4 decode after a timeout")
    assert_close(got8, oracle_full(b, fp8=True)[0], "fp8 decode after a timeout")


def test_prefix_dequant_wait_runs_out_then_recovers(run_out):
    w = workloads.custom(2, 8, 2, (200, 77), seed=62)
    b = Built(w, fp8=False)
    run_out()
    indptr = torch.tensor([0, 200], dtype=torch.int32, device=DEV)
    k = torch.zeros((277, 2, 128), dtype=torch.uint8, device=DEV)
    v = torch.zeros_like(k)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    nv.nvfp4kv_dequant_prefix_fp8(b.cache, b.bt_d, b.sl_d, indptr, k, v, dev_status=status)
    assert nv.read_device_status(status) == nv.DEV_TIMEOUT
    nv.nvfp4kv_set_wait_limit(nv.WAIT_LIMIT_DEFAULT)
    status.zero_()
    nv.nvfp4kv_dequant_prefix_fp8(b.cache, b.bt_d, b.sl_d, indptr, k, v, dev_status=status)
    assert nv.read_device_status(status) == 0
    _, pools = oracle_full(b)
    want_k = oracle.dequant_prefix_fp8(pools[0], pools[1], b.bt, np.int32(w.seq_lens), np.int32([0, 200]),
                                       out_rows=277)
    np.testing.assert_array_equal(k.cpu().numpy(), want_k)


@pytest.mark.parametrize("chunk", ["bf16", "e4m3", "bf16_long_prefix"])
@pytest.mark.parametrize("fused", [False, True])
def test_extend_wait_runs_out_then_recovers(run_out, fused, chunk):
    """The tensor-core extend kernels (bf16 chunks; E4M3 chunks, whose key
    tiles come by TMA; bf16 chunks behind long prefixes, whose chunk tiles the
    converters split and publish): their roles give up, the MMAs and TMA loads
    already issued are waited for before the CTA frees tensor memory and exits."""
    e8 = chunk == "e4m3"
    prefix = (3000, 2500) if chunk == "bf16_long_prefix" else (70, 300)
    e = workloads.extend_custom(prefix, (100, 129), 16, 2, seed=63)
    x = workloads.extend_inputs(e, chunk="e4m3" if e8 else "bf16")
    xd = {k: t.to(DEV) for k, t in x.items()}
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    cache = nv.NVFP4Cache.allocate(64, e.num_kv_heads, device=DEV)
    slots = torch.arange(e.q_rows, dtype=torch.int32, device=DEV)
    out = torch.full((e.q_rows, 16, 128), float("nan"), device=DEV)

    def call():
        args = (xd["q"], xd["q_indptr"], xd["k_prefix"], xd["v_prefix"], xd["kv_indptr"], xd["prefix_lens"],
                xd["k_chunk"], xd["v_chunk"], out)
        if fused:
            nv.nvfp4kv_extend_attention_fp8_append(cache, slots, *args, max_q_len=129, dev_status=status)
        else:
            nv.nvfp4kv_extend_attention_fp8(*args, max_q_len=129, dev_status=status)
    run_out()
    call()
    assert nv.read_device_status(status) == nv.DEV_TIMEOUT
    nv.nvfp4kv_set_wait_limit(nv.WAIT_LIMIT_DEFAULT)
    status.zero_()
    call()
    assert nv.read_device_status(status) == 0
    want = oracle.extend_attention(x["q"].float().numpy(), x["q_indptr"].numpy(), x["k_prefix"].numpy(),
                                   x["v_prefix"].numpy(), x["kv_indptr"].numpy(), x["prefix_lens"].numpy(),
                                   x["k_chunk"].numpy() if e8 else x["k_chunk"].float().numpy(),
                                   x["v_chunk"].numpy() if e8 else x["v_chunk"].float().numpy())
    assert_close(out.cpu().numpy(), want, f"extend ({chunk} chunk) after a timeout")

