"""The decode entry point for callers that cannot allocate device memory.

Such callers (a serving engine whose device memory is all reserved at
start-up, for instance) cannot hand the decode a workspace; this entry point
uses the library's own fixed scratch array instead.  It must give the same
results as the ordinary entry point, call after call, since every call reuses
the same array.  This file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import workloads
from gpu_util import Built, assert_close, oracle_full

pytestmark = pytest.mark.gpu


def static_decode(b, out, num_workers=0):
    w = b.w
    return nv.load().nvfp4kv_paged_decode_static_scratch(
        b.cache.c, b.q.data_ptr(), w.batch, w.num_q_heads, b.bt_d.data_ptr(), b.bt_d.shape[1],
        b.sl_d.data_ptr(), 1.0 / math.sqrt(128), out.data_ptr(), nv.F32, num_workers,
        b.status.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name,batch,seq_len", [("llama70b", 12, 2048), ("ctx32k", 6, 4000)])
def test_static_scratch_decode_matches_workspace_decode(name, batch, seq_len):
    w = workloads.make(name, batch=batch, seq_len=seq_len)
    b = Built(w, fp8=False)
    ref = b.decode(torch.float32)                       # ordinary entry point, own workspace
    want, _ = oracle_full(b)                            # and the oracle
    for call in range(2):                               # two calls in a row share the array
        out = torch.full_like(torch.from_numpy(ref), float("nan")).cuda()
        assert static_decode(b, out) == nv.OK
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref, f"static-scratch decode, call {call}")
        assert_close(out.cpu().numpy(), want, f"static-scratch decode against the oracle, call {call}")
    assert int(b.status.item()) == 0


def test_static_scratch_worker_limit():
    """The largest worker count fills the array to its end; one more is
    refused before anything is launched."""
    w = workloads.custom(5, 16, 4, (8000, 17, 7900, 1, 640), seed=9)   # 4,148 page-heads
    b = Built(w, fp8=False)
    want, _ = oracle_full(b)
    out = torch.full((w.batch, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
    assert static_decode(b, out, num_workers=nv.STATIC_SCRATCH_MAX_WORKERS + 1) == nv.ERR_WORKSPACE
    assert static_decode(b, out, num_workers=100000) == nv.ERR_WORKSPACE
    for call in range(2):
        out.fill_(float("nan"))
        assert static_decode(b, out, num_workers=nv.STATIC_SCRATCH_MAX_WORKERS) == nv.OK
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), want, f"static scratch at its worker limit, call {call}")
    assert int(b.status.item()) == 0
