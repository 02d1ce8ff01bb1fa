"""Decode at the largest batch one call takes (NVFP4KV_MAX_BATCH = 8,192
sequences), NVFP4 and FP8, every output against the oracle within
|d| <= 2e-3 + 1e-2 |ref|.  Kept in a file of its own that runs last."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import Built, assert_close, oracle_full

pytestmark = pytest.mark.gpu


def test_maximum_batch():
    """Short ragged lengths (0 to 39 tokens): the per-sequence offsets fill the
    decode's shared-memory table and the merge grid is 8,192 x 2 x 4 CTAs."""
    lens = np.random.default_rng(11).integers(0, 40, size=8192)
    w = workloads.custom(8192, 8, 2, lens, seed=11)
    b = Built(w, spare_pages=0)
    want, _ = oracle_full(b)
    assert_close(b.decode(torch.float32), want, "nvfp4, batch 8192")
    want8, _ = oracle_full(b, fp8=True)
    assert_close(b.decode(torch.float32, fp8=True), want8, "fp8, batch 8192")
    assert int(b.status.item()) == 0
