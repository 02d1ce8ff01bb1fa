"""Shared set-up for the GPU parity tests.

The CUDA side builds its cache with the library's own quantize_append; the
oracle side quantises the same generator output on the CPU.  Nothing the
oracle consumes comes from the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
import oracle
import workloads

DEV = "cuda"
ATOL, RTOL = 2e-3, 1e-2        # attention tolerance (allclose form)


def assert_close(got, want, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    bad = err > ATOL + RTOL * np.abs(want)
    if bad.any():
        i = np.unravel_index(np.argmax(err - RTOL * np.abs(want)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside |d| <= {ATOL} + {RTOL}|ref|; "
                             f"worst at {i}: got {got[i]:.6g} want {want[i]:.6g}; max abs {err.max():.3e}")


class Built:
    """GPU caches (NVFP4 and optionally FP8) for a workload plus its tables."""

    def __init__(self, w, spare_pages=3, fp8=True, in_dtype=torch.float32, garbage=False,
                 keep_rows=False, global_scale=1.0, head_scales=None):
        self.w = w
        self.global_scale = global_scale
        self.head_scales = head_scales
        self.bt, self.num_pages = workloads.block_table(w, spare_pages=spare_pages)
        self.cache = nv.NVFP4Cache.allocate(self.num_pages, w.num_kv_heads, device=DEV,
                                            global_scale=global_scale, head_scales=head_scales)
        self.fp8 = nv.FP8Cache.allocate(self.num_pages, w.num_kv_heads, device=DEV) if fp8 else None
        if garbage:                   # unused slots hold bytes that decode to NaN scales
            self.cache.pool.fill_(0xFF)
            if fp8:
                self.fp8.pool.fill_(0xFF)
        self.status = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.rows = {}
        for b in range(w.batch):
            L = w.seq_lens[b]
            for t0 in range(0, L, workloads.CHUNK):
                t1 = min(L, t0 + workloads.CHUNK)
                sm = torch.from_numpy(workloads.slot_mapping(w, self.bt, b, t0, t1)).to(DEV)
                k = workloads.kv_rows(w, "k", b, t0, t1, device=DEV).to(in_dtype)
                v = workloads.kv_rows(w, "v", b, t0, t1, device=DEV).to(in_dtype)
                nv.nvfp4kv_quantize_append(self.cache, k, v, sm, self.status)
                if fp8:
                    nv.fp8kv_quantize_append(self.fp8, k, v, sm, self.status)
                if keep_rows:
                    self.rows[(b, t0)] = (k.float().cpu().numpy(), v.float().cpu().numpy())
        self.bt_d = torch.from_numpy(self.bt).to(DEV)
        self.sl_d = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
        self.q = workloads.query(w, device=DEV)

    def rows_of(self, b, which, h=None):
        """The fp32 rows (as the GPU path saw them) of sequence b, optional kv head."""
        w = self.w
        L = w.seq_lens[b]
        parts = []
        for t0 in range(0, L, workloads.CHUNK):
            if (b, t0) in self.rows:
                k, v = self.rows[(b, t0)]
                x = k if which == "k" else v
            else:
                t1 = min(L, t0 + workloads.CHUNK)
                x = workloads.kv_rows(w, which, b, t0, t1, device=DEV).float().cpu().numpy()
            parts.append(x if h is None else x[:, h:h + 1])
        return np.concatenate(parts, 0) if parts else np.zeros((0, w.num_kv_heads if h is None else 1, 128),
                                                                np.float32)

    def decode(self, out_dtype=torch.float32, num_workers=0, fp8=False, q=None):
        w = self.w
        out = torch.full((w.batch, w.num_q_heads, w.head_dim), float("nan"), dtype=out_dtype, device=DEV)
        ws = nv.new_workspace(num_workers, device=DEV)
        ws.fill_(0xFF)               # NaN everywhere: a partial read before it is written shows
        q = self.q if q is None else q
        if fp8:
            nv.fp8kv_paged_decode(self.fp8, q, self.bt_d, self.sl_d, out, ws, num_workers=num_workers,
                                  dev_status=self.status)
        else:
            nv.nvfp4kv_paged_decode(self.cache, q, self.bt_d, self.sl_d, out, ws,
                                    num_workers=num_workers, dev_status=self.status)
        torch.cuda.synchronize()
        return out.float().cpu().numpy()


def oracle_single_head(built: Built, b: int, h: int, fp8=False):
    """Oracle decode of the g query heads of (sequence b, kv head h), built from
    the generator's rows of that head alone (a 1-kv-head cache, identity pages)."""
    w = built.w
    L = w.seq_lens[b]
    g = w.group
    npg = max(1, (L + 15) // 16)
    bt = np.arange(npg, dtype=np.int32)[None, :]
    sm = np.arange(L, dtype=np.int32)
    k = built.rows_of(b, "k", h)
    v = built.rows_of(b, "v", h)
    q = built.q[b:b + 1, h * g:(h + 1) * g].float().cpu().numpy()
    if fp8:
        kc = np.zeros((npg, 1, 16, 128), np.uint8)
        vc = np.zeros_like(kc)
        oracle.fp8_quantize_append(k, sm, kc)
        oracle.fp8_quantize_append(v, sm, vc)
        return oracle.fp8_paged_decode(kc, vc, q, bt, np.int32([L]))[0]
    pools = [np.zeros((npg, 1, 16, s), np.uint8) for s in (64, 8, 64, 8)]
    oracle.quantize_append(k, sm, pools[0], pools[1])
    oracle.quantize_append(v, sm, pools[2], pools[3])
    return oracle.paged_decode(*pools, q, bt, np.int32([L]))[0]


def oracle_full(built: Built, fp8=False):
    """Oracle decode of every output, from a CPU-quantised copy of the whole cache."""
    w = built.w
    if fp8:
        kc = np.zeros((built.num_pages, w.num_kv_heads, 16, 128), np.uint8)
        vc = np.zeros_like(kc)
    else:
        pools = [np.zeros((built.num_pages, w.num_kv_heads, 16, s), np.uint8) for s in (64, 8, 64, 8)]
    for b in range(w.batch):
        L = w.seq_lens[b]
        if L == 0:
            continue
        sm = workloads.slot_mapping(w, built.bt, b, 0, L)
        k, v = built.rows_of(b, "k"), built.rows_of(b, "v")
        if fp8:
            oracle.fp8_quantize_append(k, sm, kc)
            oracle.fp8_quantize_append(v, sm, vc)
        else:
            hs = built.head_scales
            oracle.quantize_append(k, sm, pools[0], pools[1], global_scale=built.global_scale,
                                   head_scales=None if hs is None else hs[0])
            oracle.quantize_append(v, sm, pools[2], pools[3], global_scale=built.global_scale,
                                   head_scales=None if hs is None else hs[1])
    q = built.q.float().cpu().numpy()
    if fp8:
        return oracle.fp8_paged_decode(kc, vc, q, built.bt, np.int32(w.seq_lens)), (kc, vc)
    return oracle.paged_decode(*pools, q, built.bt, np.int32(w.seq_lens),
                               global_scale=built.global_scale, head_scales=built.head_scales), pools
