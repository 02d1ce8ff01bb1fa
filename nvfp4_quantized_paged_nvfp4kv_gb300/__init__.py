"""Python binding of libnvfp4kv (the C ABI in include/nvfp4kv.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  There is no fallback:
if the shared library is missing or fails to load, importing the binding's
functions raises.

Functions carry the C names and take torch tensors:

  write path
    nvfp4kv_quantize_append(cache, k_new, v_new, slot_mapping, dev_status=None)
    fp8kv_quantize_append(cache, k_new, v_new, slot_mapping, dev_status=None)
  decode path
    nvfp4kv_paged_decode(cache, q, block_table, seq_lens, out, workspace, ...)
    nvfp4kv_append_paged_decode(cache, k_new, v_new, q, block_table, seq_lens, out, workspace, ...)
    nvfp4kv_paged_decode_multi(cache, q, block_table, seq_lens, out, workspace, ...)
    nvfp4kv_paged_decode_static_scratch(cache, q, block_table, seq_lens, out, ...)
    fp8kv_paged_decode / fp8kv_append_paged_decode (the FP8 comparison cache)
    nvfp4kv_decode_workspace_size(num_workers=0), new_workspace(num_workers=0)
  extend path
    nvfp4kv_dequant_prefix_fp8(cache, block_table, prefix_lens, kv_indptr, k_out, v_out)
    nvfp4kv_extend_attention_fp8(q, q_indptr, k_prefix, v_prefix, kv_indptr, prefix_lens, k_chunk, v_chunk, ...)
    nvfp4kv_extend_attention_fp8_append(cache, slot_mapping, q, q_indptr, ...)
  utilities
    nvfp4kv_read_device_status(dev_status, stream=None)
    nvfp4kv_set_wait_limit(polls) (failure detection: when bounded waits give up)
    nvfp4kv_cache_bytes / fp8kv_cache_bytes / nvfp4kv_status_string / nvfp4kv_version

``NVFP4Cache`` and ``FP8Cache`` hold the pool tensors and build the C structs.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import _build

PAGE_SIZE = 16
HEAD_DIM = 128

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_CHECK = 0, 1, 2, 3, 4, 5
DEV_BAD_PAGE, DEV_BAD_SLOT, DEV_BAD_LEN, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8
F32, BF16, E4M3 = 0, 1, 2
STATIC_SCRATCH_MAX_WORKERS = 3024   # NVFP4KV_STATIC_SCRATCH_MAX_WORKERS

_lock = threading.Lock()
_lib = None


class Nvfp4kvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


NVFP4_RECORD_BYTES = 2304      # one page-head record: K, V data and scales
FP8_RECORD_BYTES = 4096


class _Nvfp4Cache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("global_scale", ctypes.c_float), ("head_scales", ctypes.c_void_p)]


class _Fp8Cache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_st = ctypes.c_int


def library_path() -> str:
    """The library that load() opens: libnvfp4kv.so built in-tree, or a prebuilt
    copy of the same sources named by NVFP4KV_LIBRARY (for example a build with
    host-side sanitizers)."""
    return os.environ.get("NVFP4KV_LIBRARY") or _build.LIB


def load(build_if_missing: bool = True):
    """Load libnvfp4kv.so (building it in-tree first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if path == _build.LIB and not os.path.exists(path):
            if not build_if_missing:
                raise OSError(f"libnvfp4kv.so not built at {path}")
            _build.build()
        try:
            import torch  # noqa: F401  (loads the CUDA runtime torch uses first)
        except ImportError:
            pass
        lib = ctypes.CDLL(path)
        sig = {
            "nvfp4kv_quantize_append": (_st, [ctypes.POINTER(_Nvfp4Cache), _vp, _vp, _st, _i32, _vp, _vp, _vp]),
            "nvfp4kv_decode_workspace_size": (ctypes.c_size_t, [_i32]),
            "nvfp4kv_paged_decode": (_st, [ctypes.POINTER(_Nvfp4Cache), _vp, _i32, _i32, _vp, _i32, _vp,
                                           ctypes.c_float, _vp, _st, _vp, ctypes.c_size_t, _i32, _vp, _vp]),
            "nvfp4kv_append_paged_decode": (_st, [ctypes.POINTER(_Nvfp4Cache), _vp, _vp, _st, _vp, _i32, _i32,
                                                  _vp, _i32, _vp, ctypes.c_float, _vp, _st, _vp,
                                                  ctypes.c_size_t, _i32, _vp, _vp]),
            "fp8kv_append_paged_decode": (_st, [ctypes.POINTER(_Fp8Cache), _vp, _vp, _st, _vp, _i32, _i32,
                                                _vp, _i32, _vp, ctypes.c_float, _vp, _st, _vp,
                                                ctypes.c_size_t, _i32, _vp, _vp]),
            "nvfp4kv_paged_decode_multi": (_st, [ctypes.POINTER(_Nvfp4Cache), _vp, _i32, _i32, _i32, _vp, _i32,
                                                 _vp, ctypes.c_float, _vp, _st, _vp, ctypes.c_size_t, _i32, _vp,
                                                 _vp]),
            "nvfp4kv_paged_decode_static_scratch": (_st, [ctypes.POINTER(_Nvfp4Cache), _vp, _i32, _i32, _vp,
                                                          _i32, _vp, ctypes.c_float, _vp, _st, _i32, _vp,
                                                          _vp]),
            "nvfp4kv_dequant_prefix_fp8": (_st, [ctypes.POINTER(_Nvfp4Cache), _vp, _i32, _vp, _vp, _i32,
                                                 _vp, _vp, _vp, _vp]),
            "nvfp4kv_extend_attention_fp8": (_st, [_vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp,
                                                   _vp, _st, _i32, _i32, _i32, ctypes.c_float, _vp, _st, _vp,
                                                   _vp]),
            "nvfp4kv_extend_attention_fp8_append": (_st, [ctypes.POINTER(_Nvfp4Cache), _vp, _vp, _vp, _i32, _i32,
                                                          _vp, _vp, _vp, _vp, ctypes.c_int64, _vp, _vp, _st,
                                                          _i32, _i32, ctypes.c_float, _vp, _st, _vp, _vp]),
            "fp8kv_quantize_append": (_st, [ctypes.POINTER(_Fp8Cache), _vp, _vp, _st, _i32, _vp, _vp, _vp]),
            "fp8kv_paged_decode": (_st, [ctypes.POINTER(_Fp8Cache), _vp, _i32, _i32, _vp, _i32, _vp,
                                         ctypes.c_float, _vp, _st, _vp, ctypes.c_size_t, _i32, _vp, _vp]),
            "nvfp4kv_cache_bytes": (ctypes.c_int64, [_i32, _i32, _i32, _i32]),
            "fp8kv_cache_bytes": (ctypes.c_int64, [_i32, _i32, _i32, _i32]),
            "nvfp4kv_status_string": (ctypes.c_char_p, [_st]),
            "nvfp4kv_read_device_status": (_st, [_vp, _vp, ctypes.POINTER(_i32)]),
            "nvfp4kv_version": (_i32, []),
            "nvfp4kv_set_wait_limit": (ctypes.c_uint32, [ctypes.c_uint32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != OK:
        raise Nvfp4kvError(status, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


# --- caches -----------------------------------------------------------------

class NVFP4Cache:
    """An NVFP4 pool: uint8 [num_pages][num_kv_heads][NVFP4_RECORD_BYTES] page-head
    records (layout in include/nvfp4kv.h).  global_scale is the FP32 tensor
    scale G: a cached value is G * E4M3 block scale * E2M1 code.  head_scales
    (optional): per-head factors [2][num_kv_heads] (K, then V); kv head h then
    uses fl32(G * factor) as its tensor scale."""

    record_bytes = NVFP4_RECORD_BYTES

    def __init__(self, pool, global_scale: float = 1.0, head_scales=None):
        self.pool = pool
        self.num_pages, self.num_kv_heads, rb = pool.shape
        assert rb == self.record_bytes
        self.page_size, self.head_dim = PAGE_SIZE, HEAD_DIM
        self.global_scale = float(global_scale)
        self._hs = None
        if head_scales is not None:
            vals = [float(v) for row in head_scales for v in row]
            assert len(vals) == 2 * self.num_kv_heads, "head_scales: [2][num_kv_heads]"
            self._hs = (ctypes.c_float * len(vals))(*vals)     # host array the library reads per call
        self.head_scales = head_scales
        self._c = _Nvfp4Cache(pool.data_ptr(), self.num_pages, self.num_kv_heads, PAGE_SIZE, HEAD_DIM,
                              self.global_scale, None if self._hs is None else ctypes.addressof(self._hs))

    @classmethod
    def allocate(cls, num_pages, num_kv_heads, device="cuda", zero=True, **kw):
        import torch
        f = torch.zeros if zero else torch.empty
        return cls(f((num_pages, num_kv_heads, cls.record_bytes), dtype=torch.uint8, device=device), **kw)

    @property
    def c(self):
        return ctypes.byref(self._c)

    def nbytes(self) -> int:
        return self.pool.numel()


class FP8Cache(NVFP4Cache):
    """An FP8-E4M3 pool: uint8 [num_pages][num_kv_heads][FP8_RECORD_BYTES] records."""

    record_bytes = FP8_RECORD_BYTES

    def __init__(self, pool):
        self.pool = pool
        self.num_pages, self.num_kv_heads, rb = pool.shape
        assert rb == self.record_bytes
        self.page_size, self.head_dim = PAGE_SIZE, HEAD_DIM
        self._c = _Fp8Cache(pool.data_ptr(), self.num_pages, self.num_kv_heads, PAGE_SIZE, HEAD_DIM)


# --- entry points -------------------------------------------------------------

def nvfp4kv_quantize_append(cache: NVFP4Cache, k_new, v_new, slot_mapping, dev_status=None,
                            stream=None) -> None:
    st = load().nvfp4kv_quantize_append(cache.c, _ptr(k_new), _ptr(v_new), _dtype_code(k_new),
                                        k_new.shape[0], _ptr(slot_mapping), _ptr(dev_status),
                                        _stream(stream))
    _check(st, "nvfp4kv_quantize_append")


def fp8kv_quantize_append(cache: FP8Cache, k_new, v_new, slot_mapping, dev_status=None,
                          stream=None) -> None:
    st = load().fp8kv_quantize_append(cache.c, _ptr(k_new), _ptr(v_new), _dtype_code(k_new),
                                      k_new.shape[0], _ptr(slot_mapping), _ptr(dev_status),
                                      _stream(stream))
    _check(st, "fp8kv_quantize_append")


def nvfp4kv_decode_workspace_size(num_workers: int = 0) -> int:
    return int(load().nvfp4kv_decode_workspace_size(int(num_workers)))


def _decode(fn, name, cache, q, block_table, seq_lens, out, workspace, sm_scale, num_workers,
            dev_status, stream):
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    B, Hq, _ = q.shape
    st = fn(cache.c, _ptr(q), B, Hq, _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
            float(sm_scale), _ptr(out), _dtype_code(out), _ptr(workspace),
            0 if workspace is None else workspace.numel() * workspace.element_size(),
            int(num_workers), _ptr(dev_status), _stream(stream))
    _check(st, name)


def nvfp4kv_paged_decode(cache: NVFP4Cache, q, block_table, seq_lens, out, workspace,
                         sm_scale=None, num_workers=0, dev_status=None, stream=None) -> None:
    _decode(load().nvfp4kv_paged_decode, "nvfp4kv_paged_decode", cache, q, block_table, seq_lens,
            out, workspace, sm_scale, num_workers, dev_status, stream)


def nvfp4kv_paged_decode_multi(cache: NVFP4Cache, q, block_table, seq_lens, out, workspace,
                               sm_scale=None, num_workers=0, dev_status=None, stream=None) -> None:
    """q: bf16 [batch][q_len][Hq][128] (the last q_len positions of each
    sequence, causal); out: [batch][q_len][Hq][128]."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    B, T, Hq, _ = q.shape
    st = load().nvfp4kv_paged_decode_multi(
        cache.c, _ptr(q), B, T, Hq, _ptr(block_table), block_table.shape[1], _ptr(seq_lens), float(sm_scale),
        _ptr(out), _dtype_code(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), int(num_workers),
        _ptr(dev_status), _stream(stream))
    _check(st, "nvfp4kv_paged_decode_multi")


def fp8kv_paged_decode(cache: FP8Cache, q, block_table, seq_lens, out, workspace,
                       sm_scale=None, num_workers=0, dev_status=None, stream=None) -> None:
    _decode(load().fp8kv_paged_decode, "fp8kv_paged_decode", cache, q, block_table, seq_lens,
            out, workspace, sm_scale, num_workers, dev_status, stream)


def _append_decode(fn, name, cache, k_new, v_new, q, block_table, seq_lens, out, workspace, sm_scale,
                   num_workers, dev_status, stream):
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    B, Hq, _ = q.shape
    st = fn(cache.c, _ptr(k_new), _ptr(v_new), _dtype_code(k_new), _ptr(q), B, Hq, _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), float(sm_scale), _ptr(out), _dtype_code(out),
            _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
            int(num_workers), _ptr(dev_status), _stream(stream))
    _check(st, name)


def nvfp4kv_append_paged_decode(cache: NVFP4Cache, k_new, v_new, q, block_table, seq_lens, out,
                                workspace, sm_scale=None, num_workers=0, dev_status=None,
                                stream=None) -> None:
    """One decode step: append k_new/v_new [B][Hkv][128] at position seq_lens-1, then decode."""
    _append_decode(load().nvfp4kv_append_paged_decode, "nvfp4kv_append_paged_decode", cache, k_new,
                   v_new, q, block_table, seq_lens, out, workspace, sm_scale, num_workers, dev_status,
                   stream)


def fp8kv_append_paged_decode(cache: FP8Cache, k_new, v_new, q, block_table, seq_lens, out,
                              workspace, sm_scale=None, num_workers=0, dev_status=None,
                              stream=None) -> None:
    _append_decode(load().fp8kv_append_paged_decode, "fp8kv_append_paged_decode", cache, k_new,
                   v_new, q, block_table, seq_lens, out, workspace, sm_scale, num_workers, dev_status,
                   stream)


def nvfp4kv_paged_decode_static_scratch(cache: NVFP4Cache, q, block_table, seq_lens, out,
                                        sm_scale=None, num_workers=0, dev_status=None,
                                        stream=None) -> None:
    """Decode for callers that cannot allocate device memory: the split-KV
    scratch is the library's own fixed array (see include/nvfp4kv.h)."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    B, Hq, _ = q.shape
    st = load().nvfp4kv_paged_decode_static_scratch(
        cache.c, _ptr(q), B, Hq, _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
        float(sm_scale), _ptr(out), _dtype_code(out), int(num_workers), _ptr(dev_status),
        _stream(stream))
    _check(st, "nvfp4kv_paged_decode_static_scratch")


def nvfp4kv_dequant_prefix_fp8(cache: NVFP4Cache, block_table, prefix_lens, kv_indptr, k_out, v_out,
                               dev_status=None, stream=None) -> None:
    st = load().nvfp4kv_dequant_prefix_fp8(cache.c, _ptr(block_table), block_table.shape[1],
                                           _ptr(prefix_lens), _ptr(kv_indptr), prefix_lens.shape[0],
                                           _ptr(k_out), _ptr(v_out), _ptr(dev_status),
                                           _stream(stream))
    _check(st, "nvfp4kv_dequant_prefix_fp8")


def _chunk_dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return E4M3
    raise TypeError(f"unsupported chunk dtype {t.dtype}")


def nvfp4kv_extend_attention_fp8(q, q_indptr, k_prefix, v_prefix, kv_indptr, prefix_lens, k_chunk, v_chunk,
                                 out, max_q_len=None, sm_scale=None, dev_status=None, stream=None) -> None:
    """Extend attention: each chunk token attends over its sequence's FP8 prefix
    rows and the chunk up to itself.  q: bf16 [rows][Hq][128]; k_chunk, v_chunk:
    [rows][Hkv][128], bf16 or E4M3 bytes (uint8 or float8_e4m3fn: initial
    prefill on the prompt's FP8 K/V); k_prefix, v_prefix: E4M3 bytes
    [prefix rows][Hkv][128] (uint8 or float8_e4m3fn); q_indptr int32 [B+1],
    kv_indptr and prefix_lens int32 [B], all on the device; out: bf16 or fp32
    [rows][Hq][128].  max_q_len bounds every chunk length (read from q_indptr
    when None, which synchronises)."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    rows, Hq, _ = q.shape
    Hkv = k_chunk.shape[1]
    B = prefix_lens.shape[0]
    if max_q_len is None:
        max_q_len = int((q_indptr[1:] - q_indptr[:-1]).max().item()) if B > 0 else 0
    st = load().nvfp4kv_extend_attention_fp8(
        _ptr(q), _ptr(q_indptr), rows, int(max_q_len), _ptr(k_prefix), _ptr(v_prefix), _ptr(kv_indptr),
        _ptr(prefix_lens), k_prefix.shape[0], _ptr(k_chunk), _ptr(v_chunk), _chunk_dtype_code(k_chunk), B, Hq,
        Hkv, float(sm_scale), _ptr(out), _dtype_code(out), _ptr(dev_status), _stream(stream))
    _check(st, "nvfp4kv_extend_attention_fp8")


def nvfp4kv_extend_attention_fp8_append(cache: NVFP4Cache, slot_mapping, q, q_indptr, k_prefix, v_prefix,
                                        kv_indptr, prefix_lens, k_chunk, v_chunk, out, max_q_len=None,
                                        sm_scale=None, dev_status=None, stream=None) -> None:
    """nvfp4kv_extend_attention_fp8 that also writes the chunk's K/V (bf16 or
    E4M3, the values the attention reads) into the NVFP4 cache at slot_mapping
    (int32 [rows], device)."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    rows, Hq, _ = q.shape
    B = prefix_lens.shape[0]
    if max_q_len is None:
        max_q_len = int((q_indptr[1:] - q_indptr[:-1]).max().item()) if B > 0 else 0
    st = load().nvfp4kv_extend_attention_fp8_append(
        cache.c, _ptr(slot_mapping), _ptr(q), _ptr(q_indptr), rows, int(max_q_len), _ptr(k_prefix),
        _ptr(v_prefix), _ptr(kv_indptr), _ptr(prefix_lens), k_prefix.shape[0], _ptr(k_chunk), _ptr(v_chunk),
        _chunk_dtype_code(k_chunk), B, Hq, float(sm_scale), _ptr(out), _dtype_code(out), _ptr(dev_status),
        _stream(stream))
    _check(st, "nvfp4kv_extend_attention_fp8_append")


def nvfp4kv_cache_bytes(num_pages, num_kv_heads, page_size=PAGE_SIZE, head_dim=HEAD_DIM) -> int:
    return int(load().nvfp4kv_cache_bytes(num_pages, num_kv_heads, page_size, head_dim))


def fp8kv_cache_bytes(num_pages, num_kv_heads, page_size=PAGE_SIZE, head_dim=HEAD_DIM) -> int:
    return int(load().fp8kv_cache_bytes(num_pages, num_kv_heads, page_size, head_dim))


def read_device_status(dev_status, stream=None) -> int:
    """Synchronise `stream` and return the bits of the device status word
    (int32 tensor of one element); 0 when no kernel reported anything."""
    bits = _i32(0)
    st = load().nvfp4kv_read_device_status(_ptr(dev_status), _stream(stream), ctypes.byref(bits))
    if st not in (OK, ERR_DEVICE_CHECK):
        _check(st, "nvfp4kv_read_device_status")
    return int(bits.value)


nvfp4kv_read_device_status = read_device_status


def status_string(status: int) -> str:
    return load().nvfp4kv_status_string(int(status)).decode()


nvfp4kv_status_string = status_string


def nvfp4kv_version() -> int:
    return int(load().nvfp4kv_version())


WAIT_LIMIT_DEFAULT = 4194304        # NVFP4KV_WAIT_LIMIT_DEFAULT


def nvfp4kv_set_wait_limit(polls: int) -> int:
    """Polls after which a kernel's bounded waits give up (and report
    DEV_TIMEOUT), for the calls made from now on; returns the previous value."""
    return int(load().nvfp4kv_set_wait_limit(int(polls)))


def new_workspace(num_workers: int = 0, device="cuda"):
    """A decode workspace tensor of the size the library asks for."""
    import torch
    n = nvfp4kv_decode_workspace_size(num_workers)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)
