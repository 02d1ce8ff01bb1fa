"""CPU oracle for the NVFP4 paged KV-cache path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and this
package shares no code, table or constant with it.

The arithmetic lives in ``nvfp4kv_oracle.c`` (plain C, fp64 attention); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
Every function cites the page passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4kv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
# A prebuilt copy of the same source to load instead (the sanitizer test builds
# one with AddressSanitizer and UBSan); unset in normal use.
_LIB_OVERRIDE = os.environ.get("NVFP4KV_ORACLE_LIB")
CFLAGS = ["-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math, no FP contraction)."""
    if _LIB_OVERRIDE:
        return _LIB_OVERRIDE
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc"] + CFLAGS + [_SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e2m1_encode_array.argtypes = [_f32p, _u8p, ctypes.c_int64]
        lib.oracle_e4m3_encode_array.argtypes = [_f32p, _u8p, ctypes.c_int64]
        lib.oracle_quantize_block16.argtypes = [_f32p, _u8p, _u8p, ctypes.c_float]
        lib.oracle_quantize_append.argtypes = [
            _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _u8p, _u8p, _f32p]
        lib.oracle_dequant_rows.argtypes = [_u8p, _u8p, ctypes.c_int64, ctypes.c_int, _f32p, ctypes.c_float]
        lib.oracle_paged_decode.argtypes = [
            _u8p, _u8p, _u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p,
            ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _i32p, ctypes.c_double, _f64p, _f32p, _f32p]
        lib.oracle_dequant_prefix_fp8.argtypes = [
            _u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int,
            _i32p, _i32p, ctypes.c_int, _u8p, _f32p]
        lib.oracle_fp8_quantize_append.argtypes = [
            _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, _u8p]
        lib.oracle_fp8_paged_decode.argtypes = [
            _u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p, ctypes.c_int,
            ctypes.c_int, _i32p, ctypes.c_int, _i32p, ctypes.c_double, _f64p]
        lib.oracle_extend_attention.argtypes = [
            _f32p, _i32p, _u8p, _u8p, _i32p, _i32p, _f32p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_double, _f64p]
        lib.oracle_extend_attention_e4m3_chunk.argtypes = [
            _f32p, _i32p, _u8p, _u8p, _i32p, _i32p, _u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_double, _f64p]
        lib.oracle_nvfp4_bytes.restype = ctypes.c_int64
        lib.oracle_nvfp4_bytes.argtypes = [ctypes.c_int64]
        lib.oracle_fp8_bytes.restype = ctypes.c_int64
        lib.oracle_fp8_bytes.argtypes = [ctypes.c_int64]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray, ptype):
    return a.ctypes.data_as(ptype)


# --- element formats -------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e2m1_encode(y) -> np.ndarray:
    y = _c(np.atleast_1d(y), np.float32)
    out = np.empty(y.shape, np.uint8)
    _load().oracle_e2m1_encode_array(_p(y, _f32p), _p(out, _u8p), y.size)
    return out


def e4m3_encode(y) -> np.ndarray:
    y = _c(np.atleast_1d(y), np.float32)
    out = np.empty(y.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_p(y, _f32p), _p(out, _u8p), y.size)
    return out


def e2m1_table() -> np.ndarray:
    return np.array([e2m1_value(c) for c in range(16)], np.float64)


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_value(c) for c in range(256)], np.float64)


# --- NVFP4 blocks and cache ----------------------------------------------

def quantize_block16(x, global_scale: float = 1.0) -> tuple[np.ndarray, int]:
    x = _c(x, np.float32).reshape(16)
    packed = np.empty(8, np.uint8)
    scale = np.empty(1, np.uint8)
    _load().oracle_quantize_block16(_p(x, _f32p), _p(packed, _u8p), _p(scale, _u8p), float(global_scale))
    return packed, int(scale[0])


def head_tensor_scales(global_scale: float, head_scales, Hkv: int) -> np.ndarray:
    """Tensor scale of each kv head: fl32(global_scale * head_scales[h]) (one
    fp32 rounding), or global_scale for every head without per-head factors."""
    g = np.float32(global_scale)
    if head_scales is None:
        return np.full(Hkv, g, np.float32)
    f = np.asarray(head_scales, np.float32).reshape(Hkv)
    return (g * f).astype(np.float32)


def quantize_append(x, slot_mapping, data, scale, page_size: int = 16, global_scale: float = 1.0,
                    head_scales=None) -> None:
    """Quantise rows x[T][Hkv][d] into the NVFP4 pools (in place); a value of
    kv head h is stored as G_h * E4M3 scale * E2M1 with G_h =
    fl32(global_scale * head_scales[h]) (global_scale when head_scales is
    None)."""
    x = _c(x, np.float32)
    T, Hkv, d = x.shape
    sm = _c(slot_mapping, np.int32)
    assert data.flags.c_contiguous and scale.flags.c_contiguous
    assert data.dtype == np.uint8 and scale.dtype == np.uint8
    hs = head_tensor_scales(global_scale, head_scales, Hkv)
    _load().oracle_quantize_append(_p(x, _f32p), T, Hkv, d, _p(sm, _i32p), page_size,
                                   _p(data, _u8p), _p(scale, _u8p), _p(hs, _f32p))


def dequant_rows(data, scale, global_scale: float = 1.0, head_scales=None) -> np.ndarray:
    """Dequantise NVFP4 rows (data[..., d/2], scale[..., d/16]) to fp32.  With
    head_scales, data is a pool [pages][Hkv][P][d/2] and head h's rows use
    fl32(global_scale * head_scales[h])."""
    if head_scales is not None:
        Hkv = data.shape[1]
        hs = head_tensor_scales(global_scale, head_scales, Hkv)
        return np.stack([dequant_rows(np.ascontiguousarray(data[:, h]), np.ascontiguousarray(scale[:, h]),
                                      float(hs[h])) for h in range(Hkv)], 1)
    data = _c(data, np.uint8)
    scale = _c(scale, np.uint8)
    d = data.shape[-1] * 2
    rows = data.size // (d // 2)
    out = np.empty(data.shape[:-1] + (d,), np.float32)
    _load().oracle_dequant_rows(_p(data, _u8p), _p(scale, _u8p), rows, d, _p(out, _f32p), float(global_scale))
    return out


def paged_decode(k_data, k_scale, v_data, v_scale, q, block_table, seq_lens,
                 sm_scale: float | None = None, global_scale: float = 1.0, head_scales=None) -> np.ndarray:
    """fp64 GQA decode over the NVFP4 pools.  q: float32 [B][Hq][d].
    head_scales: None or per-head factors [2][Hkv] (K, then V)."""
    k_data = _c(k_data, np.uint8)
    k_scale = _c(k_scale, np.uint8)
    v_data = _c(v_data, np.uint8)
    v_scale = _c(v_scale, np.uint8)
    _, Hkv, P, half = k_data.shape
    d = half * 2
    q = _c(q, np.float32)
    B, Hq, _ = q.shape
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    out = np.empty((B, Hq, d), np.float64)
    hk = head_tensor_scales(global_scale, None if head_scales is None else np.asarray(head_scales)[0], Hkv)
    hv = head_tensor_scales(global_scale, None if head_scales is None else np.asarray(head_scales)[1], Hkv)
    _load().oracle_paged_decode(_p(k_data, _u8p), _p(k_scale, _u8p), _p(v_data, _u8p),
                                _p(v_scale, _u8p), Hkv, P, d, _p(q, _f32p), B, Hq,
                                _p(bt, _i32p), bt.shape[1], _p(sl, _i32p),
                                float(sm_scale), _p(out, _f64p), _p(hk, _f32p), _p(hv, _f32p))
    return out


def dequant_prefix_fp8(data, scale, block_table, prefix_lens, kv_indptr,
                       out_rows: int | None = None, global_scale: float = 1.0, head_scales=None) -> np.ndarray:
    """FP8 workspace rows of one tensor (K or V) of the cache; head_scales:
    None or this tensor's per-head factors [Hkv]."""
    data = _c(data, np.uint8)
    scale = _c(scale, np.uint8)
    _, Hkv, P, half = data.shape
    d = half * 2
    bt = _c(block_table, np.int32)
    pl = _c(prefix_lens, np.int32)
    ip = _c(kv_indptr, np.int32)
    if out_rows is None:
        out_rows = int(ip[-1])
    out = np.zeros((out_rows, Hkv, d), np.uint8)
    _load().oracle_dequant_prefix_fp8(_p(data, _u8p), _p(scale, _u8p), Hkv, P, d,
                                      _p(bt, _i32p), bt.shape[1], _p(pl, _i32p),
                                      _p(ip, _i32p), len(pl), _p(out, _u8p),
                                      _p(head_tensor_scales(global_scale, head_scales, Hkv), _f32p))
    return out


# --- FP8 comparison cache ---------------------------------------------------

def fp8_quantize_append(x, slot_mapping, data, page_size: int = 16) -> None:
    x = _c(x, np.float32)
    T, Hkv, d = x.shape
    sm = _c(slot_mapping, np.int32)
    assert data.flags.c_contiguous and data.dtype == np.uint8
    _load().oracle_fp8_quantize_append(_p(x, _f32p), T, Hkv, d, _p(sm, _i32p), page_size,
                                       _p(data, _u8p))


def fp8_paged_decode(k, v, q, block_table, seq_lens, sm_scale: float | None = None):
    k = _c(k, np.uint8)
    v = _c(v, np.uint8)
    _, Hkv, P, d = k.shape
    q = _c(q, np.float32)
    B, Hq, _ = q.shape
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    out = np.empty((B, Hq, d), np.float64)
    _load().oracle_fp8_paged_decode(_p(k, _u8p), _p(v, _u8p), Hkv, P, d, _p(q, _f32p), B, Hq,
                                    _p(bt, _i32p), bt.shape[1], _p(sl, _i32p),
                                    float(sm_scale), _p(out, _f64p))
    return out


# --- extend attention ---------------------------------------------------------

def extend_attention(q, q_indptr, k_prefix, v_prefix, kv_indptr, prefix_lens, k_chunk, v_chunk,
                     sm_scale: float | None = None) -> np.ndarray:
    """fp64 attention of each chunk token over its sequence's FP8 prefix rows
    and the chunk's keys up to itself.  q: float32 [rows][Hq][d]; k_chunk,
    v_chunk: float32 [rows][Hkv][d], or uint8 E4M3 bytes (the chunk in FP8, as
    initial prefill receives it); k_prefix, v_prefix: E4M3 bytes
    [rows][Hkv][d]."""
    q = _c(q, np.float32)
    rows, Hq, d = q.shape
    e4m3 = np.asarray(k_chunk).dtype == np.uint8
    assert (np.asarray(v_chunk).dtype == np.uint8) == e4m3, "k_chunk and v_chunk: same kind"
    kc = _c(k_chunk, np.uint8 if e4m3 else np.float32)
    vc = _c(v_chunk, np.uint8 if e4m3 else np.float32)
    Hkv = kc.shape[1]
    kp = _c(k_prefix, np.uint8)
    vp = _c(v_prefix, np.uint8)
    qi = _c(q_indptr, np.int32)
    ki = _c(kv_indptr, np.int32)
    pl = _c(prefix_lens, np.int32)
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    out = np.zeros((rows, Hq, d), np.float64)
    fn = _load().oracle_extend_attention_e4m3_chunk if e4m3 else _load().oracle_extend_attention
    cp = _u8p if e4m3 else _f32p
    fn(_p(q, _f32p), _p(qi, _i32p), _p(kp, _u8p), _p(vp, _u8p), _p(ki, _i32p), _p(pl, _i32p), _p(kc, cp),
       _p(vc, cp), len(pl), Hq, Hkv, d, float(sm_scale), _p(out, _f64p))
    return out


# --- storage arithmetic -----------------------------------------------------

def nvfp4_bytes(num_values: int) -> int:
    return int(_load().oracle_nvfp4_bytes(int(num_values)))


def fp8_bytes(num_values: int) -> int:
    return int(_load().oracle_fp8_bytes(int(num_values)))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (timing only; the
    results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))
