"""The C ABI without a GPU: the library loads, exports every function that
include/nvfp4kv.h declares, and rejects bad arguments on the host before it
touches the device."""
import ctypes
import os
import re
import subprocess

import pytest

import nvfp4_quantized_paged_nvfp4kv_gb300 as nv
from nvfp4_quantized_paged_nvfp4kv_gb300 import _Fp8Cache, _Nvfp4Cache

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"#[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(", text):
            name = m.group(1)
            if name not in ("sizeof",) and not name.startswith("__"):
                names.add(name)
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("nvfp4kv_quantize_append", "nvfp4kv_paged_decode", "nvfp4kv_dequant_prefix_fp8",
              "fp8kv_paged_decode", "fp8kv_quantize_append", "nvfp4kv_decode_workspace_size",
              "nvfp4kv_extend_attention_fp8", "nvfp4kv_read_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = nv.load()
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", nv.library_path()], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in exported, n


def test_binding_has_a_function_of_each_declared_name():
    """The Python binding offers every entry point under its C name."""
    for n in declared_functions():
        assert callable(getattr(nv, n, None)), n


def test_every_entry_point_cites_a_passage_or_says_it_is_a_utility():
    """Each declaration's comment names the page passage that defines the
    operation, or states that the call has no counterpart on the pages."""
    text = open(os.path.join(HEADER_DIR, "nvfp4kv.h")).read()
    cites = ("SGLang stores KV cache in 4 bits", "NVFP4-KV-Cache auf der")
    utility = ("library utility", "no counterpart")
    pos = 0
    for m in re.finditer(r"\n(?:nvfp4kv_status|size_t|int64_t|int32_t|const char \*)\s*(\w+)\(", text):
        name = m.group(1)
        # the comment block(s) between the previous declaration and this one
        chunk = text[pos:m.start()]
        pos = m.end()
        comments = " ".join(re.findall(r"/\*.*?\*/", chunk, flags=re.S))
        comments = re.sub(r"\s*\n\s*\*?\s*", " ", comments)       # join wrapped comment lines
        if name == "fp8kv_paged_decode":
            continue                      # documented together with fp8kv_quantize_append just above
        assert any(c in comments for c in cites + utility), name


FAKE = 0x7F0000000000          # a 16-byte aligned address that is never dereferenced


def cache(**kw):
    c = dict(pool=FAKE, num_pages=10, num_kv_heads=2, page_size=16, head_dim=128, global_scale=1.0)
    c.update(kw)
    return _Nvfp4Cache(**c)


def fp8cache(**kw):
    c = dict(pool=FAKE, num_pages=10, num_kv_heads=2, page_size=16, head_dim=128)
    c.update(kw)
    return _Fp8Cache(**c)


def append(c, k=FAKE, v=FAKE, n=4, slots=FAKE, dtype=nv.F32):
    return nv.load().nvfp4kv_quantize_append(ctypes.byref(c) if c is not None else None, k, v, dtype,
                                             n, slots, None, None)


def decode(c, hq=4, batch=2, bt=FAKE, mp=4, sl=FAKE, out=FAKE, ws=FAKE, wsb=1 << 30, nw=0,
           q=FAKE, scale=0.088, dtype=nv.BF16):
    return nv.load().nvfp4kv_paged_decode(ctypes.byref(c), q, batch, hq, bt, mp, sl, scale, out, dtype,
                                          ws, wsb, nw, None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(head_dim=64), nv.ERR_UNSUPPORTED),
    (dict(page_size=32), nv.ERR_UNSUPPORTED),
    (dict(global_scale=0.0), nv.ERR_UNSUPPORTED),
    (dict(global_scale=-2.0), nv.ERR_UNSUPPORTED),
    (dict(global_scale=float("inf")), nv.ERR_UNSUPPORTED),
    (dict(global_scale=float("nan")), nv.ERR_UNSUPPORTED),
    (dict(global_scale=1e-40), nv.ERR_UNSUPPORTED),           # subnormal
    (dict(num_pages=0), nv.ERR_INVALID_ARG),
    (dict(num_kv_heads=-1), nv.ERR_INVALID_ARG),
    (dict(pool=FAKE + 8), nv.ERR_INVALID_ARG),
    (dict(pool=None), nv.ERR_INVALID_ARG),
])
def test_cache_validation(kw, want):
    assert append(cache(**kw)) == want
    assert decode(cache(**kw)) == want


def test_head_scale_validation():
    """Per-head factors are checked on the host: each factor and its product
    with G must be positive normal finite, num_kv_heads at most 128."""
    def with_scales(vals, **kw):
        arr = (ctypes.c_float * len(vals))(*vals)
        c = cache(head_scales=ctypes.addressof(arr), **kw)
        return append(c, k=FAKE + 4)          # passes the cache checks, then fails on k's alignment
    assert with_scales([1.0, 2.0, 0.5, 4.0]) == nv.ERR_INVALID_ARG            # accepted
    assert with_scales([1.0, 0.0, 0.5, 4.0]) == nv.ERR_UNSUPPORTED
    assert with_scales([1.0, float("nan"), 0.5, 4.0]) == nv.ERR_UNSUPPORTED
    assert with_scales([1.0, -2.0, 0.5, 4.0]) == nv.ERR_UNSUPPORTED
    assert with_scales([1.0, 1e-40, 0.5, 4.0]) == nv.ERR_UNSUPPORTED          # subnormal factor
    assert with_scales([1.0, 1e30, 0.5, 4.0], global_scale=1e10) == nv.ERR_UNSUPPORTED   # product overflows
    many = [1.0] * 400
    assert with_scales(many, num_kv_heads=200) == nv.ERR_UNSUPPORTED           # over 128 kv heads


def test_append_validation():
    assert append(None) == nv.ERR_INVALID_ARG
    assert append(cache(), n=-1) == nv.ERR_INVALID_ARG
    assert append(cache(), k=FAKE + 4) == nv.ERR_INVALID_ARG
    assert append(cache(), slots=None) == nv.ERR_INVALID_ARG
    assert append(cache(), dtype=7) == nv.ERR_INVALID_ARG
    assert append(cache(), n=0, k=None, v=None, slots=None) == nv.OK     # nothing to do
    c8 = fp8cache(head_dim=256)
    assert nv.load().fp8kv_quantize_append(ctypes.byref(c8), FAKE, FAKE, nv.F32, 1, FAKE, None,
                                           None) == nv.ERR_UNSUPPORTED


def test_decode_validation():
    c = cache()
    assert decode(c, hq=5) == nv.ERR_INVALID_ARG            # Hq % Hkv != 0
    assert decode(c, hq=18) == nv.ERR_UNSUPPORTED           # group 9 > 8
    assert decode(c, batch=-1) == nv.ERR_INVALID_ARG
    assert decode(c, mp=0) == nv.ERR_INVALID_ARG
    assert decode(c, q=FAKE + 2) == nv.ERR_INVALID_ARG
    assert decode(c, out=None) == nv.ERR_INVALID_ARG
    assert decode(c, scale=float("nan")) == nv.ERR_INVALID_ARG
    assert decode(c, dtype=9) == nv.ERR_INVALID_ARG
    assert decode(c, ws=None) == nv.ERR_WORKSPACE
    assert decode(c, ws=FAKE + 16) == nv.ERR_WORKSPACE      # not 256-byte aligned
    assert decode(c, wsb=16) == nv.ERR_WORKSPACE
    assert decode(c, batch=0, q=None, out=None, bt=None, sl=None, ws=None) == nv.OK
    assert decode(c, batch=20000) == nv.ERR_UNSUPPORTED
    assert decode(c, batch=8193) == nv.ERR_UNSUPPORTED         # NVFP4KV_MAX_BATCH + 1


def static_decode(c, hq=4, batch=0, nw=0, scale=0.088, dtype=nv.BF16):
    return nv.load().nvfp4kv_paged_decode_static_scratch(ctypes.byref(c), None, batch, hq, None, 4, None, scale,
                                                         None, dtype, nw, None, None)


def test_static_scratch_decode_batch_zero_checks_arguments():
    """At batch 0 the static-scratch call launches nothing, but it rejects the
    same bad arguments as nvfp4kv_paged_decode does (no device is touched)."""
    c = cache()
    assert static_decode(c) == nv.OK
    for kw in (dict(hq=5), dict(hq=18), dict(dtype=9), dict(scale=float("nan"))):
        want = decode(c, batch=0, q=None, out=None, bt=None, sl=None, ws=None, **kw)
        assert want != nv.OK
        assert static_decode(c, **kw) == want, kw
    assert static_decode(c, nw=nv.STATIC_SCRATCH_MAX_WORKERS + 1) == nv.ERR_WORKSPACE
    assert static_decode(cache(head_dim=64)) == nv.ERR_UNSUPPORTED


def test_prefix_validation():
    lib = nv.load()
    c = cache()
    f = lib.nvfp4kv_dequant_prefix_fp8
    assert f(ctypes.byref(c), FAKE, 4, FAKE, FAKE, -1, FAKE, FAKE, None, None) == nv.ERR_INVALID_ARG
    assert f(ctypes.byref(c), FAKE, 0, FAKE, FAKE, 1, FAKE, FAKE, None, None) == nv.ERR_INVALID_ARG
    assert f(ctypes.byref(c), FAKE, 4, FAKE, FAKE, 1, FAKE + 1, FAKE, None, None) == nv.ERR_INVALID_ARG
    assert f(ctypes.byref(c), FAKE, 4, FAKE, None, 1, FAKE, FAKE, None, None) == nv.ERR_INVALID_ARG
    assert f(ctypes.byref(c), FAKE, 4, FAKE, FAKE, 0, FAKE, FAKE, None, None) == nv.OK


def extend(q=FAKE, qi=FAKE, rows=100, mql=50, kp=FAKE, vp=FAKE, ki=FAKE, pl=FAKE, prows=1000, kc=FAKE, vc=FAKE,
           batch=2, hq=16, hkv=2, scale=0.088, out=FAKE, dtype=nv.BF16, cdtype=nv.BF16):
    return nv.load().nvfp4kv_extend_attention_fp8(q, qi, rows, mql, kp, vp, ki, pl, prows, kc, vc, cdtype, batch,
                                                  hq, hkv, scale, out, dtype, None, None)


def test_extend_validation():
    assert extend(batch=-1) == nv.ERR_INVALID_ARG
    assert extend(rows=-1) == nv.ERR_INVALID_ARG
    assert extend(mql=-1) == nv.ERR_INVALID_ARG
    assert extend(prows=-1) == nv.ERR_INVALID_ARG
    assert extend(hq=5) == nv.ERR_INVALID_ARG                  # Hq % Hkv != 0
    assert extend(hq=18) == nv.ERR_UNSUPPORTED                 # group 9 > 8
    assert extend(batch=70000) == nv.ERR_UNSUPPORTED
    assert extend(mql=1 << 30) == nv.ERR_UNSUPPORTED           # chunk rows x group past int32
    assert extend(scale=float("inf")) == nv.ERR_INVALID_ARG
    assert extend(dtype=3) == nv.ERR_INVALID_ARG
    assert extend(q=None) == nv.ERR_INVALID_ARG
    assert extend(kp=None) == nv.ERR_INVALID_ARG               # prefix rows but no workspace
    assert extend(q=FAKE + 2) == nv.ERR_INVALID_ARG
    assert extend(kc=FAKE + 8) == nv.ERR_INVALID_ARG
    assert extend(qi=FAKE + 2) == nv.ERR_INVALID_ARG
    assert extend(batch=0, q=None, qi=None, ki=None, pl=None, kc=None, vc=None, out=None) == nv.OK
    assert extend(mql=0, q=None, out=None) == nv.OK
    # chunk K/V: bf16 or E4M3 only
    assert extend(cdtype=nv.F32, kp=None) == nv.ERR_INVALID_ARG
    assert extend(cdtype=7, kp=None) == nv.ERR_INVALID_ARG
    assert extend(cdtype=nv.F32, hq=18) == nv.ERR_INVALID_ARG       # the dtype is checked first
    assert extend(cdtype=nv.E4M3, hq=18) == nv.ERR_UNSUPPORTED      # accepted, then the group is too large
    assert extend(cdtype=nv.E4M3, batch=0, q=None, qi=None, ki=None, pl=None, kc=None, vc=None, out=None) == nv.OK
    assert extend(cdtype=nv.E4M3, kc=FAKE + 8) == nv.ERR_INVALID_ARG


def test_extend_append_validation():
    f = nv.load().nvfp4kv_extend_attention_fp8_append

    def call(c, slots=FAKE, hq=4, batch=2, mql=50, cdtype=nv.BF16):
        return f(ctypes.byref(c), slots, FAKE, FAKE, 100, mql, FAKE, FAKE, FAKE, FAKE, 1000, FAKE, FAKE, cdtype,
                 batch, hq, 0.088, FAKE, nv.BF16, None, None)
    assert call(cache(global_scale=0.0)) == nv.ERR_UNSUPPORTED
    assert call(cache(pool=None)) == nv.ERR_INVALID_ARG
    assert call(cache(), slots=None) == nv.ERR_INVALID_ARG
    assert call(cache(), slots=FAKE + 2) == nv.ERR_INVALID_ARG
    assert call(cache(), hq=5) == nv.ERR_INVALID_ARG          # Hq % Hkv (2 in the cache) != 0
    assert call(cache(), hq=18) == nv.ERR_UNSUPPORTED
    assert call(cache(), batch=0, slots=None) == nv.OK
    assert call(cache(), cdtype=nv.F32) == nv.ERR_INVALID_ARG
    assert call(cache(), cdtype=nv.F32, hq=18) == nv.ERR_INVALID_ARG
    assert call(cache(), cdtype=nv.E4M3, hq=18) == nv.ERR_UNSUPPORTED


def test_read_device_status_validation():
    bits = ctypes.c_int32(0)
    assert nv.load().nvfp4kv_read_device_status(None, None, ctypes.byref(bits)) == nv.ERR_INVALID_ARG
    assert nv.load().nvfp4kv_read_device_status(FAKE, None, None) == nv.ERR_INVALID_ARG


def test_status_strings_and_version():
    for s in range(6):
        assert nv.status_string(s)
    assert nv.status_string(99) == "unknown status"
    assert nv.nvfp4kv_version() >= 100


def test_cache_bytes_match_the_printed_figures():
    """Pool sizes for Llama 3.3 70B (80 layers x 8 kv heads x d 128): 1.25 GiB
    per 8K session in FP8 and 0.5625 of that in NVFP4 ("NVFP4-KV-Cache auf der
    NVIDIA RTX PRO 6000 Blackwell Server Edition", "Bytes pro Token" and
    "Sitzungen pro Karte"); 9 bytes per 16 values."""
    pages_8k = 8192 // 16
    nv_layer = nv.nvfp4kv_cache_bytes(pages_8k, 8)
    f8_layer = nv.fp8kv_cache_bytes(pages_8k, 8)
    assert 80 * f8_layer == 1.25 * 2 ** 30
    assert nv_layer / f8_layer == 0.5625
    assert nv.nvfp4kv_cache_bytes(1, 1) == 2 * 16 * 9 * 8           # 16 tokens x 128 ch x (K,V)
    assert nv.nvfp4kv_cache_bytes(1, 1) == nv.NVFP4_RECORD_BYTES
    assert nv.fp8kv_cache_bytes(1, 1) == nv.FP8_RECORD_BYTES
    assert 80 * nv.nvfp4kv_cache_bytes(131072 // 16, 8) == 11.25 * 2 ** 30
    assert nv.nvfp4kv_cache_bytes(1, 1, 16, 100) == -1


def test_set_wait_limit_returns_the_previous_value():
    """The process-wide poll limit of the kernels' bounded waits (host only)."""
    lib = nv.load()
    first = lib.nvfp4kv_set_wait_limit(7)
    try:
        assert first == nv.WAIT_LIMIT_DEFAULT
        assert lib.nvfp4kv_set_wait_limit(0) == 7
        assert lib.nvfp4kv_set_wait_limit(0xFFFFFFFF) == 0
    finally:
        assert lib.nvfp4kv_set_wait_limit(first) == 0xFFFFFFFF
