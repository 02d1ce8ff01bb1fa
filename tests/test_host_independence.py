"""The product path and the oracle share nothing.

The library (CUDA kernels, C ABI), its header and the Python binding must not
import, include, link or load anything under oracle/, and the oracle must not
include the library's headers or load the library: a result of one can then
never come from the other.  Only the tests, the smoke check and bench.py's CPU
legs may use the oracle.
"""
import pathlib
import re

ROOT = pathlib.Path(__file__).resolve().parents[1]
PKG = ROOT / "nvfp4_quantized_paged_nvfp4kv_gb300"


def _sources(*dirs, suffixes=(".py", ".c", ".cc", ".cpp", ".cu", ".cuh", ".h")):
    for d in dirs:
        for f in sorted(d.rglob("*")):
            if f.suffix in suffixes and "_build" not in f.parts and "__pycache__" not in f.parts:
                yield f


def test_product_sources_never_reach_the_oracle():
    pat = re.compile(r"(import\s+oracle|from\s+oracle|oracle/|liboracle|nvfp4kv_oracle)")
    hits = []
    for f in _sources(PKG, ROOT / "include"):
        for n, line in enumerate(f.read_text(errors="replace").splitlines(), 1):
            if pat.search(line):
                hits.append(f"{f.relative_to(ROOT)}:{n}: {line.strip()}")
    assert not hits, "product path refers to the oracle:\n" + "\n".join(hits)


def test_oracle_never_reaches_the_library():
    pat = re.compile(r"(nvfp4_quantized_paged_nvfp4kv_gb300|libnvfp4kv|#\s*include\s*[<\"]nvfp4kv\.h|csrc/)")
    hits = []
    for f in _sources(ROOT / "oracle"):
        for n, line in enumerate(f.read_text(errors="replace").splitlines(), 1):
            if pat.search(line):
                hits.append(f"{f.relative_to(ROOT)}:{n}: {line.strip()}")
    assert not hits, "oracle refers to the library:\n" + "\n".join(hits)


def test_binding_has_no_cpu_fallback():
    """The binding only marshals arguments into the C calls: it loads the
    shared library or raises, and contains no numerical code of its own."""
    src = (PKG / "__init__.py").read_text()
    assert "ctypes.CDLL(" in src
    for banned in ("numpy.", "np.", "torch.softmax", "torch.matmul", "scaled_dot_product", "einsum", "@ "):
        assert banned not in src, f"the binding uses {banned!r}"
