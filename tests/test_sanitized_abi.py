"""The C ABI's host code under AddressSanitizer and UBSan: the library's
sources are rebuilt with both sanitizers on the host side (device code as
usual) and the ABI test file, which exercises every argument check without a
GPU, runs against that build in a child process."""
import os
import subprocess
import sys

import pytest

from nvfp4_quantized_paged_nvfp4kv_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    path = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_abi_checks_run_clean_under_asan_and_ubsan():
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("gcc sanitizer runtimes not installed")
    out = os.path.join(_build.BUILD, "sanitized")          # in-tree, git-ignored
    os.makedirs(out, exist_ok=True)
    nvcc = _build._nvcc()
    san = "-fsanitize=address,-fsanitize=undefined,-fno-sanitize-recover=undefined"
    common = ["-std=c++17", "-O1", "-g", "-Xcompiler", f"-fPIC,-fno-omit-frame-pointer,{san}",
              "-I", _build.INCLUDE, "-I", _build.CSRC] + _build.ARCH
    procs, objs = [], []
    for src in _build._sources():
        obj = os.path.join(out, os.path.basename(src) + ".o")
        objs.append(obj)
        procs.append(subprocess.Popen([nvcc] + common + ["-c", src, "-o", obj]))
    assert all(p.wait() == 0 for p in procs)
    lib = os.path.join(out, "libnvfp4kv_sanitized.so")
    subprocess.run([nvcc, "-shared", "-o", lib] + objs + _build.ARCH +
                   ["-cudart", "shared", "-Xcompiler", san.replace(",-fno-sanitize-recover=undefined", "")],
                   check=True)
    env = dict(os.environ, NVFP4KV_LIBRARY=lib, LD_PRELOAD=f"{asan}:{ubsan}",
               ASAN_OPTIONS="detect_leaks=0:halt_on_error=1:protect_shadow_gap=0",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu",
                        "tests/test_abi.py"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert "AddressSanitizer" not in r.stderr and "runtime error" not in r.stderr, tail
