"""The oracle's C code under AddressSanitizer and UBSan: the same source is
built with both sanitizers and the oracle's own test files run against it in a
child process, so any out-of-bounds access, use of uninitialised stack
arrays through bad indexing, or undefined integer or shift arithmetic in the
checker fails here instead of passing silently."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_TESTS = ["tests/test_oracle_format.py", "tests/test_oracle_quant.py", "tests/test_oracle_attention.py",
                "tests/test_oracle_global_scale.py", "tests/test_oracle_extend.py"]


def _runtime(name):
    path = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_oracle_runs_clean_under_asan_and_ubsan():
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if asan is None or ubsan is None:
        pytest.skip("gcc sanitizer runtimes not installed")
    out = os.path.join(ROOT, "oracle", "_build")            # in-tree, git-ignored
    os.makedirs(out, exist_ok=True)
    lib = os.path.join(out, "liboracle_sanitized.so")
    flags = [f for f in oracle.CFLAGS if f != "-O2"] + ["-O1", "-g", "-fno-omit-frame-pointer",
                                                        "-fsanitize=address,undefined",
                                                        "-fno-sanitize-recover=undefined"]
    subprocess.run(["gcc"] + flags + [os.path.join(ROOT, "oracle", "nvfp4kv_oracle.c"), "-o", lib, "-lm"],
                   check=True)
    env = dict(os.environ, NVFP4KV_ORACLE_LIB=lib, LD_PRELOAD=f"{asan}:{ubsan}",
               ASAN_OPTIONS="detect_leaks=0:halt_on_error=1", UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu"]
                       + ORACLE_TESTS, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert "AddressSanitizer" not in r.stderr and "runtime error" not in r.stderr, tail
