"""Checks that stand in for a device sanitizer (closed on this pool) and add
host-side ones, none of them needing a GPU:

- the debug build of the library (liblinattn_debug.so, -DLA_DEBUG, whose
  tensor-core kernels check their computed global-memory indices and report
  a failed check as LA_ERR_INTERNAL) builds, loads and exports what
  include/linattn.h declares, and its host-side validation behaves as the
  release build's; tests/test_gpu_debug_build.py runs it on the GPU;
- the oracle, built separately with the address and undefined-behaviour
  sanitizers, passes its pins (tests/test_oracle_pins.py) with every
  sanitizer report fatal."""
import os
import re
import subprocess
import sys
import tempfile

import pytest

import linear_attention_feature_gb300 as la
from linear_attention_feature_gb300 import build as labuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")
ORACLE_SRC = os.path.join(ROOT, "oracle", "la_oracle.c")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_0-9]+)\s*\(", text)))


def test_debug_library_builds_and_exports_the_boundary():
    path = labuild.build(debug=True)
    assert path.endswith("liblinattn_debug.so") and os.path.exists(path)
    lib = la.load_library(path)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared but not exported by the debug build"
    # host-side validation is the release build's: a null pointer is
    # rejected before anything is enqueued
    assert lib.la_forward(None, None, None, None, 1, 1, 8, 64, 1, None, 1, None) == 1
    assert lib.la_status_string(6) == b"LA_ERR_INTERNAL"


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True)
    path = p.stdout.strip()
    return path if p.returncode == 0 and os.path.isabs(path) and os.path.exists(path) else None


def test_oracle_pins_under_address_and_undefined_behaviour_sanitizers():
    asan = _runtime("libasan.so")
    if asan is None or _runtime("libubsan.so") is None:
        pytest.skip("gcc has no sanitizer runtimes here")
    with tempfile.TemporaryDirectory() as tmp:
        lib = os.path.join(tmp, "liblaoracle_san.so")
        subprocess.run(["gcc", "-std=c11", "-O1", "-g", "-fPIC", "-shared",
                        "-fno-omit-frame-pointer", "-fno-fast-math", "-ffp-contract=off",
                        "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                        "-o", lib, ORACLE_SRC, "-lm", "-lpthread"], check=True)
        env = dict(os.environ, LA_ORACLE_LIB=lib, LD_PRELOAD=asan,
                   ASAN_OPTIONS="detect_leaks=0:halt_on_error=1:abort_on_error=1",
                   UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
        r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
        assert "passed" in r.stdout
