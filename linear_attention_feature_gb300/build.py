"""In-tree build of liblinattn.so for sm_103a (nvcc, no cmake).

Each .cu translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically.  Outputs go to
``linear_attention_feature_gb300/_build/`` (git-ignored).  ``build(debug=True)``
makes ``liblinattn_debug.so`` in ``_build_debug/``: the same sources with
``-DLA_DEBUG``, whose kernels check their computed global-memory indices and
report a failed check as LA_ERR_INTERNAL (a stand-in for a device sanitizer).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "liblinattn.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
DEBUG_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_DIR, "liblinattn_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu"))


def _inputs_digest(extra_flags=()) -> str:
    h = hashlib.sha256()
    files = sources() + sorted(
        os.path.join(d, f) for d in (CSRC, INCLUDE) for f in os.listdir(d)
        if f.endswith((".h", ".cuh")))
    for p in files:
        h.update(p.encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join([*NVCC_FLAGS, *extra_flags]).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link liblinattn.so (liblinattn_debug.so with `debug`);
    returns its path.  Skips the work when the sources are unchanged since
    the last build."""
    out_dir, lib_path = (DEBUG_DIR, DEBUG_LIB_PATH) if debug else (OUT_DIR, LIB_PATH)
    mode_flags = ["-DLA_DEBUG"] if debug else []
    os.makedirs(out_dir, exist_ok=True)
    stamp = os.path.join(out_dir, "inputs.sha256")
    digest = _inputs_digest(mode_flags)
    if (not force and os.path.exists(lib_path) and os.path.exists(stamp)
            and open(stamp).read() == digest):
        return lib_path
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *mode_flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
