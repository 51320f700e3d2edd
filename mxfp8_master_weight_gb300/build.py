"""Build the sm_103a CUDA library in-tree (nvcc, no cmake, no torch extension).

Produces ``mxfp8_master_weight_gb300/libmxfp8_gb300.so`` from the translation
units in ``csrc/``: each unit is compiled in parallel, then linked with the
static CUDA runtime into one shared library with a plain C ABI
(``include/mxfp8_partial.h``).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import re
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libmxfp8_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
UNITS = ["capi.cu", "amax.cu", "cast_f32.cu", "cast_bf16.cu", "cast_f32_unaligned.cu",
         "cast_bf16_unaligned.cu", "cast_bf16_unaligned_f16.cu", "fused_f32.cu", "fused_bf16.cu",
         "misc.cu", "noalloc.cu", "nvfp4.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources():
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "mxfp8_partial.h"))
    return files


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def code_text(text: str) -> str:
    """A source file's code with comments dropped and whitespace runs collapsed (the
    sources hold no comment markers inside string literals)."""
    return " ".join(_COMMENT.sub(" ", text).split())


def source_digest() -> str:
    """SHA-256 over the code of every source file of the library (names and contents,
    comments and layout excluded: editing a comment changes neither the kernels nor
    the digest that build stamps and recorded profiles refer to)."""
    h = hashlib.sha256()
    for f in _sources():
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()


# Translation units that hold host code only (argument validation, dispatch, the
# allocation-free entry point's set-up): edits there leave every kernel unchanged.
HOST_ONLY_UNITS = ("capi.cu", "noalloc.cu")


def kernel_digest() -> str:
    """SHA-256 over the code of the device-side sources only (every csrc file except the
    host-only units, comments excluded): the key of recorded per-kernel counters, which
    a host-side edit does not invalidate."""
    h = hashlib.sha256()
    for f in _sources():
        name = os.path.basename(f)
        if name in HOST_ONLY_UNITS or not f.startswith(CSRC):
            continue
        h.update(name.encode())
        with open(f, encoding="utf-8") as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()


def cflags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
                   f"-I{INCLUDE}", f"-I{CSRC}", *extra]


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if the sources changed) and return the library path."""
    digest = source_digest()
    stamp = LIB_PATH + ".sha256"
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_unit(unit):
        obj = os.path.join(BUILD_DIR, unit.replace(".cu", ".o"))
        cmd = [nvcc, *cflags(extra_flags), "-c", os.path.join(CSRC, unit), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
