"""Build libpkv.so (the sm_103a CUDA library) in-tree with nvcc.

Each .cu file is compiled to an object in parallel, then linked into a shared
library with the CUDA runtime linked statically.  Output:
``paged_kv_attention_forward_gb300/_build/libpkv.so``.
"""
from __future__ import annotations

import hashlib
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpkv.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


# the files the attention kernels are compiled from (a profile of those kernels stays
# valid while these are unchanged)
ATTENTION_SOURCES = ("pkv_attention_impl.cuh", "pkv_attention.cu", "pkv_attention_quant.cu", "pkv_ptx.cuh",
                     "pkv_internal.h", "pkv_attention_tc.cuh", "pkv_tc.cuh")


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def code_text(text: str) -> str:
    """C/C++/CUDA source with its comments removed and whitespace runs collapsed: what
    the compiler sees, up to line positions."""
    return " ".join(_COMMENT.sub(" ", text).split())


def source_digest(names=None) -> str:
    """Hash of every source and header the library is built from (the rebuild stamp), or,
    for the named files of csrc/, of their code alone (comments and layout do not count,
    so a profile of the kernels stays valid across comment edits)."""
    h = hashlib.sha256()
    if names is None:
        files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)) + [os.path.join(INCLUDE, "pkv.h")]
    else:
        files = [os.path.join(CSRC, f) for f in names]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            data = fh.read()
        h.update(data if names is None else code_text(data.decode("utf-8")).encode())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    digest = source_digest()
    stamp = os.path.join(BUILD, "libpkv.digest")
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == digest:
        return LIB
    cc = nvcc()
    srcs = sources()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(digest)
    return LIB


if __name__ == "__main__":  # pragma: no cover
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))
