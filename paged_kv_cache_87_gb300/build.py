"""Build libpagedkv.so in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel; the objects link into
``paged_kv_cache_87_gb300/libpagedkv.so``.  The build is content-addressed: a
SHA-256 over every source and header, the compile and link flags and the
output of ``nvcc --version`` is stored beside the objects, and the library is
rebuilt whenever that digest changes (a modification time is never trusted).
"""
from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv.so")
    return path


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "pagedkv.h"), __file__]


STAMP = os.path.join(BUILD, "libpagedkv.sha256")
LINK_FLAGS = ["-shared", "-cudart", "static"]
_nvcc_version: dict[str, str] = {}


def nvcc_version(cc: str) -> str:
    if cc not in _nvcc_version:
        r = subprocess.run([cc, "--version"], capture_output=True, text=True)
        _nvcc_version[cc] = r.stdout + r.stderr
    return _nvcc_version[cc]


def digest(extra_flags: list[str] | None = None, cc: str | None = None) -> str:
    """SHA-256 of what the library is built from: every input file (name and bytes),
    the architecture, compile and link flags, and the compiler's version string."""
    h = hashlib.sha256()
    for f in sorted(_inputs()):
        h.update(os.path.relpath(f, ROOT).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    for part in (ARCH, NVCC_FLAGS, extra_flags or [], LINK_FLAGS):
        h.update(("\x1f".join(part) + "\0").encode())
    h.update(nvcc_version(cc or nvcc()).encode())
    return h.hexdigest()


def up_to_date(extra_flags: list[str] | None = None) -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as f:
        return f.read().strip() == digest(extra_flags)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if not force and up_to_date(extra):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    want = digest(extra, cc)

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, *LINK_FLAGS, "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP + f".tmp{os.getpid()}", "w") as f:
        f.write(want + "\n")
    os.replace(STAMP + f".tmp{os.getpid()}", STAMP)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv))
