"""Build libmoedec.so (the C-ABI CUDA library) in-tree for sm_103a.

Each .cu translation unit is compiled by its own nvcc process (in parallel),
then linked into mixture_experts_decode_gb300/libmoedec.so with the static
CUDA runtime.  A hash of the sources and flags skips up-to-date rebuilds.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmoedec.so")
BUILD_DIR = os.path.join(ROOT, "_build")
SOURCES = ["api.cu", "gate_up.cu", "down.cu", "grouped.cu", "align.cu", "router.cu", "requant.cu", "decode_fp4.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _digest(extra) -> str:
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["../../include/moedec.h"]
    for name in files:
        path = os.path.normpath(os.path.join(CSRC, name))
        if os.path.isfile(path):
            h.update(name.encode())
            with open(path, "rb") as f:
                h.update(f.read())
    h.update(repr((ARCH, NVCC_FLAGS, extra)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str = LIB) -> str:
    """Compile every CUDA source and link the library (default: the in-tree
    libmoedec.so; extra_flags/lib_path build a variant elsewhere); returns
    the library path."""
    extra = list(extra_flags)
    want = _digest(extra)
    stamp = lib_path + ".src-sha"
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == want:
                return lib_path
    # one object folder per output library (rebuilt in place: the stamp, not
    # the folder, records which sources it holds)
    obj_dir = os.path.join(BUILD_DIR, os.path.basename(lib_path) + ".objs")
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(want + "\n")
    return lib_path


if __name__ == "__main__":
    flags = [a for a in sys.argv[1:] if a.startswith("-X")]
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, extra_flags=flags))
