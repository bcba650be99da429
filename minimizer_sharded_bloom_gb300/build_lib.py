"""Build libsbf.so in-tree with nvcc for GB300 (sm_103a).

Every .cu unit under csrc/ compiles in parallel to an object under _build/,
then nvcc links the shared library _build/libsbf.so.  Objects are rebuilt when
their source or any header is newer.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsbf.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-DSBF_WITH_SWEEP",
          f"-I{INCLUDE}"]


def have_zlib() -> bool:
    """gzip input needs zlib's header and library on the build machine."""
    return os.path.exists("/usr/include/zlib.h") and any(
        glob.glob(os.path.join(d, "libz.so*")) for d in
        ("/usr/lib/x86_64-linux-gnu", "/usr/lib/aarch64-linux-gnu", "/usr/lib64", "/usr/lib", "/lib64"))


ZLIB = have_zlib()
if ZLIB:
    CFLAGS.append("-DSBF_WITH_ZLIB")


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsbf")
    return path


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    hs.append(os.path.join(INCLUDE, "sbf.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, hdr_time: float, verbose: bool) -> str:
    obj = os.path.join(OUT, os.path.basename(src)[:-3] + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time):
        return obj
    cmd = [nvcc(), *ARCH, *CFLAGS, "-c", src, "-o", obj + ".tmp"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose and res.stderr:
        with open(obj + ".ptxas.txt", "w") as f:
            f.write(res.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(jobs: int | None = None, verbose: bool = False) -> str:
    """Compile and link libsbf.so; returns its path."""
    os.makedirs(OUT, exist_ok=True)
    hdr = _headers_mtime()
    srcs = sources()
    # the heavy specialisation units first
    srcs.sort(key=lambda s: ("sbf_inst" not in s, s))
    jobs = jobs or max(1, min(len(srcs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, hdr, verbose), srcs))
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= max(os.path.getmtime(o) for o in objs):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs] + (["-lz"] if ZLIB else [])
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    import time
    t0 = time.time()
    print(build(verbose="-v" in sys.argv), f"{time.time() - t0:.1f}s")
