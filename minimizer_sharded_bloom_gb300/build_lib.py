"""Build libsbf.so in-tree with nvcc for GB300 (sm_103a).

Every .cu unit under csrc/ compiles in parallel to an object under _build/,
then nvcc links the shared library _build/libsbf.so.  The benchmark's ceiling
probes (probes/*.cu) link into _build/libsbf_probes.so the same way.  Objects
are rebuilt when their source or any header is newer.
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
PROBES = os.path.join(HERE, "probes")
PROBE_LIB = os.path.join(OUT, "libsbf_probes.so")
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


def probe_sources():
    return sorted(glob.glob(os.path.join(PROBES, "*.cu")))


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    hs += glob.glob(os.path.join(INCLUDE, "*.h"))
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


def _link(lib: str, objs, extra) -> None:
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs):
        return
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs] + extra
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)


def build(jobs: int | None = None, verbose: bool = False) -> str:
    """Compile and link libsbf.so and libsbf_probes.so; returns libsbf's path."""
    os.makedirs(OUT, exist_ok=True)
    hdr = _headers_mtime()
    srcs = sources()
    # the heavy specialisation units first
    srcs.sort(key=lambda s: ("sbf_inst" not in s, s))
    psrcs = probe_sources()
    jobs = jobs or max(1, min(len(srcs) + len(psrcs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, hdr, verbose), srcs + psrcs))
    _link(LIB, objs[:len(srcs)], ["-lz"] if ZLIB else [])
    if psrcs:
        _link(PROBE_LIB, objs[len(srcs):], [])
    return LIB


if __name__ == "__main__":
    import sys
    import time
    t0 = time.time()
    print(build(verbose="-v" in sys.argv), f"{time.time() - t0:.1f}s")
