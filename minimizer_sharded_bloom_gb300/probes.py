"""ctypes binding of libsbf_probes (include/sbf_probes.h) and the timing of
its micro-benchmarks with CUDA events.

The probes measure, on the GPU at hand, the ceilings the filter kernels are
reported against: scattered 32-byte read-modify-writes (the insert's shard
updates), scattered 32-byte reads (the query's shard loads) and the rate of
the integer instruction mix that dominates both kernels.  PyTorch supplies
device buffers, streams and events only; the work runs in the probe kernels.
"""
from __future__ import annotations

import ctypes
import os
import statistics
import threading

from . import build_lib

_lock = threading.Lock()
_lib = None

ALU_KINDS = {"mix": 0, "lop3": 1, "shf": 2, "imad": 3, "min64": 4}
RMW_MODES = {"red4": 0, "red_lanes": 1, "ld_st": 2, "red_queue": 3}
READ_MODES = {"ld_nc": 0, "ld_nc_L2_64B": 1, "ld_nc_L2_128B": 2, "ld_nc_L2_256B": 3,
              "cp_async": 4, "cp_async_L2_64B": 5, "bulk32": 6}


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(build_lib.PROBE_LIB):
                raise ImportError(f"libsbf_probes.so not built ({build_lib.PROBE_LIB})")
            L = ctypes.CDLL(build_lib.PROBE_LIB)
            vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
            L.sbf_probe_sm_count.argtypes = [ctypes.POINTER(ctypes.c_int)]
            L.sbf_probe_alu.argtypes = [i32, i32, i32, i32, vp, vp, ctypes.POINTER(ctypes.c_double)]
            L.sbf_probe_rmw.argtypes = [i32, vp, u64, i64, u64, i32, i32, vp]
            L.sbf_probe_read.argtypes = [i32, vp, u64, i64, u64, i32, i32, vp, vp]
            for name in ("sbf_probe_sm_count", "sbf_probe_alu", "sbf_probe_rmw", "sbf_probe_read"):
                getattr(L, name).restype = i32
            _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} failed ({rc})")


def sm_count() -> int:
    n = ctypes.c_int(0)
    _check(load().sbf_probe_sm_count(ctypes.byref(n)), "sbf_probe_sm_count")
    return n.value


def _median_time(torch, launch, reps: int) -> float:
    """Median seconds per launch over `reps` launches, each bracketed by
    events on the current stream, after one untimed launch."""
    stream = torch.cuda.current_stream()
    launch()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    return statistics.median(times)


def alu_rate(torch, kind: str = "mix", iters: int = 2000, threads: int = 256, blocks_per_sm: int = 8,
             reps: int = 5) -> dict:
    """Instructions per second of one probe kind, all SMs fully occupied."""
    L = load()
    sms = sm_count()
    blocks = sms * blocks_per_sm
    sink = torch.empty(blocks * threads, dtype=torch.int32, device="cuda")
    ops = ctypes.c_double(0)
    st = torch.cuda.current_stream().cuda_stream

    def launch():
        _check(L.sbf_probe_alu(ALU_KINDS[kind], iters, blocks, threads, sink.data_ptr(), st,
                               ctypes.byref(ops)), "sbf_probe_alu")
    t = _median_time(torch, launch, reps)
    return {"kind": kind, "ops_per_s": ops.value / t, "ms": 1e3 * t, "sms": sms,
            "ops_per_sm_clock_at_2070MHz": ops.value / t / sms / 2.07e9}


def rmw_rate(torch, mode: str = "red4", gib: int = 8, n_updates: int = 100_000_000, threads: int = 256,
             blocks_per_sm: int = 8, reps: int = 3, buf=None) -> dict:
    """Rows per second of scattered 32-byte read-modify-writes over a gib-GiB
    buffer (or the given int64 device tensor, whose size must be a power of
    two times 32 bytes)."""
    L = load()
    own = buf is None
    if own:
        buf = torch.zeros((gib << 30) // 8, dtype=torch.int64, device="cuda")
    n_rows = buf.numel() // 4
    blocks = sm_count() * blocks_per_sm
    st = torch.cuda.current_stream().cuda_stream
    seed = [1]

    def launch():
        seed[0] += 0x9E3779B97F4A7C15
        _check(L.sbf_probe_rmw(RMW_MODES[mode], buf.data_ptr(), n_rows, n_updates, seed[0] % 2**64, blocks,
                               threads, st), "sbf_probe_rmw")
    t = _median_time(torch, launch, reps)
    if own:
        del buf
        torch.cuda.empty_cache()
    return {"mode": mode, "rows_per_s": n_updates / t, "ms": 1e3 * t, "buffer_gib": n_rows * 32 / 2**30,
            "updates": n_updates}


def read_rate(torch, mode: str = "ld_nc", gib: int = 8, n_reads: int = 100_000_000, threads: int = 256,
              blocks_per_sm: int = 8, reps: int = 3, buf=None) -> dict:
    """Rows per second of scattered 32-byte reads over a gib-GiB buffer."""
    L = load()
    own = buf is None
    if own:
        buf = torch.zeros((gib << 30) // 8, dtype=torch.int64, device="cuda")
    n_rows = buf.numel() // 4
    blocks = sm_count() * blocks_per_sm
    sink = torch.empty(blocks * threads, dtype=torch.int64, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    seed = [2]

    def launch():
        seed[0] += 0x9E3779B97F4A7C15
        _check(L.sbf_probe_read(READ_MODES[mode], buf.data_ptr(), n_rows, n_reads, seed[0] % 2**64, blocks,
                                threads, sink.data_ptr(), st), "sbf_probe_read")
    t = _median_time(torch, launch, reps)
    if own:
        del buf
        torch.cuda.empty_cache()
    return {"mode": mode, "rows_per_s": n_reads / t, "ms": 1e3 * t, "buffer_gib": n_rows * 32 / 2**30,
            "reads": n_reads}


def launch_each_once(torch, gib: int = 2, rows: int = 25_000_000) -> None:
    """One launch of every memory probe (each RMW and read form) over a gib-GiB
    buffer, rows rows each: the command a counter capture (ncu) profiles."""
    L = load()
    buf = torch.zeros((gib << 30) // 8, dtype=torch.int64, device="cuda")
    blocks = sm_count() * 8
    sink = torch.empty(blocks * 256, dtype=torch.int64, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for name, mode in RMW_MODES.items():
        _check(L.sbf_probe_rmw(mode, buf.data_ptr(), buf.numel() // 4, rows, 12345 + mode, blocks, 256, st), name)
    for name, mode in READ_MODES.items():
        _check(L.sbf_probe_read(mode, buf.data_ptr(), buf.numel() // 4, rows, 777 + mode, blocks, 256,
                                sink.data_ptr(), st), name)
    torch.cuda.synchronize()


def main(argv=None) -> None:
    """python -m minimizer_sharded_bloom_gb300.probes [--once]: every probe's
    rate as one JSON line (8 GiB buffer, 118 M rows), or, with --once, one
    launch of each memory probe for a counter capture."""
    import argparse
    import json
    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--once", action="store_true")
    args = ap.parse_args(argv)
    build_lib.build()
    torch.cuda.set_device(0)
    if args.once:
        launch_each_once(torch)
        return
    out = {"sms": sm_count(), "alu": [alu_rate(torch, k) for k in ALU_KINDS]}
    buf = torch.zeros((8 << 30) // 8, dtype=torch.int64, device="cuda")
    out["rmw"] = [rmw_rate(torch, m, n_updates=118_000_000, buf=buf) for m in RMW_MODES]
    out["read"] = [read_rate(torch, m, n_reads=118_000_000, buf=buf) for m in READ_MODES]
    print(json.dumps(out))


if __name__ == "__main__":
    main()
