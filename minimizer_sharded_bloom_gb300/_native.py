"""ctypes binding of libsbf (include/sbf.h), same names, argument marshalling only.

Every computation runs in the library's CUDA kernels.  If libsbf.so has not
been built, or cannot be loaded, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build_lib

SBF_OK = 0
SBF_ERR_INVALID_ARG = -1
SBF_ERR_CUDA = -2
SBF_ERR_OOM = -3
SBF_ERR_BAD_OFFSETS = -4

# every entry point the header declares: name -> (restype, argtypes)
_vp, _u64, _i64, _i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
_ip = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "sbf_create": (_vp, [_u64, _i32, _i32, _i32, _i32, _u64]),
    "sbf_create_alphabet": (_vp, [_u64, _i32, _i32, _i32, _i32, _u64, _i32]),
    "sbf_create_ex": (_vp, [_u64, _i32, _i32, _i32, _i32, _u64, _i32, _i32]),
    "sbf_get_flags": (_i32, [_vp]),
    "sbf_query_dense": (_i32, [_vp, _vp, _i64, _i64, _vp, _vp]),
    "sbf_get_alphabet": (_i32, [_vp]),
    "sbf_destroy": (None, [_vp]),
    "sbf_insert": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "sbf_query": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "sbf_insert_host": (_i32, [_vp, _vp, _vp, _i64, _vp]),
    "sbf_query_host": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "sbf_query_host_noalloc": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "sbf_set_host_chunk": (_i32, [_vp, _i64]),
    "sbf_set_host_mode": (_i32, [_vp, _i32]),
    "sbf_copy_bits": (_i32, [_vp, _vp, _u64, _vp]),
    "sbf_load_bits": (_i32, [_vp, _vp, _u64, _vp]),
    "sbf_clear": (_i32, [_vp, _vp]),
    "sbf_num_shards": (_u64, [_vp]),
    "sbf_get_params": (_i32, [_vp, _ip, _ip, _ip, _ip, ctypes.POINTER(ctypes.c_uint64)]),
    "sbf_is_specialized": (_i32, [_vp]),
    "sbf_get_status": (_i32, [_vp, _vp]),
    "sbf_test_wait_timeout": (_i32, [_vp, _i32, _vp]),
    "sbf_last_error": (ctypes.c_char_p, []),
    "sbf_fastx_open": (_vp, [ctypes.c_char_p]),
    "sbf_fastx_next": (_i64, [_vp, _vp, _i64, _vp, _i64, ctypes.POINTER(ctypes.c_int64)]),
    "sbf_fastx_pending_bases": (_i64, [_vp]),
    "sbf_fastx_close": (None, [_vp]),
    "sbf_fastx_has_gzip": (_i32, []),
    "sbf_insert_fastx": (_i32, [_vp, ctypes.c_char_p, _i64, ctypes.POINTER(ctypes.c_int64),
                                ctypes.POINTER(ctypes.c_int64)]),
    "sbf_query_fastx": (_i32, [_vp, ctypes.c_char_p, _i64, _vp, _vp]),
}

# sbf_fastx_sink: int (*)(void *user, const char *seq, const int64_t *offsets,
#                         int64_t n, const uint32_t *out_bits)
FASTX_SINK = ctypes.CFUNCTYPE(ctypes.c_int, _vp, _vp, _vp, _i64, _vp)

_lock = threading.Lock()
_lib = None


class SBFError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        super().__init__(f"{where} failed ({code}): {message}")
        self.code = code


def library_path() -> str:
    return build_lib.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libsbf.so (built by build_lib.build()); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or library_path()
            if not os.path.exists(p):
                raise ImportError(f"libsbf.so not built ({p}); run "
                                  "minimizer_sharded_bloom_gb300.build_lib.build() first")
            L = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def last_error() -> str:
    msg = load().sbf_last_error()
    return msg.decode() if msg else ""


def check(rc: int, where: str) -> None:
    if rc != SBF_OK:
        raise SBFError(rc, where, last_error())


# ---- same-name wrappers (raw pointers as Python ints) ----------------------

def sbf_create(num_bits: int, k: int, m: int, s: int, H: int, seed: int) -> int:
    h = load().sbf_create(num_bits, k, m, s, H, seed & (2**64 - 1))
    if not h:
        raise SBFError(SBF_ERR_INVALID_ARG, "sbf_create", last_error())
    return h


def sbf_destroy(f: int) -> None:
    load().sbf_destroy(f)


def sbf_insert(f: int, seq: int, offsets: int, n: int, stream: int = 0) -> None:
    check(load().sbf_insert(f, seq, offsets, n, stream), "sbf_insert")


def sbf_query(f: int, seq: int, offsets: int, n: int, out_bits: int, stream: int = 0) -> None:
    check(load().sbf_query(f, seq, offsets, n, out_bits, stream), "sbf_query")


def sbf_insert_host(f: int, seq: int, offsets: int, n: int, stream: int = 0) -> None:
    check(load().sbf_insert_host(f, seq, offsets, n, stream), "sbf_insert_host")


def sbf_query_host(f: int, seq: int, offsets: int, n: int, out_bits: int, stream: int = 0) -> None:
    check(load().sbf_query_host(f, seq, offsets, n, out_bits, stream), "sbf_query_host")


def sbf_query_host_noalloc(f: int, seq: int, offsets: int, n: int, out_bits: int,
                           stream: int = 0) -> None:
    check(load().sbf_query_host_noalloc(f, seq, offsets, n, out_bits, stream),
          "sbf_query_host_noalloc")


def sbf_set_host_chunk(f: int, positions: int) -> None:
    check(load().sbf_set_host_chunk(f, positions), "sbf_set_host_chunk")


def sbf_set_host_mode(f: int, mode: int) -> None:
    check(load().sbf_set_host_mode(f, mode), "sbf_set_host_mode")


def sbf_copy_bits(f: int, dst: int, dst_bytes: int, stream: int = 0) -> None:
    check(load().sbf_copy_bits(f, dst, dst_bytes, stream), "sbf_copy_bits")


def sbf_load_bits(f: int, src: int, src_bytes: int, stream: int = 0) -> None:
    check(load().sbf_load_bits(f, src, src_bytes, stream), "sbf_load_bits")


def sbf_clear(f: int, stream: int = 0) -> None:
    check(load().sbf_clear(f, stream), "sbf_clear")


def sbf_num_shards(f: int) -> int:
    return int(load().sbf_num_shards(f))


# Sec. IV-A alphabets (SBF_ALPHABET_* of sbf.h)
ALPHABET_DNA, ALPHABET_PROTEIN, ALPHABET_DNA_TRIPLET = 0, 1, 2
ALPHABETS = {"dna": ALPHABET_DNA, "protein": ALPHABET_PROTEIN, "dna_triplet": ALPHABET_DNA_TRIPLET,
             "triplet": ALPHABET_DNA_TRIPLET}


def alphabet_id(alphabet) -> int:
    if isinstance(alphabet, str):
        try:
            return ALPHABETS[alphabet.lower()]
        except KeyError:
            raise ValueError(f"unknown alphabet {alphabet!r}") from None
    return int(alphabet)


def sbf_create_alphabet(num_bits: int, k: int, m: int, s: int, H: int, seed: int, alphabet) -> int:
    h = load().sbf_create_alphabet(num_bits, k, m, s, H, seed & (2**64 - 1), alphabet_id(alphabet))
    if not h:
        raise SBFError(SBF_ERR_INVALID_ARG, "sbf_create_alphabet", last_error())
    return h


# creation flags (SBF_FLAG_* of sbf.h)
FLAG_HASHED_SECTORS = 1
FLAG_RUNTIME_KERNELS = 2


def sbf_create_ex(num_bits: int, k: int, m: int, s: int, H: int, seed: int, alphabet, flags: int) -> int:
    h = load().sbf_create_ex(num_bits, k, m, s, H, seed & (2**64 - 1), alphabet_id(alphabet), flags)
    if not h:
        raise SBFError(SBF_ERR_INVALID_ARG, "sbf_create_ex", last_error())
    return h


def sbf_get_flags(f: int) -> int:
    return int(load().sbf_get_flags(f))


def sbf_query_dense(f: int, seq: int, n_records: int, record_len: int, out_bits: int, stream: int = 0) -> None:
    check(load().sbf_query_dense(f, seq, n_records, record_len, out_bits, stream), "sbf_query_dense")


def sbf_get_alphabet(f: int) -> int:
    return int(load().sbf_get_alphabet(f))


def sbf_get_params(f: int):
    k, m, s, H = (ctypes.c_int() for _ in range(4))
    seed = ctypes.c_uint64()
    check(load().sbf_get_params(f, ctypes.byref(k), ctypes.byref(m), ctypes.byref(s),
                                ctypes.byref(H), ctypes.byref(seed)), "sbf_get_params")
    return k.value, m.value, s.value, H.value, seed.value


def sbf_is_specialized(f: int) -> bool:
    return bool(load().sbf_is_specialized(f))


def sbf_get_status(f: int, stream: int = 0) -> int:
    return int(load().sbf_get_status(f, stream))


def sbf_test_wait_timeout(f: int, polls: int, stream: int = 0) -> None:
    check(load().sbf_test_wait_timeout(f, polls, stream), "sbf_test_wait_timeout")


def sbf_last_error() -> str:
    return last_error()


def sbf_fastx_open(path: str) -> int:
    h = load().sbf_fastx_open(path.encode())
    if not h:
        raise SBFError(SBF_ERR_INVALID_ARG, "sbf_fastx_open", last_error())
    return h


def sbf_fastx_next(r: int, seq: int, seq_cap: int, offsets: int, max_records: int):
    bases = ctypes.c_int64(0)
    n = int(load().sbf_fastx_next(r, seq, seq_cap, offsets, max_records, ctypes.byref(bases)))
    if n < 0:
        raise SBFError(n, "sbf_fastx_next", last_error())
    return n, bases.value


def sbf_fastx_pending_bases(r: int) -> int:
    return int(load().sbf_fastx_pending_bases(r))


def sbf_fastx_close(r: int) -> None:
    load().sbf_fastx_close(r)


def sbf_fastx_has_gzip() -> bool:
    return bool(load().sbf_fastx_has_gzip())


def sbf_insert_fastx(f: int, path: str, batch_bases: int = 0):
    recs, bases = ctypes.c_int64(0), ctypes.c_int64(0)
    check(load().sbf_insert_fastx(f, path.encode(), batch_bases, ctypes.byref(recs),
                                  ctypes.byref(bases)), "sbf_insert_fastx")
    return recs.value, bases.value


def sbf_query_fastx(f: int, path: str, sink, batch_bases: int = 0) -> None:
    """sink(seq_ptr, offsets_ptr, n, bits_ptr) -> int, called per batch."""
    cb = FASTX_SINK(lambda user, s, o, n, b: int(sink(s, o, n, b) or 0))
    check(load().sbf_query_fastx(f, path.encode(), batch_bases, cb, None), "sbf_query_fastx")
