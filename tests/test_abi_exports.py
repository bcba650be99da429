"""The C-ABI library builds, loads without a GPU and exports every entry
point include/sbf.h declares; the binding covers exactly those names.  No
compute call is made here."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sbf.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sbf_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from minimizer_sharded_bloom_gb300 import build_lib
    path = build_lib.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("sbf_create", "sbf_insert", "sbf_query", "sbf_copy_bits", "sbf_destroy",
                     "sbf_get_status", "sbf_last_error", "sbf_insert_host", "sbf_query_host"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_matches_header():
    from minimizer_sharded_bloom_gb300 import _native
    assert sorted(_native.SIGNATURES) == declared_functions()
    for name in declared_functions():
        assert callable(getattr(_native, name))


def test_binding_fails_loudly_without_library(tmp_path):
    from minimizer_sharded_bloom_gb300 import _native
    with pytest.raises(ImportError):
        _native._lib = None
        try:
            _native.load(str(tmp_path / "missing.so"))
        finally:
            _native._lib = None


def test_argument_errors_need_no_gpu(lib):
    """Host-side validation returns SBF_ERR_INVALID_ARG before touching CUDA."""
    from minimizer_sharded_bloom_gb300 import _native
    L = _native.load()
    assert not L.sbf_create(0, 31, 16, 28, 4, 0)
    assert "num_bits" in _native.last_error()
    assert not L.sbf_create(1 << 20, 33, 16, 28, 4, 0)
    assert not L.sbf_create(1 << 20, 31, 16, 28, 33, 0)
    assert not L.sbf_create(1 << 20, 31, 16, 28, 0, 0)
    assert not L.sbf_create(1 << 20, 31, 32, 28, 4, 0)
    assert L.sbf_insert(None, None, None, 1, None) == _native.SBF_ERR_INVALID_ARG
    assert L.sbf_query(None, None, None, 1, None, None) == _native.SBF_ERR_INVALID_ARG
    assert L.sbf_num_shards(None) == 0
    assert L.sbf_test_wait_timeout(None, 1, None) == _native.SBF_ERR_INVALID_ARG
    L.sbf_destroy(None)


def test_create_without_gpu_fails_cleanly(lib):
    """On a machine without a CUDA device creation reports an error (no CPU
    fallback, no crash)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from minimizer_sharded_bloom_gb300 import _native
    L = _native.load()
    assert not L.sbf_create(1 << 20, 31, 16, 28, 4, 0)
    assert _native.last_error()


def test_probe_library_exports_every_declared_symbol(lib):
    """The benchmark's ceiling probes (include/sbf_probes.h) are a library of
    their own; every declared entry point is exported, the binding loads them
    all, and invalid arguments are refused before any launch."""
    from minimizer_sharded_bloom_gb300 import build_lib, probes
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "sbf_probes.h")).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(sbf_probe_[a-z_]+)\s*\(", text)))
    assert names == ["sbf_probe_alu", "sbf_probe_read", "sbf_probe_rmw", "sbf_probe_sm_count"]
    P = ctypes.CDLL(build_lib.PROBE_LIB)
    for name in names:
        assert hasattr(P, name), name
    L = probes.load()
    assert L.sbf_probe_rmw(0, None, 3, 1, 1, 1, 32, None) == -1       # no buffer, rows not a power of two
    assert L.sbf_probe_read(9, None, 4, 1, 1, 1, 32, None, None) == -1  # unknown mode
    assert L.sbf_probe_alu(7, 1, 1, 32, None, None, None) == -1         # unknown kind
