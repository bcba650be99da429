"""GB300-native Super Bloom filter (SBF) insert and query over raw DNA.

A k-mer's minimizer (the minimum-hash m-mer among its k-m+1 windows) selects a
256-bit shard; each of its k-s+1 s-mers sets (insert) or tests (query) H bits in
that shard ("cuSBF: A Minimizer-Aware Bloom Filter for Genomic Sequence Data on
Modern GPUs", Sec. II-B, IV).  The work runs in the CUDA kernels of libsbf.so
(C ABI: include/sbf.h); this package is a thin binding plus seeded synthetic
inputs (``synth``).  Nothing here falls back to the CPU.

The library is loaded lazily: importing the package (e.g. for ``synth``) needs
neither a GPU nor a built library.
"""
from __future__ import annotations

__all__ = ["SuperBloomFilter", "build", "native", "synth"]


def build(verbose: bool = False) -> str:
    from . import build_lib
    return build_lib.build(verbose=verbose)


def __getattr__(name):
    if name == "native":
        from . import _native
        return _native
    if name == "SuperBloomFilter":
        from .filter import SuperBloomFilter
        return SuperBloomFilter
    raise AttributeError(name)
