"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI (via the thin binding) and the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import pytest

import oracle

MAIN = dict(k=31, m=16, s=28, H=4)


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from minimizer_sharded_bloom_gb300 import build_lib
    build_lib.build()
    return torch


def to_dev(torch, seq: np.ndarray, offsets: np.ndarray, pad_front: int = 0):
    """Device copies; pad_front > 0 shifts the sequence start by that many
    bytes inside a larger allocation (an unaligned seq pointer)."""
    buf = torch.zeros(seq.size + pad_front + 16, dtype=torch.uint8, device="cuda")
    if seq.size:
        buf[pad_front:pad_front + seq.size] = torch.from_numpy(np.ascontiguousarray(seq)).cuda()
    dseq = buf[pad_front:]
    doff = torch.from_numpy(np.ascontiguousarray(offsets, dtype=np.int64)).cuda()
    return dseq, doff


def gpu_insert(torch, sbf, seq, offsets, pad_front=0):
    dseq, doff = to_dev(torch, seq, offsets, pad_front)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    return sbf


def gpu_query(torch, sbf, seq, offsets, pad_front=0, sentinel=None):
    dseq, doff = to_dev(torch, seq, offsets, pad_front)
    n_words = (int(offsets[-1]) + 31) // 32 + 2
    out = torch.zeros(n_words, dtype=torch.int32, device="cuda")
    if sentinel is not None:
        out.fill_(sentinel)
    sbf.query(dseq, doff, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


def oracle_image(seq, offsets, params, num_bits, seed, nthreads=8, alphabet="dna"):
    F = oracle.new_filter(num_bits)
    oracle.insert(F, seq, offsets, params["k"], params["m"], params["s"], params["H"], seed,
                  nthreads=nthreads, alphabet=alphabet)
    return F


def oracle_answers(F, seq, offsets, params, seed, nthreads=8, alphabet="dna"):
    return oracle.query(F, seq, offsets, params["k"], params["m"], params["s"], params["H"], seed,
                        nthreads=nthreads, alphabet=alphabet)


def assert_words_equal(gpu_words, oracle_words, offsets):
    """Compare the answer words the contract defines: [offsets[0] >> 5,
    (offsets[-1] + 31) >> 5)."""
    lo, hi = int(offsets[0]) >> 5, (int(offsets[-1]) + 31) >> 5
    g = gpu_words[lo:hi]
    o = oracle_words[lo:hi]
    if not np.array_equal(g, o):
        bad = np.flatnonzero(g != o)
        w = bad[0]
        raise AssertionError(f"{bad.size} answer words differ; first word {lo + w}: "
                             f"gpu {g[w]:#010x} oracle {o[w]:#010x}")


def assert_images_equal(gpu_img, oracle_img):
    if not np.array_equal(gpu_img, oracle_img):
        bad = np.flatnonzero((gpu_img != oracle_img).any(axis=1))
        s = bad[0]
        raise AssertionError(f"{bad.size} shards differ; first shard {s}: gpu "
                             f"{[hex(x) for x in gpu_img[s]]} oracle {[hex(x) for x in oracle_img[s]]}")


def answer_bits(words: np.ndarray, positions: np.ndarray) -> np.ndarray:
    positions = np.asarray(positions, dtype=np.int64)
    return ((words[positions >> 5] >> (positions & 31).astype(np.uint32)) & 1).astype(bool)
