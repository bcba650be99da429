"""GPU parity of hash-chosen sectors (SBF_FLAG_HASHED_SECTORS), an extension
of the paper's layout for H < 4: every kernel family against the oracle with
sectors = 1, image and answers bit for bit.

* the sweep points with H = 1 and 2 (k = 31), which have compiled strip
  kernels for the paper's layout: with the flag they run on the
  runtime-parameter kernels;
* the runtime-parameter kernel: H = 3 and random (k, m, s);
* the protein and triplet alphabet kernels;
* H >= 4: the flag changes nothing.
"""
import numpy as np
import pytest

import oracle
from minimizer_sharded_bloom_gb300 import synth
from _gpu_helpers import assert_images_equal, assert_words_equal, gpu_insert, gpu_query, need_gpu

pytestmark = pytest.mark.gpu


def _filter(bits, params, seed, alphabet="dna", sectors="hashed"):
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter
    return SuperBloomFilter(bits, seed=seed, alphabet=alphabet, sectors=sectors, **params)


def _check(torch, params, bits, seed, ins, qry, alphabet="dna", specialized=None):
    sbf = _filter(bits, params, seed, alphabet)
    if specialized is not None:
        assert sbf.specialized == specialized
    from minimizer_sharded_bloom_gb300 import _native as N
    assert N.sbf_get_flags(sbf.handle) == N.FLAG_HASHED_SECTORS
    gpu_insert(torch, sbf, ins.seq, ins.offsets)
    assert sbf.status() == 0
    k, m, s, H = params["k"], params["m"], params["s"], params["H"]
    F = oracle.new_filter(bits)
    oracle.insert(F, ins.seq, ins.offsets, k, m, s, H, seed, nthreads=8, alphabet=alphabet, sectors=1)
    img = sbf.to_numpy()
    assert_images_equal(img, F)
    if H < 4:
        # the option did what it is for: bits in the words the paper's layout leaves empty
        assert img[:, H:].any()
    qseq = np.concatenate([ins.seq, qry.seq])
    qoff = np.concatenate([ins.offsets, ins.offsets[-1] + qry.offsets[1:]])
    got = gpu_query(torch, sbf, qseq, qoff)
    want = oracle.query(F, qseq, qoff, k, m, s, H, seed, nthreads=8, alphabet=alphabet, sectors=1)
    assert_words_equal(got, want, qoff)
    sbf.close()


@pytest.mark.parametrize("m,s,H", [(16, 28, 1), (16, 28, 2), (12, 20, 1), (21, 31, 2), (14, 24, 2)])
def test_specialised_points_with_hashed_sectors(m, s, H):
    torch = need_gpu()
    rng = np.random.default_rng(1000 * H + m + s)
    ins = synth.random_records(rng, 12, 100, 30_000, n_prob=0.001, lower_prob=0.02)
    qry = synth.random_records(rng, 300, 31, 200, n_prob=0.002)
    _check(torch, dict(k=31, m=m, s=s, H=H), 1 << 22, 11 + H, ins, qry, specialized=False)


@pytest.mark.parametrize("case", range(6))
def test_runtime_kernel_with_hashed_sectors(case):
    torch = need_gpu()
    rng = np.random.default_rng(5100 + case)
    k = int(rng.integers(5, 33))
    m = int(rng.integers(1, k + 1))
    s = int(rng.integers(1, k + 1))
    H = 3 if case < 3 else int(rng.integers(1, 4))
    ins = synth.random_records(rng, 10, 0, 8_000, n_prob=0.003)
    qry = synth.random_records(rng, 50, 0, 300, n_prob=0.003)
    _check(torch, dict(k=k, m=m, s=s, H=H), int(2 ** rng.integers(12, 21)), int(rng.integers(1, 2**62)), ins, qry)


@pytest.mark.parametrize("alphabet", ["protein", "dna_triplet"])
@pytest.mark.parametrize("H", [1, 2, 3])
def test_alphabet_kernels_with_hashed_sectors(alphabet, H):
    torch = need_gpu()
    rng = np.random.default_rng(5300 + H + (7 if alphabet == "protein" else 0))
    if alphabet == "protein":
        params = dict(k=12, m=8, s=10, H=H)
        ins = synth.random_protein_records(rng, 30, 0, 3_000, lower_prob=0.05, junk_prob=0.005)
        qry = synth.random_protein_records(rng, 80, 0, 200)
    else:
        params = dict(k=10, m=5, s=8, H=H)
        ins = synth.random_records(rng, 30, 0, 6_000, n_prob=0.002)
        qry = synth.random_records(rng, 80, 0, 400, n_prob=0.002)
    _check(torch, params, 1 << 20, 23 + H, ins, qry, alphabet=alphabet)


def test_hashed_sectors_flag_is_inert_from_h4():
    torch = need_gpu()
    rng = np.random.default_rng(77)
    ins = synth.random_records(rng, 8, 1000, 20_000, n_prob=0.001)
    imgs = []
    for sectors in ("fixed", "hashed"):
        sbf = _filter(1 << 22, dict(k=31, m=16, s=28, H=4), 5, sectors=sectors)
        gpu_insert(torch, sbf, ins.seq, ins.offsets)
        imgs.append(sbf.to_numpy())
        sbf.close()
    assert np.array_equal(imgs[0], imgs[1]) and imgs[0].any()


def test_unknown_creation_flags_are_rejected():
    need_gpu()
    from minimizer_sharded_bloom_gb300 import _native as N
    L = N.load()
    assert not L.sbf_create_ex(1 << 20, 31, 16, 28, 2, 1, 0, 4)
    assert "flags" in N.last_error()
    f = N.sbf_create_ex(1 << 20, 31, 16, 28, 2, 1, 0, 0)
    assert N.sbf_get_flags(f) == 0
    N.sbf_destroy(f)
    f = N.sbf_create_ex(1 << 20, 31, 16, 28, 2, 1, 0, N.FLAG_HASHED_SECTORS | N.FLAG_RUNTIME_KERNELS)
    assert N.sbf_get_flags(f) == N.FLAG_HASHED_SECTORS | N.FLAG_RUNTIME_KERNELS
    assert not N.sbf_is_specialized(f)
    N.sbf_destroy(f)
    assert L.sbf_get_flags(None) == -1
