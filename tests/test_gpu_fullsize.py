"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times (the same library entry points and filter sizes): every
workload's whole filter image and every answer word of its whole query batch
against the oracle.

* genome-like: 50 Mbp into 2^30 bits; 10^6 reads of 150 bp.
* out-of-cache: 10^9 bp in 10,000 contigs into 2^36 bits (8 GiB); 6,666,666
  reads of 150 bp (run in the dense geometry through the CSR call, and once
  more through the explicit dense call).
* irregular: 2.6 Gbp of long reads with N runs into 2^32 bits; a disjoint
  set of the same recipe as the query.
* sweep: grid points at the full 50 Mbp.
* protein-like (5 x 10^8 residues, 2^33 bits; 10^7 fragments) and triplet
  (the out-of-cache data as codons, 2^33 bits), at the alphabets' benchmark
  parameters.

The oracle runs on all host cores; images are compared in slices of 2^24
shards (512 MiB) so the host holds one copy of a large image only.
"""
import os

import numpy as np
import pytest

import oracle
from minimizer_sharded_bloom_gb300 import synth
from _gpu_helpers import (MAIN, answer_bits, assert_images_equal, assert_words_equal, need_gpu,
                          oracle_answers, oracle_image, to_dev)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
NTHREADS = max(1, min(64, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _filter(num_bits, params, seed, alphabet="dna"):
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter
    return SuperBloomFilter(num_bits, seed=seed, alphabet=alphabet, **params)


def _gpu_words(torch, sbf, dseq, doff, total):
    out = torch.zeros((total + 31) // 32 + 1, dtype=torch.int32, device="cuda")
    sbf.query(dseq, doff, out=out)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


def _whole_image_equal(torch, sbf, F, step=1 << 24):
    """The GPU image equals the oracle's F shard for shard, slice by slice."""
    assert F.shape == (sbf.num_shards, 4)
    img = sbf.to_tensor()
    torch.cuda.synchronize()
    for a in range(0, sbf.num_shards, step):
        g = img[a:a + step].cpu().numpy().view(np.uint64)
        try:
            assert_images_equal(g, F[a:a + step])
        except AssertionError as e:
            raise AssertionError(f"in the slice starting at shard {a}: {e}") from None
    del img


def _whole_workload(torch, sbf, ins, qry, params, seed, alphabet="dna"):
    """Insert `ins` whole on the GPU, compare the whole image with the
    oracle's, query `qry` whole and compare every answer word.  Returns the
    GPU's answer words."""
    dseq, doff = to_dev(torch, ins.seq, ins.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    del dseq, doff
    assert sbf.status() == 0
    F = oracle_image(ins.seq, ins.offsets, params, sbf.num_shards * 256, seed, nthreads=NTHREADS,
                     alphabet=alphabet)
    _whole_image_equal(torch, sbf, F)
    dq, dqo = to_dev(torch, qry.seq, qry.offsets)
    words = _gpu_words(torch, sbf, dq, dqo, int(qry.offsets[-1]))
    del dq, dqo
    assert sbf.status() == 0
    want = oracle_answers(F, qry.seq, qry.offsets, params, seed, nthreads=NTHREADS, alphabet=alphabet)
    del F
    assert_words_equal(words, want, qry.offsets)
    return words


def test_genome_like_full(torch):
    ins, qry = synth.genome_like()
    seed = 3
    sbf = _filter(1 << 30, MAIN, seed)
    dseq, doff = to_dev(torch, ins.seq, ins.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    F = oracle_image(ins.seq, ins.offsets, MAIN, 1 << 30, seed, nthreads=NTHREADS)
    assert_images_equal(sbf.to_numpy(), F)
    dq, dqo = to_dev(torch, qry.seq, qry.offsets)
    got = _gpu_words(torch, sbf, dq, dqo, int(qry.offsets[-1]))
    want = oracle_answers(F, qry.seq, qry.offsets, MAIN, seed, nthreads=NTHREADS)
    assert_words_equal(got, want, qry.offsets)


@pytest.mark.parametrize("m,s,H", [(16, 28, 8), (12, 20, 4), (21, 31, 1), (18, 24, 6)])
def test_sweep_points_full(torch, m, s, H):
    ins = synth.Workload(synth.genome_like_reference(3), synth.csr([50_000_000]))
    params = dict(k=31, m=m, s=s, H=H)
    seed = 7
    sbf = _filter(1 << 30, params, seed)
    assert sbf.specialized
    dseq, doff = to_dev(torch, ins.seq, ins.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    F = oracle_image(ins.seq, ins.offsets, params, 1 << 30, seed, nthreads=NTHREADS)
    assert_images_equal(sbf.to_numpy(), F)
    q = synth.Workload(synth.uniform_bases(np.random.default_rng(7), 200_000 * 31),
                       synth.csr(np.full(200_000, 31)))
    dq, dqo = to_dev(torch, q.seq, q.offsets)
    got = _gpu_words(torch, sbf, dq, dqo, int(q.offsets[-1]))
    assert_words_equal(got, oracle_answers(F, q.seq, q.offsets, params, seed, nthreads=NTHREADS),
                       q.offsets)


def test_out_of_cache_full(torch):
    ins, qry = synth.out_of_cache()
    seed = 5
    sbf = _filter(1 << 36, MAIN, seed)
    assert sbf.specialized
    words = _whole_workload(torch, sbf, ins, qry, MAIN, seed)
    # the same reads through the explicit dense call (150 bp each) answer identically
    dq, _ = to_dev(torch, qry.seq, qry.offsets)
    dense = torch.zeros((int(qry.offsets[-1]) + 31) // 32 + 1, dtype=torch.int32, device="cuda")
    sbf.query_dense(dq[: qry.seq.size], 150, out=dense)
    torch.cuda.synchronize()
    assert np.array_equal(dense.cpu().numpy().view(np.uint32)[: words.size], words)
    del dq, dense
    # uniform reads give the false-positive rate (near 0 at 16 bits/k-mer)
    starts = qry.offsets[:-1][qry.meta["is_random"]][:20000]
    pos = (starts[:, None] + np.arange(150 - 31 + 1)[None, :]).reshape(-1)
    assert answer_bits(words, pos).mean() < 0.01


def test_irregular_full(torch):
    ins, qry = synth.irregular()
    seed = 8
    sbf = _filter(1 << 32, MAIN, seed)
    assert sbf.specialized
    _whole_workload(torch, sbf, ins, qry, MAIN, seed)


@pytest.mark.parametrize("alphabet", ["protein", "dna_triplet"])
def test_alphabet_workload_full(torch, alphabet):
    """The protein-like and triplet bench workloads at full size, with the
    bench's filter size and parameters (both run the strip kernel)."""
    if alphabet == "protein":
        ins, qry = synth.protein_like()
        params, seed = dict(k=12, m=8, s=10, H=4), 10
    else:
        ins, qry = synth.out_of_cache()
        params, seed = dict(k=10, m=5, s=8, H=4), 11
    sbf = _filter(1 << 33, params, seed, alphabet)
    assert sbf.specialized
    words = _whole_workload(torch, sbf, ins, qry, params, seed, alphabet)
    # uniform fragments / reads: the false-positive rate stays small
    B = 3 if alphabet == "dna_triplet" else 1
    flen = int(np.diff(qry.offsets)[0])
    starts = qry.offsets[:-1][qry.meta["is_random"]][:20000]
    pos = (starts[:, None] + B * np.arange(flen // B - params["k"] + 1)[None, :]).reshape(-1)
    assert answer_bits(words, pos).mean() < 0.01


@pytest.mark.parametrize("alphabet,params", [
    ("dna", MAIN), ("protein", dict(k=12, m=8, s=10, H=4)), ("dna_triplet", dict(k=10, m=5, s=8, H=4))])
def test_filter_beyond_2_31_shards(torch, alphabet, params):
    """The largest filters: 2^40 bits = 2^32 shards (128 GiB), past the strip
    kernels' 2^31-shard run keys, so the runtime-parameter kernel (DNA) and
    the tiled alphabet kernels take them, with shard word indices beyond 2^32.
    A few Mbp are inserted; every answer bit of a query batch that reaches
    the inserted shards (the records themselves and reads of them at 5 %
    substitution, whose s-mers test bits the image may or may not hold) and
    of uniform reads equals the oracle's answer on its sparse image of the
    same insert."""
    import oracle as orc
    free, _ = torch.cuda.mem_get_info()
    if free < (1 << 37) + (8 << 30):
        pytest.skip("needs 136 GiB of free device memory")
    k, m, s, H = params["k"], params["m"], params["s"], params["H"]
    shards, seed = 1 << 32, 41
    rng = np.random.default_rng(4100 + len(alphabet))
    if alphabet == "protein":
        ins = synth.random_protein_records(rng, 60, 5_000, 40_000, lower_prob=0.01, junk_prob=0.001)
        symbols, read_len = synth.AMINO20, 50
    else:
        ins = synth.random_records(rng, 40, 20_000, 60_000, n_prob=0.001, lower_prob=0.01)
        symbols, read_len = synth.ACGT, 150
    reads, roff, _ = synth.sample_reads(rng, ins.seq, ins.offsets, 20_000, 5_000, read_len, 0.05, symbols)
    qseq = np.concatenate([ins.seq, reads])
    qoff = np.concatenate([ins.offsets, ins.offsets[-1] + roff[1:]])
    sbf = _filter(1 << 40, params, seed, alphabet)
    try:
        assert sbf.num_shards == shards
        dseq, doff = to_dev(torch, ins.seq, ins.offsets)
        sbf.insert(dseq, doff)
        dq, dqo = to_dev(torch, qseq, qoff)
        words = _gpu_words(torch, sbf, dq, dqo, int(qoff[-1]))
        assert sbf.status() == 0
    finally:
        sbf.close()
    keys, rows = orc.insert_sparse(ins.seq, ins.offsets, k, m, s, H, shards, seed, alphabet)

    def shard_words(req):
        req = np.asarray(req, dtype=np.uint64)
        out = np.zeros((req.size, 4), dtype=np.uint64)
        if keys.size:
            idx = np.minimum(np.searchsorted(keys, req), keys.size - 1)
            found = keys[idx] == req
            out[found] = rows[idx[found]]
        return out

    positions = np.arange(int(qoff[0]), int(qoff[-1]), dtype=np.int64)
    want = orc.query_sampled(shard_words, qseq, qoff, positions, k, m, s, H, shards, seed, alphabet)
    got = answer_bits(words, positions)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} answers differ, first at position {positions[bad[0]]}"
    # the inserted records' own k-mers all answer present; some mutated ones do not
    own = positions < int(ins.offsets[-1])
    assert want[own].sum() > 0 and (want[~own] != got[~own]).sum() == 0
    assert 0 < want[~own].mean() < 1
