"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times (the same library entry points and filter sizes).

* genome-like (50 Mbp into 2^30 bits; 1 M reads): the whole image and every
  answer bit against the oracle.
* out-of-cache (1 Gbp, 2^36 bits = 8 GiB; 6.67 M reads) and irregular
  (2.6 Gbp of long reads with N runs, 2^32 bits): the oracle cannot redo
  them whole in a test, so (a) a prefix of the records inserted into a
  full-size filter is compared image-exactly, (b) after the full insert,
  sampled k-mers must be present with exactly their oracle bits set (no false
  negatives), and (c) sampled answer bits of the full query equal the
  oracle's answers computed against the same image.
* sweep: grid points at the full 50 Mbp against the oracle's whole image.
* protein-like (5 x 10^8 residues, 2^33 bits; 10^7 fragments) and triplet
  (the out-of-cache data as codons, 2^33 bits): (a)-(c) as for out-of-cache,
  at the alphabets' benchmark parameters.
"""
import numpy as np
import pytest

import oracle
from minimizer_sharded_bloom_gb300 import synth
from _gpu_helpers import (MAIN, answer_bits, assert_images_equal, assert_words_equal, need_gpu,
                          oracle_answers, oracle_image, to_dev)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
NTHREADS = 16


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


def _shard_rows(torch, sbf):
    img = sbf.to_tensor()
    torch.cuda.synchronize()

    def rows(shards):
        idx = torch.from_numpy(np.asarray(shards, dtype=np.int64)).cuda()
        return img.index_select(0, idx).cpu().numpy().view(np.uint64)
    return img, rows


def _sparse_compare(torch, sbf, seq, offsets, params, seed, alphabet="dna"):
    """GPU image == oracle image, comparing only the oracle's non-zero shards
    plus a count of the GPU's non-zero shards."""
    img, rows = _shard_rows(torch, sbf)
    sh, words = oracle.insert_sparse(seq, offsets, params["k"], params["m"], params["s"],
                                     params["H"], sbf.num_shards, seed, alphabet)
    nz = int((img != 0).any(dim=1).sum().item())
    assert nz == sh.size, (nz, sh.size)
    assert np.array_equal(rows(sh), words)


def _sampled_checks(torch, sbf, ins, qry, params, seed, rng, n_samples=100_000, alphabet="dna"):
    img, rows = _shard_rows(torch, sbf)
    # (b) no false negatives on sampled inserted k-mers, exact bits present
    pos = rng.integers(int(ins.offsets[0]), int(ins.offsets[-1]), size=n_samples)
    valid, shard, K = oracle.kmer_batch(ins.seq, ins.offsets, pos, params["k"], params["m"],
                                        params["s"], params["H"], sbf.num_shards, seed, alphabet)
    assert valid.sum() > n_samples // 4
    F = rows(shard[valid])
    assert ((K[valid] & ~F) == 0).all()
    # (c) sampled answers of the full query
    dseq, doff = to_dev(torch, qry.seq, qry.offsets)
    words = _gpu_words(torch, sbf, dseq, doff, int(qry.offsets[-1]))
    qpos = rng.integers(int(qry.offsets[0]), int(qry.offsets[-1]), size=n_samples)
    want = oracle.query_sampled(rows, qry.seq, qry.offsets, qpos, params["k"], params["m"],
                                params["s"], params["H"], sbf.num_shards, seed, alphabet)
    assert np.array_equal(answer_bits(words, qpos), want)
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


def _prefix(wl, max_bases):
    r = int(np.searchsorted(wl.offsets, max_bases, side="right")) - 1
    r = max(r, 1)
    return synth.Workload(wl.seq[:wl.offsets[r]], wl.offsets[:r + 1])


def test_out_of_cache_full(torch):
    ins, qry = synth.out_of_cache()
    seed = 5
    rng = np.random.default_rng(55)
    # (a) a 3 Mbp prefix of the contigs into the full 8 GiB filter, image-exact
    sub = _prefix(ins, 3_000_000)
    sbf = _filter(1 << 36, MAIN, seed)
    assert sbf.specialized
    dseq, doff = to_dev(torch, sub.seq, sub.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    _sparse_compare(torch, sbf, sub.seq, sub.offsets, MAIN, seed)
    # (b, c) everything
    sbf.clear()
    dseq, doff = to_dev(torch, ins.seq, ins.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    del dseq, doff
    assert sbf.status() == 0
    words = _sampled_checks(torch, sbf, ins, qry, MAIN, seed, rng)
    # the same reads as a dense batch (150 bp each) answer identically
    dq, _ = to_dev(torch, qry.seq, qry.offsets)
    dense = torch.zeros((int(qry.offsets[-1]) + 31) // 32 + 1, dtype=torch.int32, device="cuda")
    sbf.query_dense(dq[: qry.seq.size], 150, out=dense)
    torch.cuda.synchronize()
    assert np.array_equal(dense.cpu().numpy().view(np.uint32)[: words.size], words)
    del dq, dense
    # reads taken from the contigs without errors in a k-mer answer positive;
    # uniform reads give the false-positive rate (near 0 at 16 bits/k-mer).
    starts = qry.offsets[:-1][qry.meta["is_random"]][:20000]
    pos = (starts[:, None] + np.arange(150 - 31 + 1)[None, :]).reshape(-1)
    assert answer_bits(words, pos).mean() < 0.01


def test_irregular_full(torch):
    ins, qry = synth.irregular()
    seed = 8
    rng = np.random.default_rng(88)
    sub = _prefix(ins, 4_000_000)
    sbf = _filter(1 << 32, MAIN, seed)
    dseq, doff = to_dev(torch, sub.seq, sub.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    _sparse_compare(torch, sbf, sub.seq, sub.offsets, MAIN, seed)
    sbf.clear()
    dseq, doff = to_dev(torch, ins.seq, ins.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    del dseq, doff
    _sampled_checks(torch, sbf, ins, qry, MAIN, seed, rng)


@pytest.mark.parametrize("alphabet", ["protein", "dna_triplet"])
def test_alphabet_workload_full(torch, alphabet):
    """The protein-like and triplet bench workloads at full size, with the
    bench's filter size and parameters (protein runs the strip kernel)."""
    if alphabet == "protein":
        ins, qry = synth.protein_like()
        params, seed = dict(k=12, m=8, s=10, H=4), 10
    else:
        ins, qry = synth.out_of_cache()
        params, seed = dict(k=10, m=5, s=8, H=4), 11
    rng = np.random.default_rng(99)
    sub = _prefix(ins, 3_000_000)
    sbf = _filter(1 << 33, params, seed, alphabet)
    assert sbf.specialized
    dseq, doff = to_dev(torch, sub.seq, sub.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    _sparse_compare(torch, sbf, sub.seq, sub.offsets, params, seed, alphabet)
    sbf.clear()
    dseq, doff = to_dev(torch, ins.seq, ins.offsets)
    sbf.insert(dseq, doff)
    torch.cuda.synchronize()
    del dseq, doff
    assert sbf.status() == 0
    words = _sampled_checks(torch, sbf, ins, qry, params, seed, rng, alphabet=alphabet)
    # uniform fragments / reads: the false-positive rate stays small
    B = 3 if alphabet == "dna_triplet" else 1
    flen = int(np.diff(qry.offsets)[0])
    starts = qry.offsets[:-1][qry.meta["is_random"]][:20000]
    pos = (starts[:, None] + B * np.arange(flen // B - params["k"] + 1)[None, :]).reshape(-1)
    assert answer_bits(words, pos).mean() < 0.01
