"""The benchmark's k-mer accounting (the denominator of its k-mers/s) agrees
with the oracle: on clean records every counted position is a valid k-mer,
for DNA, protein and in-frame DNA triplets; and the false-positive-rate
positions are exactly the oracle's valid k-mers of the uniform records."""
import numpy as np
import pytest

import bench
import oracle
from minimizer_sharded_bloom_gb300 import synth


@pytest.mark.parametrize("alphabet,k,symbols,B", [
    ("dna", 31, synth.ACGT, 1), ("protein", 12, synth.AMINO20, 1), ("dna_triplet", 10, synth.ACGT, 3)])
def test_kmer_count_matches_oracle_valid_kmers(alphabet, k, symbols, B):
    rng = np.random.default_rng(17)
    lengths = rng.integers(0, 400, size=300)
    off = synth.csr(lengths)
    seq = synth.uniform_bases(rng, int(off[-1]), symbols)
    wl = synth.Workload(seq, off)
    valid, _, _ = oracle.count_runs(seq, off, k, k // 2, k - 2, 4, 1 << 20, 3, alphabet)
    assert bench.kmer_count(wl, k, B) == valid


def test_fpr_positions_are_the_oracle_valid_kmers():
    """fpr_of reads exactly the in-frame k-mer starts of the uniform records:
    with every word all-ones it returns 1, and fpr_count equals the oracle's
    valid k-mers of those records."""
    rng = np.random.default_rng(18)
    lengths = rng.integers(20, 200, size=50)
    off = synth.csr(lengths)
    seq = synth.uniform_bases(rng, int(off[-1]))
    is_random = rng.random(50) < 0.5
    qry = synth.Workload(seq, off, is_random=is_random)
    words = np.full((int(off[-1]) + 31) // 32 + 1, 0xFFFFFFFF, dtype=np.uint32)
    for B, k, alphabet in ((1, 31, "dna"), (3, 10, "dna_triplet")):
        assert bench.fpr_of(words, qry, k, B) == 1.0
        sub = [r for r in range(50) if is_random[r]]
        want = sum(oracle.count_runs(seq[off[r]:off[r + 1]], np.array([0, off[r + 1] - off[r]]),
                                     k, k // 2, k - 2, 4, 1 << 20, 3, alphabet)[0] for r in sub)
        assert bench.fpr_count(qry, k, B) == want
