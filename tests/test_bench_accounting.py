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


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle arm, no GPU) prints one JSON
    line with the metric, the impl tag, its cpu_baseline and an e2e object
    with no host-device bytes."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.join(os.path.dirname(os.path.abspath(__file__)), "..")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "1"], cwd=root, capture_output=True, text=True,
                         timeout=300, check=True)
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "k-mers/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["metric"].startswith("k-mers/s insert & query")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "k-mers/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # the workload is identified by the same keys as the GPU arm's line
    ins, qry = synth.tiny()
    want = bench.workload_config("tiny", bench.WORKLOADS["tiny"], bench.MAIN, ins, qry)
    assert {k: d["config"][k] for k in want} == want
    assert want["kmers_counted"].startswith("valid k-mers") and want["insert_kmers"] == 99_970


def test_kernel_hash_sees_code_not_comments():
    """The stored DRAM traffic is keyed by a hash of the kernels' code: comments
    and layout leave it as it is, any change of a token changes it."""
    src = "int a = 1; // one\n/* block\n comment */ int  b =\n 2;\n"
    assert bench.code_only(src) == "int a = 1; int b = 2;"
    assert bench.code_only(src.replace("// one", "// another note")) == bench.code_only(src)
    assert bench.code_only(src.replace("b =", "c =")) != bench.code_only(src)
    stored = bench.MEASURED_TRAFFIC["out-of-cache"]["source_sha"]
    assert len(stored) == 16 and len(bench.kernel_source_sha()) == 16


def test_stored_counts_match_only_their_own_input():
    """The bench takes the oracle's stored counts (valid k-mers, runs) only for
    the exact input they were computed on: the tiny workload matches, a copy
    with one base changed or other parameters does not."""
    ins, qry = synth.tiny()
    bits = 1 << 20
    rec = bench.stored_count("tiny", "insert", ins, bench.MAIN, bits)
    assert rec is not None and rec["valid_kmers"] == bench.kmer_count(ins)
    assert bench.stored_count("tiny", "query", qry, bench.MAIN, bits)["valid_kmers"] == bench.kmer_count(qry)
    seq = ins.seq.copy()
    seq[0] = ord("A") if seq[0] != ord("A") else ord("C")
    assert bench.stored_count("tiny", "insert", synth.Workload(seq, ins.offsets), bench.MAIN, bits) is None
    assert bench.stored_count("tiny", "insert", ins, dict(bench.MAIN, H=2), bits) is None
    assert bench.stored_count("tiny", "insert", ins, bench.MAIN, bits << 1) is None
    runs, src = bench.exact_runs("tiny", "insert", ins, bench.MAIN, bits)
    assert src.startswith("exact") and runs == rec["runs"]
