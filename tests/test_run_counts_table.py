"""The stored run counts (oracle/run_counts.json) that bench.py takes its
algorithmic bytes from: the tiny workload's entry is recomputed here with the
oracle, and every entry is checked against invariants that hold for any input
(Fig. 3: a run is a maximal stretch of consecutive valid k-mers of one record
with one shard; at H = 4 each run's mask has four non-zero words)."""
import json
import os

import numpy as np

import oracle
from minimizer_sharded_bloom_gb300 import synth

TABLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "run_counts.json")


def test_tiny_entry_matches_a_fresh_oracle_count():
    with open(TABLE) as f:
        rec = json.load(f)["tiny"]
    ins, qry = synth.tiny()
    shards = oracle.num_shards_for(rec["filter_bits"])
    for role, wl in (("insert", ins), ("query", qry)):
        e = rec[role]
        assert e["fingerprint"] == synth.fingerprint(wl.seq, wl.offsets)
        nv, runs, words = oracle.count_runs(wl.seq, wl.offsets, rec["k"], rec["m"], rec["s"], rec["H"], shards,
                                            rec["seed"], rec["alphabet"])
        assert (nv, runs, words) == (e["valid_kmers"], e["runs"], e["nonzero_words"])


def test_every_entry_is_consistent():
    with open(TABLE) as f:
        table = json.load(f)
    assert {"tiny", "genome-like", "out-of-cache", "out-of-cache-small", "irregular", "protein-like",
            "triplet"} <= set(table)
    for name, rec in table.items():
        sym = 3 if rec["alphabet"] == "dna_triplet" else 1
        w = rec["k"] - rec["m"] + 1
        for role in ("insert", "query"):
            e = rec[role]
            positions = e["bytes"] // sym
            assert 0 < e["runs"] <= e["valid_kmers"] <= positions, (name, role)
            # at least one run per record that holds a valid k-mer, at most one per k-mer
            assert e["runs"] <= e["valid_kmers"]
            # H = 4 (word i mod 4): every run sets a bit in each of the four words
            if rec["H"] >= 4:
                assert e["nonzero_words"] == 4 * e["runs"], (name, role)
            # density (Sec. II-B1): on these inputs runs per k-mer lie near 2/(w+1),
            # plus a run start per record
            per_kmer = e["runs"] / e["valid_kmers"]
            assert 0.7 * 2 / (w + 1) < per_kmer < 1.3 * (2 / (w + 1) + e["records"] / e["valid_kmers"]), (name, role)
