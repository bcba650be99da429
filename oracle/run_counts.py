"""Exact run counts of the benchmark workloads, from the oracle.

TEST AND MEASUREMENT INFRASTRUCTURE ONLY (like the rest of ``oracle/``).

A run is a maximal stretch of consecutive valid k-mers of one record that
share a shard ("cuSBF", Fig. 3 and Algorithm 1: the insert issues one atomic
update per non-zero word of each run; the query reads one shard per run).
The benchmark's algorithmic bytes count one 32-byte shard read (query) or
read plus write-back (insert) per run, so it needs each workload's exact run
count.  This script computes them with ``oracle.count_runs`` (every k-mer
from scratch) split over worker processes by records, and writes
``run_counts.json`` beside it, keyed by workload name with a fingerprint of
the generated input so a reader can tell whether its own input is the same.

    python -m oracle.run_counts [workload ...]
"""
from __future__ import annotations

import json
import multiprocessing as mp
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "run_counts.json")


def _count_group(args):
    import oracle
    seq, off, k, m, s, H, shards, seed, alphabet = args
    return oracle.count_runs(seq, off, k, m, s, H, shards, seed, alphabet)


def count_runs_parallel(seq, offsets, k, m, s, H, num_shards, seed, alphabet="dna", procs=None):
    """oracle.count_runs over the whole batch, records split into groups of
    about equal size (runs never cross records, so the counts add up)."""
    procs = procs or os.cpu_count() or 1
    n = offsets.size - 1
    groups = max(1, min(n, 8 * procs))
    target = np.linspace(int(offsets[0]), int(offsets[-1]), groups + 1)
    cuts = np.unique(np.concatenate([[0], np.searchsorted(offsets, target[1:-1]), [n]]))
    jobs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b <= a:
            continue
        lo, hi = int(offsets[a]), int(offsets[b])
        jobs.append((seq[lo:hi], offsets[a:b + 1] - lo, k, m, s, H, num_shards, seed, alphabet))
    if len(jobs) == 1 or procs == 1:
        parts = [_count_group(j) for j in jobs]
    else:
        with mp.get_context("spawn").Pool(procs) as pool:
            parts = pool.map(_count_group, jobs, chunksize=1)
    return tuple(int(sum(p[i] for p in parts)) for i in range(3))


def workloads():
    """name -> (make, filter bits, params, seed): the benchmark's workloads,
    with their generators' defaults."""
    from minimizer_sharded_bloom_gb300 import synth
    dna = dict(k=31, m=16, s=28, H=4, alphabet="dna")
    protein = dict(k=12, m=8, s=10, H=4, alphabet="protein")
    triplet = dict(k=10, m=5, s=8, H=4, alphabet="dna_triplet")
    return {
        "tiny": (synth.tiny, 1 << 20, dna, 5),
        "genome-like": (synth.genome_like, 1 << 30, dna, 5),
        "out-of-cache": (synth.out_of_cache, 1 << 36, dna, 5),
        "out-of-cache-small": (lambda: synth.out_of_cache(total=200_000_000, n_contigs=2_000), 1 << 34, dna, 5),
        "irregular": (synth.irregular, 1 << 32, dna, 5),
        "protein-like": (synth.protein_like, 1 << 33, protein, 5),
        "triplet": (synth.out_of_cache, 1 << 33, triplet, 5),
    }


def main(names):
    import oracle
    from minimizer_sharded_bloom_gb300 import synth
    table = {}
    if os.path.exists(OUT):
        with open(OUT) as f:
            table = json.load(f)
    specs = workloads()
    for name in names or list(specs):
        make, bits, p, seed = specs[name]
        t0 = time.time()
        ins, qry = make()
        shards = oracle.num_shards_for(bits)
        rec = {"filter_bits": bits, "seed": seed, **p}
        for role, wl in (("insert", ins), ("query", qry)):
            nv, runs, atomics = count_runs_parallel(wl.seq, wl.offsets, p["k"], p["m"], p["s"], p["H"], shards,
                                                    seed, p["alphabet"])
            rec[role] = {"fingerprint": synth.fingerprint(wl.seq, wl.offsets), "valid_kmers": nv, "runs": runs,
                         "nonzero_words": atomics, "bytes": int(wl.seq.size), "records": int(wl.offsets.size - 1)}
        table[name] = rec
        with open(OUT, "w") as f:
            json.dump(table, f, indent=1, sort_keys=True)
        print(f"{name}: {rec['insert']['runs']:,} / {rec['query']['runs']:,} runs "
              f"({time.time() - t0:.0f} s)", flush=True)


if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(HERE))
    main(sys.argv[1:])
