#!/usr/bin/env python
"""Benchmark: SBF insert + query throughput on one GB300 (or N replicas).

One step = the whole hot path over one batch: insert every k-mer of the
workload's reference records, then query every k-mer of its reads, with the
paper's operating point k=31, m=16, s=28, H=4.  The default workload is the
out-of-cache configuration (1 Gbp in 10,000 contigs into a 2^36-bit = 8 GiB
filter; 6,666,666 reads of 150 bp), the stand-in for the paper's T2T-CHM13
experiment on which its headline throughput is quoted.

Printed: one JSON line with the device-resident throughput (CUDA events on the
launching stream, inputs already in HBM and larger than L2), the same metric
end to end through the host-facing C-ABI calls (pinned host buffers, copies
inside the timed region), the false-positive rate of the uniform reads, the
roofline of the dominant kernel, SM clocks sampled during the timed region and
the CPU oracle timed on the host cores.

The protein-like and triplet workloads measure the other two alphabets of the
paper's Sec. IV-A with their own parameters (stated in each workload).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle arm
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from minimizer_sharded_bloom_gb300 import synth  # noqa: E402

METRIC = "k-mers/s insert & query (k=31,s=28,m=16,H=4); FPR; % HBM roofline"
K, M, S, H = 31, 16, 28, 4
SEED = 5
MAIN = dict(k=K, m=M, s=S, H=H, alphabet="dna")
# the other alphabets (Sec. IV-A): k at the 64-bit packing limit, s = k - 2
# (three s-mers per k-mer); m = 8 for proteins (at m = 6 only 20^6 = 64 M
# distinct m-mers exist, each recurring in a 500 M-residue set, and the
# minimizers pile onto few shards: FPR 4 %), m = 5 for codons (64^5 m-mers)
PROTEIN = dict(k=12, m=8, s=10, H=4, alphabet="protein")
TRIPLET = dict(k=10, m=5, s=8, H=4, alphabet="dna_triplet")


def metric_of(p):
    if p == MAIN:
        return METRIC
    return (f"k-mers/s insert & query ({p['alphabet']}, k={p['k']},s={p['s']},m={p['m']},"
            f"H={p['H']}); FPR; % roofline")


def sym_bytes(p) -> int:
    return 3 if p["alphabet"] == "dna_triplet" else 1

WORKLOADS = {
    "out-of-cache": dict(bits=1 << 36, make=lambda: synth.out_of_cache(),
                         desc="out-of-cache: 1 Gbp in 10,000 log-normal contigs (median 50 kbp) "
                              "into a 2^36-bit (8 GiB) filter; query 6,666,666 x 150 bp reads "
                              "(50% from the contigs at 1% error, 50% uniform)"),
    "out-of-cache-small": dict(bits=1 << 34, make=lambda: synth.out_of_cache(total=200_000_000,
                                                                               n_contigs=2_000),
                               desc="out-of-cache, profiling size: 200 Mbp in 2,000 log-normal contigs "
                                    "into a 2^34-bit (2 GiB) filter; query 1,333,333 x 150 bp reads"),
    "genome-like": dict(bits=1 << 30, make=lambda: synth.genome_like(),
                        desc="genome-like: 50 Mbp with 20% copied 1-10 kbp segments at 1% error "
                             "into a 2^30-bit (128 MiB) filter; query 1,000,000 x 150 bp reads"),
    "irregular": dict(bits=1 << 32, make=lambda: synth.irregular(),
                      desc="irregular: 200,000 log-normal long reads (median 8 kbp, 0.1% N in "
                           "runs of 1-50) into a 2^32-bit filter; query a disjoint equal set"),
    "tiny": dict(bits=1 << 20, make=lambda: synth.tiny(),
                 desc="tiny: 100 kbp into 2^20 bits; query it plus 100 kbp uniform"),
    "protein-like": dict(bits=1 << 33, make=lambda: synth.protein_like(), p=PROTEIN,
                         desc="protein-like: 500 M residues uniform over the 20 amino acids in "
                              "log-normal proteins (median 300) into a 2^33-bit (1 GiB) filter; "
                              "query 10,000,000 x 50-residue fragments (50% from the proteins at "
                              "1% substitution, 50% uniform); protein alphabet, k=12 m=8 s=10 H=4"),
    "protein-like-small": dict(bits=1 << 31, make=lambda: synth.protein_like(total=100_000_000),
                               p=PROTEIN,
                               desc="protein-like, profiling size: 100 M residues into a 2^31-bit "
                                    "(256 MiB) filter; query 2,000,000 x 50-residue fragments"),
    "triplet-small": dict(bits=1 << 31, make=lambda: synth.out_of_cache(total=200_000_000,
                                                                         n_contigs=2_000),
                          p=TRIPLET,
                          desc="DNA triplets, profiling size: 200 Mbp in 2,000 contigs into a "
                               "2^31-bit (256 MiB) filter; query 1,333,333 x 150 bp reads"),
    "triplet": dict(bits=1 << 33, make=lambda: synth.out_of_cache(), p=TRIPLET,
                    desc="DNA triplets: the out-of-cache data (1 Gbp in 10,000 contigs; "
                         "6,666,666 x 150 bp reads) read as in-frame codons into a 2^33-bit "
                         "(1 GiB) filter; triplet alphabet, k=10 m=5 s=8 H=4"),
}

# Algorithmic integer operations per k-mer of the rolling formulation
# (k=31, m=16, s=28, H=4) that run on the ALU pipe (logic, shift, compare,
# select), counted in the design notes: shared front end 39 (decode 1,
# validity 1, m-mer and s-mer extraction 3, minimizer-hash xor + fold 2,
# three 64-bit sliding-window minimums 12, shard 1, s-mer-hash xors and
# xorshifts 7, four bit positions to one-hot word halves 12); insert adds 10
# (run compare, select, OR of the newest s-mer into the run's eight
# half-words); query adds 26 (k-mer mask from four s-mer masks 16, subset test
# 9, answer bit 1).  The multiplies of the two hashes (11 per k-mer) run on
# the FMA pipe and are not counted.
ALU_OPS_PER_KMER = {"insert": 49, "query": 65}


def alu_ops(p):
    """The same count for any (k, s, alphabet): the k-mer mask costs 4 ops per
    s-mer (k-s+1 of them); a codon decodes from three bases (+2)."""
    front = 39 + (2 if p["alphabet"] == "dna_triplet" else 0)
    return {"insert": front + 10, "query": front + 4 * (p["k"] - p["s"] + 1) + 10}
# The ALU-pipe ceiling is measured in each run (probe kernels of
# libsbf_probes.so: a LOP3 / funnel-shift / compare / select / min mix on
# every SM, SM count from the device properties); see measure_ceilings().

# The form of the shard updates and loads in the current kernel source, whose
# probe rate is the pattern ceiling the insert and query are reported against:
# the DNA insert flushes a run with four 64-bit OR reductions from its lane
# ("red4"), or, on filters larger than 8x the L2 (where the library takes the
# queued insert), through its warp's run queue ("red_queue"; the protein and
# triplet inserts' cooperative flush is of that form too); the query copies
# each run head's shard with two 16-byte cp.async.cg.
QUEUED_INSERT_L2_MULTIPLE = 8
QUERY_SHARD_FORM = "cp_async"


def insert_flush_form(torch, filter_bits: int, alphabet: str) -> str:
    """The RMW probe form of the insert's run flush: the protein and triplet
    strip kernels flush a warp's runs cooperatively (one 32-byte request per
    run, like the queue); DNA queues them on filters larger than 8x the L2 and
    otherwise sends four reductions from the run's lane."""
    if alphabet != "dna":
        return "red_queue"
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    if filter_bits // 8 > QUEUED_INSERT_L2_MULTIPLE * l2:
        return "red_queue"
    return "red4"

# ncu DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per k-mer,
# valid only for the kernel source they were measured on (summaries under
# profiles/).  Out-of-cache: measured on its profiling size (200 Mbp into a
# 2 GiB filter, one kernel and two launches per capture) and applied per
# k-mer to the full workload -- both filters are many times larger than L2,
# where each run costs one DRAM read-modify-write of its shard at either
# size (the earlier full-size and profiling-size captures agreed within 3 %).
MEASURED_TRAFFIC = {
    "out-of-cache": {"source_sha": "858ff6c614669673", "insert": 14.1465, "query": 9.7808},
}

def code_only(text: str) -> str:
    """C++ source without its comments, whitespace runs collapsed: what the
    compiler sees of it (the kernels hold no string with '//' or '/*')."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(p=MAIN) -> str:
    """Hash of the code (comments and layout aside) of the source files the
    workload's kernels are built from."""
    files = {"dna": ("sbf_strip.cuh", "sbf_device.cuh", "sbf_inst_main.cu"),
             "protein": ("sbf_strip.cuh", "sbf_device.cuh", "sbf_inst_protein.cu"),
             "dna_triplet": ("sbf_strip.cuh", "sbf_alphabet.cu", "sbf_device.cuh",
                             "sbf_inst_triplet.cu")}[p["alphabet"]]
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "minimizer_sharded_bloom_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(pg, values):
    """Element-wise maximum of a list of floats over all ranks (gloo, CPU
    tensors); the values themselves on a single rank."""
    if pg is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(x) for x in t]


def throughput(world: int, steps: int, kmers_per_step: int, seconds: float) -> float:
    """Whole-job k-mers/s: every rank processes the same per-step work
    (weak scaling, replicas) within the slowest rank's time."""
    return world * steps * kmers_per_step / seconds


def kmer_count(wl, k=K, B=1):
    """k-mer positions: per record floor(len / B) - k + 1 (B bytes per symbol)."""
    return int(np.maximum(np.diff(wl.offsets) // B - k + 1, 0).sum())


def runs_estimate(wl, k=K, m=M, B=1):
    """Expected runs: density 2/(w+1) per k-mer (Sec. II-B1) plus one run
    start per record."""
    w = k - m + 1
    return kmer_count(wl, k, B) * 2.0 / (w + 1) + wl.n_records


def stored_count(workload: str, role: str, wl, p, bits):
    """The oracle's counts of this input (valid k-mers, runs, ...) from
    oracle/run_counts.json, or None when no stored entry matches its
    fingerprint and parameters."""
    try:
        with open(os.path.join(ROOT, "oracle", "run_counts.json")) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not (rec and role in rec and rec.get("filter_bits") == bits
            and all(rec.get(x) == p[x] for x in ("k", "m", "s", "H"))
            and rec.get("alphabet") == p["alphabet"] and rec.get("seed") == SEED):
        return None
    return rec[role] if rec[role]["fingerprint"] == synth.fingerprint(wl.seq, wl.offsets) else None


def exact_runs(workload: str, role: str, wl, p, bits, k=K, m=M, B=1):
    """(runs, source): the oracle's exact run count of this input (stored in
    oracle/run_counts.json by oracle/run_counts.py, matched by the input's
    fingerprint and parameters), else the 2/(w+1) estimate."""
    rec = stored_count(workload, role, wl, p, bits)
    if rec:
        return float(rec["runs"]), "exact (oracle run count of this input)"
    return runs_estimate(wl, k, m, B), "estimate 2/(w+1) per k-mer + 1 per record (no stored count matches)"


def fpr_count(qry, k=K, B=1) -> int:
    rnd = qry.meta.get("is_random")
    if rnd is None:
        return 0
    return int(np.maximum(np.diff(qry.offsets)[rnd] // B - k + 1, 0).sum())


def fpr_of(words: np.ndarray, qry, k=K, B=1) -> float | None:
    rnd = qry.meta.get("is_random")
    if rnd is None or not rnd.any():
        return None
    starts = qry.offsets[:-1][rnd]
    lens = np.diff(qry.offsets)[rnd]
    hits = total = 0
    for c in range(0, starts.size, 1 << 16):
        st, ln = starts[c:c + (1 << 16)], lens[c:c + (1 << 16)]
        nk = np.maximum(ln // B - k + 1, 0)
        if nk.sum() == 0:
            continue
        pos = np.repeat(st, nk) + B * (np.arange(nk.sum()) - np.repeat(np.cumsum(nk) - nk, nk))
        bits = (words[pos >> 5] >> (pos & 31).astype(np.uint32)) & 1
        hits += int(bits.sum())
        total += int(pos.size)
    return hits / total if total else None


def cpu_baseline(ins, qry, bits: int, budget_bases: int = 40_000_000, reads: int = 300_000, p=MAIN,
                 single_thread: bool = False):
    """The CPU oracle, as it stands, on a bounded prefix sample of the same
    workload, all host cores."""
    import oracle
    cores = os.cpu_count() or 1
    # the first budget_bases positions of the insert stream (records clipped
    # there) and the first `reads` query records
    end = int(ins.offsets[0]) + budget_bases
    off = np.minimum(ins.offsets, end)
    r = int(np.searchsorted(off, end, side="left"))
    r = max(1, min(r, ins.n_records))
    s_ins = synth.Workload(ins.seq[:off[r]], off[:r + 1])
    rq = max(1, min(reads, qry.n_records))
    s_q = synth.Workload(qry.seq[:qry.offsets[rq]], qry.offsets[:rq + 1])
    F = oracle.new_filter(bits)
    t0 = time.perf_counter()
    k, m, s, h, B = p["k"], p["m"], p["s"], p["H"], sym_bytes(p)
    oracle.insert(F, s_ins.seq, s_ins.offsets, k, m, s, h, SEED, nthreads=cores, alphabet=p["alphabet"])
    t1 = time.perf_counter()
    oracle.query(F, s_q.seq, s_q.offsets, k, m, s, h, SEED, nthreads=cores, alphabet=p["alphabet"])
    t2 = time.perf_counter()
    nk_i, nk_q = kmer_count(s_ins, k, B), kmer_count(s_q, k, B)
    nk = nk_i + nk_q
    res = {"value": nk / (t2 - t0), "unit": "k-mers/s", "cores": cores, "kind": "oracle",
           "sample": f"first {s_ins.n_bases:,} bytes ({r} records) inserted, first {rq:,} reads "
                     f"queried; {nk:,} k-mers in {t2 - t0:.1f} s",
           "insert_kmers_per_s": nk_i / (t1 - t0),
           "query_kmers_per_s": nk_q / (t2 - t1)}
    if single_thread:
        # the same loops on one thread, on a tenth of the sample
        e1 = int(ins.offsets[0]) + budget_bases // 10
        o1 = np.minimum(ins.offsets, e1)
        r1 = max(1, min(int(np.searchsorted(o1, e1, side="left")), ins.n_records))
        w_ins = synth.Workload(ins.seq[:o1[r1]], o1[:r1 + 1])
        rq1 = max(1, min(reads // 10, qry.n_records))
        w_q = synth.Workload(qry.seq[:qry.offsets[rq1]], qry.offsets[:rq1 + 1])
        F1 = oracle.new_filter(bits)
        u0 = time.perf_counter()
        oracle.insert(F1, w_ins.seq, w_ins.offsets, k, m, s, h, SEED, nthreads=1, alphabet=p["alphabet"])
        u1 = time.perf_counter()
        oracle.query(F1, w_q.seq, w_q.offsets, k, m, s, h, SEED, nthreads=1, alphabet=p["alphabet"])
        u2 = time.perf_counter()
        n1, n2 = kmer_count(w_ins, k, B), kmer_count(w_q, k, B)
        res["single_thread"] = {"kmers_per_s": (n1 + n2) / (u2 - u0), "cores": 1,
                                "insert_kmers_per_s": n1 / (u1 - u0), "query_kmers_per_s": n2 / (u2 - u1),
                                "sample": f"first {w_ins.n_bases:,} bytes inserted, first {rq1:,} reads queried"}
        res["single_thread_kmers_per_s"] = res["single_thread"]["kmers_per_s"]
    return res


def workload_config(workload: str, spec, p, ins, qry) -> dict:
    """The keys of a line's `config` that identify its workload, the same in
    both arms: parameters, filter size, and the batches' bases, k-mer
    positions, valid k-mers (the oracle's stored count where it matches) and
    records, plus which of the counts the k-mers/s divide by."""
    B = sym_bytes(p)
    pos_ins, pos_q = kmer_count(ins, p["k"], B), kmer_count(qry, p["k"], B)
    st_ins = stored_count(workload, "insert", ins, p, spec["bits"])
    st_q = stored_count(workload, "query", qry, p, spec["bits"])
    return {"workload": spec["desc"], "k": p["k"], "m": p["m"], "s": p["s"], "H": p["H"],
            "alphabet": p["alphabet"], "seed": SEED, "filter_bits": spec["bits"],
            "insert_kmers": st_ins["valid_kmers"] if st_ins else pos_ins,
            "query_kmers": st_q["valid_kmers"] if st_q else pos_q,
            "kmers_counted": ("valid k-mers (the oracle's count of this input)" if st_ins and st_q
                              else "k-mer positions (no stored oracle count of this input)"),
            "insert_bases": int(ins.offsets[-1] - ins.offsets[0]),
            "query_bases": int(qry.offsets[-1] - qry.offsets[0]),
            "insert_kmer_positions": pos_ins, "query_kmer_positions": pos_q,
            "insert_valid_kmers": st_ins["valid_kmers"] if st_ins else None,
            "query_valid_kmers": st_q["valid_kmers"] if st_q else None,
            "insert_records": int(ins.n_records), "query_records": int(qry.n_records)}


def run_reference(args, workload):
    """The reference arm: the CPU oracle on the host cores, one bounded sample
    of the workload per step."""
    spec = WORKLOADS[workload]
    p = spec.get("p", MAIN)
    ins, qry = spec["make"]()
    for _ in range(args.warmup):
        cpu_baseline(ins, qry, spec["bits"], budget_bases=2_000_000, reads=20_000, p=p)
    vals, secs = [], []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        cb = cpu_baseline(ins, qry, spec["bits"], budget_bases=10_000_000, reads=100_000, p=p)
        secs.append(time.perf_counter() - t0)
        vals.append(cb["value"])
    value = float(np.mean(vals))
    cb["value"] = value
    line = {"metric": metric_of(p), "value": value, "unit": "k-mers/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(secs)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8/u64",
            "data": "synthetic", "impl": "reference",
            "config": dict(workload_config(workload, spec, p, ins, qry),
                           timing="host wall clock per sample (the oracle on a bounded sample of "
                                  "the workload; cpu_baseline.sample says which)"),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "k-mers/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="out-of-cache", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--host-mode", type=int, default=None, choices=[0, 1, 2],
                    help="e2e leg: 0 the library default, 1 stages chunks, 2 reads host buffers in place")
    ap.add_argument("--host-chunk", type=int, default=None,
                    help="e2e leg: positions per staged chunk (default: the library's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--suite", action="store_true",
                    help="measure every configuration and the sweep grid (one JSON line each)")
    ap.add_argument("--fig4", action="store_true",
                    help="the paper's Fig. 4 grid: s 16..31 x m 8..31 x H in {4, 8, 12, 16} at k = 31 "
                         "(one JSON line per point, then the orderings the paper reports)")
    ap.add_argument("--fig4-h", default="4,8,12,16")
    ap.add_argument("--fig4-s", default="16-31")
    ap.add_argument("--fig4-m", default="8-31")
    args = ap.parse_args()
    if args.suite:
        run_suite(args)
        return
    if args.fig4:
        run_fig4(args)
        return
    rank, world, local = dist_info()

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, args.workload)
        return

    import torch
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter, build_lib, _native as N

    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    torch.cuda.set_device(local)
    build_lib.build()
    spec = WORKLOADS[args.workload]
    p = spec.get("p", MAIN)
    B = sym_bytes(p)
    ins, qry = spec["make"]()
    # k-mers/s counts valid k-mers: the oracle's count of this input where a
    # stored one matches (the k-mer positions of clean records are all valid)
    wcfg = workload_config(args.workload, spec, p, ins, qry)
    nk_ins, nk_q = wcfg["insert_kmers"], wcfg["query_kmers"]

    dseq = torch.from_numpy(ins.seq).cuda()
    doff = torch.from_numpy(ins.offsets).cuda()
    dq = torch.from_numpy(qry.seq).cuda()
    dqo = torch.from_numpy(qry.offsets).cuda()
    out = torch.zeros((qry.n_bases + 31) // 32 + 1, dtype=torch.int32, device="cuda")
    sbf = SuperBloomFilter(spec["bits"], k=p["k"], m=p["m"], s=p["s"], H=p["H"], seed=SEED,
                           alphabet=p["alphabet"])
    if p["alphabet"] == "dna" and not sbf.specialized:
        raise RuntimeError("the benchmark configuration must run its specialised kernel")
    # which kernel runs each call: DNA and the protein and triplet points on
    # the strip kernel, other alphabet points on the tiled alphabet kernel
    pt = f"{p['k']},{p['m']},{p['s']},{p['H']}"
    an = "protein" if p["alphabet"] == "protein" else "triplet"

    def kname(kind):
        if p["alphabet"] == "dna":
            return f"strip_kernel<{pt},{kind}>"
        if sbf.specialized:
            return f"strip_kernel<{pt},{kind},{an}>"
        return f"alphabet_kernel<{an},{pt},{kind}>"
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    n_ins, n_q = ins.n_records, qry.n_records

    def clear():
        # untimed: every insert starts from an empty filter (the 2^36-bit
        # memset also evicts the inputs and the filter from L2)
        N.sbf_clear(sbf.handle, sh)

    def step():
        N.sbf_insert(sbf.handle, dseq.data_ptr(), doff.data_ptr(), n_ins, sh)
        N.sbf_query(sbf.handle, dq.data_ptr(), dqo.data_ptr(), n_q, out.data_ptr(), sh)

    # hardware ceilings of this GPU, measured before the timed region
    ceil = measure_ceilings(torch, spec["bits"], small=args.workload.endswith("-small") or spec["bits"] < (1 << 30))
    for _ in range(max(args.warmup, 0)):
        clear()
        step()
    torch.cuda.synchronize()
    if sbf.status() != 0:
        raise RuntimeError("device status error during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        clear()
        ev[i][0].record(stream)
        N.sbf_insert(sbf.handle, dseq.data_ptr(), doff.data_ptr(), n_ins, sh)
        ev[i][1].record(stream)
        N.sbf_query(sbf.handle, dq.data_ptr(), dqo.data_ptr(), n_q, out.data_ptr(), sh)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t_wall = time.perf_counter() - t_wall0
    clocks = sampler.stop() if sampler else None
    t_ins = [ev[i][0].elapsed_time(ev[i][1]) / 1e3 for i in range(args.steps)]
    t_q = [ev[i][1].elapsed_time(ev[i][2]) / 1e3 for i in range(args.steps)]
    # per call: the median of the event-timed calls (the slowest rank's);
    # the means are kept for the roofline's average launch duration
    med_ins, med_q, mean_ins, mean_q = max_over_ranks(
        pg, [statistics.median(t_ins), statistics.median(t_q), statistics.mean(t_ins), statistics.mean(t_q)])
    step_s = med_ins + med_q
    if sbf.status() != 0:
        raise RuntimeError("device status error in the timed region")

    words = out.cpu().numpy().view(np.uint32)
    fpr = fpr_of(words, qry, p["k"], B)

    # the query batch as a dense record batch (all reads of one length, DNA):
    # sbf_query_dense, timed apart from the step, its answers checked equal
    dense = None
    lens = np.diff(qry.offsets)
    alu_peak = ceil["alu"]["ops_per_s"] / 1e12
    if p["alphabet"] == "dna" and lens.size and (lens == lens[0]).all() and qry.offsets[0] == 0:
        rl = int(lens[0])
        dout = torch.zeros_like(out)

        def dq_call():
            N.sbf_query_dense(sbf.handle, dq.data_ptr(), n_q, rl, dout.data_ptr(), sh)
        t_dense = _timed(torch, dq_call, warmup=2, reps=max(args.steps, 3))
        same = bool(torch.equal(dout[: (qry.n_bases + 31) // 32], out[: (qry.n_bases + 31) // 32]))
        dense = {"call": "sbf_query_dense", "record_len": rl, "kmers_per_s": nk_q / t_dense,
                 "ms": 1e3 * t_dense, "answers_equal_csr": same,
                 "alu_frac": alu_ops(p)["query"] * nk_q / t_dense / 1e12 / alu_peak,
                 "note": "one strip per read (skips the k-1 tail positions of each read); "
                         "not part of `value`, which uses the CSR query (it runs this batch dense too)"}
        del dout
    value = throughput(world, 1, nk_ins + nk_q, step_s)

    # rooflines: insert against HBM (one 32-byte sector read and written per
    # run), query against the ALU pipe; "roofline" is the dominant (longer) one.
    peaks, peak_src = measured_peaks()
    sha = kernel_source_sha(p)
    runs_i, runs_i_src = exact_runs(args.workload, "insert", ins, p, spec["bits"], p["k"], p["m"], B)
    runs_q, runs_q_src = exact_runs(args.workload, "query", qry, p, spec["bits"], p["k"], p["m"], B)
    ops = alu_ops(p)
    bytes_ins = ins.n_bases + 8 * (n_ins + 1) + 64 * runs_i
    bytes_q = qry.n_bases + 8 * (n_q + 1) + 32 * runs_q + 4 * ((qry.n_bases + 31) // 32)

    def traffic_of(name, nk):
        rec = MEASURED_TRAFFIC.get(args.workload)
        if rec and rec["source_sha"] == sha and rec[name] is not None:
            return rec[name] * nk
        return None

    ins_ach = bytes_ins / mean_ins / 1e9
    roof_ins = {"bound": "hbm", "kernel": kname("insert"),
                "achieved": ins_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ins_ach / peaks["hbm_gbs"], "traffic": traffic_of("insert", nk_ins),
                "peak_source": f"{peak_src} hbm_gbs (copy)",
                "algorithmic_bytes_per_kmer": bytes_ins / nk_ins,
                "runs_per_launch": runs_i, "runs_source": runs_i_src,
                "avg_launch_ms": 1e3 * mean_ins, "median_launch_ms": 1e3 * med_ins}
    flush_form = insert_flush_form(torch, spec["bits"], p["alphabet"])
    rmw = ceil["rmw"].get(flush_form)
    if rmw:
        roof_ins["pattern_peak"] = {
            "what": f"random 32-byte row read-modify-writes over a {rmw['buffer_gib']:.0f} GiB buffer, "
                    f"hand-written probe in the insert's flush form ({flush_form}), measured in this run",
            "form": flush_form, "rows_per_s": rmw["rows_per_s"], "runs_per_s": runs_i / mean_ins,
            "frac": runs_i / mean_ins / rmw["rows_per_s"],
            "all_forms_rows_per_s": {k: v["rows_per_s"] for k, v in ceil["rmw"].items()}}
    q_ach = ops["query"] * nk_q / mean_q / 1e12
    roof_q = {"bound": "alu", "kernel": kname("query"),
              "achieved": q_ach, "peak": alu_peak, "unit": "Tops/s (ALU pipe)",
              "frac": q_ach / alu_peak, "traffic": traffic_of("query", nk_q),
              "peak_source": f"measured in this run: probe of a LOP3/SHF/ISETP/SEL/IMNMX mix on all "
                             f"{ceil['sms']} SMs ({ceil['alu']['ops_per_sm_clock_at_2070MHz']:.1f} ops/SM/clock "
                             f"at 2.07 GHz)",
              "ops_per_kmer": ops["query"], "avg_launch_ms": 1e3 * mean_q, "median_launch_ms": 1e3 * med_q,
              "algorithmic_bytes_per_kmer": bytes_q / nk_q, "runs_per_launch": runs_q, "runs_source": runs_q_src,
              "hbm_frac": bytes_q / mean_q / 1e9 / peaks["hbm_gbs"]}
    rd = ceil["read"].get(QUERY_SHARD_FORM)
    if rd:
        roof_q["pattern_peak"] = {
            "what": f"random 32-byte row reads over a {rd['buffer_gib']:.0f} GiB buffer, hand-written probe in "
                    f"the query's shard-load form ({QUERY_SHARD_FORM}), measured in this run",
            "form": QUERY_SHARD_FORM, "rows_per_s": rd["rows_per_s"], "runs_per_s": runs_q / mean_q,
            "frac": runs_q / mean_q / rd["rows_per_s"],
            "all_forms_rows_per_s": {k: v["rows_per_s"] for k, v in ceil["read"].items()}}
    ins_alu = ops["insert"] * nk_ins / mean_ins / 1e12
    roof_ins["alu_frac"] = ins_alu / alu_peak
    roofline, roofline_other = (roof_ins, roof_q) if mean_ins >= mean_q else (roof_q, roof_ins)

    e2e = None
    if not args.no_e2e:
        if args.host_mode is not None:
            N.sbf_set_host_mode(sbf.handle, args.host_mode)
        if args.host_chunk is not None:
            N.sbf_set_host_chunk(sbf.handle, args.host_chunk)
        e2e = run_e2e(torch, N, sbf, ins, qry, nk_ins + nk_q, pg, world, max(args.steps, 10))

    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(ins, qry, spec["bits"], p=p, single_thread=True)

    if rank == 0:
        line = {
            "metric": metric_of(p), "value": value, "unit": "k-mers/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * step_s, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8/u64 (integer)",
            "data": "synthetic",
            "config": dict(wcfg, **{
                       "l2": {"out-of-cache": "inputs larger than L2 (sequences 1 GB each, filter 8 GiB)",
                              "protein-like": "inputs larger than L2 (sequences 0.5 GB each, filter 1 GiB)",
                              "triplet": "inputs larger than L2 (sequences 1 GB each, filter 1 GiB)"}
                             .get(args.workload, "see workload"),
                       "filter_between_steps": "zeroed before every insert (sbf_clear, untimed, outside "
                                               "the events; it also flushes L2)",
                       "timing": "CUDA events around each call on the launching stream; value and "
                                 "ms_per_step from the median insert + median query",
                       "replicas": world}),
            "insert_kmers_per_s": throughput(world, 1, nk_ins, med_ins),
            "query_kmers_per_s": throughput(world, 1, nk_q, med_q),
            "insert_ms": {"median": 1e3 * med_ins, "mean": 1e3 * mean_ins, "all": [1e3 * t for t in t_ins]},
            "query_ms": {"median": 1e3 * med_q, "mean": 1e3 * mean_q, "all": [1e3 * t for t in t_q]},
            "value_from_means": throughput(world, 1, nk_ins + nk_q, mean_ins + mean_q),
            "fpr": fpr, "fpr_definition": "answer-positive fraction of the valid k-mers of the uniform reads",
            "query_dense": dense,
            "roofline": roofline, "roofline_other_kernel": roofline_other,
            "ceilings": ceil,
            "gpu_launches": 4 * args.steps,
            "gpu_launches_note": "per step: offsets check + insert kernel, offsets check + query kernel "
                                 "(the untimed filter clear is a memset)",
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cb,
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    sbf.close()
    if pg:
        pg.destroy_process_group()


def measure_ceilings(torch, filter_bits: int, small: bool = False) -> dict:
    """The ceilings of this GPU, from the hand-written probe kernels
    (libsbf_probes.so): the ALU instruction rate of the mix the filter
    kernels issue, on all SMs; scattered 32-byte row read-modify-writes and
    reads over a buffer of the filter's size (at least 1 GiB, so not
    L2-resident), in every form the kernels may use; ~120 M rows each (the
    out-of-cache insert's run count)."""
    from minimizer_sharded_bloom_gb300 import probes
    res = {"sms": probes.sm_count(), "alu": probes.alu_rate(torch, "mix")}
    res["alu_imad"] = probes.alu_rate(torch, "imad")
    gib = max(1, filter_bits >> 33)
    n = 30_000_000 if small else 118_000_000
    buf = torch.zeros((gib << 30) // 8, dtype=torch.int64, device="cuda")
    res["rmw"] = {m: probes.rmw_rate(torch, m, n_updates=n, buf=buf) for m in ("red4", "red_queue")}
    res["read"] = {m: probes.read_rate(torch, m, n_reads=n, buf=buf) for m in ("ld_nc", "cp_async", "bulk32")}
    del buf
    torch.cuda.empty_cache()
    return res


def _timed(torch, fn, warmup=2, reps=3, before=None):
    """Seconds per call of `fn`: the mean of `reps` back-to-back calls, or, with
    `before` (run untimed ahead of every call, e.g. zeroing the filter), the
    median of `reps` calls each bracketed by its own events."""
    for _ in range(warmup):
        if before is not None:
            before()
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if before is not None:
        times = []
        for _ in range(reps):
            before()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / 1e3)
        return statistics.median(times)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def run_suite(args):
    """One JSON line per configuration (tiny, genome-like, irregular, the
    protein-like and triplet alphabets) and per point of the (s, m, H) sweep at
    k = 31 and 2^30 bits: insert and query
    k-mers/s (CUDA events, device-resident inputs) and the false-positive
    rate.  Parity of every point is covered by the tests."""
    import torch
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter, build_lib, _native as N
    build_lib.build()
    torch.cuda.set_device(0)
    st = int(torch.cuda.current_stream().cuda_stream)

    def dev(wl):
        return torch.from_numpy(wl.seq).cuda(), torch.from_numpy(wl.offsets).cuda()

    def measure(name, ins, qry, bits, k=K, m=M, s=S, H=H, fpr_qry=None, extra=None, p=None, sectors="fixed"):
        alphabet = "dna"
        if p is not None:
            k, m, s, H, alphabet = p["k"], p["m"], p["s"], p["H"], p["alphabet"]
        B = 3 if alphabet == "dna_triplet" else 1
        sbf = SuperBloomFilter(bits, k=k, m=m, s=s, H=H, seed=SEED, alphabet=alphabet, sectors=sectors)
        di, dio = dev(ins)
        dq, dqo = dev(qry)
        out = torch.zeros((qry.n_bases + 31) // 32 + 2, dtype=torch.int32, device="cuda")
        # the filter is zeroed before every timed insert, as in the main bench
        t_ins = _timed(torch, lambda: N.sbf_insert(sbf.handle, di.data_ptr(), dio.data_ptr(),
                                                    ins.n_records, st),
                       reps=5, before=lambda: N.sbf_clear(sbf.handle, st))
        t_q = _timed(torch, lambda: N.sbf_query(sbf.handle, dq.data_ptr(), dqo.data_ptr(),
                                                 qry.n_records, out.data_ptr(), st))
        words = out.cpu().numpy().view(np.uint32)
        fq = fpr_qry or qry
        if fpr_qry is not None:
            df, dfo = dev(fpr_qry)
            fout = torch.zeros((fpr_qry.n_bases + 31) // 32 + 2, dtype=torch.int32, device="cuda")
            N.sbf_query(sbf.handle, df.data_ptr(), dfo.data_ptr(), fpr_qry.n_records, fout.data_ptr(), st)
            torch.cuda.synchronize()
            words = fout.cpu().numpy().view(np.uint32)
            del df, dfo, fout
        if name == "irregular":
            # every record is uniform-random and holds N runs: count the valid
            # k-mers by querying against an all-ones image (each valid k-mer
            # answers 1), then FPR = positives / valid k-mers
            lo_w, hi_w = int(qry.offsets[0]) >> 5, (int(qry.offsets[-1]) + 31) >> 5
            positives = int(np.unpackbits(words[lo_w:hi_w].view(np.uint8)).sum())
            ones = torch.full((sbf.num_shards, 4), -1, dtype=torch.int64, device="cuda")
            sbf.load(ones)
            out.zero_()
            N.sbf_query(sbf.handle, dq.data_ptr(), dqo.data_ptr(), qry.n_records, out.data_ptr(), st)
            torch.cuda.synchronize()
            allw = out.cpu().numpy().view(np.uint32)
            n_valid = int(np.unpackbits(allw[lo_w:hi_w].view(np.uint8)).sum())
            fpr, n_fpr = positives / max(n_valid, 1), n_valid
            del ones
        else:
            fpr, n_fpr = fpr_of(words, fq, k, B), fpr_count(fq, k, B)
        # valid k-mers where the oracle's count of this input is stored, else positions
        pp = dict(k=k, m=m, s=s, H=H, alphabet=alphabet)
        st_i = stored_count(name, "insert", ins, pp, bits) if sectors == "fixed" else None
        st_q = stored_count(name, "query", qry, pp, bits) if sectors == "fixed" else None
        n_i = st_i["valid_kmers"] if st_i else kmer_count(ins, k, B)
        n_q = st_q["valid_kmers"] if st_q else kmer_count(qry, k, B)
        line = {"suite": name, "alphabet": alphabet, "k": k, "m": m, "s": s, "H": H, "sectors": sectors,
                "filter_bits": bits, "specialized": sbf.specialized,
                "insert_kmers": n_i, "query_kmers": n_q,
                "kmers_counted": "valid k-mers (oracle count)" if st_i and st_q else "k-mer positions",
                "insert_kmers_per_s": n_i / t_ins,
                "query_kmers_per_s": n_q / t_q, "fpr": fpr,
                "fpr_kmers": n_fpr}
        line.update(extra or {})
        print(json.dumps(line), flush=True)
        sbf.close()

    ins, qry = synth.tiny()
    measure("tiny", ins, qry, 1 << 20)
    g_ins, g_qry = synth.genome_like()
    measure("genome-like", g_ins, g_qry, 1 << 30)
    sweep_q = synth.sweep_queries(g_ins)
    for s_ in (20, 24, 28, 31):
        for m_ in (12, 14, 16, 18, 21):
            for H_ in (1, 2, 4, 6, 8):
                measure("sweep", g_ins, g_qry, 1 << 30, m=m_, s=s_, H=H_, fpr_qry=sweep_q,
                        extra={"fpr_queries": "10,000,000 uniform 31-mers absent from the inserted set"})
    for H_ in (12, 16):  # the paper's larger hash counts (salted multiply, Sec. IV-G)
        measure("sweep", g_ins, g_qry, 1 << 30, m=16, s=28, H=H_, fpr_qry=sweep_q,
                extra={"fpr_queries": "10,000,000 uniform 31-mers absent from the inserted set"})
    # hash-chosen sectors (SBF_FLAG_HASHED_SECTORS) against the paper's layout
    # where it applies (H < 4)
    for s_ in (20, 24, 28, 31):
        for H_ in (1, 2):
            measure("sweep", g_ins, g_qry, 1 << 30, m=16, s=s_, H=H_, fpr_qry=sweep_q, sectors="hashed",
                    extra={"fpr_queries": "10,000,000 uniform 31-mers absent from the inserted set"})
    del g_ins, g_qry, sweep_q
    i_ins, i_qry = synth.irregular()
    i_qry.meta["is_random"] = np.ones(i_qry.n_records, dtype=bool)
    measure("irregular", i_ins, i_qry, 1 << 32)
    del i_ins, i_qry
    for name in ("protein-like", "triplet"):
        spec = WORKLOADS[name]
        a_ins, a_qry = spec["make"]()
        measure(name, a_ins, a_qry, spec["bits"], p=spec["p"])
        del a_ins, a_qry


def _int_range(spec: str):
    out = []
    for part in spec.split(","):
        a, _, b = part.partition("-")
        out += list(range(int(a), int(b or a) + 1))
    return out


def run_fig4(args):
    """The paper's parameter study (Sec. V-B, Fig. 4) at k = 31: every (s, m, H)
    of the grid inserts the 50 Mbp genome-like reference into its own 2^30-bit
    filter (the paper: C. elegans into 256 MiB, ~21 bits per k-mer here and
    there), queries its 10^6 reads (timing) and 10^7 uniform 31-mers absent
    from the reference (FPR).  Every point is timed on the runtime-parameter
    kernels (one kernel family for the whole heatmap); points with a compiled
    strip kernel are timed on it too ("strip").  Times are CUDA-event means
    of two calls after one untimed call."""
    import torch
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter, build_lib, _native as N
    build_lib.build()
    torch.cuda.set_device(0)
    st = int(torch.cuda.current_stream().cuda_stream)
    g_ins, g_qry = synth.genome_like()
    fq = synth.sweep_queries(g_ins)
    dev = [torch.from_numpy(x).cuda() for x in (g_ins.seq, g_ins.offsets, g_qry.seq, g_qry.offsets, fq.seq,
                                                  fq.offsets)]
    di, dio, dq, dqo, df, dfo = dev
    out = torch.zeros((g_qry.n_bases + 31) // 32 + 2, dtype=torch.int32, device="cuda")
    fout = torch.zeros((fq.n_bases + 31) // 32 + 2, dtype=torch.int32, device="cuda")
    nk_i, nk_q = kmer_count(g_ins), kmer_count(g_qry)
    def timed_pair(sbf):
        t_i = _timed(torch, lambda: N.sbf_insert(sbf.handle, di.data_ptr(), dio.data_ptr(), g_ins.n_records, st),
                     warmup=1, reps=2)
        t_q = _timed(torch, lambda: N.sbf_query(sbf.handle, dq.data_ptr(), dqo.data_ptr(), g_qry.n_records,
                                                 out.data_ptr(), st), warmup=1, reps=2)
        return t_i, t_q

    res = {}
    for H_ in _int_range(args.fig4_h):
        for s_ in _int_range(args.fig4_s):
            for m_ in _int_range(args.fig4_m):
                # every point on the runtime-parameter kernels (one kernel family
                # for the whole time heatmap); its FPR is the method's, whatever
                # the kernel
                sbf = SuperBloomFilter(1 << 30, k=31, m=m_, s=s_, H=H_, seed=SEED, runtime_kernels=True)
                t_i, t_q = timed_pair(sbf)
                N.sbf_query(sbf.handle, df.data_ptr(), dfo.data_ptr(), fq.n_records, fout.data_ptr(), st)
                torch.cuda.synchronize()
                if sbf.status() != 0:
                    raise RuntimeError(f"device status error at s={s_} m={m_} H={H_}")
                fpr = fpr_of(fout.cpu().numpy().view(np.uint32), fq)
                sbf.close()
                line = {"fig4": True, "s": s_, "m": m_, "H": H_, "k": 31, "kernel": "runtime",
                        "insert_kmers_per_s": nk_i / t_i, "query_kmers_per_s": nk_q / t_q,
                        "insert_ms": 1e3 * t_i, "query_ms": 1e3 * t_q, "fpr": fpr}
                spec = SuperBloomFilter(1 << 30, k=31, m=m_, s=s_, H=H_, seed=SEED)
                if spec.specialized:
                    u_i, u_q = timed_pair(spec)
                    line["strip"] = {"insert_kmers_per_s": nk_i / u_i, "query_kmers_per_s": nk_q / u_q,
                                     "insert_ms": 1e3 * u_i, "query_ms": 1e3 * u_q}
                spec.close()
                res[(s_, m_, H_)] = line
                print(json.dumps(line), flush=True)
    print(json.dumps({"fig4_orderings": fig4_orderings(res)}), flush=True)


def fig4_orderings(res) -> dict:
    """The paper's Sec. V-B statements about Fig. 4, each as (ours, the
    paper's), where the grid holds the points; FPR ratios are exact results
    of the method, times those of this GPU's runtime-parameter kernels (one
    kernel family for every point)."""
    def get(s_, m_, H_, key):
        r = res.get((s_, m_, H_))
        return None if r is None else r[key]

    def ratio(a, b):
        return None if a is None or b is None or not b else a / b
    tot = {k: r["insert_ms"] + r["query_ms"] for k, r in res.items()}
    out = {
        "fpr H=8 / H=4 at (28,16)": (ratio(get(28, 16, 8, "fpr"), get(28, 16, 4, "fpr")), 2.0),
        "fpr H=16 / H=4 at (28,16)": (ratio(get(28, 16, 16, "fpr"), get(28, 16, 4, "fpr")), 5.2),
        "time H=8 / H=4 at (28,16)": (ratio(tot.get((28, 16, 8)), tot.get((28, 16, 4))), 1.076),
        "time H=16 / H=4 at (28,16)": (ratio(tot.get((28, 16, 16)), tot.get((28, 16, 4))), 1.659),
        "fpr s=30 / s=28 at (m,H)=(16,4)": (ratio(get(30, 16, 4, "fpr"), get(28, 16, 4, "fpr")), 1.256),
        "fpr s=31 / s=28 at (m,H)=(16,4)": (ratio(get(31, 16, 4, "fpr"), get(28, 16, 4, "fpr")), 2.29),
        "fpr s=28 / s=16 at (m,H)=(16,4)": (ratio(get(28, 16, 4, "fpr"), get(16, 16, 4, "fpr")), 1 - 0.374),
        "time s=28 / s=16 at (m,H)=(16,4)": (ratio(tot.get((28, 16, 4)), tot.get((16, 16, 4))), 1 - 0.291),
        "fpr m=12 / m=8 at (s,H)=(28,4)": (ratio(get(28, 12, 4, "fpr"), get(28, 8, 4, "fpr")), 1 - 0.917),
        "fpr m=16 / m=12 at (s,H)=(28,4)": (ratio(get(28, 16, 4, "fpr"), get(28, 12, 4, "fpr")), 1 - 0.908),
        "fpr m=18 / m=16 at (s,H)=(28,4)": (ratio(get(28, 18, 4, "fpr"), get(28, 16, 4, "fpr")), 1.035),
        "time m=18 / m=16 at (s,H)=(28,4)": (ratio(tot.get((28, 18, 4)), tot.get((28, 16, 4))), 1.085),
        "fpr m=31 / m=16 at (s,H)=(28,4)": (ratio(get(28, 31, 4, "fpr"), get(28, 16, 4, "fpr")), 4.8),
    }
    # Pareto set (minimise FPR and insert+query time jointly)
    pts = sorted(res, key=lambda k: (res[k]["fpr"], tot[k]))
    pareto, best_t = [], float("inf")
    for k in pts:
        if tot[k] < best_t:
            pareto.append(k)
            best_t = tot[k]
    return {"ratios (ours, paper)": out, "pareto (s, m, H)": pareto}


def run_e2e(torch, N, sbf, ins, qry, nk_total, pg, world, steps):
    """Same metric through the host-facing C-ABI calls: pinned host inputs,
    host-to-device copies and the answer's device-to-host copy inside the
    timed region (each call synchronizes).  The filter is zeroed before each
    step, outside the timed region.  Each call is timed on the host clock;
    the value uses the median step, and the per-call medians and maxima plus
    the host link's copy rate (1 GiB from the same kind of pinned buffer,
    CUDA events) are reported beside it."""
    h_seq = torch.from_numpy(ins.seq).pin_memory()
    h_off = torch.from_numpy(ins.offsets).pin_memory()
    h_q = torch.from_numpy(qry.seq).pin_memory()
    h_qo = torch.from_numpy(qry.offsets).pin_memory()
    h_out = torch.zeros((qry.n_bases + 31) // 32 + 1, dtype=torch.int32).pin_memory()
    sh = int(torch.cuda.current_stream().cuda_stream)

    def one():
        N.sbf_clear(sbf.handle, sh)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        N.sbf_insert_host(sbf.handle, h_seq.data_ptr(), h_off.data_ptr(), ins.n_records, sh)
        t1 = time.perf_counter()
        N.sbf_query_host(sbf.handle, h_q.data_ptr(), h_qo.data_ptr(), qry.n_records, h_out.data_ptr(), sh)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    for _ in range(3):  # the first calls size the staging buffers
        one()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ti, tq = [], []
    for _ in range(steps):
        a, b = one()
        ti.append(a)
        tq.append(b)
    tstep = [a + b for a, b in zip(ti, tq)]
    med, mean, worst = max_over_ranks(pg, [statistics.median(tstep), statistics.mean(tstep), max(tstep)])
    # the host link, measured now: 1 GiB from pinned memory to the device
    hb = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    db = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    link = []
    for _ in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        db.copy_(hb, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        link.append((1 << 30) / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del hb, db
    h2d = ins.seq.nbytes + ins.offsets.nbytes + qry.seq.nbytes + qry.offsets.nbytes
    d2h = 4 * ((qry.n_bases + 31) // 32)
    ms = [1e3 * x for x in (statistics.median(ti), max(ti), statistics.median(tq), max(tq))]
    return {"value": throughput(world, 1, nk_total, med), "unit": "k-mers/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "ms_per_step": 1e3 * med, "ms_per_step_mean": 1e3 * mean,
            "ms_per_step_max": 1e3 * worst, "value_from_mean": throughput(world, 1, nk_total, mean),
            "insert_host_ms": {"median": ms[0], "max": ms[1], "all": [round(1e3 * x, 3) for x in ti]},
            "query_host_ms": {"median": ms[2], "max": ms[3], "all": [round(1e3 * x, 3) for x in tq]},
            "link_h2d_gbs": statistics.median(link),
            "link_bound_ms_per_step": 1e3 * h2d / (statistics.median(link) * 1e9),
            "path": "sbf_insert_host + sbf_query_host, pinned host buffers, host clock per call; "
                    "filter zeroed before each step (untimed)"}


if __name__ == "__main__":
    main()
