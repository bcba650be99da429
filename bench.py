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
# ALU-pipe peak: 152 SMs x 4 sub-partitions x 16 lanes x 2.07 GHz (maximum SM
# clock).  ncu reports the ALU pipe at 16 lanes per sub-partition: with the
# pipe ~75 % busy the issue rate is ~53 %, i.e. one ALU warp-instruction per
# two cycles at most.
ALU_PEAK_TOPS = 152 * 64 * 2.07e9 / 1e12

# ncu DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per k-mer of
# the full-size launches of each workload (summaries under profiles/), valid
# only for the kernel source they were measured on.
MEASURED_TRAFFIC = {
    "out-of-cache": {"source_sha": "81fea15e301fb957", "insert": 14.4073, "query": 18.2213},
    "protein-like": {"source_sha": "5a8e9ca5e801e671", "insert": 37.0033, "query": 52.7077},
    "triplet": {"source_sha": "5ec40e89a3fe204a", "insert": 33.3874, "query": 45.4888},
}


def kernel_source_sha(p=MAIN) -> str:
    """Hash of the source files the workload's kernels are built from."""
    files = {"dna": ("sbf_strip.cuh", "sbf_device.cuh", "sbf_inst_main.cu"),
             "protein": ("sbf_strip.cuh", "sbf_device.cuh", "sbf_inst_protein.cu"),
             "dna_triplet": ("sbf_strip.cuh", "sbf_alphabet.cu", "sbf_device.cuh",
                             "sbf_inst_triplet.cu")}[p["alphabet"]]
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "minimizer_sharded_bloom_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
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


def cpu_baseline(ins, qry, bits: int, budget_bases: int = 40_000_000, reads: int = 300_000, p=MAIN):
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
    return {"value": nk / (t2 - t0), "unit": "k-mers/s", "cores": cores, "kind": "oracle",
            "sample": f"first {s_ins.n_bases:,} bytes ({r} records) inserted, first {rq:,} reads "
                      f"queried; {nk:,} k-mers in {t2 - t0:.1f} s",
            "insert_kmers_per_s": nk_i / (t1 - t0),
            "query_kmers_per_s": nk_q / (t2 - t1)}


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
            "config": {"workload": spec["desc"], "k": p["k"], "m": p["m"], "s": p["s"], "H": p["H"],
                       "alphabet": p["alphabet"],
                       "filter_bits": spec["bits"], "timing": "host wall clock per sample"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "k-mers/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
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
    args = ap.parse_args()
    if args.suite:
        run_suite(args)
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
    nk_ins, nk_q = kmer_count(ins, p["k"], B), kmer_count(qry, p["k"], B)

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

    def step():
        N.sbf_insert(sbf.handle, dseq.data_ptr(), doff.data_ptr(), n_ins, sh)
        N.sbf_query(sbf.handle, dq.data_ptr(), dqo.data_ptr(), n_q, out.data_ptr(), sh)

    # the random-RMW ceiling (an 8 GiB probe) for filters larger than L2,
    # except at the profiling sizes
    rmw_gib = max(1, spec["bits"] >> 33)  # the probe spans the filter's size
    rmw_ceiling = (random_rmw_ceiling(torch, gib=rmw_gib)
                   if spec["bits"] > 8 * (129 << 20) and not args.workload.endswith("-small") else None)
    for _ in range(max(args.warmup, 0)):
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
    total = sum(t_ins) + sum(t_q)
    total, s_ins, s_q = max_over_ranks(pg, [total, sum(t_ins), sum(t_q)])
    if sbf.status() != 0:
        raise RuntimeError("device status error in the timed region")

    words = out.cpu().numpy().view(np.uint32)
    fpr = fpr_of(words, qry, p["k"], B)

    # the query batch as a dense record batch (all reads of one length, DNA):
    # sbf_query_dense, timed apart from the step, its answers checked equal
    dense = None
    lens = np.diff(qry.offsets)
    if p["alphabet"] == "dna" and lens.size and (lens == lens[0]).all() and qry.offsets[0] == 0:
        rl = int(lens[0])
        dout = torch.zeros_like(out)

        def dq_call():
            N.sbf_query_dense(sbf.handle, dq.data_ptr(), n_q, rl, dout.data_ptr(), sh)
        t_dense = _timed(torch, dq_call, warmup=2, reps=max(args.steps, 3))
        same = bool(torch.equal(dout[: (qry.n_bases + 31) // 32], out[: (qry.n_bases + 31) // 32]))
        dense = {"call": "sbf_query_dense", "record_len": rl, "kmers_per_s": nk_q / t_dense,
                 "ms": 1e3 * t_dense, "answers_equal_csr": same,
                 "alu_frac": alu_ops(p)["query"] * nk_q / t_dense / 1e12 / ALU_PEAK_TOPS,
                 "note": "one strip per read (skips the k-1 tail positions of each read); "
                         "not part of `value`, which uses the CSR query"}
        del dout
    value = throughput(world, args.steps, nk_ins + nk_q, total)

    # rooflines: insert against HBM (one 32-byte sector read and written per
    # run), query against the ALU pipe; "roofline" is the dominant (longer) one.
    peaks, peak_src = measured_peaks()
    avg_ins, avg_q = s_ins / args.steps, s_q / args.steps
    sha = kernel_source_sha(p)
    runs_i = runs_estimate(ins, p["k"], p["m"], B)
    runs_q = runs_estimate(qry, p["k"], p["m"], B)
    ops = alu_ops(p)
    bytes_ins = ins.n_bases + 8 * (n_ins + 1) + 64 * runs_i
    bytes_q = qry.n_bases + 8 * (n_q + 1) + 32 * runs_q + 4 * ((qry.n_bases + 31) // 32)

    def traffic_of(name, nk):
        rec = MEASURED_TRAFFIC.get(args.workload)
        if rec and rec["source_sha"] == sha and rec[name] is not None:
            return rec[name] * nk
        return None

    ins_ach = bytes_ins / avg_ins / 1e9
    roof_ins = {"bound": "hbm", "kernel": kname("insert"),
                "achieved": ins_ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ins_ach / peaks["hbm_gbs"], "traffic": traffic_of("insert", nk_ins),
                "peak_source": f"{peak_src} hbm_gbs (copy)",
                "algorithmic_bytes_per_kmer": bytes_ins / nk_ins,
                "runs_per_launch": runs_i, "avg_launch_ms": 1e3 * avg_ins}
    if rmw_ceiling:
        roof_ins["pattern_peak"] = {
            "what": "random 32-byte row read-modify-write (4 x 64-bit atomic add per row, "
                    f"torch index_add_) over a {rmw_gib} GiB tensor (the filter's size), measured in this run",
            "rows_per_s": rmw_ceiling, "runs_per_s": runs_i / avg_ins,
            "frac": runs_i / avg_ins / rmw_ceiling}
    q_ach = ops["query"] * nk_q / avg_q / 1e12
    roof_q = {"bound": "alu", "kernel": kname("query"),
              "achieved": q_ach, "peak": ALU_PEAK_TOPS, "unit": "Tops/s (ALU pipe)",
              "frac": q_ach / ALU_PEAK_TOPS, "traffic": traffic_of("query", nk_q),
              "peak_source": "152 SMs x 64 ALU lanes x 2.07 GHz (recipe SM count and clock)",
              "ops_per_kmer": ops["query"], "avg_launch_ms": 1e3 * avg_q,
              "algorithmic_bytes_per_kmer": bytes_q / nk_q,
              "hbm_frac": bytes_q / avg_q / 1e9 / peaks["hbm_gbs"]}
    ins_alu = ops["insert"] * nk_ins / avg_ins / 1e12
    roof_ins["alu_frac"] = ins_alu / ALU_PEAK_TOPS
    roofline, roofline_other = (roof_ins, roof_q) if avg_ins >= avg_q else (roof_q, roof_ins)

    e2e = None
    if not args.no_e2e:
        if args.host_mode is not None:
            N.sbf_set_host_mode(sbf.handle, args.host_mode)
        if args.host_chunk is not None:
            N.sbf_set_host_chunk(sbf.handle, args.host_chunk)
        e2e = run_e2e(torch, N, sbf, ins, qry, nk_ins + nk_q, pg, world, min(args.steps, 3))

    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(ins, qry, spec["bits"], p=p)

    if rank == 0:
        line = {
            "metric": metric_of(p), "value": value, "unit": "k-mers/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8/u64 (integer)",
            "data": "synthetic",
            "config": {"workload": spec["desc"], "k": p["k"], "m": p["m"], "s": p["s"], "H": p["H"],
                       "alphabet": p["alphabet"], "seed": SEED,
                       "filter_bits": spec["bits"], "insert_kmers": nk_ins, "query_kmers": nk_q,
                       "insert_records": n_ins, "query_records": n_q,
                       "l2": {"out-of-cache": "inputs larger than L2 (sequences 1 GB each, filter 8 GiB)",
                              "protein-like": "inputs larger than L2 (sequences 0.5 GB each, filter 1 GiB)",
                              "triplet": "inputs larger than L2 (sequences 1 GB each, filter 1 GiB)"}
                             .get(args.workload, "see workload"),
                       "filter_between_steps": "not cleared (insert is idempotent; same work)",
                       "replicas": world},
            "insert_kmers_per_s": throughput(world, args.steps, nk_ins, s_ins),
            "query_kmers_per_s": throughput(world, args.steps, nk_q, s_q),
            "fpr": fpr, "fpr_definition": "answer-positive fraction of the valid k-mers of the uniform reads",
            "query_dense": dense,
            "roofline": roofline, "roofline_other_kernel": roofline_other,
            "gpu_launches": 4 * args.steps,
            "gpu_launches_note": "per step: offsets check + insert kernel, offsets check + query kernel",
            "clocks": clocks, "e2e": e2e, "cpu_baseline": cb,
            "wall_s_timed": t_wall,
        }
        print(json.dumps(line), flush=True)
    sbf.close()
    if pg:
        pg.destroy_process_group()


def random_rmw_ceiling(torch, gib: int = 8, rows_touched: int = 25_000_000) -> float:
    """Rows per second of random 32-byte read-modify-writes over a gib-GiB
    tensor (torch index_add_: four 64-bit atomic adds per row) -- the memory
    system's ceiling for the insert's per-run shard update."""
    n_rows = (gib << 30) // 32
    F = torch.zeros(n_rows, 4, dtype=torch.int64, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(1)
    idx = torch.randint(0, n_rows, (rows_touched,), device="cuda", generator=g)
    src = torch.ones(rows_touched, 4, dtype=torch.int64, device="cuda")
    for _ in range(2):
        F.index_add_(0, idx, src)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        F.index_add_(0, idx, src)
    e1.record()
    torch.cuda.synchronize()
    rate = 3 * rows_touched / (e0.elapsed_time(e1) / 1e3)
    del F, idx, src
    torch.cuda.empty_cache()
    return rate


def _timed(torch, fn, warmup=2, reps=3):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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

    def measure(name, ins, qry, bits, k=K, m=M, s=S, H=H, fpr_qry=None, extra=None, p=None):
        alphabet = "dna"
        if p is not None:
            k, m, s, H, alphabet = p["k"], p["m"], p["s"], p["H"], p["alphabet"]
        B = 3 if alphabet == "dna_triplet" else 1
        sbf = SuperBloomFilter(bits, k=k, m=m, s=s, H=H, seed=SEED, alphabet=alphabet)
        di, dio = dev(ins)
        dq, dqo = dev(qry)
        out = torch.zeros((qry.n_bases + 31) // 32 + 2, dtype=torch.int32, device="cuda")
        t_ins = _timed(torch, lambda: N.sbf_insert(sbf.handle, di.data_ptr(), dio.data_ptr(),
                                                    ins.n_records, st))
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
        line = {"suite": name, "alphabet": alphabet, "k": k, "m": m, "s": s, "H": H,
                "filter_bits": bits, "specialized": sbf.specialized,
                "insert_kmers": kmer_count(ins, k, B), "query_kmers": kmer_count(qry, k, B),
                "insert_kmers_per_s": kmer_count(ins, k, B) / t_ins,
                "query_kmers_per_s": kmer_count(qry, k, B) / t_q, "fpr": fpr,
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


def run_e2e(torch, N, sbf, ins, qry, nk_total, pg, world, steps):
    """Same metric through the host-facing C-ABI calls: pinned host inputs,
    host-to-device copies and the answer's device-to-host copy inside the
    timed region (each call synchronizes)."""
    h_seq = torch.from_numpy(ins.seq).pin_memory()
    h_off = torch.from_numpy(ins.offsets).pin_memory()
    h_q = torch.from_numpy(qry.seq).pin_memory()
    h_qo = torch.from_numpy(qry.offsets).pin_memory()
    h_out = torch.zeros((qry.n_bases + 31) // 32 + 1, dtype=torch.int32).pin_memory()

    def one():
        N.sbf_insert_host(sbf.handle, h_seq.data_ptr(), h_off.data_ptr(), ins.n_records, 0)
        N.sbf_query_host(sbf.handle, h_q.data_ptr(), h_qo.data_ptr(), qry.n_records,
                         h_out.data_ptr(), 0)

    for _ in range(2):  # the first calls size the staging buffers
        one()
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    dt = max_over_ranks(pg, [dt])[0]
    h2d = ins.seq.nbytes + ins.offsets.nbytes + qry.seq.nbytes + qry.offsets.nbytes
    d2h = 4 * ((qry.n_bases + 31) // 32)
    return {"value": throughput(world, steps, nk_total, dt), "unit": "k-mers/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "ms_per_step": 1e3 * dt / steps,
            "path": "sbf_insert_host + sbf_query_host, pinned host buffers, host wall clock"}


if __name__ == "__main__":
    main()
