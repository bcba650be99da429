"""CPU tests of the host-facing calls' chunk planner (csrc/sbf_chunks.h), the
host logic that cuts a staged insert or query into chunks: every k-mer start
is answered by exactly one chunk, from exactly its own bytes and record, in
its own codon frame; chunks end on answer-word boundaries, at record starts
where one is near; chunk sizes follow the growth policy.  The planner runs in
a small C++ driver compiled here with g++ (no GPU)."""
import os
import shutil
import subprocess
import zlib

import numpy as np
import pytest

from minimizer_sharded_bloom_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "minimizer_sharded_bloom_gb300", "csrc")
FIELDS = ("cs", "ce", "data_lo", "data_hi", "r0", "r1", "first", "last", "whole", "empty", "final")


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    gxx = shutil.which("g++")
    if not gxx:
        pytest.skip("g++ not found")
    exe = str(tmp_path_factory.mktemp("chunkplan") / "chunk_plan_driver")
    subprocess.run([gxx, "-std=c++17", "-O2", "-I", CSRC, os.path.join(HERE, "chunk_plan_driver.cpp"),
                    "-o", exe], check=True)
    return exe


def plan(driver, off, host_chunk, kb, sb, query):
    off = np.asarray(off, dtype=np.int64)
    n = off.size - 1
    text = f"{n} {host_chunk} {kb} {sb} {int(query)}\n" + " ".join(map(str, off.tolist())) + "\n"
    res = subprocess.run([driver], input=text, capture_output=True, text=True, check=True)
    lines = res.stdout.split("\n")
    chunk_max = int(lines[0])
    chunks = [dict(zip(FIELDS, map(int, ln.split()))) for ln in lines[1:] if ln.strip()]
    return chunk_max, chunks


def kmer_starts(starts, ends, kb, sb, a, b):
    """Positions g in [a, b) that start a k-mer inside one record
    [starts[i], ends[i]) at a multiple of sb from the record's start."""
    hit = np.zeros(max(b - a, 0), dtype=bool)
    for s, e in zip(starts.tolist(), ends.tolist()):
        lo_g, hi_g = max(s, a), min(e - kb + 1, b)
        if hi_g <= lo_g:
            continue
        first = lo_g + (-(lo_g - s)) % sb
        hit[first - a:hi_g - a:sb] = True
    return hit


def check_plan(off, chunk_max, chunks, host_chunk, kb, sb, query, per_position=True):
    off = np.asarray(off, dtype=np.int64)
    lo, hi = int(off[0]), int(off[-1])
    assert chunks, "no chunk"
    # contiguity and word-aligned edges
    assert chunks[0]["cs"] == lo & ~31
    for c, d in zip(chunks, chunks[1:]):
        assert d["cs"] == c["ce"]
    assert chunks[-1]["ce"] == hi and chunks[-1]["final"] == 1
    for c in chunks:
        assert c["ce"] > c["cs"]
        if not c["final"]:
            assert c["ce"] % 32 == 0 and c["ce"] < hi
            assert c["ce"] - c["cs"] <= chunk_max
        assert c["data_lo"] == max(c["cs"], lo)
        assert c["data_hi"] - c["cs"] <= chunk_max + kb
    assert chunk_max <= max(host_chunk, 32)
    for c in chunks:
        if c["empty"]:
            continue
        r0, r1 = c["r0"], c["r1"]
        assert 0 <= r0 < r1 <= off.size - 1
        # the chunk's view of its records: the caller's offsets with both ends replaced
        starts = off[r0:r1].copy()
        ends = off[r0 + 1:r1 + 1].copy()
        starts[0], ends[-1] = c["first"], c["last"]
        if r1 - r0 >= 2:
            assert c["first"] <= ends[0]
        # no record grows, none leaves the shipped bytes, frames are kept
        assert (starts >= off[r0:r1]).all() and (ends <= off[r0 + 1:r1 + 1]).all()
        assert ((starts - off[r0:r1]) % sb == 0).all()
        nonempty = ends > starts
        assert (starts[nonempty] >= c["data_lo"]).all() and (ends[nonempty] <= c["data_hi"]).all()
        assert bool(c["whole"]) == (c["first"] == off[r0] and c["last"] == off[r1])
        if not c["final"]:
            if c["data_hi"] == c["ce"]:
                assert off[r1] == c["ce"]  # ends at a record start: nothing shipped past ce
            else:
                assert c["data_hi"] == min(c["ce"] + kb - 1, hi)  # cut inside a record
        if per_position:
            # the k-mer starts this chunk answers are exactly the batch's in [cs, ce)
            want = kmer_starts(off[:-1], off[1:], kb, sb, c["cs"], c["ce"])
            got = kmer_starts(starts, ends, kb, sb, c["cs"], c["ce"])
            assert np.array_equal(want, got), f"chunk {c}: k-mer starts differ"


CASES = {
    "reads150": lambda rng: synth.csr(np.full(3000, 150)),
    "reads97": lambda rng: synth.csr(np.full(3000, 97)),
    "mixed_with_empty": lambda rng: synth.csr(rng.integers(0, 3000, size=300)),
    "long_records": lambda rng: synth.csr(rng.integers(5000, 20000, size=40)),
    "one_record": lambda rng: synth.csr([100_000]),
    "offset_start": lambda rng: 7 + synth.csr(rng.integers(1, 900, size=400)),
    "aligned_start": lambda rng: 4096 + synth.csr(rng.integers(1, 900, size=400)),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("kb,sb", [(31, 1), (12, 1), (30, 3)])
@pytest.mark.parametrize("query", [False, True])
@pytest.mark.parametrize("host_chunk", [4096, 10_016])
def test_chunks_cover_every_kmer_once(driver, case, kb, sb, query, host_chunk):
    """Every chunk answers exactly the batch's k-mer starts in [cs, ce), from
    records clipped only inside the bytes it ships and only at symbol
    boundaries (DNA, protein and DNA triplets, reads, long records cut across
    chunks, empty records, unaligned and aligned first offsets)."""
    rng = np.random.default_rng(zlib.crc32(f"{case}/{kb}/{sb}/{query}/{host_chunk}".encode()))
    off = CASES[case](rng)
    chunk_max, chunks = plan(driver, off, host_chunk, kb, sb, query)
    check_plan(off, chunk_max, chunks, host_chunk, kb, sb, query)


def test_uniform_reads_give_whole_dense_ready_chunks(driver):
    """A batch of equal-length reads is cut only at reads that start on a
    32-position boundary, so every chunk is a uniform batch whose first offset
    is a multiple of 32 (the condition for the query's dense geometry)."""
    for R in (31, 100, 150, 160):
        off = synth.csr(np.full(5000, R))
        chunk_max, chunks = plan(driver, off, 8192, 31, 1, True)
        assert len(chunks) > 10
        for c in chunks:
            assert c["whole"] == 1 and c["first"] % 32 == 0 and (c["first"] % R) == 0


def test_chunk_sizes_grow_and_a_query_tail_shrinks(driver):
    """Full-size policy on 2,000,000 reads of 150 bp (3 * 10^8 positions,
    a 2^26 chunk setting): chunks start near 2^22 positions and double up to
    an eighth of the batch (37.5 M positions, under 2^26); a query's last
    chunks shrink again, an insert's do not; every chunk stays whole."""
    off = synth.csr(np.full(2_000_000, 150))
    for query in (False, True):
        chunk_max, chunks = plan(driver, off, 1 << 26, 31, 1, query)
        assert chunk_max == 300_000_000 // 8
        check_plan(off, chunk_max, chunks, 1 << 26, 31, 1, query, per_position=False)
        sizes = [c["ce"] - c["cs"] for c in chunks]
        assert sizes[0] <= 1 << 22 and sizes[0] > (1 << 22) - 64 * 150
        assert max(sizes) <= chunk_max and max(sizes) > chunk_max - 64 * 150
        assert all(c["whole"] for c in chunks)
        tail = sizes[-4:]
        if query:
            assert tail[-1] < 1 << 24 and tail == sorted(tail, reverse=True)
        else:
            assert sizes[-2] > chunk_max - 64 * 150


def test_library_default_chunk_on_the_benchmark_read_batch(driver):
    """The library's default chunk setting (2^25 positions) on the benchmark's
    6,666,666 reads of 150 bp: chunks are capped at 2^25 positions (under an
    eighth of the batch), stay whole and end at read starts, so every chunk
    runs as a uniform batch; the query's tail shrinks below 2^23."""
    off = synth.csr(np.full(6_666_666, 150))
    chunk_max, chunks = plan(driver, off, 1 << 25, 31, 1, True)
    assert chunk_max == 1 << 25
    check_plan(off, chunk_max, chunks, 1 << 25, 31, 1, True, per_position=False)
    sizes = [c["ce"] - c["cs"] for c in chunks]
    assert max(sizes) <= 1 << 25 and all(c["whole"] for c in chunks)
    assert all(c["cs"] % 150 == 0 for c in chunks)
    assert sizes[-1] < 1 << 23


def test_small_batch_is_one_chunk(driver):
    off = synth.csr([120, 0, 33, 5000])
    chunk_max, chunks = plan(driver, off, 1 << 26, 31, 1, True)
    assert len(chunks) == 1 and chunks[0]["whole"] == 1 and chunks[0]["final"] == 1
    check_plan(off, chunk_max, chunks, 1 << 26, 31, 1, True)


@pytest.mark.parametrize("seed", range(6))
def test_malformed_offsets_still_plan_inside_the_batch(driver, seed):
    """Offsets that decrease somewhere (the device check rejects them, but the
    copies are issued before its verdict) still give a finite plan whose byte
    ranges, record ranges and clipped ends all stay inside the batch."""
    rng = np.random.default_rng(700 + seed)
    n = 500
    off = synth.csr(rng.integers(1, 400, size=n))
    bad = rng.choice(np.arange(1, n), size=20, replace=False)
    off[bad] = rng.integers(off[0], off[-1], size=bad.size)  # out of order
    lo, hi = int(off[0]), int(off[-1])
    chunk_max, chunks = plan(driver, off, 4096, 31, 1, True)
    assert chunks and chunks[-1]["ce"] == hi
    assert len(chunks) <= (hi - (lo & ~31)) // 32 + 1
    for c in chunks:
        assert lo & ~31 <= c["cs"] < c["ce"] <= hi
        assert lo <= c["data_lo"] <= c["data_hi"] <= hi
        assert c["data_hi"] - c["cs"] <= chunk_max + 31
        if not c["empty"]:
            assert 0 <= c["r0"] < c["r1"] <= n
            assert c["data_lo"] <= c["first"] <= c["data_hi"] and c["data_lo"] <= c["last"] <= c["data_hi"]
