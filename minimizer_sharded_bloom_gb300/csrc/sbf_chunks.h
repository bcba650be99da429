// sbf_chunks.h -- how a staged host-facing call cuts its CSR batch into chunks.
//
// Pure host arithmetic (no CUDA), shared by sbf_host.cu and a CPU test driver.
// A chunk answers the k-mers that start in positions [cs, ce): cs and ce are
// multiples of 32 (answer-word boundaries) except ce at the batch's end.
//   - Where a record starts on a 32-position boundary within the last
//     kEdgeSearch records before the nominal end, the chunk ends there: its
//     records are whole and no bytes overlap the next chunk.
//   - Otherwise it ends at the nominal position and ships kb - 1 bytes more
//     (kb = bytes of one k-mer); its last record is clipped at data_hi, so the
//     k-mers that start at or after ce fall off its end and belong to the next
//     chunk.
// A record cut at a chunk's start begins, in that chunk, at its next symbol
// boundary (sb bytes per symbol), which keeps the codon frame of DNA triplets.
// The chunk's offsets are the caller's offsets[r0 .. r1] with the two ends
// replaced by `first` and `last`.
#pragma once

#include <algorithm>
#include <cstdint>

namespace sbf {

// First record r with offsets[r + 1] > g (n >= 1).
inline int64_t record_at(const int64_t *off, int64_t n, int64_t g) {
    int64_t lo = 0, hi = n - 1;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (off[mid + 1] > g) hi = mid; else lo = mid + 1;
    }
    return lo;
}

// Records searched back from a nominal chunk end for one that starts on an
// answer-word boundary.
constexpr int kEdgeSearch = 64;

struct Chunk {
    int64_t cs = 0, ce = 0;            // k-mer starts answered: [cs, ce)
    int64_t data_lo = 0, data_hi = 0;  // bytes shipped: [data_lo, data_hi)
    int64_t r0 = 0, r1 = 0;            // records r0 .. r1 - 1 (offsets r0 .. r1)
    int64_t first = 0, last = 0;       // the chunk's offsets[r0] and offsets[r1]
    bool whole = false;                // first == offsets[r0] and last == offsets[r1]
    bool empty = false;                // no record (only with offsets the check rejects)
    bool final = false;                // ce is the batch's end
};

// Walks a batch of n >= 1 records with offsets[n] > offsets[0] >= 0.
// Chunks start at 2^22 positions and double, up to an eighth of the batch and
// at most host_chunk: the first copy, which no kernel overlaps, stays short.
// A query's chunks also shrink towards the end (at most half of what is
// left), so that its last kernel, which no copy overlaps, is short too.
class ChunkPlan {
  public:
    ChunkPlan(const int64_t *off, int64_t n, int64_t host_chunk, int64_t kb, int sb, bool query)
        : off_(off), n_(n), lo_(off[0]), hi_(off[n]), kb_(kb), sb_(sb), query_(query) {
        chunk_max_ = std::min<int64_t>(
            host_chunk, std::max<int64_t>(((hi_ - lo_) / 8 + 31) & ~int64_t(31), int64_t(1) << 22));
        chunk_ = std::min<int64_t>(chunk_max_, int64_t(1) << 22);
        cs_ = lo_ & ~int64_t(31);
    }

    // the largest chunk, for sizing buffers once: at most this + kb bytes
    int64_t chunk_max() const { return chunk_max_; }

    // The next chunk; false when the batch is done.
    bool next(Chunk &c) {
        if (cs_ >= hi_) return false;
        c = Chunk();
        c.cs = cs_;
        c.data_lo = std::max<int64_t>(cs_, lo_);
        const int64_t cur =
            query_ ? std::min<int64_t>(chunk_, std::max<int64_t>(((hi_ - cs_) / 2 + 31) & ~int64_t(31),
                                                                 std::min<int64_t>(chunk_, int64_t(1) << 22)))
                   : chunk_;
        c.ce = std::min<int64_t>(cs_ + cur, hi_);
        c.data_hi = hi_;
        if (c.ce < hi_) {
            int64_t P = -1;
            int64_t r = record_at(off_, n_, c.ce);
            for (int t = 0; t < kEdgeSearch && r > 0; ++t, --r) {
                const int64_t p = off_[r];
                if (p <= c.data_lo) break;
                if (p <= c.ce && (p & 31) == 0) {
                    P = p;
                    break;
                }
            }
            if (P > 0) c.ce = c.data_hi = P;
            else c.data_hi = std::min<int64_t>(c.ce + kb_ - 1, hi_);
        }
        c.final = c.ce >= hi_;
        cs_ = c.ce;
        chunk_ = std::min<int64_t>(2 * chunk_, chunk_max_);
        c.r0 = record_at(off_, n_, c.data_lo);
        c.r1 = record_at(off_, n_, c.data_hi - 1) + 1;
        if (c.r1 <= c.r0) {
            c.empty = true;
            return true;
        }
        auto clip = [&](int64_t v) { return std::min<int64_t>(std::max<int64_t>(v, c.data_lo), c.data_hi); };
        c.last = clip(off_[c.r1]);
        const int64_t next = c.r1 - c.r0 >= 2 ? clip(off_[c.r0 + 1]) : c.last;
        int64_t first = off_[c.r0] < c.data_lo ? c.data_lo + (sb_ - (c.data_lo - off_[c.r0]) % sb_) % sb_
                                               : off_[c.r0];
        c.first = std::min<int64_t>(clip(first), next);
        c.whole = c.first == off_[c.r0] && c.last == off_[c.r1];
        return true;
    }

  private:
    const int64_t *off_;
    int64_t n_, lo_, hi_, kb_;
    int sb_;
    bool query_;
    int64_t chunk_max_ = 0, chunk_ = 0, cs_ = 0;
};

}  // namespace sbf
