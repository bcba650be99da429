// sbf_fastx.cu -- FASTA/FASTQ input ("cuSBF", Sec. IV-A: streamed FASTA/FASTQ
// input with transparent gzip decompression; Sec. IV-F: sequence-native
// records).  Host code only.
//
// A reader turns a file into CSR batches of whole records: the bases of each
// record (sequence lines joined, line breaks dropped, every other byte kept as
// is -- bytes outside ACGTacgt are invalid k-mer symbols downstream) and the
// record offsets.  FASTA records start with '>'; FASTQ records with '@', their
// sequence lines run until the '+' line and are followed by as many quality
// characters as bases.  With zlib available the file is read through gzread,
// which decompresses gzip (including concatenated members) and passes plain
// files through; without it gzip input is rejected.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "sbf_internal.h"

#ifdef SBF_WITH_ZLIB
#include <zlib.h>
#endif

struct sbf_fastx {
#ifdef SBF_WITH_ZLIB
    gzFile gz = nullptr;
#else
    FILE *fp = nullptr;
#endif
    std::vector<char> buf;  // raw input buffer
    size_t pos = 0, len = 0;
    bool eof = false;
    int format = 0;         // 0 unknown, 1 FASTA, 2 FASTQ
    std::string pending;    // bases of a record that did not fit the caller's buffer
    bool has_pending = false;
    int64_t line = 0;
};

namespace {

bool refill(sbf_fastx *r) {
    if (r->eof) return false;
#ifdef SBF_WITH_ZLIB
    const int got = gzread(r->gz, r->buf.data(), (unsigned)r->buf.size());
    if (got < 0) {
        r->eof = true;
        return false;
    }
    r->len = (size_t)got;
#else
    r->len = fread(r->buf.data(), 1, r->buf.size(), r->fp);
#endif
    r->pos = 0;
    if (r->len == 0) r->eof = true;
    return r->len > 0;
}

// Next line without its terminator ('\n', optional '\r'); false at end of input.
bool next_line(sbf_fastx *r, std::string &out) {
    out.clear();
    bool any = false;
    for (;;) {
        if (r->pos >= r->len && !refill(r)) {
            if (any) ++r->line;
            return any;
        }
        const char *start = r->buf.data() + r->pos;
        const char *nl = static_cast<const char *>(memchr(start, '\n', r->len - r->pos));
        if (nl) {
            out.append(start, nl - start);
            r->pos += (size_t)(nl - start) + 1;
            if (!out.empty() && out.back() == '\r') out.pop_back();
            ++r->line;
            return true;
        }
        out.append(start, r->len - r->pos);
        r->pos = r->len;
        any = true;
    }
}

// Peek at the next byte without consuming it; -1 at end of input.
int peek(sbf_fastx *r) {
    if (r->pos >= r->len && !refill(r)) return -1;
    return (unsigned char)r->buf[r->pos];
}

// One record's bases into `bases`; 1 = record, 0 = end of input, < 0 = error.
int read_record(sbf_fastx *r, std::string &bases) {
    bases.clear();
    std::string line;
    // skip blank lines before the header
    int c;
    while ((c = peek(r)) == '\n' || c == '\r') next_line(r, line);
    if (c < 0) return 0;
    if (!next_line(r, line)) return 0;
    if (r->format == 0) r->format = line[0] == '@' ? 2 : 1;
    if (r->format == 1) {
        if (line[0] != '>')
            return sbf::set_error(SBF_ERR_INVALID_ARG, "FASTA line %lld: expected '>'", (long long)r->line);
        while ((c = peek(r)) >= 0 && c != '>') {
            next_line(r, line);
            bases += line;
        }
        return 1;
    }
    if (line[0] != '@')
        return sbf::set_error(SBF_ERR_INVALID_ARG, "FASTQ line %lld: expected '@'", (long long)r->line);
    for (;;) {
        if (!next_line(r, line))
            return sbf::set_error(SBF_ERR_INVALID_ARG, "FASTQ: record without a '+' line");
        if (!line.empty() && line[0] == '+') break;
        bases += line;
    }
    size_t qual = 0;
    while (qual < bases.size()) {
        if (!next_line(r, line))
            return sbf::set_error(SBF_ERR_INVALID_ARG, "FASTQ: quality shorter than the sequence");
        qual += line.size();
    }
    if (qual != bases.size())
        return sbf::set_error(SBF_ERR_INVALID_ARG, "FASTQ line %lld: quality length differs from the sequence",
                              (long long)r->line);
    return 1;
}

}  // namespace

extern "C" {

sbf_fastx *sbf_fastx_open(const char *path) {
    if (!path) {
        sbf::set_error(SBF_ERR_INVALID_ARG, "sbf_fastx_open: NULL path");
        return nullptr;
    }
    auto *r = new sbf_fastx;
    r->buf.resize(1 << 20);
#ifdef SBF_WITH_ZLIB
    r->gz = gzopen(path, "rb");
    if (!r->gz) {
        sbf::set_error(SBF_ERR_INVALID_ARG, "cannot open %s", path);
        delete r;
        return nullptr;
    }
    gzbuffer(r->gz, 1 << 20);
#else
    r->fp = fopen(path, "rb");
    if (!r->fp) {
        sbf::set_error(SBF_ERR_INVALID_ARG, "cannot open %s", path);
        delete r;
        return nullptr;
    }
    unsigned char magic[2] = {0, 0};
    if (fread(magic, 1, 2, r->fp) == 2 && magic[0] == 0x1f && magic[1] == 0x8b) {
        sbf::set_error(SBF_ERR_INVALID_ARG, "%s is gzip-compressed but libsbf was built without zlib", path);
        fclose(r->fp);
        delete r;
        return nullptr;
    }
    rewind(r->fp);
#endif
    return r;
}

void sbf_fastx_close(sbf_fastx *r) {
    if (!r) return;
#ifdef SBF_WITH_ZLIB
    if (r->gz) gzclose(r->gz);
#else
    if (r->fp) fclose(r->fp);
#endif
    delete r;
}

int sbf_fastx_has_gzip(void) {
#ifdef SBF_WITH_ZLIB
    return 1;
#else
    return 0;
#endif
}

int64_t sbf_fastx_pending_bases(const sbf_fastx *r) {
    return r && r->has_pending ? (int64_t)r->pending.size() : 0;
}

int64_t sbf_fastx_next(sbf_fastx *r, char *seq, int64_t seq_cap, int64_t *offsets, int64_t max_records,
                       int64_t *bases_out) {
    if (!r || !seq || !offsets || seq_cap < 0 || max_records < 1)
        return sbf::set_error(SBF_ERR_INVALID_ARG, "sbf_fastx_next: bad arguments");
    int64_t n = 0, used = 0;
    offsets[0] = 0;
    std::string rec;
    while (n < max_records) {
        if (r->has_pending) {
            rec.swap(r->pending);
            r->has_pending = false;
        } else {
            const int rc = read_record(r, rec);
            if (rc < 0) return rc;
            if (rc == 0) break;
        }
        if (used + (int64_t)rec.size() > seq_cap) {
            // keep the record for the next call (with a larger buffer if it is alone)
            r->pending.swap(rec);
            r->has_pending = true;
            if (n == 0)
                return sbf::set_error(SBF_ERR_INVALID_ARG, "a %lld-base record does not fit %lld bytes",
                                      (long long)r->pending.size(), (long long)seq_cap);
            break;
        }
        memcpy(seq + used, rec.data(), rec.size());
        used += (int64_t)rec.size();
        offsets[++n] = used;
    }
    if (bases_out) *bases_out = used;
    return n;
}

// Insert every record of a FASTA/FASTQ file, in batches of about batch_bases.
int sbf_insert_fastx(sbf_filter *f, const char *path, int64_t batch_bases, int64_t *records, int64_t *bases) {
    if (!f) return sbf::set_error(SBF_ERR_INVALID_ARG, "NULL filter");
    sbf_fastx *r = sbf_fastx_open(path);
    if (!r) return SBF_ERR_INVALID_ARG;
    if (batch_bases <= 0) batch_bases = int64_t(1) << 28;
    std::vector<char> seq((size_t)batch_bases);
    std::vector<int64_t> off((size_t)(batch_bases / 2 + 2));
    int64_t nrec = 0, nbase = 0;
    int rc = SBF_OK;
    for (;;) {
        int64_t got_bases = 0;
        int64_t n = sbf_fastx_next(r, seq.data(), (int64_t)seq.size(), off.data(), (int64_t)off.size() - 1,
                                   &got_bases);
        if (n < 0 && r->has_pending) {  // one record larger than the batch: grow and retry
            seq.resize(r->pending.size());
            continue;
        }
        if (n < 0) {
            rc = (int)n;
            break;
        }
        if (n == 0) break;
        rc = sbf_insert_host(f, seq.data(), off.data(), n, nullptr);
        if (rc != SBF_OK) break;
        nrec += n;
        nbase += got_bases;
    }
    sbf_fastx_close(r);
    if (records) *records = nrec;
    if (bases) *bases = nbase;
    return rc;
}

// Query every record of a FASTA/FASTQ file; for each batch, `sink` receives the
// batch's bases, offsets and answer bits (sbf_query's layout, batch-relative
// positions).  A non-zero return from sink stops the scan and is returned.
int sbf_query_fastx(const sbf_filter *f, const char *path, int64_t batch_bases, sbf_fastx_sink sink, void *user) {
    if (!f || !sink) return sbf::set_error(SBF_ERR_INVALID_ARG, "sbf_query_fastx: bad arguments");
    sbf_fastx *r = sbf_fastx_open(path);
    if (!r) return SBF_ERR_INVALID_ARG;
    if (batch_bases <= 0) batch_bases = int64_t(1) << 28;
    std::vector<char> seq((size_t)batch_bases);
    std::vector<int64_t> off((size_t)(batch_bases / 2 + 2));
    std::vector<uint32_t> bits;
    int rc = SBF_OK;
    for (;;) {
        int64_t got_bases = 0;
        int64_t n = sbf_fastx_next(r, seq.data(), (int64_t)seq.size(), off.data(), (int64_t)off.size() - 1,
                                   &got_bases);
        if (n < 0 && r->has_pending) {
            seq.resize(r->pending.size());
            continue;
        }
        if (n < 0) {
            rc = (int)n;
            break;
        }
        if (n == 0) break;
        bits.assign((size_t)((got_bases + 31) / 32 + 1), 0u);
        rc = sbf_query_host(f, seq.data(), off.data(), n, bits.data(), nullptr);
        if (rc != SBF_OK) break;
        rc = sink(user, seq.data(), off.data(), n, bits.data());
        if (rc != 0) break;
    }
    sbf_fastx_close(r);
    return rc;
}

}  // extern "C"
