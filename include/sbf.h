/*
 * sbf.h -- C ABI of libsbf, a GB300 (sm_103a) Super Bloom filter for raw DNA
 * (and, through sbf_create_alphabet, protein and DNA-triplet sequences).
 *
 * The method is the one of "cuSBF: A Minimizer-Aware Bloom Filter for Genomic
 * Sequence Data on Modern GPUs" (Dortmann, Vieth, Schmidt):
 *   - Sec. II-B1: each k-mer's minimizer -- the m-mer of minimum hash among
 *     its w = k-m+1 windows -- selects one 256-bit shard;
 *   - Sec. II-B2, Eq. 2 (Findere): inside that shard all k-s+1 overlapping
 *     s-mers of the k-mer set (insert) or test (query) H bits each;
 *   - Sec. IV-B: the filter is 2^P shards of four 64-bit words, hash index i
 *     addresses word i mod 4;
 *   - Sec. IV-G: bit i of an s-mer is slice i of its 64-bit hash.
 *
 * Fixed readings of points the paper leaves open (the CPU oracle and the CUDA
 * kernels follow the same ones):
 *   - bases: A/a=0, C/c=1, G/g=2, T/t=3; any other byte is invalid and a k-mer
 *     containing one is skipped on insert and answers 0 on query (Sec. IV-F);
 *   - a t-mer packs with its first base most significant;
 *   - C1 = 0x9E3779B97F4A7C15 (floor(2^64/phi)), C2 = 0x6A09E667F3BCC909
 *     (floor((sqrt2-1)*2^64) | 1); minimizer hash t = (x ^ seed) * C1,
 *     hm = t ^ (t >> 32); s-mer hash t = (x ^ ~seed) * C1, t ^= t >> 32,
 *     t *= C2, t ^= t >> 29 (all mod 2^64); shard = min hm & (num_shards-1);
 *   - hash i of an s-mer sets, in word i mod 4, bit ((hs >> (i * floor(64/H)))
 *     & 63) while floor(64/H) >= 6 (H <= 10), else bit (hs * salt(i)) >> 58
 *     with salt(i) = SplitMix64 output i from state 0, made odd;
 *   - records are CSR slices of one buffer; a k-mer never spans two records;
 *   - forward strand only.
 *
 * Threading and streams.  Device-facing calls (sbf_insert, sbf_query,
 * sbf_copy_bits, sbf_load_bits, sbf_clear) only enqueue work on the given
 * stream (a cudaStream_t passed as void*; NULL = the legacy default stream)
 * and return without synchronizing, as the paper's device-facing entry points
 * do (Sec. IV-A).  Host-facing calls (sbf_insert_host, sbf_query_host)
 * return after their work is complete.  A filter may be used from one host
 * thread at a time; calls that modify a filter must be ordered by the caller
 * with respect to every other call on it.  The filter lives on the device that
 * was current at sbf_create; callers must make that device current.
 *
 * Errors.  Functions returning int return SBF_OK (0) or a negative
 * sbf_status; sbf_create returns NULL on error.  The message of the calling
 * thread's last error is available from sbf_last_error().  Argument errors are
 * found on the host before anything is enqueued.  Malformed offsets (not
 * nondecreasing, or offsets[0] < 0) can only be seen on the device: a check
 * kernel then sets the filter's sticky status, the insert/query kernels of
 * that call and of every later call skip all work (query output is then left
 * unwritten), and sbf_get_status() reports SBF_ERR_BAD_OFFSETS and clears it.
 * No kernel traps or asserts, and there is no CPU fallback: without a usable
 * CUDA device every compute call fails with SBF_ERR_CUDA.
 */
#ifndef SBF_H
#define SBF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sbf_filter sbf_filter; /* opaque; owns the device bit array */

typedef enum {
    SBF_OK = 0,
    SBF_ERR_INVALID_ARG = -1, /* a NULL pointer, an out-of-range parameter or size */
    SBF_ERR_CUDA = -2,        /* a CUDA runtime call or kernel launch failed */
    SBF_ERR_OOM = -3,         /* device memory for the filter could not be allocated */
    SBF_ERR_BAD_OFFSETS = -4  /* reported by sbf_get_status: malformed CSR offsets */
} sbf_status;

/* Create an all-zero filter of at least num_bits bits on the current device.
 * Shard count = ceil(num_bits / 256) rounded up to a power of two (Sec. IV-B);
 * the device array holds num_shards * 32 bytes.
 * Requires num_bits >= 1, num_shards <= 2^40, 1 <= m <= k <= 32,
 * 1 <= s <= k and 1 <= H <= 32 (H > 10 uses the salted multiply, Sec. IV-G).
 * seed selects the hash functions (minimizer seed = seed, s-mer seed = ~seed).
 * Returns NULL on error (SBF_ERR_INVALID_ARG / _OOM / _CUDA in sbf_last_error). */
sbf_filter *sbf_create(uint64_t num_bits, int k, int m, int s, int H, uint64_t seed);

/* Sec. IV-A alphabet encodings. */
#define SBF_ALPHABET_DNA 0         /* 4 symbols, 2 bits: A/a C/c G/g T/t = 0..3; k <= 32 */
#define SBF_ALPHABET_PROTEIN 1     /* 26 symbols, 5 bits: letters A..Z, either case = 0..25; k <= 12 */
#define SBF_ALPHABET_DNA_TRIPLET 2 /* 64 symbols, 6 bits: codons, 3 bytes each; k <= 10 */

/* sbf_create for any of the three alphabets of Sec. IV-A (sbf_create is this
 * call with SBF_ALPHABET_DNA).  A k-mer packs into one 64-bit word (Sec.
 * IV-C), so k * bits-per-symbol <= 64: k <= 32 (DNA), 12 (protein), 10
 * (triplet); 1 <= m <= k, 1 <= s <= k, 1 <= H <= 32 as for sbf_create.
 *   - Protein: any byte other than a letter is an invalid symbol.
 *   - DNA triplet: a symbol is a codon of three bases read in frame from the
 *     start of its record, code 16*c0 + 4*c1 + c2 (2-bit base codes, first
 *     base most significant); a codon holding an invalid base is invalid; the
 *     1 or 2 bytes after a record's last whole codon start no symbol.
 * The packed value of a t-mer is sum_i code_i * 2^(b*(t-1-i)), b the symbol
 * width; hashing, sharding and bit addressing are those of sbf_create.  Insert
 * and query keep their contracts with "position" meaning a byte of the
 * concatenated input: the k-mer starting at a symbol's first byte g answers at
 * bit g, and (triplets) bits of other bytes are 0.  Protein (12, 8, 10, 4) and
 * triplet (10, 5, 8, 4) have compile-time specialised kernels
 * (sbf_is_specialized returns 1); every other valid (k, m, s, H) runs the
 * runtime-parameter alphabet kernel with the same results.
 * Returns NULL on error, like sbf_create. */
sbf_filter *sbf_create_alphabet(uint64_t num_bits, int k, int m, int s, int H, uint64_t seed, int alphabet);

/* Creation flags of sbf_create_ex. */
#define SBF_FLAG_HASHED_SECTORS 1  /* hash-chosen sectors for H < 4 (see sbf_create_ex) */
#define SBF_FLAG_RUNTIME_KERNELS 2 /* always the runtime-parameter kernels (see sbf_create_ex) */

/* sbf_create_alphabet with creation flags (sbf_create_alphabet is this call
 * with flags = 0).  SBF_FLAG_HASHED_SECTORS is an extension of the paper's
 * layout (Sec. IV-B, Algorithm 2: hash i of an s-mer sets a bit in word
 * i mod 4 of the shard), which leaves words H..3 of every shard empty when
 * H < 4.  With the flag and H < 4, hash i sets its bit in the word given by
 * the two bits of its slice just above its six position bits:
 * (hs >> (i * floor(64/H) + 6)) & 3 (slices are >= 21 bits wide there), so a
 * k-mer's bits spread over all 256 bits of its shard; the position is
 * unchanged.  Such a filter runs on the runtime-parameter kernels (the
 * compile-time specialisations keep the paper's layout), so
 * sbf_is_specialized returns 0.  For H >= 4 the flag has no effect.  SBF_FLAG_RUNTIME_KERNELS
 * runs every call on the runtime-parameter kernels even where a compile-time
 * specialisation of (k, m, s, H) exists (same results, slower; for comparing
 * parameter points on one kernel family, or the two families on one point);
 * sbf_is_specialized then returns 0.  Any other flag bit is
 * SBF_ERR_INVALID_ARG.  Returns NULL on error, like sbf_create. */
sbf_filter *sbf_create_ex(uint64_t num_bits, int k, int m, int s, int H, uint64_t seed, int alphabet, int flags);

/* The creation flags of f (SBF_FLAG_*), or -1 for NULL. */
int sbf_get_flags(const sbf_filter *f);

/* The filter's alphabet (SBF_ALPHABET_*), or -1 for NULL. */
int sbf_get_alphabet(const sbf_filter *f);

/* Free the device memory of f after the device finished all work (this call
 * synchronizes the device).  NULL-safe. */
void sbf_destroy(sbf_filter *f);

/* Insert (Algorithm 1; Sec. IV-D).  seq: device pointer to bytes; offsets:
 * device pointer to n+1 int64, nondecreasing; record r is
 * seq[offsets[r] .. offsets[r+1]), so seq must be readable on
 * [offsets[0], offsets[n]).  Every valid k-mer of every record is ORed into
 * the filter; the result does not depend on record order or on how records
 * are split across calls.  n == 0 is a no-op.  Caller keeps ownership of
 * seq/offsets and must keep them alive until the stream reaches this work.
 * Asynchronous on `stream`. */
int sbf_insert(sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n, void *stream);

/* Query (Algorithm 2; Sec. IV-E).  Same seq/offsets contract as sbf_insert.
 * out_bits: device pointer to uint32 words, at least ceil(offsets[n] / 32) of
 * them (absolute indexing).  Bit g (word g >> 5, bit g & 31, LSB first) answers
 * the k-mer that starts at absolute position g: 1 iff it is valid (inside one
 * record, all k bases valid) and every bit of all its k-s+1 s-mers is set in
 * its shard.  Every word in [offsets[0] >> 5, (offsets[n] + 31) >> 5) is
 * written (positions without a valid k-mer get 0); other words are untouched.
 * Asynchronous on `stream`.  Where the filter has a dense-batch kernel (the
 * operating point k=31 m=16 s=28 H=4), a batch whose records all have one
 * length R with k <= R <= 160 and offsets[0] == 0 runs as sbf_query_dense
 * would run it, with identical answers; the call then takes one 4-byte
 * stream-ordered allocation from a memory pool of the filter's own (kept
 * between calls) for the device-side uniformity flag, and frees it on
 * `stream`.  Concurrent queries of one filter on several streams are safe. */
int sbf_query(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
              uint32_t *out_bits, void *stream);

/* Host-facing insert: seq and offsets are HOST pointers (pageable or
 * pinned), same layout as sbf_insert.  Returns when the filter holds every
 * k-mer; the work is ordered after earlier work on `stream` (may be NULL).
 * A page-locked sequence is staged (below).  A pageable one is read in place
 * when the device can access it -- pageable-memory access through the host
 * page tables (Grace systems over NVLink-C2C) -- with no copies.  Otherwise
 * (or after sbf_set_host_mode(f, 1)) the records are staged to the device in
 * chunks on eight rotating streams, overlapping copies with kernels (Sec. IV-G,
 * host FASTX staging): page-locked buffers are copied from directly, pageable
 * ones through pinned staging buffers.  Chunks end at record starts where possible; a record
 * longer than a chunk is cut, with the k-1 bytes of overlap its k-mers need.
 * The offsets are checked once before any chunk runs: on the device where it
 * can read them, else on the host. */
int sbf_insert_host(sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                    void *stream);

/* Host-facing query: seq/offsets/out_bits are HOST pointers, same layout and
 * output contract as sbf_query.  Returns when out_bits is complete.  Reads and
 * writes the host buffers in place or stages them, as sbf_insert_host.
 * Staged answers are written straight into out_bits where the device can
 * write it.  With
 * malformed offsets (SBF_ERR_BAD_OFFSETS) no answer word is written, except
 * when out_bits is pageable memory the device cannot access: the staged
 * chunks' words may then hold anything. */
int sbf_query_host(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                   uint32_t *out_bits, void *stream);

/* Host-facing query that allocates nothing (the paper has no counterpart).
 * For callers that cannot allocate device memory at call time -- code running
 * under an allocator that owns the whole device (a framework's caching
 * allocator, a fixed memory budget), or loops that cannot accept the implicit
 * device synchronisation of cudaMalloc/cudaFree.  Same inputs, outputs and
 * results as sbf_query_host (HOST seq/offsets/out_bits, same layout), but the
 * batch is staged through one fixed device array that the library holds on
 * every device that loads it until the process exits (about 26 MiB).
 * Limits: offsets[n] - offsets[0] <= 2^24 positions and n <= 2^20 records;
 * larger batches fail with SBF_ERR_INVALID_ARG and nothing is copied.  Calls
 * no cudaMalloc/cudaFree or any other allocating routine.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.
 * All calls share the array: calls whose work overlaps on the GPU (e.g. on two
 * streams) race.  Work is ordered on `stream`; returns when out_bits is
 * complete.  Like sbf_query_host it ends by reading and clearing the filter's
 * sticky status: if that status was set (this batch's offsets, or an earlier
 * device call's not yet reported with sbf_get_status), the kernel skipped its
 * work, the call returns SBF_ERR_BAD_OFFSETS (or SBF_ERR_CUDA after a device
 * wait gave up), and the words copied to out_bits are not answers. */
int sbf_query_host_noalloc(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                           uint32_t *out_bits, void *stream);

/* Host-facing access mode: 0 (default) stages a page-locked sequence (the copy
 * engine moves it over the host link faster than kernel loads) and reads a
 * pageable one in place when the device can, else stages it; 1 always stages;
 * 2 reads in place whenever the device can. */
int sbf_set_host_mode(sbf_filter *f, int mode);

/* Largest chunk of the staged host-facing calls, in sequence positions (default 2^25;
 * rounded down to a multiple of 32; at least 32).  A call cuts its batch into
 * chunks of up to about an eighth of it, at least 2^22 positions and at most this
 * setting; the first chunks are smaller (from 2^22 positions, doubling).
 * Smaller chunks overlap copies and kernels at a finer grain and need smaller
 * staging buffers. */
int sbf_set_host_chunk(sbf_filter *f, int64_t positions);

/* ---- FASTA / FASTQ input (Sec. IV-A: streamed FASTA/FASTQ with transparent
 * gzip; Sec. IV-F: sequence-native records).  Host code; no GPU needed to read.
 * A record's bases are its sequence lines joined without line breaks; every
 * byte is kept as is (bytes outside ACGTacgt are invalid k-mer symbols).
 * FASTA records start with '>', FASTQ records with '@' (sequence lines up to
 * the '+' line, then as many quality characters as bases). */
typedef struct sbf_fastx sbf_fastx; /* an open reader */

/* Open a plain or gzip-compressed FASTA/FASTQ file (gzip needs a libsbf built
 * with zlib; see sbf_fastx_has_gzip).  NULL on error (sbf_last_error). */
sbf_fastx *sbf_fastx_open(const char *path);

/* Next batch of whole records: bases into seq (seq_cap bytes), CSR offsets into
 * offsets (room for max_records + 1 entries, offsets[0] = 0).  Returns the
 * number of records (0 at end of input) and *bases_out the bytes used, or a
 * negative sbf_status.  A record that does not fit is kept for the next call;
 * if it does not fit an empty buffer the call fails with SBF_ERR_INVALID_ARG
 * and sbf_fastx_pending_bases() gives the size needed. */
int64_t sbf_fastx_next(sbf_fastx *r, char *seq, int64_t seq_cap, int64_t *offsets, int64_t max_records,
                       int64_t *bases_out);

/* Bases of the record kept back by sbf_fastx_next (0 if none). */
int64_t sbf_fastx_pending_bases(const sbf_fastx *r);

void sbf_fastx_close(sbf_fastx *r); /* NULL-safe */

/* 1 if the library was compiled with zlib and reads gzip input, else 0. */
int sbf_fastx_has_gzip(void);

/* Insert every record of a FASTA/FASTQ file through sbf_insert_host, in
 * batches of about batch_bases bases (<= 0: 2^28).  *records / *bases (may be
 * NULL) receive the totals.  Returns when done. */
int sbf_insert_fastx(sbf_filter *f, const char *path, int64_t batch_bases, int64_t *records, int64_t *bases);

/* Called once per batch by sbf_query_fastx with the batch's bases, offsets
 * (n + 1 entries, batch-relative) and answer bits (sbf_query's layout, bit g
 * for batch position g).  A non-zero return stops the scan. */
typedef int (*sbf_fastx_sink)(void *user, const char *seq, const int64_t *offsets, int64_t n,
                              const uint32_t *out_bits);

/* Query every record of a FASTA/FASTQ file through sbf_query_host, in batches
 * of about batch_bases bases, handing each batch's answers to sink.  Returns
 * SBF_OK, a negative sbf_status, or sink's non-zero value. */
int sbf_query_fastx(const sbf_filter *f, const char *path, int64_t batch_bases, sbf_fastx_sink sink,
                    void *user);

/* Copy the raw image (num_shards * 32 bytes: shard-major, four little-endian
 * uint64 words per shard, bit b of word j = (word >> b) & 1) to dst, host or
 * device memory (cudaMemcpyDefault).  dst_bytes must be >= the image size.
 * Asynchronous on `stream` (for pageable host dst the copy is synchronous). */
int sbf_copy_bits(const sbf_filter *f, void *dst, uint64_t dst_bytes, void *stream);

/* Replace the image with src (same layout and size as sbf_copy_bits; host or
 * device memory).  Saves a filter together with sbf_copy_bits.  Async. */
int sbf_load_bits(sbf_filter *f, const void *src, uint64_t src_bytes, void *stream);

/* Query a dense record batch (Sec. IV-A's "dense record batches"): n_records
 * records of record_len bytes each, back to back, record r = seq[r*record_len,
 * (r+1)*record_len); seq is a device pointer to n_records*record_len bytes and
 * no offsets array is read.  The answers are those of sbf_query with offsets
 * r*record_len, in the same layout: out_bits (device, at least
 * ceil(n_records*record_len / 32) words) gets bit g for the k-mer starting at
 * byte g, every word in [0, ceil(n_records*record_len / 32)) is written.
 * DNA filters only.  For record_len <= 160 and a filter at k=31, m=16, s=28,
 * H=4 with at most 2^31 shards the query runs one strip per record, which
 * skips the k-1 positions at each record's end that start no k-mer; otherwise
 * it runs the runtime-parameter kernel.  Asynchronous on `stream`; no offsets
 * check is needed, so the sticky status is not involved. */
int sbf_query_dense(const sbf_filter *f, const char *seq, int64_t n_records, int64_t record_len,
                    uint32_t *out_bits, void *stream);

/* Zero the image (an empty filter).  Asynchronous on `stream`. */
int sbf_clear(sbf_filter *f, void *stream);

/* Number of 256-bit shards (a power of two); 0 for NULL. */
uint64_t sbf_num_shards(const sbf_filter *f);

/* The filter's parameters; any output pointer may be NULL. */
int sbf_get_params(const sbf_filter *f, int *k, int *m, int *s, int *H, uint64_t *seed);

/* 1 if insert/query of f run a kernel specialised at compile time for its
 * (k, m, s, H), 0 if they run the runtime-parameter kernel (same results). */
int sbf_is_specialized(const sbf_filter *f);

/* Failure-detection test hook (the paper has no counterpart).  Launches the
 * filter's insert kernel once so that one thread waits on an mbarrier that
 * nothing completes (no copy attached), giving up after `polls` polls
 * (>= 1); the kernel then sets the filter's sticky timeout status and
 * returns.  The next sbf_get_status reports SBF_ERR_CUDA ("a bounded device
 * wait timed out") and clears the status; the filter is unchanged.  Every
 * other launch uses the kernels' normal bound (about 2^22 polls).  Async on
 * `stream`.  SBF_ERR_INVALID_ARG when polls < 1 or the filter's kernels are
 * not the strip kernels (the only ones with bounded waits). */
int sbf_test_wait_timeout(sbf_filter *f, int polls, void *stream);

/* Synchronize `stream`, then return and clear the sticky device status:
 * SBF_OK, SBF_ERR_BAD_OFFSETS, or SBF_ERR_CUDA if the stream reported an
 * error. */
int sbf_get_status(sbf_filter *f, void *stream);

/* Message of the calling thread's last error ("" if none). */
const char *sbf_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SBF_H */
