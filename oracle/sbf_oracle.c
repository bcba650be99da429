/*
 * sbf_oracle.c -- plain, slow CPU oracle for Super Bloom filter (SBF)
 * insert and query over raw DNA, protein and DNA-triplet sequences.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA path.
 *
 * Every k-mer is recomputed from scratch: its validity, its w = k-m+1 m-mer
 * hashes, its minimum, its k-s+1 s-mer hashes and their bits.  Nothing is
 * rolled, cached or merged into runs.  The optional worker threads only split
 * the list of k-mer positions; OR is commutative, so the filter image does not
 * depend on the split.
 *
 * Source: "cuSBF: A Minimizer-Aware Bloom Filter for Genomic Sequence Data on
 * Modern GPUs" (Dortmann, Vieth, Schmidt, arXiv 2606.24417):
 *   - Sec. II-B1 (minimizers, w = k-m+1 m-mers per k-mer),
 *   - Sec. II-B2 / Eq. 2 (Findere: all k-s+1 s-mers set or tested),
 *   - Sec. IV-B (2^P shards of four 64-bit words; hash index i -> word i mod 4),
 *   - Sec. IV-C (2-bit DNA packing, shift-and-OR),
 *   - Sec. IV-D / Algorithm 1 (insert: minimum m-mer hash selects the shard),
 *   - Sec. IV-E / Algorithm 2 (query: a k-mer is present iff every bit is set;
 *     an invalid k-mer answers false),
 *   - Sec. IV-F (a k-mer holding an invalid symbol is filtered out),
 *   - Sec. IV-G (bit-slicing of the s-mer hash; role-specialised hashing:
 *     one multiplicative mix for m-mers, a stronger mix with an extra
 *     xorshift for s-mers).
 *
 * Readings where the paper leaves a step open (each one is listed in the
 * design notes):
 *   - code map A/a=0, C/c=1, G/g=2, T/t=3; every other byte is invalid;
 *   - protein symbols are the 26 letters, either case, A/a=0 .. Z/z=25;
 *     every other byte is invalid;
 *   - a DNA-triplet symbol is three consecutive bases read in frame from the
 *     start of its record, code 16*c0 + 4*c1 + c2 (the three 2-bit codes,
 *     first base most significant); a codon holding an invalid base is
 *     invalid, and the 1 or 2 bytes after a record's last whole codon start
 *     no symbol.  A triplet k-mer therefore starts only at record-relative
 *     byte offsets divisible by 3 and covers 3k bytes; its answer goes to the
 *     bit of its first byte, the other bits are 0;
 *   - a t-mer packs with its first symbol most significant (Sec. IV-E's
 *     "left-shift, OR in the trailing symbol"), b bits per symbol;
 *   - hash constants: C1 = floor(2^64 / golden ratio), C2 = floor((sqrt2-1)
 *     * 2^64) | 1; minimizer hash hm(x) = t ^ (t >> 32) with
 *     t = (x ^ seed) * C1; s-mer hash hs(x): t = (x ^ ~seed) * C1,
 *     t ^= t >> 32, t *= C2, t ^= t >> 29 (all mod 2^64);
 *   - bit position of hash i: slice width W = floor(64/H), position =
 *     (hs >> (i*W)) & 63, in word i mod 4, while W >= 6 (H <= 10); for
 *     11 <= H <= 32, position = top 6 bits of hs * salt(i) mod 2^64, salt(i)
 *     = SplitMix64 output i from state 0 (golden-ratio increment), made odd;
 *   - optional hash-chosen sectors (sectors = 1, an extension, not the
 *     paper's layout): for H < 4, where "i mod 4" leaves words H..3 of every
 *     shard empty, hash i goes to word (hs >> (i*W + 6)) & 3 -- the two bits
 *     of slice i just above its position bits (W >= 21 there); H >= 4 keeps
 *     word i mod 4;
 *   - records are given as CSR offsets; a k-mer never spans two records;
 *   - the minimum's tie-break is the leftmost window (it cannot change the
 *     result: hm is a bijection, equal hashes mean equal m-mers).
 *
 * Parity pins: see tests/test_oracle_pins.py (brute force, closed forms,
 * the figures' worked examples, Eq. 1 / Eq. 2 false-positive rates and the
 * 2/(w+1) minimizer density).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define ORC_C1 0x9E3779B97F4A7C15ULL /* floor(2^64 / phi) */
#define ORC_C2 0x6A09E667F3BCC909ULL /* floor((sqrt(2)-1) * 2^64) | 1 */

uint64_t orc_const_c1(void) { return ORC_C1; }
uint64_t orc_const_c2(void) { return ORC_C2; }

/* Sec. IV-C: 2-bit DNA alphabet; -1 marks an invalid symbol (Sec. IV-F). */
int orc_base_code(uint8_t c)
{
    switch (c) {
    case 'A': case 'a': return 0;
    case 'C': case 'c': return 1;
    case 'G': case 'g': return 2;
    case 'T': case 't': return 3;
    default: return -1;
    }
}

/* Packed value of the t bases at p, first base most significant:
 * sum_i code(p[i]) * 4^(t-1-i).  The caller guarantees validity. */
uint64_t orc_pack(const uint8_t *p, int t)
{
    uint64_t v = 0;
    for (int i = 0; i < t; i++)
        v = v * 4u + (uint64_t)orc_base_code(p[i]);
    return v;
}

/* Sec. IV-A alphabets: bits per symbol and input bytes per symbol. */
enum { ORC_DNA = 0, ORC_PROTEIN = 1, ORC_TRIPLET = 2 };

int orc_symbol_bits(int alphabet)
{
    return alphabet == ORC_PROTEIN ? 5 : alphabet == ORC_TRIPLET ? 6 : 2;
}

int orc_symbol_bytes(int alphabet)
{
    return alphabet == ORC_TRIPLET ? 3 : 1;
}

/* Code of the symbol whose first byte is p, or -1 when it is invalid. */
int orc_symbol_code(int alphabet, const uint8_t *p)
{
    if (alphabet == ORC_PROTEIN) {
        if (p[0] >= 'A' && p[0] <= 'Z')
            return p[0] - 'A';
        if (p[0] >= 'a' && p[0] <= 'z')
            return p[0] - 'a';
        return -1;
    }
    if (alphabet == ORC_TRIPLET) {
        int c0 = orc_base_code(p[0]), c1 = orc_base_code(p[1]), c2 = orc_base_code(p[2]);
        if (c0 < 0 || c1 < 0 || c2 < 0)
            return -1;
        return c0 * 16 + c1 * 4 + c2;
    }
    return orc_base_code(p[0]);
}

/* Packed value of the t symbols starting at p (symbol i at byte
 * i * bytes-per-symbol), first symbol most significant:
 * sum_i code_i * 2^(b*(t-1-i)).  The caller guarantees validity. */
uint64_t orc_pack_symbols(int alphabet, const uint8_t *p, int t)
{
    const int b = orc_symbol_bits(alphabet), B = orc_symbol_bytes(alphabet);
    uint64_t v = 0;
    for (int i = 0; i < t; i++)
        v = (v << b) | (uint64_t)orc_symbol_code(alphabet, p + (size_t)i * B);
    return v;
}

/* Sec. IV-G, minimizer role: one multiplicative mix (plus an xor-fold so that
 * the low bits, which pick the shard, depend on every base). */
uint64_t orc_hash_m(uint64_t x, uint64_t seed_m)
{
    uint64_t t = (x ^ seed_m) * ORC_C1;
    return t ^ (t >> 32);
}

/* Sec. IV-G, s-mer role: a stronger mix with an additional xorshift. */
uint64_t orc_hash_s(uint64_t x, uint64_t seed_s)
{
    uint64_t t = (x ^ seed_s) * ORC_C1;
    t ^= t >> 32;
    t *= ORC_C2;
    t ^= t >> 29;
    return t;
}

/* Salt of hash index i for the large-H fallback: output i of the SplitMix64
 * generator started at state 0 (its state advances by the golden-ratio
 * constant C1), made odd. */
uint64_t orc_salt(int i)
{
    uint64_t z = (uint64_t)(i + 1) * ORC_C1;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z | 1u;
}

/* Sec. IV-B + IV-G: the H bits of one s-mer hash, hash i in word i mod 4.
 * Bit-slicing while a slice is at least 6 bits wide (64/H >= 6): the position
 * is the low 6 bits of slice i (slice width floor(64/H)).  For larger H the
 * paper multiplies by a per-index golden-ratio-derived salt and keeps the
 * upper bits: position = top 6 bits of hs * salt(i) mod 2^64.
 * sectors = 1 (hash-chosen sectors, H < 4 only): hash i's word is the two
 * bits of slice i above its six position bits instead of i mod 4. */
void orc_smer_bits_sectors(uint64_t hs, int H, int sectors, uint64_t words[4])
{
    int W = 64 / H;
    for (int i = 0; i < H; i++) {
        int pos;
        if (W >= 6)
            pos = (int)((hs >> (i * W)) & 63u);
        else
            pos = (int)((hs * orc_salt(i)) >> 58);
        int word = i % 4;
        if (sectors && H < 4)
            word = (int)((hs >> (i * W + 6)) & 3u);
        words[word] |= (uint64_t)1 << pos;
    }
}

void orc_smer_bits(uint64_t hs, int H, uint64_t words[4])
{
    orc_smer_bits_sectors(hs, H, 0, words);
}

typedef struct {
    int k, m, s, H;
    uint64_t num_shards; /* a power of two */
    uint64_t seed;
    int alphabet;
    int sectors;         /* 0: hash i in word i mod 4; 1: hash-chosen words for H < 4 */
} orc_params;

/* One k-mer, from scratch.  seq is the whole concatenated buffer, g an
 * absolute position, [rec_start, rec_end) the byte range of g's record.
 * Returns 1 and fills shard/K when the k-mer is valid: it starts on a symbol
 * boundary of its record, its k symbols lie inside the record and all are
 * valid (Sec. IV-F). */
static int kmer_info(const uint8_t *seq, int64_t g, int64_t rec_start, int64_t rec_end,
                     const orc_params *P, uint64_t *shard, uint64_t K[4])
{
    const int k = P->k, m = P->m, s = P->s, A = P->alphabet;
    const int B = orc_symbol_bytes(A);
    if ((g - rec_start) % B != 0 || g + (int64_t)B * k > rec_end)
        return 0;
    for (int i = 0; i < k; i++)
        if (orc_symbol_code(A, seq + g + (int64_t)B * i) < 0)
            return 0;
    /* Algorithm 1: the minimizer is the minimum hash over the k-m+1 m-mer
     * windows ... */
    uint64_t mu = UINT64_MAX;
    for (int i = 0; i <= k - m; i++) {
        uint64_t h = orc_hash_m(orc_pack_symbols(A, seq + g + (int64_t)B * i, m), P->seed);
        if (h < mu)
            mu = h;
    }
    /* ... its low bits select the shard (minHash & (NumShards - 1)) ... */
    *shard = mu & (P->num_shards - 1);
    /* ... and the bits of all k-s+1 s-mers are OR-ed into four word masks. */
    K[0] = K[1] = K[2] = K[3] = 0;
    for (int j = 0; j <= k - s; j++)
        orc_smer_bits_sectors(orc_hash_s(orc_pack_symbols(A, seq + g + (int64_t)B * j, s), ~P->seed), P->H,
                              P->sectors, K);
    return 1;
}

/* First record r with offsets[r+1] > g (records may be empty). */
static int64_t record_of(const int64_t *off, int64_t n, int64_t g)
{
    int64_t lo = 0, hi = n - 1;
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (off[mid + 1] > g)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

typedef struct {
    const uint8_t *seq;
    const int64_t *off;
    int64_t n;
    orc_params P;
    uint64_t *filter;  /* num_shards * 4 words */
    uint32_t *out;     /* query output bits, absolute positions */
    int64_t g0, g1;    /* this worker's position range */
    int atomic;
} job;

static void *insert_worker(void *arg)
{
    job *J = (job *)arg;
    if (J->g0 >= J->g1)
        return NULL;
    int64_t r = record_of(J->off, J->n, J->g0);
    for (int64_t g = J->g0; g < J->g1; g++) {
        while (J->off[r + 1] <= g)
            r++;
        uint64_t shard, K[4];
        if (!kmer_info(J->seq, g, J->off[r], J->off[r + 1], &J->P, &shard, K))
            continue;
        for (int w = 0; w < 4; w++) {
            if (!K[w])
                continue;
            if (J->atomic)
                __atomic_fetch_or(&J->filter[shard * 4 + w], K[w], __ATOMIC_RELAXED);
            else
                J->filter[shard * 4 + w] |= K[w];
        }
    }
    return NULL;
}

static void *query_worker(void *arg)
{
    job *J = (job *)arg;
    if (J->g0 >= J->g1)
        return NULL;
    int64_t r = record_of(J->off, J->n, J->g0);
    for (int64_t g = J->g0; g < J->g1; g++) {
        while (J->off[r + 1] <= g)
            r++;
        uint64_t shard, K[4];
        int present = 0;
        if (kmer_info(J->seq, g, J->off[r], J->off[r + 1], &J->P, &shard, K)) {
            /* Algorithm 2: present iff every required bit is set. */
            present = 1;
            for (int w = 0; w < 4; w++)
                if (K[w] & ~J->filter[shard * 4 + w])
                    present = 0;
        }
        if (present)
            J->out[g >> 5] |= (uint32_t)1 << (g & 31);
    }
    return NULL;
}

static int valid_params(const orc_params *P)
{
    if (P->alphabet < ORC_DNA || P->alphabet > ORC_TRIPLET)
        return 0;
    /* Sec. IV-C: a k-mer packs into one 64-bit word. */
    if (P->k < 1 || P->k * orc_symbol_bits(P->alphabet) > 64 || P->m < 1 || P->m > P->k ||
        P->s < 1 || P->s > P->k)
        return 0;
    if (P->H < 1 || P->H > 32 || P->sectors < 0 || P->sectors > 1)
        return 0;
    if (P->num_shards == 0 || (P->num_shards & (P->num_shards - 1)))
        return 0;
    return 1;
}

/* Split [g0, g1) into nthreads ranges whose inner cut points are multiples
 * of 32, so that query workers never share an output word. */
static int run_jobs(void *(*fn)(void *), job *base, int nthreads)
{
    int64_t g0 = base->g0, g1 = base->g1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if (nthreads == 1) {
        base->atomic = 0;
        fn(base);
        return 0;
    }
    job jobs[256];
    pthread_t th[256];
    int64_t span = g1 - g0;
    int64_t prev = g0;
    for (int t = 0; t < nthreads; t++) {
        int64_t cut = (t == nthreads - 1) ? g1 : g0 + span * (t + 1) / nthreads;
        if (t != nthreads - 1) {
            cut &= ~(int64_t)31;
            if (cut < prev)
                cut = prev;
        }
        jobs[t] = *base;
        jobs[t].g0 = prev;
        jobs[t].g1 = cut;
        jobs[t].atomic = 1;
        prev = cut;
    }
    int started = 0;
    for (int t = 0; t < nthreads; t++) {
        if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0)
            break;
        started++;
    }
    for (int t = started; t < nthreads; t++)
        fn(&jobs[t]);
    for (int t = 0; t < started; t++)
        pthread_join(th[t], NULL);
    return 0;
}

static int check_offsets(const int64_t *off, int64_t n)
{
    if (n < 0)
        return 0;
    for (int64_t r = 0; r < n; r++)
        if (off[r + 1] < off[r])
            return 0;
    return off[0] >= 0;
}

/* Insert every valid k-mer of every record.  filter: num_shards*4 u64,
 * caller-zeroed or holding an earlier image.  Returns 0, or -1 on bad
 * arguments. */
int orc_insert(uint64_t *filter, const uint8_t *seq, const int64_t *off, int64_t n,
               int k, int m, int s, int H, uint64_t num_shards, uint64_t seed, int alphabet, int sectors,
               int nthreads)
{
    orc_params P = {k, m, s, H, num_shards, seed, alphabet, sectors};
    if (!valid_params(&P) || !check_offsets(off, n))
        return -1;
    if (n == 0)
        return 0;
    job J = {seq, off, n, P, filter, NULL, off[0], off[n], 0};
    return run_jobs(insert_worker, &J, nthreads);
}

/* Query every position of [off[0], off[n]).  out: u32 words covering
 * [off[0]>>5, (off[n]+31)>>5); the words are zeroed here and bit g is set iff
 * the k-mer at absolute position g is valid and present. */
int orc_query(const uint64_t *filter, const uint8_t *seq, const int64_t *off, int64_t n,
              int k, int m, int s, int H, uint64_t num_shards, uint64_t seed, int alphabet, int sectors,
              uint32_t *out, int nthreads)
{
    orc_params P = {k, m, s, H, num_shards, seed, alphabet, sectors};
    if (!valid_params(&P) || !check_offsets(off, n))
        return -1;
    if (n == 0)
        return 0;
    for (int64_t w = off[0] >> 5; w < (off[n] + 31) >> 5; w++)
        out[w] = 0;
    job J = {seq, off, n, P, (uint64_t *)filter, out, off[0], off[n], 0};
    return run_jobs(query_worker, &J, nthreads);
}

/* The k-mer at absolute position g (one record lookup, then from scratch).
 * Returns 1 if valid (shard and K filled), 0 if not, -1 on bad arguments. */
int orc_kmer_info(const uint8_t *seq, const int64_t *off, int64_t n, int64_t g,
                  int k, int m, int s, int H, uint64_t num_shards, uint64_t seed, int alphabet, int sectors,
                  uint64_t *shard, uint64_t K[4])
{
    orc_params P = {k, m, s, H, num_shards, seed, alphabet, sectors};
    if (!valid_params(&P) || n <= 0 || g < off[0] || g >= off[n])
        return -1;
    int64_t r = record_of(off, n, g);
    return kmer_info(seq, g, off[r], off[r + 1], &P, shard, K);
}

/* Fig. 3 structure: counts valid k-mers and runs, a run being a maximal
 * stretch of consecutive valid k-mers of one record with one shard
 * (consecutive: one symbol apart).  The
 * paper's insert issues one atomicOr per non-zero word per run; *atomics
 * receives that count.  Single-threaded, from scratch per k-mer. */
int orc_count_runs(const uint8_t *seq, const int64_t *off, int64_t n,
                   int k, int m, int s, int H, uint64_t num_shards, uint64_t seed, int alphabet, int sectors,
                   int64_t *valid_kmers, int64_t *runs, int64_t *atomics)
{
    orc_params P = {k, m, s, H, num_shards, seed, alphabet, sectors};
    if (!valid_params(&P) || !check_offsets(off, n))
        return -1;
    int64_t nv = 0, nr = 0, na = 0;
    for (int64_t r = 0; r < n; r++) {
        int have = 0;
        uint64_t cur = 0, acc[4] = {0, 0, 0, 0};
        /* consecutive k-mers of a record are one symbol apart */
        for (int64_t g = off[r]; g < off[r + 1]; g += orc_symbol_bytes(alphabet)) {
            uint64_t shard, K[4];
            int v = kmer_info(seq, g, off[r], off[r + 1], &P, &shard, K);
            if (v && have && shard == cur) {
                for (int w = 0; w < 4; w++)
                    acc[w] |= K[w];
            } else {
                if (have)
                    for (int w = 0; w < 4; w++)
                        na += acc[w] != 0;
                have = v;
                if (v) {
                    nr++;
                    cur = shard;
                    for (int w = 0; w < 4; w++)
                        acc[w] = K[w];
                }
            }
            nv += v;
        }
        if (have)
            for (int w = 0; w < 4; w++)
                na += acc[w] != 0;
    }
    *valid_kmers = nv;
    *runs = nr;
    *atomics = na;
    return 0;
}

/* Per-position evaluation for sampled checks on inputs too large for a full
 * oracle pass: for each absolute position pos[i] (any order), valid[i],
 * shard[i] and K[4i..4i+3] as kmer_info computes them.  Positions outside
 * [off[0], off[n]) are reported invalid.  Returns 0, or -1 on bad
 * arguments. */
int orc_kmer_batch(const uint8_t *seq, const int64_t *off, int64_t n,
                   const int64_t *pos, int64_t count,
                   int k, int m, int s, int H, uint64_t num_shards, uint64_t seed, int alphabet, int sectors,
                   uint8_t *valid, uint64_t *shard, uint64_t *K)
{
    orc_params P = {k, m, s, H, num_shards, seed, alphabet, sectors};
    if (!valid_params(&P) || n <= 0)
        return -1;
    for (int64_t i = 0; i < count; i++) {
        int64_t g = pos[i];
        valid[i] = 0;
        shard[i] = 0;
        K[4 * i] = K[4 * i + 1] = K[4 * i + 2] = K[4 * i + 3] = 0;
        if (g < off[0] || g >= off[n])
            continue;
        int64_t r = record_of(off, n, g);
        valid[i] = (uint8_t)kmer_info(seq, g, off[r], off[r + 1], &P, &shard[i], &K[4 * i]);
    }
    return 0;
}

/* Every valid k-mer as (shard, K) rows, in position order, for building a
 * sparse image.  rows must hold one entry per k-mer position; *count
 * receives the number of valid k-mers written. */
int orc_kmer_rows(const uint8_t *seq, const int64_t *off, int64_t n,
                  int k, int m, int s, int H, uint64_t num_shards, uint64_t seed, int alphabet, int sectors,
                  uint64_t *shard, uint64_t *K, int64_t *count)
{
    orc_params P = {k, m, s, H, num_shards, seed, alphabet, sectors};
    if (!valid_params(&P) || !check_offsets(off, n))
        return -1;
    int64_t c = 0;
    for (int64_t r = 0; r < n; r++)
        for (int64_t g = off[r]; g < off[r + 1]; g++)
            if (kmer_info(seq, g, off[r], off[r + 1], &P, &shard[c], &K[4 * c]))
                c++;
    *count = c;
    return 0;
}
