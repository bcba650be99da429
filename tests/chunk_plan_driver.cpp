// Test driver: runs the host-facing calls' chunk planner (sbf_chunks.h) over
// a CSR batch read from stdin and prints every chunk, for tests/test_chunk_plan.py.
//
// stdin:  n host_chunk kb sb query
//         offsets[0] .. offsets[n]
// stdout: chunk_max
//         one line per chunk: cs ce data_lo data_hi r0 r1 first last whole empty final
#include <cstdint>
#include <cstdio>
#include <vector>

#include "sbf_chunks.h"

int main() {
    long long n = 0, host_chunk = 0, kb = 0;
    int sb = 0, query = 0;
    if (std::scanf("%lld %lld %lld %d %d", &n, &host_chunk, &kb, &sb, &query) != 5 || n < 1) return 2;
    std::vector<int64_t> off(n + 1);
    for (long long i = 0; i <= n; ++i) {
        long long v = 0;
        if (std::scanf("%lld", &v) != 1) return 2;
        off[i] = v;
    }
    sbf::ChunkPlan plan(off.data(), n, host_chunk, kb, sb, query != 0);
    std::printf("%lld\n", (long long)plan.chunk_max());
    sbf::Chunk c;
    while (plan.next(c)) {
        std::printf("%lld %lld %lld %lld %lld %lld %lld %lld %d %d %d\n", (long long)c.cs, (long long)c.ce,
                    (long long)c.data_lo, (long long)c.data_hi, (long long)c.r0, (long long)c.r1,
                    (long long)c.first, (long long)c.last, c.whole ? 1 : 0, c.empty ? 1 : 0, c.final ? 1 : 0);
    }
    return 0;
}
