// Exhaustive check of the stream-K partition used by the tensor-core prefill
// GEMM (weight_only_quantized_i4g_gb300/csrc/streamk.h) against brute force:
// ranges tile [0, U) exactly, owner() names the block holding each unit, the
// contributor interval of every tile is the set of blocks touching it, and no
// two partial segments (a tile's K range shared by several blocks) share a
// partial slot, and every contributor after a tile's first uses slot 2c.
// Prints "ok <cases>" or the first failure.
#include <cstdio>
#include <set>
#include <utility>
#include <vector>

#include "../weight_only_quantized_i4g_gb300/csrc/streamk.h"

using namespace qg::sk;

static int fail(const char *what, long T, long Kt, long P) {
    std::printf("FAIL %s T=%ld Kt=%ld P=%ld\n", what, T, Kt, P);
    return 1;
}

int main() {
    long cases = 0;
    for (long T = 1; T <= 40; ++T)
        for (long Kt = 1; Kt <= 40; ++Kt)
            for (long P = 1; P <= 160; ++P) {
                const long U = T * Kt;
                if (P > U) continue;   // the launcher never starts more blocks than units
                ++cases;
                std::vector<long> own(U, -1);
                for (long c = 0; c < P; ++c) {
                    const long b = range_begin(c, U, P), e = range_begin(c + 1, U, P);
                    if (b > e) return fail("range order", T, Kt, P);
                    for (long u = b; u < e; ++u) {
                        if (own[u] != -1) return fail("overlap", T, Kt, P);
                        own[u] = c;
                    }
                }
                if (range_begin(0, U, P) != 0 || range_begin(P, U, P) != U) return fail("ends", T, Kt, P);
                for (long u = 0; u < U; ++u)
                    if (own[u] != owner(u, U, P)) return fail("owner", T, Kt, P);
                std::set<long> used;
                for (long t = 0; t < T; ++t) {
                    std::set<long> blocks;
                    for (long k = 0; k < Kt; ++k) blocks.insert(own[t * Kt + k]);
                    const long cf = first_contributor(t, Kt, U, P), cl = last_contributor(t, Kt, U, P);
                    if (*blocks.begin() != cf || *blocks.rbegin() != cl || (long)blocks.size() != cl - cf + 1)
                        return fail("contributors", T, Kt, P);
                    if (blocks.size() == 1) continue;
                    for (long c : blocks) {
                        const long s = partial_slot(c, t, Kt, U, P);
                        if (s < 2 * c || s > 2 * c + 1) return fail("slot range", T, Kt, P);
                        if (!used.insert(s).second) return fail("slot reuse", T, Kt, P);
                        // The kernel relies on this shortcut for all but the first contributor.
                        if (c > cf && s != 2 * c) return fail("slot shortcut", T, Kt, P);
                    }
                }
            }
    std::printf("ok %ld\n", cases);
    return 0;
}
