// Host-side brute-force check of the stream-K partition arithmetic in
// token_decode_attention_gb300/csrc/streamk.h (compiled and run by
// tests/test_streamk_host.py with g++; no GPU involved).
//
// For random batches (live lengths L_b, head groups NHG) and partition counts
// G it checks that: the ranges tile [0, W) in order and differ by at most one
// position; range_owner(x) is the partition whose range holds x, for every x;
// walking the flattened positions the way the kernels do yields pieces whose
// slots c + u are unique and below G + U; and the first / last owners of each
// unit (what the combine kernel computes) bracket exactly the partitions that
// hold a piece of it.
#include <cstdio>
#include <cstdlib>
#include <random>
#include <set>
#include <vector>

#include "streamk.h"

using dattn::piece_slot;
using dattn::range_begin;
using dattn::range_begin_split;
using dattn::range_owner;

static int fail(const char *what, long long a, long long b) {
    std::fprintf(stderr, "FAIL %s (%lld, %lld)\n", what, a, b);
    return 1;
}

int main() {
    std::mt19937_64 rng(20260001);
    for (int trial = 0; trial < 3000; ++trial) {
        const int B = 1 + static_cast<int>(rng() % 40);
        const int S = 1 + static_cast<int>(rng() % 300);
        const int NHG = 1 + static_cast<int>(rng() % 3);
        std::vector<long long> L(B), Pb(B + 1, 0);
        for (int b = 0; b < B; ++b) {
            L[b] = 1 + static_cast<long long>(rng() % S);
            Pb[b + 1] = Pb[b] + L[b];
        }
        const long long W = NHG * Pb[B];
        const long long U = static_cast<long long>(B) * NHG;
        const long long Gs[] = {1, 2, 3, 7, static_cast<long long>(1 + rng() % 400), W, W + 5};
        for (long long G : Gs) {
            // ranges tile [0, W) and are balanced
            if (range_begin(0, W, G) != 0) return fail("begin(0)", G, W);
            if (range_begin(G, W, G) != W) return fail("begin(G)", G, W);
            for (long long c = 0; c < G; ++c) {
                const long long n = range_begin(c + 1, W, G) - range_begin(c, W, G);
                if (n < W / G || n > W / G + 1) return fail("balance", c, n);
            }
            for (long long c = 0; c <= G; ++c) {
                if (range_begin_split(static_cast<unsigned>(c), W / G,
                                      static_cast<unsigned>(W % G),
                                      static_cast<unsigned>(G)) != range_begin(c, W, G))
                    return fail("split begin", c, G);
            }
            // owner of every position
            for (long long x = 0; x < W; ++x) {
                const long long c = range_owner(x, W, G);
                if (c < 0 || c >= G) return fail("owner range", x, c);
                if (!(range_begin(c, W, G) <= x && x < range_begin(c + 1, W, G)))
                    return fail("owner", x, c);
            }
            // walk the pieces partition by partition, as the kernels do
            std::set<long long> slots;
            std::vector<long long> first(U, -1), last(U, -1);
            std::vector<std::set<long long>> holders(U);
            for (long long c = 0; c < G; ++c) {
                long long x = range_begin(c, W, G);
                const long long x1 = range_begin(c + 1, W, G);
                long long b = 0, base = 0;
                while (x < x1) {
                    while (x >= base + NHG * L[b]) {
                        base += NHG * L[b];
                        ++b;
                    }
                    const long long rel = x - base;
                    const long long g = rel / L[b];
                    const long long off = rel - g * L[b];
                    const long long len = std::min(L[b] - off, x1 - x);
                    const long long u = b * NHG + g;
                    const long long s = piece_slot(c, u);
                    if (s < 0 || s >= G + U) return fail("slot range", c, u);
                    if (!slots.insert(s).second) return fail("slot unique", c, u);
                    if (first[u] < 0) first[u] = c;
                    last[u] = c;
                    holders[u].insert(c);
                    x += len;
                }
            }
            for (int b = 0; b < B; ++b) {
                for (int g = 0; g < NHG; ++g) {
                    const long long u = static_cast<long long>(b) * NHG + g;
                    const long long Pu = NHG * Pb[b] + g * L[b];
                    if (range_owner(Pu, W, G) != first[u]) return fail("first owner", u, G);
                    if (range_owner(Pu + L[b] - 1, W, G) != last[u]) return fail("last owner", u, G);
                    // between its first and last partition, a unit's pieces are held
                    // exactly by the partitions whose range is not empty (the merge
                    // skips the empty ones, which exist only when W < G)
                    for (long long c = first[u]; c <= last[u]; ++c) {
                        const bool empty = range_begin(c + 1, W, G) == range_begin(c, W, G);
                        if (empty == (holders[u].count(c) != 0)) return fail("holders", u, c);
                        if (empty && W >= G) return fail("empty range with W >= G", c, W);
                    }
                }
            }
        }
    }
    // the 32-bit split form at the largest partition counts and big W
    for (int trial = 0; trial < 200000; ++trial) {
        const long long G = 1 + static_cast<long long>(rng() % 65535);
        const long long W = static_cast<long long>(rng() % (1ULL << 40)) + 1;
        const long long c = static_cast<long long>(rng() % (G + 1));
        if (range_begin_split(static_cast<unsigned>(c), W / G, static_cast<unsigned>(W % G),
                              static_cast<unsigned>(G)) != range_begin(c, W, G))
            return fail("split begin (large)", c, G);
    }
    std::printf("streamk partition checks passed\n");
    return 0;
}
