// Host build of the prefill's row-gather planner (hs_rowgather.cuh), for the
// CPU tests.  Two modes:
//   selfcheck   random and adversarial union masks; every plan is checked for
//               the invariants the down product relies on (each live neuron
//               listed exactly once, ascending; a group's entries start on an
//               8-entry boundary; an entry takes the slab of gA before
//               8 * split8 and of gB after; at most NG k-steps, else the
//               identity plan).  Prints "ok ..." or aborts.
//   plan        reads "NG m0 m1 ... m(NG-1)" lines (hex masks) from stdin and
//               prints, per line, the k-step count and 1 if the identity plan
//               was taken.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>
#include <vector>

#include "hs_rowgather.cuh"

using namespace rowgather;

#define CHECK(c)                                                        \
    do {                                                                \
        if (!(c)) {                                                     \
            std::fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__); \
            std::exit(1);                                               \
        }                                                               \
    } while (0)

static int plan_or_identity(const uint64_t* mask, int NG, uint32_t* ksd, int* ofs, bool* ident) {
    int n = plan_tile(mask, NG, ksd, ofs);
    *ident = n < 0;
    if (n < 0) n = plan_identity(NG, ksd, ofs);
    return n;
}

static bool check(const uint64_t* mask, int NG) {
    uint32_t ksd[64];
    int ofs[64];
    bool ident = false;
    const int nks = plan_or_identity(mask, NG, ksd, ofs, &ident);
    CHECK(nks >= 0 && nks <= NG);
    std::vector<uint16_t> L(64 * nks, kPad);
    int prev_end = 0;
    for (int g = 0; g < NG; ++g) {
        const int c = ident ? 64 : popc64(mask[g]);
        if (c == 0) {
            CHECK(ofs[g] == -1);
            continue;
        }
        CHECK(ofs[g] % 8 == 0 && ofs[g] >= prev_end);
        prev_end = ofs[g] + ((c + 7) & ~7);
        CHECK(prev_end <= 64 * nks);
        int k = 0;
        for (int i = 0; i < 64; ++i)
            if (ident || ((mask[g] >> i) & 1)) L[ofs[g] + k++] = (uint16_t)(64 * g + i);
    }
    int last = -1, nlive = 0, want = 0;
    for (size_t e = 0; e < L.size(); ++e) {
        if (L[e] == kPad) continue;
        const int n = L[e], g = n / 64;
        CHECK(ident || ((mask[g] >> (n % 64)) & 1));
        CHECK(n > last);
        last = n;
        ++nlive;
        const uint32_t d = ksd[e / 64];
        const int pos = (int)(e % 64), s8 = ksd_split8(d);
        CHECK(s8 >= 0 && s8 <= 8);
        CHECK(g == (pos < 8 * s8 ? ksd_gA(d) : ksd_gB(d)));
        if (ksd_gA(d) == ksd_gB(d)) CHECK(s8 == 8);
    }
    for (int g = 0; g < NG; ++g) want += ident ? 64 : popc64(mask[g]);
    CHECK(nlive == want);
    return ident;
}

static int selfcheck() {
    std::mt19937_64 rng(1);
    int fallbacks = 0, plans = 0;
    for (int NG : {1, 2, 3, 29, 58, 64}) {
        std::vector<uint64_t> m(NG);
        for (auto& v : m) v = 0;
        CHECK(!check(m.data(), NG));
        for (auto& v : m) v = ~0ull;
        CHECK(!check(m.data(), NG));
        for (int k : {1, 8, 9, 31, 33, 57}) {
            for (int g = 0; g < NG; ++g) m[g] = ((1ull << k) - 1) << (g % (65 - k));
            fallbacks += check(m.data(), NG);
        }
        for (int g = 0; g < NG; ++g) m[g] = (g % 2) ? 0xFFull : ~0ull;
        fallbacks += check(m.data(), NG);
        for (int g = 0; g < NG; ++g) m[g] = (g % 3 == 0) ? ~0ull : (g % 3 == 1 ? 0x1ull : 0x3FFull);
        fallbacks += check(m.data(), NG);
        for (double q : {0.02, 0.1, 0.3, 0.5, 0.7, 0.9, 0.99}) {
            std::bernoulli_distribution bern(q);
            for (int it = 0; it < 300; ++it) {
                for (int g = 0; g < NG; ++g) {
                    uint64_t v = 0;
                    for (int i = 0; i < 64; ++i) v |= (uint64_t)bern(rng) << i;
                    m[g] = v;
                }
                fallbacks += check(m.data(), NG);
                ++plans;
            }
        }
    }
    std::printf("ok %d plans, %d identity fallbacks\n", plans, fallbacks);
    return 0;
}

static int plan_stdin() {
    int NG;
    while (std::scanf("%d", &NG) == 1) {
        CHECK(NG >= 1 && NG <= 64);
        uint64_t m[64];
        for (int g = 0; g < NG; ++g) {
            unsigned long long v;
            CHECK(std::scanf("%llx", &v) == 1);
            m[g] = v;
        }
        uint32_t ksd[64];
        int ofs[64];
        bool ident = false;
        const int n = plan_or_identity(m, NG, ksd, ofs, &ident);
        std::printf("%d %d\n", n, ident ? 1 : 0);
    }
    return 0;
}

int main(int argc, char** argv) {
    if (argc > 1 && std::strcmp(argv[1], "plan") == 0) return plan_stdin();
    return selfcheck();
}
