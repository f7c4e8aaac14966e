// Host-side checks of the split-schedule planner (fa2_split_ranges.h), built and
// run by tests/test_split_ranges.py.  For a sweep of (units, n_kv, grid) it checks
// that the ranges tile [0, I) in order, that none costs more than the reported
// bound T, that T is the smallest bound any cut into at most G ranges can meet,
// and it prints the whole-vs-split decision for a few named shapes.
#include <cstdio>
#include <vector>

#include "fa2_split_ranges.h"

using namespace fa2;

// Smallest makespan over all cuts of [0, I) into at most G ranges, by dynamic
// programming over range ends (small I only).
static long long brute_force(long long units, long long n_kv, int G)
{
    const long long I = units * n_kv;
    const long long INF = 1ll << 60;
    auto cost = [&](long long a, long long b) { return (b - a) + SEGMENT_COST * ((b - 1) / n_kv - a / n_kv + 1); };
    std::vector<long long> best(I + 1, INF), next(I + 1, INF);
    best[0] = 0;
    long long answer = INF;
    for (int g = 1; g <= G; ++g) {
        for (long long b = 0; b <= I; ++b)
            next[b] = INF;
        for (long long a = 0; a < I; ++a) {
            if (best[a] == INF)
                continue;
            for (long long b = a + 1; b <= I; ++b) {
                const long long c = best[a] > cost(a, b) ? best[a] : cost(a, b);
                if (c < next[b])
                    next[b] = c;
            }
        }
        if (next[I] < answer)
            answer = next[I];
        best.swap(next);
    }
    return answer;
}

int main()
{
    int failures = 0, cases = 0;
    for (long long units = 1; units <= 40; units += 3)
        for (long long n_kv = 1; n_kv <= 33; n_kv += 4)
            for (int sms : {1, 2, 5, 16, 152}) {
                const int G = static_cast<int>(split_grid(units, n_kv, sms));
                int begin[MAX_SPLIT_CTAS + 1];
                long long T = 0;
                const int k = cut_ranges(units, n_kv, G, begin, &T);
                const long long I = units * n_kv;
                bool ok = k >= 1 && k <= G && begin[0] == 0 && begin[k] == I;
                for (int i = 0; ok && i < k; ++i) {
                    const long long a = begin[i], b = begin[i + 1];
                    ok = b > a && (b - a) + SEGMENT_COST * ((b - 1) / n_kv - a / n_kv + 1) <= T;
                }
                if (ok && I <= 400)
                    ok = T == brute_force(units, n_kv, G);
                ++cases;
                if (!ok) {
                    ++failures;
                    std::printf("FAIL units=%lld n_kv=%lld sms=%d G=%d k=%d T=%lld\n", units, n_kv, sms, G, k, T);
                }
            }
    std::printf("checked %d cases, %d failures\n", cases, failures);
    // whole-vs-split decisions on 152 SMs (units, n_kv of the five workloads' tilings)
    struct Named { const char *name; long long units, n_kv; } named[] = {
        {"c2", 256, 8}, {"c3", 512, 32}, {"c4", 2048, 128}, {"c5", 256, 47}, {"one_long_head", 4, 32}};
    for (const Named &n : named)
        std::printf("pays %s %d\n", n.name, split_pays(n.units, n.n_kv, 152) ? 1 : 0);
    return failures == 0 ? 0 : 1;
}
