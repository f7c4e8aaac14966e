// fa2_split_ranges.h -- host-side planning of the split schedule (plain C++, no
// CUDA): how the K/V-tile iterations of a non-causal pass are cut into one range
// per CTA, and whether that beats dealing out whole work units.
#pragma once

#include <climits>

namespace fa2 {

// Largest grid of the split schedule (one CTA per SM at most).
constexpr int MAX_SPLIT_CTAS = 256;

// Cost model of the split schedule, in K/V-tile times.  Every segment a CTA works
// on (a whole unit or a cut part of one) costs SEGMENT_COST on top of its tiles:
// its epilogue, the wait for the next unit's first S and, for cut parts, writing or
// merging the part (on GB300 a boundary costs two to three tile times, and four fit
// the measured finishing times best).  Cutting units also costs MERGE_COST once.
#ifndef FA2_SEGMENT_COST
#define FA2_SEGMENT_COST 4
#endif
constexpr long long SEGMENT_COST = FA2_SEGMENT_COST;
constexpr long long MERGE_COST = 2;

// End of the range that starts at iteration a and costs at most T, in an iteration
// space of I tiles cut into units of n_kv; a when not even one tile fits.
inline long long range_end(long long a, long long T, long long I, long long n_kv)
{
    long long rem = T - SEGMENT_COST;   // the first segment's own cost
    if (rem <= 0 || a >= I)
        return a;
    long long len = n_kv - a % n_kv;
    if (len > I - a)
        len = I - a;
    if (len >= rem)
        return a + rem;
    long long b = a + len;
    rem -= len;
    while (b < I && rem > SEGMENT_COST) {
        len = n_kv < I - b ? n_kv : I - b;
        const long long take = len < rem - SEGMENT_COST ? len : rem - SEGMENT_COST;
        b += take;
        rem -= SEGMENT_COST + take;
        if (take < len)
            break;
    }
    return b;
}

// Number of ranges of cost <= T that cover [0, I) greedily (limit + 1 if more).
inline int count_ranges(long long T, long long I, long long n_kv, int limit)
{
    long long a = 0;
    int k = 0;
    while (a < I) {
        const long long b = range_end(a, T, I, n_kv);
        if (b == a || ++k > limit)
            return limit + 1;
        a = b;
    }
    return k;
}

// Cut the I = n_units * n_kv tile iterations into at most G ranges whose largest cost
// (tiles + SEGMENT_COST per segment) is as small as possible.  Writes the range starts
// to begin[0..k] (begin[k] = I) when begin is given; returns the number of ranges k
// and the largest cost in *T_out.
inline int cut_ranges(long long n_units, long long n_kv, int G, int *begin, long long *T_out)
{
    const long long I = n_units * n_kv;
    const long long L = (I + G - 1) / G;
    long long lo = L + SEGMENT_COST;
    long long hi = L + SEGMENT_COST * (L / n_kv + 2) + 1;
    while (count_ranges(hi, I, n_kv, G) > G)   // not expected; widen until feasible
        hi *= 2;
    while (lo < hi) {
        const long long mid = (lo + hi) / 2;
        if (count_ranges(mid, I, n_kv, G) <= G)
            hi = mid;
        else
            lo = mid + 1;
    }
    long long a = 0;
    int k = 0;
    while (a < I) {
        if (begin)
            begin[k] = static_cast<int>(a);
        a = range_end(a, lo, I, n_kv);
        ++k;
    }
    if (begin)
        begin[k] = static_cast<int>(I);
    if (T_out)
        *T_out = lo;
    return k;
}

// Grid bound of the split schedule: one CTA per SM, at most one per K/V-tile iteration.
inline long long split_grid(long long n_units, long long n_kv, int num_sms)
{
    const long long iters = n_units * n_kv;
    long long g = iters < num_sms ? iters : num_sms;
    return g < MAX_SPLIT_CTAS ? g : MAX_SPLIT_CTAS;
}

// Whether the cost-balanced ranges beat dealing out whole units by at least 5 %:
// whole units finish after ceil(units / SMs) segments of n_kv tiles; the ranges
// after the balanced cost plus the merge.
// (T: the largest range cost cut_ranges found for split_grid(units, n_kv, num_sms) CTAs.)
inline bool split_pays_given(long long units, long long n_kv, int num_sms, long long T)
{
    const long long whole = (units + num_sms - 1) / num_sms * (n_kv + SEGMENT_COST);
    return (T + MERGE_COST) * 100 < whole * 95;
}

inline bool split_pays(long long units, long long n_kv, int num_sms)
{
    if (units * n_kv > INT_MAX)
        return false;
    long long T = 0;
    cut_ranges(units, n_kv, static_cast<int>(split_grid(units, n_kv, num_sms)), nullptr, &T);
    return split_pays_given(units, n_kv, num_sms, T);
}

}  // namespace fa2
