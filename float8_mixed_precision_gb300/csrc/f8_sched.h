// Static tile schedule for one persistent GEMM launch that runs several
// independent problems (a linear's dgrad and wgrad, which both read q(dY);
// the forward GEMMs of linears that share their input X).  Plain integer
// code, usable from host and device.
//
// The problems of a launch fall into two cost classes: every tile of class
// 0 costs c0, every tile of class 1 costs c1 (a model of the tile's run
// time: its K blocks plus a fixed share; the host puts the costlier class
// first).  Within a class the problems' tiles are numbered one after the
// other.  U workers (CTAs, or CTA pairs) share the T0 tiles of class 0 and
// the T1 tiles of class 1.  Class 0 is dealt round-robin: worker u takes
// tiles u, u + U, u + 2U, ...  and is then free at T_u = n0(u) c0.  Class
// 1's tiles are then handed out in order, each to the worker that is free
// first (ties: lower worker index first); a worker is free again c1 after it
// took one.  That is list scheduling of the second class behind the first,
// and it keeps consecutive tiles on concurrently running workers (the raster
// order's L2 reuse).
//
// Nothing is communicated: the free-time events form two arithmetic
// sequences (workers u < T0 mod U start at (q0 + 1) c0, the rest at q0 c0,
// q0 = T0 div U), so worker u ranks its own k-th event among all events in
// closed form.  With T1 = 0 the schedule is plain round-robin.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define F8_SCHED_FN __host__ __device__ __forceinline__
#else
#define F8_SCHED_FN static inline
#endif

namespace f8 {

struct TileSched {
    int units;    // U >= 1
    int tiles0;   // T0 >= 0
    int tiles1;   // T1 >= 0
    int cost0;    // c0 >= 1
    int cost1;    // c1 >= 1
};

// Most problems one launch runs.
constexpr int kMaxLaunchProblems = 4;

// Problem slot of a launch-global tile index g, and g's index within that
// problem: first_tile[i] is the global index of slot i's first tile
// (first_tile[nprob] = the launch's tile count).
F8_SCHED_FN int sched_slot(const int *first_tile, int nprob, int g, int &local)
{
    int slot = 0;
    for (int i = 1; i < kMaxLaunchProblems; ++i)
        slot += (i < nprob && g >= first_tile[i]) ? 1 : 0;
    local = g - first_tile[slot];
    return slot;
}

// events start, start + c, start + 2c, ... that fall strictly before t
F8_SCHED_FN int64_t sched_events_before(int64_t t, int64_t start, int64_t c)
{
    return t > start ? (t - start + c - 1) / c : 0;
}

F8_SCHED_FN bool sched_event_at(int64_t t, int64_t start, int64_t c)
{
    return t >= start && (t - start) % c == 0;
}

// Index, among problem 1's tiles, of worker u's k-th problem-1 tile (may be
// >= tiles1: the worker has no such tile).  Increasing in k.
F8_SCHED_FN int64_t sched_rank1(const TileSched &s, int u, int k)
{
    const int q0 = s.tiles0 / s.units;
    const int r0 = s.tiles0 % s.units;  // workers 0 .. r0-1 hold one more problem-0 tile
    const int64_t th = static_cast<int64_t>(q0 + 1) * s.cost0;
    const int64_t tl = static_cast<int64_t>(q0) * s.cost0;
    const int64_t t = (u < r0 ? th : tl) + static_cast<int64_t>(k) * s.cost1;
    int64_t j = static_cast<int64_t>(r0) * sched_events_before(t, th, s.cost1) +
                static_cast<int64_t>(s.units - r0) * sched_events_before(t, tl, s.cost1);
    if (r0 > 0 && sched_event_at(t, th, s.cost1))
        j += u < r0 ? u : r0;
    if (sched_event_at(t, tl, s.cost1))
        j += u > r0 ? u - r0 : 0;
    return j;
}

// Worker u's i-th tile (i = 0, 1, ...) as a global index: [0, tiles0) are
// problem 0's tiles, [tiles0, tiles0 + tiles1) problem 1's; -1 once the
// worker has no more.
F8_SCHED_FN int sched_tile(const TileSched &s, int u, int i)
{
    const int n0 = u < s.tiles0 ? (s.tiles0 - 1 - u) / s.units + 1 : 0;
    if (i < n0)
        return u + i * s.units;
    const int64_t j = sched_rank1(s, u, i - n0);
    return j < s.tiles1 ? s.tiles0 + static_cast<int>(j) : -1;
}

// Finishing time of the busiest worker under the schedule (host use: the
// launch decides whether two problems share a launch).
static inline int64_t sched_makespan(const TileSched &s)
{
    int64_t worst = 0;
    for (int u = 0; u < s.units; ++u) {
        int64_t t = 0;
        for (int i = 0;; ++i) {
            const int g = sched_tile(s, u, i);
            if (g < 0)
                break;
            t += g < s.tiles0 ? s.cost0 : s.cost1;
        }
        worst = t > worst ? t : worst;
    }
    return worst;
}

// ------------------------------------------------------------ host planning

// Bytes of K per pipeline stage (one K block), as the GEMM kernel stages them.
constexpr int kSchedBlockK = 128;

// Per-tile cost in the schedule, in K blocks: the tile's K blocks plus a
// fixed share for handing over the accumulator and draining it (measured: a
// short-K tile costs about four K blocks more than its MMAs).
constexpr int kSchedTileOverheadKb = 4;

// Smallest gain, in percent of the two launches' predicted time, for which
// two GEMMs share one launch.  Measured: the attention projections'
// backward GEMMs (predicted 6-8%) gain 2-10%; the FFN ones (predicted
// 0-2%, power-capped) lose up to 2% when grouped.
constexpr int kSchedMinGainPct = 4;

// Per-launch cost in the same unit (K blocks): the ramp of a persistent
// launch (pipeline fill, the first tiles' loads) and its drain (the last
// tiles' epilogues).  Measured: the 128 tiles of an 8192 x 1024 x 4096 GEMM
// take 28.8 us alone, two rounds of 36 K blocks, where the 512-tile
// 8192 x 4096 x 4096 GEMM spends 11.4 us a round: about 6 us, 19 K blocks,
// more than its rounds.
constexpr int kSchedLaunchOverheadKb = 16;

// The extents of one GEMM C[M,N] = A[M,K] B[N,K]^T.
struct SchedProblem {
    int64_t M, N, K;
};

// One launch over nprob (1 .. kMaxLaunchProblems) problems in tile_m x bn
// output tiles: the schedule, the caller's problem index of each slot
// (class 0's problems first, each class in the caller's order), and the
// first global tile of each slot.
struct LaunchPlan {
    TileSched s;
    int nprob;
    int nclass0;                          // slots [0, nclass0) are class 0
    int order[kMaxLaunchProblems];
    int first_tile[kMaxLaunchProblems + 1];
    bool ok;                              // false: more than two tile costs
};

static inline int64_t sched_tiles(const SchedProblem &p, int tile_m, int bn)
{
    return ((p.M + tile_m - 1) / tile_m) * ((p.N + bn - 1) / bn);
}

static inline int sched_cost(const SchedProblem &p)
{
    return static_cast<int>((p.K + kSchedBlockK - 1) / kSchedBlockK) + kSchedTileOverheadKb;
}

// The plan of one launch over problems p[idx[0 .. n)] on at most max_units
// workers.  ok = false if their tiles have more than two costs.
static inline LaunchPlan sched_plan_idx(const SchedProblem *p, const int *idx, int n, int tile_m,
                                        int bn, int64_t max_units)
{
    LaunchPlan pl;
    pl.nprob = n;
    pl.nclass0 = 0;
    pl.ok = n >= 1 && n <= kMaxLaunchProblems;
    // the distinct tile costs: at most two
    int c_hi = 0, c_lo = 0;
    for (int i = 0; i < n && pl.ok; ++i) {
        const int c = sched_cost(p[idx[i]]);
        if (c == c_hi || c == c_lo)
            continue;
        if (c_hi == 0)
            c_hi = c;
        else if (c_lo == 0)
            c_lo = c;
        else
            pl.ok = false;
    }
    if (c_lo > c_hi) {
        const int t = c_hi;
        c_hi = c_lo;
        c_lo = t;
    }
    int k = 0;
    int64_t t0 = 0, t1 = 0;
    pl.first_tile[0] = 0;
    for (int pass = 0; pass < 2 && pl.ok; ++pass) {
        for (int i = 0; i < n; ++i) {
            const bool hi = sched_cost(p[idx[i]]) == c_hi;
            if (hi != (pass == 0))
                continue;
            const int64_t t = sched_tiles(p[idx[i]], tile_m, bn);
            pl.order[k] = idx[i];
            pl.first_tile[k + 1] = static_cast<int>(pl.first_tile[k] + t);
            (pass == 0 ? t0 : t1) += t;
            ++k;
        }
        if (pass == 0)
            pl.nclass0 = k;
    }
    const int64_t total = t0 + t1;
    pl.s.units = static_cast<int>(total < max_units ? (total > 0 ? total : 1) : max_units);
    pl.s.tiles0 = static_cast<int>(t0);
    pl.s.tiles1 = static_cast<int>(t1);
    pl.s.cost0 = c_hi > 0 ? c_hi : 1;
    pl.s.cost1 = c_lo > 0 ? c_lo : pl.s.cost0;
    return pl;
}

static inline LaunchPlan sched_plan(const SchedProblem *p, int n, int tile_m, int bn,
                                    int64_t max_units)
{
    int idx[kMaxLaunchProblems];
    for (int i = 0; i < n && i < kMaxLaunchProblems; ++i)
        idx[i] = i;
    return sched_plan_idx(p, idx, n, tile_m, bn, max_units);
}

// Predicted time of a launch: its busiest worker plus the launch's own cost.
static inline int64_t sched_launch_time(const LaunchPlan &pl)
{
    return sched_makespan(pl.s) + kSchedLaunchOverheadKb;
}

// Whether two GEMMs should share one launch: the schedule's predicted
// makespan beats the two launches' by at least kSchedMinGainPct percent.
static inline bool sched_should_group(const SchedProblem &p0, const SchedProblem &p1, int tile_m,
                                      int bn, int64_t max_units)
{
    const SchedProblem both[2] = {p0, p1};
    const int64_t grouped = sched_launch_time(sched_plan(both, 2, tile_m, bn, max_units));
    const int64_t apart = sched_launch_time(sched_plan(&p0, 1, tile_m, bn, max_units)) +
                          sched_launch_time(sched_plan(&p1, 1, tile_m, bn, max_units));
    return grouped * 100 <= apart * (100 - kSchedMinGainPct);
}

// ------------------------------------------------ partition into launches

// Most problems a partition takes (e.g. the dgrad and wgrad GEMMs of four
// linears).
constexpr int kMaxPartitionProblems = 8;

struct Partition {
    int nlaunch;
    int nprob[kMaxPartitionProblems];                   // problems of launch j
    int idx[kMaxPartitionProblems][kMaxLaunchProblems];  // their caller indices
    int64_t predicted;                                  // sum of launch times
};

// Splits n (<= kMaxPartitionProblems) independent GEMMs into launches.
// Problems of equal tile cost form a class (split into chunks of at most
// kMaxLaunchProblems); a launch takes one class chunk or two of different
// costs.  Every pairing of the chunks is tried and the one with the least
// predicted time kept, provided it beats one launch per problem by at least
// kSchedMinGainPct percent; otherwise every problem gets its own launch.
static inline Partition sched_partition(const SchedProblem *p, int n, int tile_m, int bn,
                                        int64_t max_units)
{
    Partition alone;
    alone.nlaunch = n;
    alone.predicted = 0;
    for (int i = 0; i < n; ++i) {
        alone.nprob[i] = 1;
        alone.idx[i][0] = i;
        alone.predicted += sched_launch_time(sched_plan_idx(p, &i, 1, tile_m, bn, max_units));
    }
    if (n <= 1 || n > kMaxPartitionProblems)
        return alone;
    // chunks: problems of one cost, at most kMaxLaunchProblems each
    int nch = 0, ch_n[kMaxPartitionProblems], ch_idx[kMaxPartitionProblems][kMaxLaunchProblems],
        ch_cost[kMaxPartitionProblems];
    bool used[kMaxPartitionProblems] = {};
    for (int i = 0; i < n; ++i) {
        if (used[i])
            continue;
        const int c = sched_cost(p[i]);
        ch_n[nch] = 0;
        ch_cost[nch] = c;
        for (int j = i; j < n; ++j) {
            if (!used[j] && sched_cost(p[j]) == c) {
                if (ch_n[nch] == kMaxLaunchProblems) {
                    ++nch;
                    ch_n[nch] = 0;
                    ch_cost[nch] = c;
                }
                ch_idx[nch][ch_n[nch]++] = j;
                used[j] = true;
            }
        }
        ++nch;
    }
    // every matching of the chunks (a chunk alone, or with one of another
    // cost whose problems fit in the launch), by depth-first search
    Partition best = alone;
    Partition cur;
    cur.nlaunch = 0;
    cur.predicted = 0;
    bool taken[kMaxPartitionProblems] = {};
    struct Search {
        static void go(const SchedProblem *p, int tile_m, int bn, int64_t max_units, int nch,
                       const int *ch_n, const int (*ch_idx)[kMaxLaunchProblems], const int *ch_cost,
                       bool *taken, Partition &cur, Partition &best)
        {
            int first = -1;
            for (int c = 0; c < nch && first < 0; ++c)
                if (!taken[c])
                    first = c;
            if (first < 0) {
                if (cur.predicted < best.predicted)
                    best = cur;
                return;
            }
            taken[first] = true;
            for (int other = -1; other < nch; ++other) {
                if (other >= 0 && (taken[other] || ch_cost[other] == ch_cost[first] ||
                                   ch_n[first] + ch_n[other] > kMaxLaunchProblems))
                    continue;
                int idx[kMaxLaunchProblems], k = 0;
                for (int i = 0; i < ch_n[first]; ++i)
                    idx[k++] = ch_idx[first][i];
                if (other >= 0)
                    for (int i = 0; i < ch_n[other]; ++i)
                        idx[k++] = ch_idx[other][i];
                const LaunchPlan pl = sched_plan_idx(p, idx, k, tile_m, bn, max_units);
                const int64_t t = sched_launch_time(pl);
                if (other >= 0)
                    taken[other] = true;
                const int j = cur.nlaunch++;
                cur.nprob[j] = k;
                for (int i = 0; i < k; ++i)
                    cur.idx[j][i] = idx[i];
                cur.predicted += t;
                go(p, tile_m, bn, max_units, nch, ch_n, ch_idx, ch_cost, taken, cur, best);
                cur.predicted -= t;
                --cur.nlaunch;
                if (other >= 0)
                    taken[other] = false;
            }
            taken[first] = false;
        }
    };
    Search::go(p, tile_m, bn, max_units, nch, ch_n, ch_idx, ch_cost, taken, cur, best);
    if (best.predicted * 100 <= alone.predicted * (100 - kSchedMinGainPct))
        return best;
    return alone;
}

}  // namespace f8
