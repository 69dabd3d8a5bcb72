// Static tile schedule for one persistent GEMM launch that runs two
// independent problems (the dgrad and wgrad GEMMs of a linear's backward
// pass, which both read q(dY)).  Plain integer code, usable from host and
// device.
//
// U workers (CTAs, or CTA pairs) share T0 tiles of problem 0, each costing
// c0, and T1 tiles of problem 1, each costing c1 (a model of the tile's run
// time; the host puts the problem with the larger cost first).  Problem 0 is
// dealt round-robin: worker u takes tiles u, u + U, u + 2U, ...  and is then
// free at T_u = n0(u) c0.  Problem 1's tiles are then handed out in order,
// each to the worker that is free first (ties: lower worker index first);
// a worker is free again c1 after it took one.  That is list scheduling of
// the second problem behind the first, and it keeps consecutive tiles of
// problem 1 on concurrently running workers (the raster order's L2 reuse).
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

// The extents of one GEMM C[M,N] = A[M,K] B[N,K]^T.
struct SchedProblem {
    int64_t M, N, K;
};

// The schedule of one launch over `nprob` (1 or 2) problems in tile_m x bn
// output tiles on at most max_units workers; `first` is the index of the
// problem dealt round-robin (the one with the costlier tiles).
struct SchedPlan {
    TileSched s;
    int first;
};

static inline SchedPlan sched_plan(const SchedProblem *p, int nprob, int tile_m, int bn,
                                   int64_t max_units)
{
    int tiles[2] = {0, 0};
    int cost[2] = {1, 1};
    for (int i = 0; i < nprob; ++i) {
        tiles[i] = static_cast<int>(((p[i].M + tile_m - 1) / tile_m) * ((p[i].N + bn - 1) / bn));
        cost[i] = static_cast<int>((p[i].K + kSchedBlockK - 1) / kSchedBlockK) +
                  kSchedTileOverheadKb;
    }
    const int64_t total = static_cast<int64_t>(tiles[0]) + tiles[1];
    const int units = static_cast<int>(total < max_units ? total : max_units);
    const int first = (nprob == 2 && cost[1] > cost[0]) ? 1 : 0;
    const int second = nprob == 2 ? 1 - first : first;
    SchedPlan plan;
    plan.s.units = units;
    plan.s.tiles0 = tiles[first];
    plan.s.tiles1 = nprob == 2 ? tiles[second] : 0;
    plan.s.cost0 = cost[first];
    plan.s.cost1 = cost[second];
    plan.first = first;
    return plan;
}

// Whether two GEMMs should share one launch: the schedule's predicted
// makespan beats the two launches' by at least kSchedMinGainPct percent.
static inline bool sched_should_group(const SchedProblem &p0, const SchedProblem &p1, int tile_m,
                                      int bn, int64_t max_units)
{
    const SchedProblem both[2] = {p0, p1};
    const int64_t grouped = sched_makespan(sched_plan(both, 2, tile_m, bn, max_units).s);
    const int64_t apart = sched_makespan(sched_plan(&p0, 1, tile_m, bn, max_units).s) +
                          sched_makespan(sched_plan(&p1, 1, tile_m, bn, max_units).s);
    return grouped * 100 <= apart * (100 - kSchedMinGainPct);
}

}  // namespace f8
