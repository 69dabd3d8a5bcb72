// Checks the closed-form two-class tile schedule (f8_sched.h) against a
// direct simulation of the list scheduler it stands for: class 0 dealt
// round-robin, then each class-1 tile, in order, to the worker that is
// free first (lowest worker index among equals).  Every worker's tile list
// must be identical, which also makes every tile appear exactly once, and
// sched_makespan must equal the simulated busiest worker's finishing time.
// A launch of up to four problems numbers their tiles one after the other
// (class 0's problems first): every (problem, tile) must come out of the
// slot map exactly once.  The planner's tile counts, costs and grouping
// decisions for the Llama-3.1 linears are checked against the values worked
// out by hand (a launch is shared only where that is predicted to gain
// >= 4%).
// Usage: sched_check [cases]; prints "<n> cases, <m> mismatches".
#include <cstdio>
#include <cstdlib>
#include <map>
#include <queue>
#include <utility>
#include <vector>

#include "../../float8_mixed_precision_gb300/csrc/f8_sched.h"

using f8::TileSched;

static std::vector<std::vector<int>> simulate(const TileSched &s)
{
    std::vector<std::vector<int>> lists(s.units);
    std::vector<long long> free_at(s.units, 0);
    for (int t = 0; t < s.tiles0; ++t) {
        lists[t % s.units].push_back(t);
        free_at[t % s.units] += s.cost0;
    }
    typedef std::pair<long long, int> Ev;  // (free time, worker): smallest first
    std::priority_queue<Ev, std::vector<Ev>, std::greater<Ev>> q;
    for (int u = 0; u < s.units; ++u)
        q.push(Ev(free_at[u], u));
    for (int t = 0; t < s.tiles1; ++t) {
        Ev e = q.top();
        q.pop();
        lists[e.second].push_back(s.tiles0 + t);
        q.push(Ev(e.first + s.cost1, e.second));
    }
    return lists;
}

static std::vector<std::vector<int>> closed_form(const TileSched &s)
{
    std::vector<std::vector<int>> lists(s.units);
    for (int u = 0; u < s.units; ++u)
        for (int i = 0;; ++i) {
            const int g = f8::sched_tile(s, u, i);
            if (g < 0)
                break;
            lists[u].push_back(g);
            if (i > s.tiles0 + s.tiles1)  // a runaway list is a mismatch
                break;
        }
    return lists;
}

static long long simulated_makespan(const TileSched &s, const std::vector<std::vector<int>> &l)
{
    long long worst = 0;
    for (const std::vector<int> &v : l) {
        long long t = 0;
        for (int g : v)
            t += g < s.tiles0 ? s.cost0 : s.cost1;
        worst = t > worst ? t : worst;
    }
    return worst;
}

static int check(const TileSched &s)
{
    const std::vector<std::vector<int>> sim = simulate(s);
    if (sim == closed_form(s) && simulated_makespan(s, sim) == f8::sched_makespan(s))
        return 0;
    std::printf("mismatch: U=%d T0=%d T1=%d c0=%d c1=%d\n", s.units, s.tiles0, s.tiles1, s.cost0,
                s.cost1);
    return 1;
}

int main(int argc, char **argv)
{
    const int cases = argc > 1 ? std::atoi(argv[1]) : 20000;
    int bad = 0, n = 0;
    // the launches a linear's backward pass makes on 76 CTA pairs, with the
    // tile cost model K blocks + 4 (Llama-3.1 8B/70B attention and FFN shapes)
    const TileSched shapes[] = {
        {76, 256, 512, 68, 36},   {76, 64, 512, 68, 12},    {76, 512, 896, 116, 68},
        {76, 448, 512, 68, 60},   {76, 1792, 1024, 228, 68}, {76, 1024, 1792, 68, 228},
        {76, 0, 100, 1, 5},       {76, 100, 0, 5, 1},        {1, 7, 9, 3, 2},
        {152, 512, 512, 36, 36},
    };
    for (const TileSched &s : shapes) {
        bad += check(s);
        ++n;
    }
    // exhaustive over small parameters (equal-time ties of both classes)
    for (int U = 1; U <= 9; ++U)
        for (int t0 = 0; t0 <= 20; ++t0)
            for (int t1 = 0; t1 <= 20; t1 += 3)
                for (int c0 = 1; c0 <= 6; ++c0)
                    for (int c1 = 1; c1 <= 6; ++c1) {
                        bad += check(TileSched{U, t0, t1, c0, c1});
                        ++n;
                    }
    unsigned r = 12345u;
    for (int i = 0; i < cases; ++i) {
        r = r * 1103515245u + 12345u;
        const int U = 1 + static_cast<int>((r >> 8) % 160u);
        r = r * 1103515245u + 12345u;
        const int t0 = static_cast<int>((r >> 8) % 2000u);
        r = r * 1103515245u + 12345u;
        const int t1 = static_cast<int>((r >> 8) % 2000u);
        r = r * 1103515245u + 12345u;
        const int c0 = 1 + static_cast<int>((r >> 8) % 300u);
        r = r * 1103515245u + 12345u;
        const int c1 = 1 + static_cast<int>((r >> 8) % 300u);
        bad += check(TileSched{U, t0, t1, c0, c1});
        ++n;
    }
    // the planner on the backward pass of the Llama-3.1 linears (M = 8192
    // tokens; dgrad [M, K] over N, wgrad [N, K] over M; 256 x 256 tiles on 76
    // CTA pairs): tile counts and costs, and the decision to share a launch
    struct Lin {
        const char *name;
        int64_t N, K;
        bool group;
    };
    const Lin lins[] = {{"wq/wo", 4096, 4096, true},      {"wk/wv", 1024, 4096, true},
                        {"8B w1/w3", 14336, 4096, false}, {"8B w2", 4096, 14336, false},
                        {"70B w1/w3", 28672, 8192, false}, {"70B w2", 8192, 28672, false}};
    for (const Lin &l : lins) {
        const f8::SchedProblem dgrad{8192, l.K, l.N}, wgrad{l.N, l.K, 8192};
        const bool g = f8::sched_should_group(dgrad, wgrad, 256, 256, 76);
        if (g != l.group) {
            std::printf("decision mismatch: %s grouped=%d\n", l.name, g);
            ++bad;
        }
        ++n;
    }
    {
        // wq: wgrad (K = 8192: 64 K blocks + 4) is dealt first, 256 tiles;
        // then dgrad's 512 tiles of 32 + 4
        const f8::SchedProblem p[2] = {{8192, 4096, 4096}, {4096, 4096, 8192}};
        const f8::LaunchPlan pl = f8::sched_plan(p, 2, 256, 256, 76);
        if (!(pl.ok && pl.order[0] == 1 && pl.order[1] == 0 && pl.nclass0 == 1 &&
              pl.s.units == 76 && pl.s.tiles0 == 256 && pl.s.cost0 == 68 && pl.s.tiles1 == 512 &&
              pl.s.cost1 == 36 && pl.first_tile[1] == 256 && pl.first_tile[2] == 768)) {
            std::printf("plan mismatch (wq)\n");
            ++bad;
        }
        // one small problem: round-robin over as many workers as tiles
        const f8::LaunchPlan one = f8::sched_plan(p + 1, 1, 256, 256, 76);
        const f8::SchedProblem tiny{300, 520, 400};
        const f8::LaunchPlan t = f8::sched_plan(&tiny, 1, 256, 256, 76);
        if (!(one.s.tiles1 == 0 && one.s.units == 76 && t.s.units == 6 && t.s.tiles0 == 6 &&
              t.s.cost0 == 8)) {
            std::printf("plan mismatch (one problem)\n");
            ++bad;
        }
        // three K extents cannot share a launch
        const f8::SchedProblem three[3] = {{256, 256, 128}, {256, 256, 256}, {256, 256, 384}};
        if (f8::sched_plan(three, 3, 256, 256, 76).ok) {
            std::printf("plan mismatch (three costs accepted)\n");
            ++bad;
        }
        n += 3;
    }
    {
        // the slot map: random launches of 1-4 problems with at most two K
        // extents; every (problem, tile) exactly once over all workers
        unsigned r2 = 777u;
        auto rnd = [&](unsigned m) {
            r2 = r2 * 1103515245u + 12345u;
            return static_cast<int>((r2 >> 8) % m);
        };
        for (int it = 0; it < 4000; ++it) {
            const int np = 1 + rnd(4);
            const int64_t k0 = 128 * (1 + rnd(40)), k1 = 128 * (1 + rnd(40));
            f8::SchedProblem p[4];
            for (int i = 0; i < np; ++i)
                p[i] = f8::SchedProblem{1 + rnd(3000), 1 + rnd(3000), rnd(2) ? k0 : k1};
            const int tile_m = rnd(2) ? 256 : 128;
            const int units = 1 + rnd(160);
            const f8::LaunchPlan pl = f8::sched_plan(p, np, tile_m, 256, units);
            std::map<std::pair<int, int>, int> seen;
            bool ok = pl.ok;
            for (int u = 0; u < pl.s.units && ok; ++u)
                for (int i = 0;; ++i) {
                    const int g = f8::sched_tile(pl.s, u, i);
                    if (g < 0)
                        break;
                    int local = -1;
                    const int slot = f8::sched_slot(pl.first_tile, pl.nprob, g, local);
                    ++seen[std::make_pair(pl.order[slot], local)];
                }
            int64_t want = 0;
            for (int i = 0; i < np && ok; ++i) {
                const int64_t tiles = f8::sched_tiles(p[i], tile_m, 256);
                want += tiles;
                for (int64_t t = 0; t < tiles && ok; ++t)
                    ok = seen.count(std::make_pair(i, static_cast<int>(t))) &&
                         seen[std::make_pair(i, static_cast<int>(t))] == 1;
            }
            ok = ok && static_cast<int64_t>(seen.size()) == want;
            // class 0 holds the costlier problems, each class in caller order
            for (int i = 1; i < pl.nprob && ok; ++i) {
                const int ci = f8::sched_cost(p[pl.order[i]]), cp = f8::sched_cost(p[pl.order[i - 1]]);
                ok = ci < cp || (ci == cp && pl.order[i] > pl.order[i - 1]);
            }
            if (!ok) {
                std::printf("slot map mismatch (case %d, %d problems)\n", it, np);
                ++bad;
            }
            ++n;
        }
    }
    {
        // partitions of the Llama-3.1-8B groups' GEMMs (M = 8192)
        struct Case {
            const char *name;
            int np;
            f8::SchedProblem p[6];
            int nlaunch;
            int first_launch[4];  // problem indices of the first launch (-1 ends)
        };
        const int M = 8192;
        const Case cases_[] = {
            // q, k, v forward (one K): one launch of 768 tiles
            {"qkv fwd", 3, {{M, 4096, 4096}, {M, 1024, 4096}, {M, 1024, 4096}}, 1, {0, 1, 2, -1}},
            // w1, w3 forward: 2 x 1792 tiles, no gain
            {"w1+w3 fwd", 2, {{M, 14336, 4096}, {M, 14336, 4096}}, 2, {0, -1}},
            // q, k, v backward: dgrad_q with the three wgrads (K = M), then
            // dgrad_k with dgrad_v (K = 1024)
            {"qkv bwd", 6,
             {{M, 4096, 4096}, {4096, 4096, M}, {M, 4096, 1024}, {1024, 4096, M}, {M, 4096, 1024},
              {1024, 4096, M}},
             2, {0, 1, 3, 5}},
            {"w1+w3 bwd", 4,
             {{M, 4096, 14336}, {14336, 4096, M}, {M, 4096, 14336}, {14336, 4096, M}}, 4, {0, -1}},
        };
        for (const Case &c : cases_) {
            const f8::Partition pt = f8::sched_partition(c.p, c.np, 256, 256, 76);
            bool ok = pt.nlaunch == c.nlaunch;
            for (int i = 0; i < 4 && ok; ++i) {
                if (c.first_launch[i] < 0) {
                    ok = pt.nprob[0] == i;
                    break;
                }
                ok = i < pt.nprob[0] && pt.idx[0][i] == c.first_launch[i];
            }
            // every problem in exactly one launch
            int count[8] = {};
            for (int j = 0; j < pt.nlaunch; ++j)
                for (int i = 0; i < pt.nprob[j]; ++i)
                    ++count[pt.idx[j][i]];
            for (int i = 0; i < c.np; ++i)
                ok = ok && count[i] == 1;
            if (!ok) {
                std::printf("partition mismatch: %s (%d launches)\n", c.name, pt.nlaunch);
                ++bad;
            }
            ++n;
        }
    }
    std::printf("%d cases, %d mismatches\n", n, bad);
    return bad != 0;
}
