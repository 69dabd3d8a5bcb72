// E4M3 x E4M3 -> fp32 -> bf16 GEMM on the 5th-generation tensor cores:
// C[M,N] = bf16( A[M,K] B[N,K]^T * 1/(sa sb) ), both operands K-major.
//
// Persistent, warp-specialised, 192 threads per CTA, one CTA per SM:
//   warp 0      TMA producer: A and B tiles of 128 bytes of K (128-byte
//               swizzle) into a STAGES-deep shared-memory ring; completion
//               is counted in transaction bytes on full[s];
//   warp 1      TMEM allocator and MMA issuer: 4 tcgen05.mma kind::f8f6f4
//               (K = 32 each) per stage into one of two TMEM accumulators;
//               tcgen05.commit releases the stage (empty[s]) and, after the
//               last K block of a tile, hands the accumulator to the
//               epilogue (tfull[a]);
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 64 columns, x fl32(1/(sa sb)),
//               round to bf16, stage 32 rows x 128 bytes in swizzled shared
//               memory and write it with one TMA tensor store; the
//               accumulator is released (tempty[a]) as soon as it has been
//               read, so the MMAs of tile i+1 overlap the epilogue of tile i.
// GLU = true is the W13 GEMM of a SwiGLU FFN: B holds W1 and W3 interleaved
// by 128 rows, so the 256 columns of a tile are 128 columns of a = X W1^T and
// the matching 128 of b = X W3^T.  The epilogue stores a and b (bf16) and
// h = bf16(silu(a) b), formed from those bf16 values, into a second [M, N/2]
// output, all by TMA stores, and keeps the largest |h|: one partial maximum
// per CTA is written at the end for the cast of h (or, with hatomic, one
// atomicMax per CTA into a zeroed fp32 amax).
// Two shapes of the same kernel:
//   PAIR = false  one CTA computes a 128 x BN tile (tcgen05 cta_group::1);
//   PAIR = true   a cluster of two CTAs on neighbouring SMs computes a
//                 256 x BN tile with cta_group::2: each CTA loads its own
//                 128 rows of A and BN/2 rows of B, so each SM stages half
//                 the B tile it would need alone.  The even CTA issues the
//                 MMAs; its full[s] barriers count the bytes of both CTAs;
//                 commits are multicast to the barriers of both CTAs; both
//                 epilogues arrive on the even CTA's tempty barriers.
// A launch runs one GEMM (NP = 1), or up to four independent ones (NP = 4:
// a linear's dgrad and wgrad; the forward GEMMs of linears that share their
// input) whose tiles share the persistent CTAs under the static list
// schedule of f8_sched.h: every role of every CTA derives the same tile
// sequence from (CTA, i), so nothing is communicated.
// Tiles are visited in groups of `group_m` M-blocks so that concurrently
// running CTAs share operand tiles in L2.  M, N and K edges are zero-filled
// by TMA loads and clipped by TMA stores (or masked on the direct-store path
// used when a C row is not a multiple of 16 bytes).
//
// Every wait is bounded (global-timer limit).  A wait that gives up sets a
// CTA-wide abort flag and the device status word; the roles leave their
// loops, the producer waits for copies still in flight, the MMA thread for
// its own MMAs, and TMEM is released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <map>
#include <mutex>
#include <vector>

#include "f8_internal.h"
#include "f8_ptx.cuh"
#include "f8_sched.h"
#include "f8_swiglu.cuh"

namespace f8 {
namespace {

constexpr int kBM = 128;   // accumulator rows per CTA (TMEM lanes)
constexpr int kBK = 128;   // bytes of K per stage = one 128-byte swizzle row
constexpr int kEpiWarps = 4;       // one per TMEM lane quarter
constexpr int kGluCols = 32;       // GLU: h columns per epilogue step
constexpr int kGluBoxBytes = 32 * kGluCols * 2;  // one 32 x 64-byte box, 64-byte swizzle
constexpr int kEpiCols = 64;                       // columns per epilogue step
constexpr int kEpiBufBytes = 32 * kEpiCols * 2;    // 32 rows x 128 bytes
constexpr uint64_t kDrainLimitNs = 1000000000ull;

template <int BN, int STAGES, bool PAIR, bool GLU = false>
struct Cfg {
    static constexpr int kTileM = PAIR ? 2 * kBM : kBM;
    static constexpr int kBRows = PAIR ? BN / 2 : BN;  // rows of B each CTA loads
    static constexpr int kABytes = kBM * kBK;
    static constexpr int kBBytes = kBRows * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = (2 * BN <= 256) ? 256 : 512;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue
    // per epilogue warp: plain, two 32 x 128-byte swizzled store buffers;
    // GLU, one set of three 32 x 64-byte boxes (a, b, h)
    static constexpr int kWarpStaging = GLU ? 3 * kGluBoxBytes : 2 * kEpiBufBytes;
    static constexpr int kStagingBytes = kEpiWarps * kWarpStaging;
    static constexpr int kBarBytes = 8 * (2 * STAGES + 5) + 16;
    static constexpr int kSmemBytes = STAGES * kStageBytes + kStagingBytes + kBarBytes + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(BN % kEpiCols == 0, "epilogue steps");
    static_assert(!GLU || BN == 256, "a GLU tile is 128 columns of a and 128 of b");
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group_m, int &mb,
                                            int &nb)
{
    const int per_group = group_m * num_n;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int gm = min(group_m, num_m - first_m);
    const int r = tile - g * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

__device__ __forceinline__ void note_timeout(volatile int *abort_flag, unsigned *status)
{
    *abort_flag = 1;
    atomicOr(status, kStatusTimeout);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __float22bfloat162_rn(make_float2(lo, hi));
    return *reinterpret_cast<uint32_t *>(&h);
}

// eight fp32 accumulators x inv (one packed fp32x2 multiply per pair, per
// lane the scalar round-to-nearest product), rounded to bf16 and packed
__device__ __forceinline__ uint32_t scale2(const uint32_t *r, float2 inv2)
{
    const float2 v = __fmul2_rn(make_float2(__uint_as_float(r[0]), __uint_as_float(r[1])), inv2);
    return pack_bf16x2(v.x, v.y);
}

__device__ __forceinline__ uint4 pack8(const uint32_t *r, float inv)
{
    const float2 inv2 = make_float2(inv, inv);
    return make_uint4(scale2(r, inv2), scale2(r + 2, inv2), scale2(r + 4, inv2),
                      scale2(r + 6, inv2));
}

// One warp's share of an accumulator: TMEM lanes [32q, 32q + 32) x BN
// columns starting at `taddr`, i.e. C rows row0 .. row0 + 31 and columns
// col_base .. col_base + BN - 1.
template <int BN>
__device__ __forceinline__ void epilogue_rows(uint32_t taddr, int row0, int col_base, int M, int N,
                                              float inv, __nv_bfloat16 *__restrict__ c,
                                              const CUtensorMap *tma_c, bool tma_store,
                                              uint8_t *stage, uint32_t &buf, int lane,
                                              unsigned *status)
{
#pragma unroll 1
    for (int j = 0; j < BN / kEpiCols; ++j) {
        uint32_t r[kEpiCols];
        tc_ld_32x32b_x32(taddr + j * kEpiCols, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tc_ld_32x32b_x32(taddr + j * kEpiCols + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tc_wait_ld();
        const int col0 = col_base + j * kEpiCols;
        if (tma_store) {
            // nothing of this box lies in C: no staging, no store, no bulk
            // group (row0 and col0 are warp-uniform)
            if (row0 >= M || col0 >= N)
                continue;
            uint8_t *b = stage + buf * kEpiBufBytes;
            if (lane == 0)
                bulk_wait_group_read<1>();  // the store issued from b two stores ago has read it
            __syncwarp();
            // row `lane` of the box, 16-byte chunk q at (q ^ row % 8): the 128-byte swizzle
#pragma unroll
            for (int q = 0; q < kEpiCols / 8; ++q)
                *reinterpret_cast<uint4 *>(b + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                    pack8(&r[8 * q], inv);
            fence_proxy_async_shared();
            __syncwarp();
            // every use of a buffer ends in one store and one bulk group, so
            // the read wait above always refers to this buffer's last store
            if (lane == 0) {
                tma_store_2d(tma_c, b, col0, row0);
                bulk_commit_group();
            }
            buf ^= 1u;
        } else {
            const int row = row0 + lane;
            if (row < M) {
                __nv_bfloat16 *dst = c + static_cast<int64_t>(row) * N + col0;
                const bool vec = (N % 8) == 0 && col0 + kEpiCols <= N;
                const int64_t o = static_cast<int64_t>(row) * N + col0;
                const int64_t mn = static_cast<int64_t>(M) * N;
                if (vec) {
#pragma unroll
                    for (int q = 0; q < kEpiCols / 8; ++q)
                        if (in_range(o + 8 * q, 8, mn, status))
                            *reinterpret_cast<uint4 *>(dst + 8 * q) = pack8(&r[8 * q], inv);
                } else {
                    for (int e = 0; e < kEpiCols; ++e)
                        if (col0 + e < N && in_range(o + e, 1, mn, status))
                            dst[e] = __float2bfloat16_rn(__uint_as_float(r[e]) * inv);
                }
            }
        }
    }
}

// The GLU epilogue of one warp: TMEM lanes [32q, 32q + 32) of a W13 tile,
// accumulator columns [0, 128) = a and [128, 256) = the matching b.  Per
// step of 32 h columns: a and b are scaled and rounded exactly as in
// epilogue_rows, h = bf16(silu(a) b) is formed from those bf16 values, and
// the three 32 x 32 blocks (row = lane, 64 bytes each) are staged in boxes
// laid out in the TMA 64-byte swizzle (16-byte chunk q of row r at chunk
// q ^ ((r / 2) % 4), which keeps each 8-lane phase of a 16-byte shared store
// on 8 distinct bank groups) and written with three TMA stores (AB columns col_base +
// c and col_base + 128 + c, h columns col_base / 2 + c): whole-line bulk
// writes, which keep the L2 request rate of the epilogue at the plain
// epilogue's.  The box set is reused once the previous step's stores have
// read it; the next accumulator load is issued before that wait.
__device__ __forceinline__ void epilogue_rows_glu(uint32_t taddr, int row0, int col_base, int M,
                                                  float inv, const CUtensorMap *tma_ab,
                                                  const CUtensorMap *tma_h, uint8_t *stage,
                                                  uint32_t &hmax2, int lane)
{
    uint8_t *sa = stage;
    uint8_t *sb = stage + kGluBoxBytes;
    uint8_t *sh = stage + 2 * kGluBoxBytes;
#pragma unroll 1
    for (int c = 0; c < 128; c += kGluCols) {
        uint32_t ra[32], rb[32];
        tc_ld_32x32b_x32(taddr + c, ra);
        tc_ld_32x32b_x32(taddr + 128 + c, rb);
        if (lane == 0)
            bulk_wait_group_read<0>();  // the previous step's stores have read the boxes
        __syncwarp();
        tc_wait_ld();
        uint4 a8[4], b8[4], h8[4];
        uint32_t amag = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            a8[q] = pack8(&ra[8 * q], inv);
            b8[q] = pack8(&rb[8 * q], inv);
            amag = swiglu::fold_abs(amag, a8[q]);
        }
        // one branch per 32 elements, so that their chains interleave
        if (swiglu::small87(amag)) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                h8[q] = swiglu::swiglu8<false>(a8[q], b8[q]);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                h8[q] = swiglu::swiglu8<true>(a8[q], b8[q]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            hmax2 = swiglu::max_abs2(hmax2, h8[q].x);
            hmax2 = swiglu::max_abs2(hmax2, h8[q].y);
            hmax2 = swiglu::max_abs2(hmax2, h8[q].z);
            hmax2 = swiglu::max_abs2(hmax2, h8[q].w);
            const int off = lane * (kGluCols * 2) + ((q ^ ((lane >> 1) & 3)) << 4);
            *reinterpret_cast<uint4 *>(sa + off) = a8[q];
            *reinterpret_cast<uint4 *>(sb + off) = b8[q];
            *reinterpret_cast<uint4 *>(sh + off) = h8[q];
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && row0 < M) {
            tma_store_2d(tma_ab, sa, col_base + c, row0);
            tma_store_2d(tma_ab, sb, col_base + 128 + c, row0);
            tma_store_2d(tma_h, sh, col_base / 2 + c, row0);
            bulk_commit_group();
        }
    }
}

// One GEMM problem of a launch.
struct GemmProb {
    __nv_bfloat16 *c;
    const float *sa;
    const float *sb;
    int M, N;
    int num_m, num_n, num_kb;
    int tma_store;
    uint32_t idesc;
};

// The problems of one launch and their tensor maps (C's map unused when the
// problem stores directly).  NP = 1: one problem, its tiles dealt
// round-robin.  NP > 1: nprob problems in the slot order of f8_sched.h's
// LaunchPlan; first_tile[i] is slot i's first launch-global tile and sched
// the list schedule over them.
template <int NP>
struct GemmSet {
    CUtensorMap a[NP], b[NP], c[NP];
    GemmProb p[NP];
    int first_tile[NP + 1];
    int nprob;
    TileSched sched;
};

// This unit's i-th tile as a launch-global index, or -1.
template <int NP>
__device__ __forceinline__ int unit_tile(const GemmSet<NP> &set, int unit, int i)
{
    if (NP == 1) {
        const int t = unit + i * set.sched.units;
        return t < set.sched.tiles0 ? t : -1;
    }
    return sched_tile(set.sched, unit, i);
}

// The slot of launch-global tile g, and g's tile index within that problem.
template <int NP>
__device__ __forceinline__ int tile_slot(const GemmSet<NP> &set, int g, int &local)
{
    if (NP == 1) {
        local = g;
        return 0;
    }
    return sched_slot(set.first_tile, set.nprob, g, local);
}

// v[slot] for a slot held in a register, by selects (no local memory).
template <int NP>
__device__ __forceinline__ float pick(const float (&v)[NP], int slot)
{
    float r = v[0];
#pragma unroll
    for (int j = 1; j < NP; ++j)
        r = slot == j ? v[j] : r;
    return r;
}

template <int BN, int STAGES, bool PAIR, bool GLU, int NP>
__global__ void __launch_bounds__(Cfg<BN, STAGES, PAIR, GLU>::kThreads, 1)
gemm_kernel(const __grid_constant__ GemmSet<NP> set, const __grid_constant__ CUtensorMap tma_h,
            unsigned *__restrict__ status, uint64_t limit_ns, int group_m,
            unsigned *__restrict__ hparts, int hatomic)
{
    using C = Cfg<BN, STAGES, PAIR, GLU>;
    static_assert(!GLU || NP == 1, "the SwiGLU epilogue runs single-problem launches");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *smA = smem;
    uint8_t *smB = smem + STAGES * C::kABytes;
    uint8_t *staging = smem + STAGES * C::kStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(staging + C::kStagingBytes);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    unsigned *hmax_cta = reinterpret_cast<unsigned *>(tmem_slot + 2);  // GLU: largest |h| bits

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], PAIR ? 2 * kEpiWarps : kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *hmax_cta = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            if (j < set.nprob) {
                tma_prefetch_desc(&set.a[j]);
                tma_prefetch_desc(&set.b[j]);
                if (set.p[j].tma_store)
                    tma_prefetch_desc(&set.c[j]);
            }
        }
        if (GLU)
            tma_prefetch_desc(&tma_h);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(tmem_slot, C::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, C::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    if (PAIR)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // everything above overlaps the previous kernel in the stream; the
    // operands and scales may come from it
    griddep_wait();
    griddep_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint32_t full_leader = PAIR ? cluster_map(smem_addr(&full[0]), 0) : 0u;
            uint32_t stage = 0, phase = 0;
            int64_t issued = 0;
            bool stop = false;
            for (int i = 0; !stop; ++i) {
                const int g = unit_tile<NP>(set, unit, i);
                if (g < 0)
                    break;
                int tile;
                const int slot = tile_slot<NP>(set, g, tile);
                const CUtensorMap *ma = &set.a[slot];
                const CUtensorMap *mb_ = &set.b[slot];
                const GemmProb &pr = set.p[slot];
                const int num_kb = pr.num_kb;
                int mb, nb;
                tile_coords(tile, pr.num_m, pr.num_n, group_m, mb, nb);
                const int arow = mb * C::kTileM + static_cast<int>(rank) * kBM;
                const int brow = nb * BN + static_cast<int>(rank) * C::kBRows;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, limit_ns)) {
                        note_timeout(abort_flag, status);
                        stop = true;
                        break;
                    }
                    uint8_t *sa_dst = smA + stage * C::kABytes;
                    uint8_t *sb_dst = smB + stage * C::kBBytes;
                    if (PAIR) {
                        if (leader)
                            mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
                        const uint32_t fb = full_leader + 8u * stage;
                        tma_load_2d_pair(sa_dst, ma, fb, kb * kBK, arow);
                        tma_load_2d_pair(sb_dst, mb_, fb, kb * kBK, brow);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
                        tma_load_2d(sa_dst, ma, &full[stage], kb * kBK, arow);
                        tma_load_2d(sb_dst, mb_, &full[stage], kb * kBK, brow);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!*abort_flag) {
                // every stage filled must be released (its commit arrivals
                // have landed here) before the CTA may exit
                for (int i = 0; i < STAGES; ++i) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, limit_ns)) {
                        note_timeout(abort_flag, status);
                        break;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            } else if (leader) {
                // copies still in flight land on these barriers
                int64_t n = issued < STAGES ? issued : STAGES;
                uint32_t s = stage, p = phase;
                for (int64_t i = 0; i < n; ++i) {
                    if (s == 0) {
                        s = STAGES - 1;
                        p ^= 1u;
                    } else {
                        --s;
                    }
                    mbar_wait(&full[s], p, nullptr, kDrainLimitNs);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------------------ MMA issuer
            uint32_t stage = 0, phase = 0;
            bool stop = false;
            int local = 0;
            for (;; ++local) {
                const int g = unit_tile<NP>(set, unit, local);
                if (g < 0)
                    break;
                int tile;
                const int slot = tile_slot<NP>(set, g, tile);
                const int num_kb = set.p[slot].num_kb;
                const uint32_t idesc = set.p[slot].idesc;
                const uint32_t acc = local & 1;
                const uint32_t aph = (local >> 1) & 1;
                if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, limit_ns)) {
                    note_timeout(abort_flag, status);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem_base + acc * BN;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, limit_ns)) {
                        note_timeout(abort_flag, status);
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_addr(smA + stage * C::kABytes));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_addr(smB + stage * C::kBBytes));
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k) {
                        if (PAIR)
                            tc_mma_f8_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
                        else
                            tc_mma_f8(d, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0);
                    }
                    if (PAIR)
                        tc_commit_pair_mc(&empty[stage], 0x3);
                    else
                        tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (stop)
                    break;
                if (PAIR)
                    tc_commit_pair_mc(&tfull[acc], 0x3);
                else
                    tc_commit(&tfull[acc]);
            }
            if (*abort_flag) {
                if (PAIR)
                    tc_commit_pair(drain);
                else
                    tc_commit(drain);
                mbar_wait(drain, 0, nullptr, kDrainLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue
        const int quad = warp & 3;  // the TMEM lane quarter this warp may read
        float inv[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j)
            inv[j] = j < set.nprob ? static_cast<float>(1.0 / (static_cast<double>(*set.p[j].sa) *
                                                               static_cast<double>(*set.p[j].sb)))
                                   : 0.0f;
        uint8_t *my_stage = staging + (warp - 2) * C::kWarpStaging;
        uint32_t hmax2 = 0;
        const uint32_t tempty_leader = PAIR ? cluster_map(smem_addr(&tempty[0]), 0) : 0u;
        uint32_t buf = 0;
        for (int local = 0;; ++local) {
            const int g = unit_tile<NP>(set, unit, local);
            if (g < 0)
                break;
            int tile;
            const int slot = tile_slot<NP>(set, g, tile);
            const GemmProb &pr = set.p[slot];
            const uint32_t acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            bool ok = mbar_wait(&tfull[acc], aph, abort_flag, limit_ns);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                if (lane == 0)
                    note_timeout(abort_flag, status);
                break;
            }
            tc_fence_after_sync();
            int mb, nb;
            tile_coords(tile, pr.num_m, pr.num_n, group_m, mb, nb);
            const int row0 = mb * C::kTileM + static_cast<int>(rank) * kBM + quad * 32;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
            if (GLU)
                epilogue_rows_glu(taddr, row0, nb * BN, pr.M, inv[0], &set.c[0], &tma_h, my_stage,
                                  hmax2, lane);
            else
                epilogue_rows<BN>(taddr, row0, nb * BN, pr.M, pr.N, pick<NP>(inv, slot), pr.c,
                                  &set.c[slot], pr.tma_store != 0, my_stage, buf, lane, status);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (!PAIR || leader)
                    mbar_arrive(&tempty[acc]);
                else
                    mbar_arrive_remote(tempty_leader + 8u * acc);
            }
        }
        if (lane == 0)
            bulk_wait_group_all();
        __syncwarp();
        if (GLU) {
            const unsigned m = __reduce_max_sync(0xFFFFFFFFu, max(hmax2 & 0xFFFFu, hmax2 >> 16));
            if (lane == 0)
                atomicMax(hmax_cta, m);
        }
    }

    tc_fence_before_sync();
    if (PAIR)
        cluster_sync();
    else
        __syncthreads();
    if (GLU && threadIdx.x == 0) {
        const unsigned m = *hmax_cta;
        if (m >= 0x7F80u)
            atomicOr(status, kStatusNonfinite);
        if (hatomic)
            atomicMax(hparts, m << 16);  // fp32 bits of the bf16 |h|: integer order = numeric
        else
            hparts[blockIdx.x] = m << 16;
    }
    if (warp == 1) {
        tc_fence_after_sync();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, C::kTmemCols);
        else
            tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

__global__ void wait_selftest_kernel(unsigned *status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, nullptr, limit_ns))
        atomicOr(status, kStatusTimeout);
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D row-major tensor [rows, cols] of `esize`-byte elements with a
// box_cols x box_rows box and the 128-byte swizzle (box_cols * esize == 128).
bool make_map(CUtensorMap *map, CUtensorMapDataType dtype, int esize, const void *ptr,
              int64_t rows, int64_t cols, int box_cols, int box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static_assert(kBK == kSchedBlockK, "the schedule's tile costs count the kernel's K blocks");

// One launch of gemm_kernel over the problems probs[plan.order[0 .. n)]
// (n = 1 for NP = 1), in the plan's slot order.
template <int BN, int STAGES, bool PAIR, bool GLU = false, int NP = 1>
cudaError_t run_gemm(const GemmDesc *probs, const LaunchPlan &plan, const DeviceInfo &dev,
                     cudaStream_t stream, void *h = nullptr, unsigned *hparts = nullptr,
                     int *nparts = nullptr, int hatomic = 0)
{
    using C = Cfg<BN, STAGES, PAIR, GLU>;
    if (!plan.ok || plan.nprob < 1 || plan.nprob > NP)
        return cudaErrorInvalidValue;
    GemmSet<NP> set;
    CUtensorMap mh;
    for (int i = 0; i < plan.nprob; ++i) {
        const GemmDesc &p = probs[plan.order[i]];
        if (!make_map(&set.a[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.a, p.M, p.K, kBK, kBM) ||
            !make_map(&set.b[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.b, p.N, p.K, kBK, C::kBRows))
            return cudaErrorNotSupported;
        // TMA stores need every C row to start on a 16-byte boundary
        int tma_store;
        if (GLU) {
            // AB and h through 32-row x 32-column boxes in the 64-byte swizzle
            tma_store = 1;
            if (p.N % 256 != 0 ||
                !make_tensor_map_2d(&set.c[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.c, p.M, p.N,
                                    kGluCols, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
                !make_tensor_map_2d(&mh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h, p.M, p.N / 2,
                                    kGluCols, 32, CU_TENSOR_MAP_SWIZZLE_64B))
                return cudaErrorNotSupported;
        } else {
            tma_store = (p.N % 8 == 0) && make_map(&set.c[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                                   p.c, p.M, p.N, kEpiCols, 32);
            if (!tma_store)
                set.c[i] = set.a[i];  // not used by the kernel
        }
        const int num_m = static_cast<int>((p.M + C::kTileM - 1) / C::kTileM);
        const int num_n = static_cast<int>((p.N + BN - 1) / BN);
        const int num_kb = static_cast<int>((p.K + kBK - 1) / kBK);
        set.p[i] = GemmProb{static_cast<__nv_bfloat16 *>(p.c), p.sa, p.sb, static_cast<int>(p.M),
                            static_cast<int>(p.N), num_m, num_n, num_kb, tma_store,
                            idesc_f8_f32(C::kTileM, BN, static_cast<uint32_t>(p.fa),
                                         static_cast<uint32_t>(p.fb))};
    }
    for (int i = plan.nprob; i < NP; ++i) {  // unused slots: copies, never read
        set.a[i] = set.a[0];
        set.b[i] = set.b[0];
        set.c[i] = set.c[0];
        set.p[i] = set.p[0];
    }
    for (int i = 0; i <= NP; ++i)
        set.first_tile[i] = i <= plan.nprob ? plan.first_tile[i] : plan.first_tile[plan.nprob];
    set.nprob = plan.nprob;
    set.sched = plan.s;
    if (!GLU)
        mh = set.a[0];  // not used by the kernel
    static std::once_flag attr_once[64];
    static cudaError_t attr_err[64];
    const int dv = dev.ordinal & 63;
    std::call_once(attr_once[dv], [&] {
        attr_err[dv] = cudaFuncSetAttribute(gemm_kernel<BN, STAGES, PAIR, GLU, NP>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            C::kSmemBytes);
    });
    if (attr_err[dv] != cudaSuccess)
        return attr_err[dv];
    const int units = plan.s.units;
    const int group_m = PAIR ? 8 : 16;
    if (nparts != nullptr)
        *nparts = (PAIR ? 2 : 1) * units;
    return launch_pdl_cluster(gemm_kernel<BN, STAGES, PAIR, GLU, NP>, dim3((PAIR ? 2 : 1) * units),
                              dim3(C::kThreads), C::kSmemBytes, stream, PAIR ? 2u : 1u, set, mh,
                              dev.status, wait_limit_ns(), group_m, hparts, hatomic);
}

constexpr int kVariantSingle = 1;
constexpr int kVariantPair = 2;

// Kernel choice: the CTA-pair kernel for every shape with at least two
// 128-row blocks; F8_GEMM_VARIANT=1|2 forces one kernel (for measurement).
int gemm_variant(int64_t M, const DeviceInfo &dev)
{
    const char *e = std::getenv("F8_GEMM_VARIANT");
    const int forced = e ? std::atoi(e) : 0;
    if (forced == kVariantSingle || forced == kVariantPair)
        return forced;
    if (dev.sm_count < 2 || M < 2 * kBM)
        return kVariantSingle;
    return kVariantPair;
}

} // namespace

bool make_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, int esize, const void *ptr,
                        int64_t rows, int64_t cols, int box_cols, int box_rows,
                        CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Tile geometry of a kernel variant.
int variant_tile_m(int v) { return v == kVariantPair ? 2 * kBM : kBM; }

int64_t variant_units(int v, const DeviceInfo &dev)
{
    return v == kVariantPair ? dev.sm_count / 2 : dev.sm_count;
}

SchedProblem sched_problem(const GemmDesc &g) { return SchedProblem{g.M, g.N, g.K}; }

// sched_partition's plans, keyed by the problems' extents and the launch
// geometry: a training step asks for the same few plans every step, and a
// plan costs tens of microseconds of host time to search.
std::mutex g_plan_mutex;
std::map<std::vector<int64_t>, Partition> g_plan_cache;

Partition cached_partition(const SchedProblem *sp, int n, int tile_m, int64_t units)
{
    std::vector<int64_t> key;
    key.reserve(3 * n + 2);
    for (int i = 0; i < n; ++i) {
        key.push_back(sp[i].M);
        key.push_back(sp[i].N);
        key.push_back(sp[i].K);
    }
    key.push_back(tile_m);
    key.push_back(units);
    {
        std::lock_guard<std::mutex> lock(g_plan_mutex);
        auto it = g_plan_cache.find(key);
        if (it != g_plan_cache.end())
            return it->second;
    }
    const Partition part = sched_partition(sp, n, tile_m, 256, units);
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    if (g_plan_cache.size() >= 1024)
        g_plan_cache.clear();
    g_plan_cache.emplace(std::move(key), part);
    return part;
}

// One launch over probs[idx[0 .. n)], all of kernel variant v.
cudaError_t launch_set(const GemmDesc *probs, const int *idx, int n, int v, const DeviceInfo &dev,
                       cudaStream_t stream)
{
    SchedProblem sp[kMaxLaunchProblems];
    for (int i = 0; i < n; ++i)
        sp[i] = sched_problem(probs[idx[i]]);
    int local[kMaxLaunchProblems];
    for (int i = 0; i < n; ++i)
        local[i] = i;
    LaunchPlan plan = sched_plan_idx(sp, local, n, variant_tile_m(v), 256, variant_units(v, dev));
    if (!plan.ok)
        return cudaErrorInvalidValue;
    GemmDesc g[kMaxLaunchProblems];
    for (int i = 0; i < n; ++i)
        g[i] = probs[idx[i]];
    if (n == 1)
        return v == kVariantPair ? run_gemm<256, 6, true>(g, plan, dev, stream)
                                 : run_gemm<256, 4, false>(g, plan, dev, stream);
    return v == kVariantPair ? run_gemm<256, 6, true, false, kMaxLaunchProblems>(g, plan, dev, stream)
                             : run_gemm<256, 4, false, false, kMaxLaunchProblems>(g, plan, dev, stream);
}

} // namespace

cudaError_t launch_gemm(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                        const float *sa, const float *sb, void *c, const DeviceInfo &dev,
                        cudaStream_t stream, int fa, int fb)
{
    const GemmDesc g{a, b, M, N, K, sa, sb, c, fa, fb};
    const int idx = 0;
    return launch_set(&g, &idx, 1, gemm_variant(M, dev), dev, stream);
}

cudaError_t launch_gemm_multi(const GemmDesc *g, int n, const DeviceInfo &dev, cudaStream_t stream)
{
    if (n < 1 || n > kMaxPartitionProblems)
        return cudaErrorInvalidValue;
    // problems of different kernel variants never share a launch
    const int v0 = gemm_variant(g[0].M, dev);
    bool same = true;
    for (int i = 1; i < n; ++i)
        same = same && gemm_variant(g[i].M, dev) == v0;
    const int mode = gemm_group_mode();
    if (n == 1 || !same || mode == kGroupNever) {
        for (int i = 0; i < n; ++i) {
            const cudaError_t e = launch_set(g, &i, 1, gemm_variant(g[i].M, dev), dev, stream);
            if (e != cudaSuccess)
                return e;
        }
        return cudaSuccess;
    }
    SchedProblem sp[kMaxPartitionProblems];
    for (int i = 0; i < n; ++i)
        sp[i] = sched_problem(g[i]);
    Partition part;
    int all[kMaxLaunchProblems];
    for (int i = 0; i < n && i < kMaxLaunchProblems; ++i)
        all[i] = i;
    if (mode == kGroupAlways && n <= kMaxLaunchProblems &&
        sched_plan_idx(sp, all, n, variant_tile_m(v0), 256, variant_units(v0, dev)).ok) {
        part.nlaunch = 1;
        part.nprob[0] = n;
        for (int i = 0; i < n; ++i)
            part.idx[0][i] = i;
    } else {
        part = cached_partition(sp, n, variant_tile_m(v0), variant_units(v0, dev));
    }
    for (int j = 0; j < part.nlaunch; ++j) {
        const cudaError_t e = launch_set(g, part.idx[j], part.nprob[j], v0, dev, stream);
        if (e != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm2(const GemmDesc &g0, const GemmDesc &g1, const DeviceInfo &dev,
                         cudaStream_t stream)
{
    const GemmDesc g[2] = {g0, g1};
    return launch_gemm_multi(g, 2, dev, stream);
}

cudaError_t launch_gemm_w13_swiglu(const uint8_t *x_q, const uint8_t *w13_q, int64_t M, int64_t F,
                                   int64_t K, const float *sx, const float *sw, void *ab, void *h,
                                   unsigned *hparts, int *nparts, const DeviceInfo &dev,
                                   cudaStream_t stream, bool hatomic)
{
    if (F % 128 != 0)
        return cudaErrorInvalidValue;
    const GemmDesc g{x_q, w13_q, M, 2 * F, K, sx, sw, ab, 0, 0};
    const int v = gemm_variant(M, dev);
    const SchedProblem sp = sched_problem(g);
    const LaunchPlan plan = sched_plan(&sp, 1, variant_tile_m(v), 256, variant_units(v, dev));
    if (v == kVariantPair)
        return run_gemm<256, 6, true, true>(&g, plan, dev, stream, h, hparts, nparts,
                                            hatomic ? 1 : 0);
    return run_gemm<256, 4, false, true>(&g, plan, dev, stream, h, hparts, nparts, hatomic ? 1 : 0);
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, const DeviceInfo &dev, cudaStream_t stream)
{
    count_launch();
    wait_selftest_kernel<<<1, 32, 0, stream>>>(dev.status, limit_ns);
    return cudaGetLastError();
}

} // namespace f8
