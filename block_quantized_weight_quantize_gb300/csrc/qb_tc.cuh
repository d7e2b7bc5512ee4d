// qb_tc.cuh -- the Q4_K-like and Q6_K-like products for many activation
// columns on the fifth-generation tensor cores (tcgen05): the weights decoded
// into tensor memory as the A operand, the activation codes in shared memory
// as the B operand, f32 accumulators in tensor memory.
//
// What the tensor core computes, and why it is exact (the lane page,
// block_sums):
//   * Q4_K-like, C = sum_s sc_s * sum_{i in s} q_i a_i: A holds the
//     coefficients sc_s*q_i (integers 0..945, exact in f16), B the codes a
//     (-127..127, exact in f16).  Products are exact in f32 and every partial
//     sum over a 128-element half block is an integer below
//     945*127*128 < 2^24, so one accumulator per half block holds its sum
//     exactly in any order of accumulation; the halves are added as integers.
//     O = sum_s mn_s * S_s (S_s the activation's sub-block sums) is one more
//     16-deep product: A = (mn_0..mn_7, mn_0..mn_7), B = (S mod 64 for the
//     eight sub-blocks, 64*floor(S/64) for the eight again) -- every operand
//     an integer exact in f16, |O| <= 8*63*4064 < 2^24.
//   * Q6_K-like, C = sum_u sc_u * sum_{i in u} (q_i - 32) a_i with sc_u an int8:
//     sc_u*(q-32) reaches 4096 in magnitude and is not exact in f16, so sc_u
//     is split as 16*hi + lo (hi in -8..7, lo in 0..15) and A holds both
//     hi*(q-32) and lo*(q-32) (|.| <= 480): two accumulators per block,
//     each below 480*127*256 < 2^24, and C = 16*D_hi + D_lo.
// Each block's C (and O) then goes through the same exact combine and single
// rounding as the other kernels, and each row's values are added in block
// order from +0, so every output has the bits the one-column product gives.
//
// Organisation: a CTA takes a tile of 128 rows (tensor-memory lane r = row
// r) and a contiguous range of its blocks; the KS CTAs that share a tile form
// a cluster and split its blocks.  Per block (Q6_K-like: per half block) the
// 256 threads decode the rows' weights from the staged records (bulk copies,
// the TMA engine) into tensor memory, one thread issues the MMAs (M = 128
// rows, N = 16 columns, K = 16 a step), and the MMAs of one block run while
// the threads combine the previous block and decode the next (two A and two
// accumulator buffers).  A block value goes to the shared memory of the
// cluster CTA that folds its column (distributed shared memory); after a
// cluster barrier each CTA folds its columns' values in block order.
//
// The k order inside an MMA step is free as long as A and B agree: a 32-bit
// word of nibbles (bytes b0..b3) yields the f16 pairs (b0, b2) and (b1, b3)
// in one masked OR each, so within every group of four k slots the middle
// two elements trade places, on both operands.
#pragma once

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"
#include "qb_tmap.cuh"

namespace qb {

// ---------------------------------------------------------------- tcgen05 wrappers

__device__ __forceinline__ void tc_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) = A (tensor memory) * B (shared memory, descriptor) [+ D]
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// The mbarrier gets one arrival once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Three 8-column loads of this warp's 32 lanes and the wait for them, in one
// statement so that nothing reads the registers before the data is there.
__device__ __forceinline__ void tc_ld3x8(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t (&a)[8], uint32_t (&b)[8],
                                         uint32_t (&c)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%24];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%25];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16, %17, %18, %19, %20, %21, %22, %23}, [%26];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
          "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3]), "=r"(c[4]), "=r"(c[5]), "=r"(c[6]), "=r"(c[7])
        : "r"(t0), "r"(t1), "r"(t2)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand without swizzling:
// 8-row x 16-byte core matrices (128 contiguous bytes each), `lbo` bytes
// between core matrices along K, `sbo` bytes between them along M/N.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, both
// K-major, N = 16, M = 128.
constexpr uint32_t kTcIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// ---------------------------------------------------------------- cluster helpers

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// The address of this CTA's shared variable at `saddr` in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---------------------------------------------------------------- f16 pairs

__device__ __forceinline__ uint32_t tc_hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t tc_hadd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// (lo, hi) f32 -> f16x2, round to nearest (exact for the integers used here)
__device__ __forceinline__ uint32_t tc_pack2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t tc_prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ---------------------------------------------------------------- exact combine

template <int KIND>
static __device__ __noinline__ float lane_value_cold(int C, int O, uint32_t s1, uint32_t s2, int m, int e) {
    return lane_value<KIND>(C, O, s1, s2, m, e);
}

// The per-(row, block) part of a block's combine: the weight scales as
// A1*2^Eb and A2*2^Eb at their common (lower) exponent, when their exponents
// are within 11 places (|A| < 2^22, so A*m fits 30 bits).  Q6_K-like: A1 = d,
// A2 = 0.
struct TcScales {
    int A1, A2, Eb;
    bool fast;
};
template <int F>
__device__ __forceinline__ TcScales tc_scales(uint32_t dd) {
    TcScales t;
    int s1, x1;
    const bool f1 = f16_scale(dd & 0xFFFFu, s1, x1);
    if (F == kQ6K) {
        t.A1 = s1;
        t.A2 = 0;
        t.Eb = x1;
        t.fast = f1;
        return t;
    }
    int s2, x2;
    const bool fin = f1 & f16_scale(dd >> 16, s2, x2);
    const int dx = x1 - x2;
    t.fast = fin && dx >= -11 && dx <= 11;
    t.A1 = dx > 0 ? s1 * (1 << dx) : s1;
    t.A2 = dx < 0 ? s2 * (1 << (-dx)) : s2;
    t.Eb = dx > 0 ? x2 : x1;
    return t;
}

// A block's value m*2^e*(d*C - dmin*O) (Q6_K-like: m*2^e*d*C) rounded once
// (lane page: lane).  Fast path: n = m*(A1*C - A2*O) exactly in 64 bits with
// |n| < 2^45 and 2^(Eb+e) within [2^-126, 2^82]: n = H*2^23 + L with
// H = floor(n / 2^23) (|H| < 2^22) and L in [0, 2^23) are exact f32 values
// (built from their bits), one fused multiply-add H*2^23 + L rounds the exact
// n to nearest even, and the product with 2^(Eb+e) is exact (the result is a
// normal number).  Everything else goes to the exact routine.
template <int F>
__device__ __forceinline__ float tc_value(int C, int O, uint32_t dd, const TcScales &t, uint32_t scl) {
    const int m = (int)(scl & 0xFFu), e = (int)(int16_t)(scl >> 16);
    const int E = t.Eb + e;
    if (t.fast && m != 0 && (unsigned)(E + 126) <= 208u) {
        const long long n = (long long)(t.A1 * m) * C - (long long)(t.A2 * m) * O;
        const int hi = (int)(n >> 32);
        if ((unsigned)(hi + 0x2000) < 0x4000u) {
            const int H = (int)(n >> 23);
            const float hf = __int_as_float(0x4B400000 + H) - 12582912.0f;
            const float lf = __uint_as_float(0x4B000000u | ((uint32_t)n & 0x7FFFFFu)) - 8388608.0f;
            return __fmaf_rn(hf, 8388608.0f, lf) * __int_as_float((E + 127) << 23);
        }
    }
    return F == kQ4K ? lane_value_cold<1>(C, O, dd & 0xFFFFu, dd >> 16, m, e) : lane_value_cold<0>(C, 0, dd, 0, m, e);
}

// tc_value with the range checks of a (row, block) done once for its columns
// (blk_fast: finite scales within 11 places, every column scaled, 2^(Eb+e)
// normal for every column): n = m*(A1*C - A2*O) rounded by the fused
// multiply-add as above, then scaled exactly by 2^Eb and 2^e (each product a
// normal number).
template <int F>
__device__ __forceinline__ float tc_value2(int C, int O, uint32_t dd, const TcScales &t, uint32_t scl, bool blk_fast,
                                           float pEb) {
    const int m = (int)(scl & 0xFFu), e = (int)(int16_t)(scl >> 16);
    if (blk_fast) {
        const long long n = (long long)(t.A1 * m) * C - (long long)(t.A2 * m) * O;
        const int hi = (int)(n >> 32);
        if ((unsigned)(hi + 0x2000) < 0x4000u) {
            const int H = (int)(n >> 23);
            const float hf = __int_as_float(0x4B400000 + H) - 12582912.0f;
            const float lf = __uint_as_float(0x4B000000u | ((uint32_t)n & 0x7FFFFFu)) - 8388608.0f;
            return __fmaf_rn(hf, 8388608.0f, lf) * pEb * __int_as_float((e + 127) << 23);
        }
    }
    return F == kQ4K ? lane_value_cold<1>(C, O, dd & 0xFFFFu, dd >> 16, m, e) : lane_value_cold<0>(C, 0, dd, 0, m, e);
}

// ---------------------------------------------------------------- layout

constexpr int kTcRows = 128;     // rows of a tile (tensor-memory lanes)
constexpr int kTcThreads = 800;  // 8 decoder warps, 16 combiner warps, 1 MMA/copy warp
constexpr int kTcMaxKS = 8;      // CTAs of a cluster
constexpr int kTcMinSmem = 116 * 1024;  // at most one CTA a SM (each allocates all 512 columns)
constexpr int kTcMinCols = 9;           // columns from which the dispatch takes this kernel (measured crossover)

struct TcK {
    CUtensorMap tmap[kMaxMats];  // each matrix as [rows][rec] bytes, boxes of 128 rows x one block
    CUtensorMap dmap[kMaxMats];  // Q6_K-like: the same, boxes of 128 rows x 64 bytes (the d plane)
    MatTable mt;
    int64_t tstart[kMaxMats + 1];  // tiles of 128 rows: matrix i holds tiles [tstart[i], tstart[i+1])
    int K, nb, rec;
    int ncols;  // real columns, 1..16 (B's other columns are zero)
    int KS;     // cluster size: the CTAs that split a tile's blocks
    int nbq;    // the most blocks a CTA takes
    int cpc;    // the most columns a CTA folds
    const int8_t *codes;
    const qb_scale *scales;
    const int16_t *sums16;
    int *fault;
};

struct TcSmem {
    int bars, tptr, bact, bo, scl, vals, slab, dreg, total;
};
// bars: 8 pipeline mbarriers, then one per staged block; tptr: the
// tensor-memory address; bact: B, 16 columns x 16 k per 512-byte step,
// nbq*16 steps; bo: the O-term B steps (Q4_K-like), one a block; scl:
// activation scales [16][nbq]; vals: block values [cpc][nb][128] (row
// fastest); slab: the rows' blocks as landed, [nbq][128][block bytes] (a
// block's 144 or 208 bytes are an odd number of 16-B units, so eight
// consecutive rows' 16-B loads hit eight bank groups); dreg (Q6_K-like): each
// row's 64 bytes of the d plane.
__host__ __device__ inline TcSmem tc_smem(int F, int nb, int nbq, int cpc) {
    TcSmem s;
    s.bars = 0;
    s.tptr = 8 * (8 + nbq);
    s.bact = (s.tptr + 4 + 127) & ~127;
    s.bo = s.bact + nbq * 16 * 512;
    s.scl = s.bo + (F == kQ4K ? nbq * 512 : 0);
    s.vals = s.scl + ((16 * nbq * 4 + 127) & ~127);
    s.slab = s.vals + ((cpc * nb * kTcRows * 4 + 127) & ~127);
    s.dreg = s.slab + nbq * kTcRows * (F == kQ4K ? 144 : 208);
    s.total = s.dreg + (F == kQ6K ? kTcRows * 64 : 0);
    return s;
}

// tensor-memory columns
constexpr uint32_t kTcA = 0;         // A buffers: 0 and 128 (128 columns each)
constexpr uint32_t kTcAO = 256;      // Q4_K-like O-term A buffers: 256 and 264
constexpr uint32_t kTcD4 = 288;      // Q4_K-like accumulators: C half 0, C half 1, O (16 each) at 288 and 352
constexpr uint32_t kTcD6 = 256;      // Q6_K-like accumulators: hi, lo (16 each) at 256 and 320

// The B operand of k step T (16 k x 16 columns): core matrix (column group g,
// k group kg) at T*512 + kg*256 + g*128, column n's 8 k values at + (n%8)*16.
__device__ __forceinline__ uint32_t tc_b_off(int T, int kg, int n) {
    return (uint32_t)(T * 512 + kg * 256 + (n >> 3) * 128 + (n & 7) * 16);
}

__device__ __forceinline__ uint32_t tc_hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ void tc_ld4(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t (&a)[4], uint32_t (&b)[4],
                                       uint32_t (&c)[4]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%12];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4, %5, %6, %7}, [%13];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8, %9, %10, %11}, [%14];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]),
          "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3])
        : "r"(t0), "r"(t1), "r"(t2)
        : "memory");
}

// Waits for phase `parity` of `bar`, the thread suspended in hardware between
// checks (no spinning issue slots), for at most ~`limit_cycles` SM cycles;
// false (and the device fault word raised) if the wait ran out.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, int *fault,
                                                long long limit_cycles = 4000000000LL) {
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > limit_cycles) {
            atomicOr(fault, kFaultMbarTimeout);
            return false;
        }
    }
}
// One lane of the converged warp (the others false): tcgen05 instructions
// issued under it keep the warp's operands uniform.
__device__ __forceinline__ bool elect_one() {
    uint32_t e;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(e));
    return e != 0;
}

// Roles: warps 0-7 decode weights into tensor memory (two threads a row),
// warps 8-15 combine and send block values (two threads a row, eight columns
// each), warp 16 stages the rows (bulk copies), owns the tensor memory and
// issues the MMAs from one lane.  They meet at mbarriers only:
//   full[jb]   the slab's block jb has landed          (bulk copies -> decoders)
//   afull[s]   stage buffer s is decoded              (8 decoder warps -> MMA)
//   mdone[s]   the MMAs reading stage buffer s are done (commit -> decoders)
//   dfull[t]   accumulator t holds a finished block    (commit -> combiners)
//   dempty[t]  accumulator t has been read             (8 combiner warps -> MMA)
__device__ __forceinline__ void st_cluster_f32_nc(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v));
}

// Roles: warps 0-7 decode weights into tensor memory (two threads a row),
// warps 8-15 combine and send block values (two threads a row, eight columns
// each), warp 16 stages the blocks (tensor-map copies), owns the tensor
// memory and issues the MMAs from one lane.  They meet at mbarriers only:
//   full[jb]   block jb of the tile's rows has landed      (copies -> decoders, combiners)
//   afull[s]   stage buffer s is decoded                   (8 decoder warps -> MMA)
//   mdone[s]   the MMAs reading stage buffer s are done    (commit -> decoders)
//   dfull[t]   accumulator t holds a finished block        (commit -> combiners)
//   dempty[t]  accumulator t has been read                 (8 combiner warps -> MMA)
template <int F>
__global__ void __launch_bounds__(kTcThreads, 1) tc_kernel(const __grid_constant__ TcK p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const TcSmem Lo = tc_smem(F, p.nb, p.nbq, p.cpc);
    // the warp index through a broadcast, so the compiler sees it (and the
    // tensor-memory addresses made from it) as uniform across the warp
    const int tid = threadIdx.x, lane = tid & 31, w = __shfl_sync(0xFFFFFFFFu, tid >> 5, 0);
    uint64_t *afull = reinterpret_cast<uint64_t *>(smem + Lo.bars);  // [2]
    uint64_t *mdone = afull + 2;                                      // [2]
    uint64_t *dfull = afull + 4;                                      // [2]
    uint64_t *dempty = afull + 6;                                     // [2]
    uint64_t *full = afull + 8;                                       // [nbq]
    uint32_t *tptr = reinterpret_cast<uint32_t *>(smem + Lo.tptr);
    uint8_t *bact = smem + Lo.bact;
    uint8_t *bo = smem + Lo.bo;
    uint32_t *scl = reinterpret_cast<uint32_t *>(smem + Lo.scl);
    float *vals = reinterpret_cast<float *>(smem + Lo.vals);
    uint8_t *slab = smem + Lo.slab;

    const int q = blockIdx.x;  // rank in the cluster
    const int64_t tile = blockIdx.y;
    int mi = 0;  // the matrix this tile belongs to
#pragma unroll
    for (int i = 1; i < kMaxMats; ++i) mi = (i < p.mt.n && tile >= p.tstart[i]) ? i : mi;
    const int64_t mrows = p.mt.start[mi + 1] - p.mt.start[mi];
    const int64_t row0 = (tile - p.tstart[mi]) * kTcRows;  // within matrix mi
    const int count = (int)min((int64_t)kTcRows, mrows - row0);
    const int b0 = q * p.nb / p.KS, b1 = (q + 1) * p.nb / p.KS, nbq = b1 - b0;
    const int c0 = q * p.ncols / p.KS, c1 = (q + 1) * p.ncols / p.KS;  // the columns this CTA folds
    constexpr int BB = F == kQ4K ? 144 : 208;                          // bytes of a block
    const int dlo = (2 * b0) & ~15;  // Q6_K-like: where my blocks' d values start in the d plane (16-B aligned)

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(afull + i, 8);
            mbar_init(mdone + i, 1);
            mbar_init(dfull + i, 1);
            mbar_init(dempty + i, 16);
        }
        for (int jb = 0; jb < nbq; ++jb) mbar_init(full + jb, 1);
        fence_mbar_init();
        // the tile's blocks, one box each (rows past the matrix read as zero; weights depend on no earlier kernel)
        for (int jb = 0; jb < nbq; ++jb) {
            mbar_arrive_expect_tx(full + jb, (uint32_t)(kTcRows * BB + (F == kQ6K && jb == 0 ? kTcRows * 64 : 0)));
            if (F == kQ6K && jb == 0) tma_box_2d(smem + Lo.dreg, &p.dmap[mi], 208 * p.nb + dlo, (int)row0, full);
            tma_box_2d(slab + jb * kTcRows * BB, &p.tmap[mi], BB * (b0 + jb), (int)row0, full + jb);
        }
    }
    cluster_arrive_relaxed();  // every CTA of the cluster has started (waited on before the first remote store)
    pdl_launch_dependents();
    pdl_wait();
    __syncthreads();  // the mbarriers are initialised
    if (w == 24) {
        tc_alloc(tptr, 512);
        tc_relinquish();
    }

    // ---- B: the activation codes of my blocks as f16, in the MMA's k order
    {
        const int units = nbq * 16 * 32;  // (k step, k group, column)
        constexpr int UN = 4;
        for (int u0 = tid; u0 < units; u0 += UN * kTcThreads) {
            uint2 cw[UN];
#pragma unroll
            for (int k = 0; k < UN; ++k) {  // the loads first
                const int u = u0 + k * kTcThreads;
                const int n = (u & 7) | (((u >> 4) & 1) << 3), kg = (u >> 3) & 1, T = u >> 5;
                const int64_t e0 = 256 * (int64_t)(b0 + (T >> 4)) + 32 * ((T & 15) >> 1) + 16 * (T & 1) + 8 * kg;
                cw[k] = (u < units && n < p.ncols) ? *reinterpret_cast<const uint2 *>(p.codes + (int64_t)n * p.K + e0)
                                                   : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < UN; ++k) {
                const int u = u0 + k * kTcThreads;
                if (u >= units) break;
                const int n = (u & 7) | (((u >> 4) & 1) << 3), kg = (u >> 3) & 1, T = u >> 5;
                const uint32_t w0 = cw[k].x ^ 0x80808080u, w1 = cw[k].y ^ 0x80808080u;
                constexpr uint32_t M1152 = 0xE480E480u;  // (-1152, -1152): 0x64xx is 1024 + xx
                uint4 o;
                o.x = tc_hadd2(tc_prmt(w0, 0x64646464u, 0x4240u), M1152);
                o.y = tc_hadd2(tc_prmt(w0, 0x64646464u, 0x4341u), M1152);
                o.z = tc_hadd2(tc_prmt(w1, 0x64646464u, 0x4240u), M1152);
                o.w = tc_hadd2(tc_prmt(w1, 0x64646464u, 0x4341u), M1152);
                *reinterpret_cast<uint4 *>(bact + tc_b_off(T, kg, n)) = o;
            }
        }
        // the O-term B (Q4_K-like): k 0..7 = S_s mod 64, k 8..15 = 64*floor(S_s/64)
        if (F == kQ4K)
            for (int u = tid; u < nbq * 16; u += kTcThreads) {
                const int n = u & 15, jb = u >> 4;
                uint32_t lo[4] = {0, 0, 0, 0}, hi[4] = {0, 0, 0, 0};
                if (n < p.ncols) {
                    const uint4 *sp = reinterpret_cast<const uint4 *>(p.sums16 + (int64_t)n * (p.K / 16) + 16 * (b0 + jb));
                    const uint4 sa = sp[0], sb = sp[1];
                    const uint32_t sw[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
                    int S[8];
#pragma unroll
                    for (int s = 0; s < 8; ++s) S[s] = (int)(int16_t)(sw[s] & 0xFFFFu) + (int)(int16_t)(sw[s] >> 16);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        lo[i] = tc_pack2((float)(S[2 * i] & 63), (float)(S[2 * i + 1] & 63));
                        hi[i] = tc_pack2((float)(64 * (S[2 * i] >> 6)), (float)(64 * (S[2 * i + 1] >> 6)));
                    }
                }
                *reinterpret_cast<uint4 *>(bo + tc_b_off(jb, 0, n)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4 *>(bo + tc_b_off(jb, 1, n)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
        for (int u = tid; u < 16 * nbq; u += kTcThreads) {
            const int n = u / nbq, jb = u - n * nbq;
            scl[u] = n < p.ncols ? reinterpret_cast<const uint32_t *>(p.scales)[(int64_t)n * p.nb + b0 + jb] : 0u;
        }
    }
    fence_proxy_async_smem();  // the generic-proxy writes of B, seen by the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = __shfl_sync(0xFFFFFFFFu, *tptr, 0);  // (uniform, as above)
    const int S = F == kQ4K ? nbq : 2 * nbq;  // stages: a block (Q4_K-like) or a half block (Q6_K-like)

    if (w < 8) {
        // ---- decoders: stage j's weights into A buffer j&1
        const int qw = w & 3, h = w >> 2, r = 32 * qw + lane;
        const uint32_t tl = tb + ((uint32_t)(32 * qw) << 16);
        for (int j = 0; j < S; ++j) {
            const int jb = F == kQ4K ? j : j >> 1;
            mbar_wait_sleep(full + jb, 0, p.fault);  // a timeout raises the fault word (the values are then garbage)
            if (j >= 2) mbar_wait_sleep(mdone + (j & 1), ((j - 2) >> 1) & 1, p.fault);  // stage j-2's MMAs read it
            const uint32_t ab = tl + kTcA + 128u * (j & 1);
            const uint8_t *blk = slab + (jb * kTcRows + r) * BB;
            if (F == kQ4K) {
                const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
                uint4 qv[4];
#pragma unroll
                for (int ss = 0; ss < 4; ++ss) qv[ss] = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * (4 * h + ss));
                const unsigned long long sc48 =
                    (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
                const uint32_t scp = (uint32_t)(sc48 >> (24 * h));  // my four sub-blocks' fields
#pragma unroll
                for (int ss = 0; ss < 4; ++ss) {
                    const uint32_t sc = (scp >> (6 * ss)) & 63u;
                    const uint32_t klo = tc_hadd2(sc * 0x10001u + 0x64006400u, 0xE400E400u);  // (sc, sc)
                    const uint32_t nlo = tc_hmul2(klo, 0xE400E400u);                           // -1024 sc
                    const uint32_t khi = tc_hmul2(klo, 0x2C002C00u);                           // sc / 16
                    const uint32_t nhi = tc_hmul2(klo, 0xD400D400u);                           // -64 sc
                    const uint32_t wv[4] = {qv[ss].x, qv[ss].y, qv[ss].z, qv[ss].w};
                    uint32_t v[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t x = wv[i], x8 = wv[i] >> 8;
                        v[2 * i] = tc_hfma2((x & 0x000F000Fu) | 0x64006400u, klo, nlo);
                        v[2 * i + 1] = tc_hfma2((x8 & 0x000F000Fu) | 0x64006400u, klo, nlo);
                        v[8 + 2 * i] = tc_hfma2((x & 0x00F000F0u) | 0x64006400u, khi, nhi);
                        v[8 + 2 * i + 1] = tc_hfma2((x8 & 0x00F000F0u) | 0x64006400u, khi, nhi);
                    }
                    tc_st16(ab + 16 * (4 * h + ss), v);  // k steps 2s (low nibbles) and 2s+1 (high)
                }
                if (h == 0) {
                    const unsigned long long mn48 =
                        (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
                    uint32_t ao[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t pr = (uint32_t)((mn48 >> (12 * i)) & 63u) |
                                            ((uint32_t)((mn48 >> (12 * i + 6)) & 63u) << 16);
                        ao[i] = ao[i + 4] = tc_hadd2(pr | 0x64006400u, 0xE400E400u);  // (mn, mn') exactly
                    }
                    tc_st8(tl + kTcAO + 8u * (j & 1), ao);
                }
            } else {
                uint4 ql[2];
                uint2 hb[2];
                uint32_t scp[2];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 4 * (j & 1) + 2 * h + cc;  // 32-element chunk: units 2c, 2c+1
                    ql[cc] = *reinterpret_cast<const uint4 *>(blk + 16 * c);
                    hb[cc] = *reinterpret_cast<const uint2 *>(blk + 128 + 8 * c);
                    scp[cc] = *reinterpret_cast<const uint16_t *>(blk + 192 + 2 * c);
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const uint32_t wl[4] = {ql[cc].x, ql[cc].y, ql[cc].z, ql[cc].w};
#pragma unroll
                    for (int uu = 0; uu < 2; ++uu) {
                        const int sc = (int)(int8_t)((scp[cc] >> (8 * uu)) & 0xFFu);
                        const uint32_t sh8 = (uint32_t)((sc >> 4) + 8), sl = (uint32_t)(sc & 15);
                        const uint32_t kh = tc_hadd2(sh8 * 0x10001u + 0x64006400u, 0xE408E408u);  // (hi, hi): hi in -8..7
                        const uint32_t nh = tc_hmul2(kh, 0xE420E420u);                             // -1056 hi
                        const uint32_t kl = tc_hadd2(sl * 0x10001u + 0x64006400u, 0xE400E400u);   // (lo, lo)
                        const uint32_t nl = tc_hmul2(kl, 0xE420E420u);                             // -1056 lo
                        const uint32_t hw = uu ? hb[cc].y : hb[cc].x;
                        uint32_t vh[8], vl[8];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint32_t hi2 = (i < 3) ? (hw << (4 - 2 * i)) : (hw >> 2);
                            const uint32_t qb = ((uu ? (wl[i] >> 4) : wl[i]) & 0x0F0F0F0Fu) | (hi2 & 0x30303030u);
                            const uint32_t x02 = tc_prmt(qb, 0x64646464u, 0x4240u);  // (1024 + q0, 1024 + q2)
                            const uint32_t x13 = tc_prmt(qb, 0x64646464u, 0x4341u);
                            vh[2 * i] = tc_hfma2(x02, kh, nh);
                            vh[2 * i + 1] = tc_hfma2(x13, kh, nh);
                            vl[2 * i] = tc_hfma2(x02, kl, nl);
                            vl[2 * i + 1] = tc_hfma2(x13, kl, nl);
                        }
                        const int ui = 4 * h + 2 * cc + uu;  // unit within the stage
                        tc_st8(ab + 8 * ui, vh);
                        tc_st8(ab + 64 + 8 * ui, vl);
                    }
                }
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(afull + (j & 1));
        }
    } else if (w < 24) {
        // ---- combiners: block jb's accumulators -> values -> the CTAs that fold them
        const int qw = w & 3, h = (w - 8) >> 2, r = 32 * qw + lane;  // four threads a row, four columns each
        const uint32_t tl = tb + ((uint32_t)(32 * qw) << 16);
        const bool live = r < count;
        uint32_t rb[4];  // where my columns' values go
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = min(4 * h + i, p.ncols - 1);
            const int owner = ((n + 1) * p.KS - 1) / p.ncols;
            const int nl = n - owner * p.ncols / p.KS;
            rb[i] = cluster_map(smem_u32(vals + ((int64_t)nl * p.nb * kTcRows + r)), (uint32_t)owner);
        }
        cluster_wait();
        for (int jb = 0; jb < nbq; ++jb) {
            mbar_wait_sleep(dfull + (jb & 1), (jb >> 1) & 1, p.fault);
            mbar_wait_sleep(full + jb, 0, p.fault);  // (done long ago: makes the staged scales visible here)
            tc_fence_after();
            uint32_t x0[4], x1[4], x2[4];
            const uint32_t D = tl + (F == kQ4K ? kTcD4 : kTcD6) + 64u * (jb & 1) + 4u * h;
            tc_ld4(D, D + 16u, F == kQ4K ? D + 32u : D, x0, x1, x2);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty + (jb & 1));
            const int bg = b0 + jb;
            const uint32_t dd = F == kQ4K ? *reinterpret_cast<const uint32_t *>(slab + (jb * kTcRows + r) * 144)
                                          : *reinterpret_cast<const uint16_t *>(smem + Lo.dreg + r * 64 + 2 * bg - dlo);
            // the block's activation scales: exponent range and whether every column has one (warp-wide)
            const uint32_t ms = scl[min(lane, p.ncols - 1) * nbq + jb];
            const int me = (int)(int16_t)(ms >> 16);
            const int emin = __reduce_min_sync(0xFFFFFFFFu, me), emax = __reduce_max_sync(0xFFFFFFFFu, me);
            const bool allm = __all_sync(0xFFFFFFFFu, (ms & 0xFFu) != 0u);
            uint32_t sv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) sv[i] = scl[min(4 * h + i, 15) * nbq + jb];
            const TcScales ts = tc_scales<F>(dd);
            // every value of this (row, block) is a normal number after the scaling below when:
            const bool blk_fast = ts.fast && allm && ts.Eb >= -126 && emin >= -126 && emax <= 127 &&
                                  ts.Eb + emin >= -126 && ts.Eb + emax <= 82;
            const float pEb = __int_as_float((min(max(ts.Eb, -126), 127) + 127) << 23);
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                int C, O = 0;
                if (F == kQ4K) {
                    C = __float2int_rn(__uint_as_float(x0[i])) + __float2int_rn(__uint_as_float(x1[i]));
                    O = __float_as_int(__uint_as_float(x2[i]) + 12582912.0f) - 0x4B400000;  // |O| < 2^22
                } else {
                    C = 16 * __float2int_rn(__uint_as_float(x0[i])) + __float2int_rn(__uint_as_float(x1[i]));
                }
                v[i] = tc_value2<F>(C, O, dd, ts, sv[i], blk_fast, pEb);
            }
            if (live) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (4 * h + i < p.ncols) st_cluster_f32_nc(rb[i] + (uint32_t)bg * (kTcRows * 4), v[i]);
            }
        }
    } else {
        // ---- the MMA issuer: the whole warp waits and stays converged; one
        // elected lane issues each MMA and commit
        const uint32_t sb = smem_u32(bact);
        for (int j = 0; j < S; ++j) {
            const int jb = F == kQ4K ? j : j >> 1;
            mbar_wait_sleep(afull + (j & 1), (j >> 1) & 1, p.fault);
            if (jb >= 2 && (F == kQ4K || (j & 1) == 0))  // the accumulator's previous block has been read
                mbar_wait_sleep(dempty + (jb & 1), ((jb - 2) >> 1) & 1, p.fault);
            __syncwarp();
            tc_fence_after();
            const uint32_t A = tb + kTcA + 128u * (j & 1);
            if (F == kQ4K) {
                const uint32_t D = tb + kTcD4 + 64u * (jb & 1);
#pragma unroll
                for (int tt = 0; tt < 16; ++tt) {
                    if (elect_one())
                        tc_mma_ts(D + (tt >= 8 ? 16u : 0u), A + 8u * tt,
                                  tc_desc(sb + (uint32_t)(jb * 16 + tt) * 512u, 256, 128), kTcIdesc, (tt & 7) != 0);
                    __syncwarp();
                }
                if (elect_one())
                    tc_mma_ts(D + 32u, tb + kTcAO + 8u * (j & 1),
                              tc_desc(smem_u32(bo) + (uint32_t)jb * 512u, 256, 128), kTcIdesc, 0u);
                __syncwarp();
            } else {
                const int hh = j & 1;
                const uint32_t D = tb + kTcD6 + 64u * (jb & 1);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int u = 8 * hh + i;
                    const uint64_t bd = tc_desc(sb + (uint32_t)(jb * 16 + u) * 512u, 256, 128);
                    if (elect_one()) tc_mma_ts(D, A + 8u * i, bd, kTcIdesc, u != 0);
                    __syncwarp();
                    if (elect_one()) tc_mma_ts(D + 16u, A + 64u + 8u * i, bd, kTcIdesc, u != 0);
                    __syncwarp();
                }
            }
            if (elect_one()) {
                tc_commit(mdone + (j & 1));
                if (F == kQ4K || (j & 1)) tc_commit(dfull + (jb & 1));
            }
            __syncwarp();
        }
    }
    if (w < 8 || w == 24) cluster_wait();  // (the combiners waited before their first remote store)
    // every tensor-memory access done: free it; every value delivered: fold
    tc_fence_before();
    __syncthreads();
    if (w == 24) tc_dealloc(tb, 512);
    cluster_arrive();
    cluster_wait();
    const int nown = c1 - c0;
    float *outm = p.mt.out[mi];
    for (int pi = tid; pi < nown * kTcRows; pi += kTcThreads) {
        const int nl = pi >> 7, rr = pi & 127;
        if (rr >= count) continue;
        const float *vr = vals + (int64_t)nl * p.nb * kTcRows + rr;
        float acc = 0.0f;
        for (int b = 0; b < p.nb; ++b) acc = fadd_ftz(acc, vr[b * kTcRows]);
        if (acc != acc) acc = __uint_as_float(kEngineNaN);
        outm[(int64_t)(c0 + nl) * mrows + row0 + rr] = acc;
    }
}

// CTAs of cluster size ks that run at once on this device (cached per device and size).
template <int F>
inline int tc_active_ctas(int ks, int smem) {
    static std::atomic<int> cache[kMaxDevices][kTcMaxKS + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int v = cache[dev][ks].load(std::memory_order_relaxed);
    if (v) return v;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ks, 64);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, tc_kernel<F>, &cfg) != cudaSuccess || nc <= 0) {
        (void)cudaGetLastError();
        nc = std::max(1, num_sms() / ks / 2);
    }
    v = nc * ks;
    cache[dev][ks].store(v, std::memory_order_relaxed);
    return v;
}

// The Q4_K-like / Q6_K-like product of 1..16 columns on the tensor cores;
// QB_E_ARG where it does not take the shape (the caller then uses another kernel).
template <int F>
int launch_tc(const GemvArgs &a, cudaStream_t stream) {
    if ((F != kQ4K && F != kQ6K) || a.mode != 0 || a.ncols < 1 || a.ncols > 16 || a.K < 256 || a.K % 256 != 0 ||
        reinterpret_cast<uintptr_t>(a.codes) % 8 != 0 || reinterpret_cast<uintptr_t>(a.scales) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(a.sums16) % 16 != 0)
        return QB_E_ARG;
    TcK k;
    memset(&k, 0, sizeof(k));
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.K = (int)a.K;
    k.nb = (int)(a.K / 256);
    k.rec = (int)record_bytes(F, a.K);
    k.ncols = a.ncols;
    int64_t tiles = 0;
    for (int i = 0; i < k.mt.n; ++i) {
        const int64_t ri = k.mt.start[i + 1] - k.mt.start[i];
        k.tstart[i] = tiles;
        if (ri > 0 && (reinterpret_cast<uintptr_t>(k.mt.W[i]) % 16 != 0 || ri > (int64_t(1) << 31))) return QB_E_ARG;
        if (ri > 0 && !tmap_rows(&k.tmap[i], k.mt.W[i], ri, k.rec, F == kQ4K ? 144 : 208, kTcRows)) return QB_E_ARG;
        if (ri > 0 && F == kQ6K && !tmap_rows(&k.dmap[i], k.mt.W[i], ri, k.rec, 64, kTcRows)) return QB_E_ARG;
        tiles += (ri + kTcRows - 1) / kTcRows;
    }
    for (int i = k.mt.n; i <= kMaxMats; ++i) k.tstart[i] = tiles;
    if (tiles < 1 || tiles > 65535) return QB_E_ARG;
    const int budget = 227 * 1024;
    if (ensure_smem_limit(reinterpret_cast<const void *>(tc_kernel<F>), budget) != QB_OK) return QB_E_CUDA;
    // the cluster size: the least estimated time (waves x blocks a CTA), fewer CTAs on a tie
    int best = 0;
    long long best_cost = 0;
    for (int ks = 1; ks <= std::min(kTcMaxKS, k.nb); ++ks) {
        const int nbq = (k.nb + ks - 1) / ks, cpc = (k.ncols + ks - 1) / ks;
        if (tc_smem(F, k.nb, nbq, cpc).total > budget) continue;
        if (F == kQ6K && 2 * nbq + 14 > 64) continue;  // a CTA's d values within its 64-byte box
        const int act = tc_active_ctas<F>(ks, budget);
        if (act < ks) continue;
        const long long waves = (tiles * ks + act - 1) / act;
        const long long cost = waves * nbq;
        if (!best || cost < best_cost) {
            best = ks;
            best_cost = cost;
        }
    }
    if (!best) return QB_E_ARG;
    k.KS = best;
    k.nbq = (k.nb + best - 1) / best;
    k.cpc = (k.ncols + best - 1) / best;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    const int smem = std::max(tc_smem(F, k.nb, k.nbq, k.cpc).total, kTcMinSmem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(best, (unsigned)tiles);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = best;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_kernel<F>, k) == cudaSuccess ? QB_OK : QB_E_CUDA;
}

}  // namespace qb
