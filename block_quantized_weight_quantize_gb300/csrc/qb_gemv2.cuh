// qb_gemv2.cuh -- the streaming product kernel (one activation column).
//
// Same arithmetic as qb_gemv.cuh (the decode engine's dot under PerBlock:
// exact block sums, exact two-term combine, one rounding per block, in-order
// row fold), organised for throughput on a weight stream:
//   * persistent CTAs of "teams": a team of K/128 threads covers one row, and
//     thread j of a team owns the 128-element half-slice j of K in every row
//     the team visits.  Its activation codes (32 registers), unit sums and
//     scale are loaded once per launch;
//   * a team takes two rows per iteration.  For 256-element blocks the two
//     threads of a block each form partial sums for both rows, swap one pair
//     of partials, and each finishes one row's block -- one exact combine per
//     thread per iteration, none duplicated;
//   * rows reach shared memory through a ring of D slots (two row records per
//     team), filled by bulk asynchronous copies (the TMA engine) completing on
//     the slot's mbarrier.  The first D fills are issued before the
//     programmatic-dependent-launch wait, so a launch streams its weights
//     while the previous kernel finishes;
//   * CTA c owns a contiguous range of rows (the ranges differ by at most one
//     row), so each ring slot fills with a single bulk copy;
//   * the rounded block values of H iterations are kept in shared memory and
//     folded in block order from +0 (f32 round-to-nearest-even, ftz) by one
//     thread per row, with vector loads.
// Shared-memory reads are conflict-free: consecutive threads read blocks at
// strides that are odd multiples of 16 B (Q4_K 144 B, Q6_K 208 B), and the
// activation and the Q8_0 codes are visited in a per-thread XOR order.
#pragma once

#include <algorithm>
#include <type_traits>

#include "qb_common.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"
#include "qb_quant.cuh"

namespace qb {

struct Gemv2K {
    const uint8_t *W;  // the matrix (one-matrix launches)
    int64_t rows;      // rows of the whole range
    int K;
    int rec;       // bytes per row record
    int nt;        // teams per CTA
    int ts;        // threads per team = K / 128
    int D;         // ring slots
    int H;         // iterations of block values kept before a fold
    int nb;        // weight blocks per row
    int vstride;   // floats per row line of block values (an odd number of 16-B units)
    int n_iter;    // iterations (two rows per team each)
    int wfold;     // one iteration and whole teams per warp: each warp folds its own rows
    int64_t base;  // rows per CTA, and how many CTAs own one more
    int64_t rem;
    const int8_t *codes;
    const qb_scale *scales;
    const int16_t *sums16;
    const float *x;  // single-launch form: the f32 activation, quantized in the kernel
    float *out;      // one-matrix launches
    int *fault;
};
// A launch over several matrices sharing the activation: the same fields and
// the matrix table (W and out unused).
struct Gemv2KM : Gemv2K {
    MatTable mt;
};

struct Gemv2Smem {
    int bars, act, scl, sums, val, ring, total;
};

__host__ __device__ inline Gemv2Smem gemv2_smem(int K, int rec, int nt, int D, int H, int vstride) {
    Gemv2Smem s;
    s.bars = 0;                                            // D mbarriers
    s.act = 128;                                           // K activation codes
    s.scl = s.act + ((K + 127) & ~127);                    // up to K/32 activation scales
    s.sums = s.scl + ((K / 32 * 4 + 127) & ~127);          // K/16 unit sums (single-launch form)
    s.val = s.sums + ((K / 16 * 2 + 127) & ~127);          // H * nt * 2 rows of block values
    s.ring = s.val + ((H * nt * 2 * vstride * 4 + 127) & ~127);
    s.total = s.ring + D * nt * 2 * rec;
    return s;
}

// lane (block-scale lane page): the block's value rounded once.  Fast path:
// the exact integer n*2^E with n in 64 bits is rounded by the hardware's
// round-to-nearest-even int64 -> f32 conversion, then scaled by 2^E through
// the exponent field, which is exact while the result stays a normal f32;
// any other case (zero, a subnormal or infinite result) goes to the exact
// integer routine round_to_f32.  (That conversion issues at 2 a clock per SM
// on this part, but it overlaps other issue: an equivalent built from 32-bit
// operations measured slower.)
static __device__ __noinline__ float round_to_f32_cold(long long n, int E) { return round_to_f32(n, E); }

__device__ __forceinline__ float round_fast(long long n, int E) {
    const float f = __ll2float_rn(n);
    const uint32_t b = __float_as_uint(f);
    const int ex = (int)((b >> 23) & 0xFFu) + E;
    if (n != 0 && ex >= 1 && ex <= 254) return __uint_as_float(b + ((uint32_t)E << 23));
    return round_to_f32_cold(n, E);  // out of line: rare
}

// The two terms of a block whose scale exponents lie more than 17 (or 21)
// places apart: combined in 128 bits.  Out of line: rare.
static __device__ __noinline__ float lane_value_spread(long long t1, long long t2, int d, int ex1, int ex2, int e) {
    const __int128 w = d >= 0 ? ((__int128)t1 << d) + t2 : (__int128)t1 + ((__int128)t2 << (-d));
    return round_to_f32_wide(w, (d >= 0 ? ex2 : ex1) + e);
}

template <int KIND>
__device__ __forceinline__ float lane_value_fast(int C, int O, uint32_t s1, uint32_t s2, int m, int e) {
    int sig1, ex1;
    bool ok = f16_scale(s1, sig1, ex1) && m != 0;
    if (KIND == 0) {
        if (!ok) return __uint_as_float(kEngineNaN);
        return round_fast((long long)(sig1 * m) * (long long)C, ex1 + e);
    } else {
        int sig2, ex2;
        ok = f16_scale(s2, sig2, ex2) && ok;
        if (!ok) return __uint_as_float(kEngineNaN);
        const long long t1 = (long long)(sig1 * m) * (long long)C;   // |t1| < 2^44
        const long long t2 = -(long long)(sig2 * m) * (long long)O;  // |t2| < 2^40
        const int d = ex1 - ex2;
        if (d > 17 || d < -21) return lane_value_spread(t1, t2, d, ex1, ex2, e);
        // the term of the larger exponent shifted up to the other's: no branch
        // on the sign of d, whose lanes (rows) would otherwise take both forms
        const int sh1 = d > 0 ? d : 0, sh2 = d < 0 ? -d : 0;
        return round_fast((t1 << sh1) + (t2 << sh2), (d >= 0 ? ex2 : ex1) + e);
    }
}

// ------------------------------------------------------------------ half-slice sums
// a[k] holds activation 16-B unit 8j+k of the thread's half-slice j (elements
// 128j + 16k .. +15).

// Q4_K-like half block h of the block at blk: sub-blocks 4h..4h+3.  C is
// returned as 16*C: per sub-block 16*(sum lo*a) + (sum 16*hi*a) in one
// multiply-add (|16*C| <= 16 * 63 * 15 * 127 * 256 < 2^31 over a whole
// block).  O = sum mn_s * S_s by two dp2a over the packed 16-bit sub-block
// sums S01, S23 and the four mn fields spread to bytes.
__device__ __forceinline__ void half_q4k(const uint8_t *blk, int h, const uint4 (&a)[8], uint32_t S01, uint32_t S23,
                                         int &C16, int &O, uint32_t &dd) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    dd = meta.x;
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
    const uint32_t scm = (uint32_t)(sc48 >> (24 * h)), mnm = (uint32_t)(mn48 >> (24 * h));  // my four fields
    const uint8_t *qs = blk + 16 + 64 * h;
    int c = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint4 w = *reinterpret_cast<const uint4 *>(qs + 16 * s);
        int pl = dp4a_ss(w.x & 0x0F0F0F0Fu, a[2 * s].x, 0);
        pl = dp4a_ss(w.y & 0x0F0F0F0Fu, a[2 * s].y, pl);
        pl = dp4a_ss(w.z & 0x0F0F0F0Fu, a[2 * s].z, pl);
        pl = dp4a_ss(w.w & 0x0F0F0F0Fu, a[2 * s].w, pl);
        int ph = dp4a_us(w.x & 0xF0F0F0F0u, a[2 * s + 1].x, 0);  // 16*q against a: a multiple of 16
        ph = dp4a_us(w.y & 0xF0F0F0F0u, a[2 * s + 1].y, ph);
        ph = dp4a_us(w.z & 0xF0F0F0F0u, a[2 * s + 1].z, ph);
        ph = dp4a_us(w.w & 0xF0F0F0F0u, a[2 * s + 1].w, ph);
        c += (int)((scm >> (6 * s)) & 63u) * (16 * pl + ph);
    }
    const uint32_t mnb = spread6(mnm);
    C16 = c;
    O = dp2a_hi_su(S23, mnb, dp2a_lo_su(S01, mnb, 0));
}

// Q6_K-like half block h: 32-element chunks 4h..4h+3 (units 8h..8h+7).
__device__ __forceinline__ int half_q6k(const uint8_t *blk, int h, const uint4 (&a)[8], const uint32_t (&S)[4]) {
    const uint2 scw = *reinterpret_cast<const uint2 *>(blk + 192 + 8 * h);  // sc of my eight units
    int c = 0;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 64 * h + 16 * ch);
        const uint2 hb = *reinterpret_cast<const uint2 *>(blk + 128 + 32 * h + 8 * ch);
        const uint32_t wl[4] = {w.x, w.y, w.z, w.w};
        const uint32_t al[4] = {a[2 * ch].x, a[2 * ch].y, a[2 * ch].z, a[2 * ch].w};
        const uint32_t ah[4] = {a[2 * ch + 1].x, a[2 * ch + 1].y, a[2 * ch + 1].z, a[2 * ch + 1].w};
        int pl = 0, ph = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t hl = (k < 3) ? (hb.x << (4 - 2 * k)) : (hb.x >> 2);
            const uint32_t hh = (k < 3) ? (hb.y << (4 - 2 * k)) : (hb.y >> 2);
            pl = dp4a_ss((wl[k] & 0x0F0F0F0Fu) | (hl & 0x30303030u), al[k], pl);
            ph = dp4a_ss(((wl[k] >> 4) & 0x0F0F0F0Fu) | (hh & 0x30303030u), ah[k], ph);
        }
        const uint32_t sw = (ch < 2) ? scw.x : scw.y;
        const int sc_lo = (int)(int8_t)((sw >> (16 * (ch & 1))) & 0xFFu);
        const int sc_hi = (int)(int8_t)((sw >> (16 * (ch & 1) + 8)) & 0xFFu);
        // sum over a unit of (q - 32) * a = sum q*a - 32 * S_u
        c += sc_lo * (pl - 32 * (int)(int16_t)(S[ch] & 0xFFFFu)) + sc_hi * (ph - 32 * (int)(int16_t)(S[ch] >> 16));
    }
    return c;
}

// Q8_0 half-slice: four blocks of 32; the thread visits its eight 16-B units in
// the order k ^ jj (a[k] holds activation unit k ^ jj), so eight lanes of a
// shared-memory phase hit eight banks.  vl[i] receives block i's value.
__device__ __forceinline__ void half_q8_0(const uint8_t *q, const uint8_t *dptr, const uint32_t *scl,
                                          const uint4 (&a)[8], int jj, float *vl) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int u0 = (2 * kk) ^ jj, u1 = u0 ^ 1;
        const int i = u0 >> 1;
        const uint4 w0 = *reinterpret_cast<const uint4 *>(q + 16 * u0);
        const uint4 w1 = *reinterpret_cast<const uint4 *>(q + 16 * u1);
        int p = dp4a_ss(w0.x, a[2 * kk].x, 0);
        p = dp4a_ss(w0.y, a[2 * kk].y, p);
        p = dp4a_ss(w0.z, a[2 * kk].z, p);
        p = dp4a_ss(w0.w, a[2 * kk].w, p);
        p = dp4a_ss(w1.x, a[2 * kk + 1].x, p);
        p = dp4a_ss(w1.y, a[2 * kk + 1].y, p);
        p = dp4a_ss(w1.z, a[2 * kk + 1].z, p);
        p = dp4a_ss(w1.w, a[2 * kk + 1].w, p);
        const uint32_t d = *reinterpret_cast<const uint16_t *>(dptr + 2 * i);
        const uint32_t sw = scl[i];
        vl[i] = lane_value_fast<0>(p, 0, d, 0, (int)(sw & 0xFFu), (int)(int16_t)(sw >> 16));
    }
}

// Global loads whose issue order the compiler keeps (volatile asm).
__device__ __forceinline__ uint4 ldg_v4_ordered(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ldg_f4_ordered(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u32_ordered(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// CTA c owns the contiguous rows [row0, row0 + count): the rows split as evenly
// as whole rows allow.  Iteration it covers rows row0 + 2*nt*it ... of them;
// team t takes the two consecutive rows 2t and 2t+1 of the iteration.
__device__ __forceinline__ void cta_rows(const Gemv2K &p, int64_t &row0, int64_t &count) {
    const int64_t c = blockIdx.x;
    row0 = c * p.base + (c < p.rem ? c : p.rem);
    count = p.base + (c < p.rem ? 1 : 0);
}

// Issue the fill of iteration `it` -- its rows are contiguous in memory, so
// one bulk copy -- into ring slot it % D, completing on that slot's mbarrier.
template <bool MULTI, typename P>
__device__ __forceinline__ void issue_fill(const P &p, uint8_t *ring, uint64_t *bars, int it, int64_t row0,
                                           int64_t count) {
    const int slot = it % p.D;
    const int64_t first = (int64_t)it * 2 * p.nt;
    const int64_t n = (count - first < 2 * p.nt) ? count - first : (int64_t)(2 * p.nt);
    const uint32_t bytes = n > 0 ? (uint32_t)(n * p.rec) : 0u;
    mbar_arrive_expect_tx(bars + slot, bytes);
    uint8_t *dst = ring + (int64_t)slot * 2 * p.nt * p.rec;
    if (!bytes) return;
    if constexpr (MULTI) fill_rows(p.mt, dst, row0 + first, n, p.rec, bars + slot);
    else bulk_g2s(dst, p.W + (row0 + first) * p.rec, bytes, bars + slot);
}

// Two CTAs per SM (<= 64 registers) for the product with a staged activation,
// so a following launch's CTA fits beside this one and streams its weights
// early; one (more registers, more overlap inside a warp) for the
// single-launch form, which measures faster that way.
// MULTI: several matrices through the table (mats.cuh); otherwise entry 0
// alone, with plain address arithmetic.
template <int F, bool FUSED, bool MULTI>
__global__ void __launch_bounds__(512, FUSED ? 1 : 2) gemv2_kernel(const typename std::conditional<MULTI, Gemv2KM, Gemv2K>::type p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const Gemv2Smem L = gemv2_smem(p.K, p.rec, p.nt, p.D, p.H, p.vstride);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint8_t *act = smem + L.act;
    uint32_t *ascl = reinterpret_cast<uint32_t *>(smem + L.scl);
    int16_t *asum = reinterpret_cast<int16_t *>(smem + L.sums);
    float *val = reinterpret_cast<float *>(smem + L.val);
    uint8_t *ring = smem + L.ring;

    const int tid = threadIdx.x;
    const int team = tid / p.ts, j = tid - team * p.ts;
    const bool live = team < p.nt;
    const int sb = j >> 1, h = j & 1, jj = j & 7;

    if (tid == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    int64_t row0, count;
    cta_rows(p, row0, count);
    if (tid == 0)
        for (int it = 0; it < p.D && it < p.n_iter; ++it) issue_fill<MULTI>(p, ring, bars, it, row0, count);  // no dependency
    pdl_wait();

    // ---- the activation, in one round trip: every thread first issues its
    // loads (codes units, unit sums, scale), then stores the codes to shared
    // memory (256-element formats: unit 8j+k at 8j + (k ^ (j & 7)), read back
    // in order; Q8_0: linear, read back in the XOR order).
    uint32_t S[4] = {0, 0, 0, 0};
    int m0 = 0, e0 = 0;
    if constexpr (FUSED) {
        // quantize_blocks of x in this kernel: a thread takes 8 consecutive
        // elements (a group); a block of B elements is B/8 consecutive lanes.
        // All loads first (one round trip), then the quantizer.
        constexpr int kB = fmt_block(F), kL = kB / 8, kMaxG = 4;  // groups per thread: K/8 <= 4 * blockDim
        const int G = p.K / 8;
        float4 xv[2 * kMaxG];
#pragma unroll
        for (int r = 0; r < kMaxG; ++r) {
            const int g = tid + r * (int)blockDim.x;
            const bool in = g < G;
            xv[2 * r] = in ? ldg_f4_ordered(reinterpret_cast<const float4 *>(p.x) + 2 * g) : make_float4(0, 0, 0, 0);
            xv[2 * r + 1] = in ? ldg_f4_ordered(reinterpret_cast<const float4 *>(p.x) + 2 * g + 1)
                               : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < kMaxG; ++r) {
            if (r * (int)blockDim.x >= G) break;  // uniform: whole warps are in or out (G % 32 == 0)
            const int g = tid + r * (int)blockDim.x;
            const uint32_t xb[8] = {__float_as_uint(xv[2 * r].x), __float_as_uint(xv[2 * r].y),
                                    __float_as_uint(xv[2 * r].z), __float_as_uint(xv[2 * r].w),
                                    __float_as_uint(xv[2 * r + 1].x), __float_as_uint(xv[2 * r + 1].y),
                                    __float_as_uint(xv[2 * r + 1].z), __float_as_uint(xv[2 * r + 1].w)};
            uint2 c;
            int usum;
            uint32_t scale;
            quantize8<kL>(xb, c, usum, scale);
            if (g < G) {
                const int u = g >> 1;
                const int pos = (F == kQ8_0) ? u : ((u & ~7) | ((u & 7) ^ ((u >> 3) & 7)));
                *reinterpret_cast<uint2 *>(act + 16 * pos + 8 * (g & 1)) = c;
                if ((g & 1) == 0) asum[u] = (int16_t)usum;
                if ((g & (kL - 1)) == 0) ascl[g / kL] = scale;
            }
        }
        __syncthreads();
        if (live && F != kQ8_0) {
            const uint4 sw = *reinterpret_cast<const uint4 *>(asum + 8 * j);  // my 8 unit sums
            const uint32_t pw[4] = {sw.x, sw.y, sw.z, sw.w};
            if (F == kQ4K) {
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2) {
                    const int Sv = (int)(int16_t)(pw[s2] & 0xFFFFu) + (int)(int16_t)(pw[s2] >> 16);
                    S[s2 >> 1] |= ((uint32_t)Sv & 0xFFFFu) << (16 * (s2 & 1));
                }
            } else {
                S[0] = pw[0]; S[1] = pw[1]; S[2] = pw[2]; S[3] = pw[3];
            }
            const uint32_t scl0 = ascl[sb];
            m0 = (int)(scl0 & 0xFFu);
            e0 = (int)(int16_t)(scl0 >> 16);
        }
    } else {
    constexpr int kMaxU = 8;  // staged units per thread: K/16 <= 8 * blockDim since blockDim >= K/128
    // the scale and unit sums first, then the codes; volatile loads keep this
    // order, so all of them are in flight together
    uint4 sw = make_uint4(0, 0, 0, 0);
    uint32_t scl0 = 0;
    if (live && F != kQ8_0) {
        sw = ldg_v4_ordered(reinterpret_cast<const uint4 *>(p.sums16) + j);  // my 8 unit sums
        scl0 = ldg_u32_ordered(reinterpret_cast<const uint32_t *>(p.scales) + sb);
    }
    uint32_t sq8[4] = {0, 0, 0, 0};  // Q8_0 block scales: K/32 <= 4 * blockDim
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = tid + q * (int)blockDim.x;
        if (F == kQ8_0 && b < p.K / 32) sq8[q] = ldg_u32_ordered(reinterpret_cast<const uint32_t *>(p.scales) + b);
    }
    uint4 stg[kMaxU];
#pragma unroll
    for (int q = 0; q < kMaxU; ++q) {
        const int u = tid + q * (int)blockDim.x;
        stg[q] = u < p.K / 16 ? ldg_v4_ordered(reinterpret_cast<const uint4 *>(p.codes) + u) : make_uint4(0, 0, 0, 0);
    }
    if (F == kQ4K) {  // per-32 sums of my 4 sub-blocks from the per-16 ones
        const uint32_t pw[4] = {sw.x, sw.y, sw.z, sw.w};
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) {
            const int Sv = (int)(int16_t)(pw[s2] & 0xFFFFu) + (int)(int16_t)(pw[s2] >> 16);
            S[s2 >> 1] |= ((uint32_t)Sv & 0xFFFFu) << (16 * (s2 & 1));
        }
    } else if (F == kQ6K) {  // per-16 sums of my eight units
        S[0] = sw.x; S[1] = sw.y; S[2] = sw.z; S[3] = sw.w;
    }
    m0 = (int)(scl0 & 0xFFu);
    e0 = (int)(int16_t)(scl0 >> 16);
#pragma unroll
    for (int q = 0; q < kMaxU; ++q) {
        const int u = tid + q * (int)blockDim.x;
        if (u < p.K / 16) {
            const int pos = (F == kQ8_0) ? u : ((u & ~7) | ((u & 7) ^ ((u >> 3) & 7)));
            *reinterpret_cast<uint4 *>(act + 16 * pos) = stg[q];
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = tid + q * (int)blockDim.x;
        if (F == kQ8_0 && b < p.K / 32) ascl[b] = sq8[q];
    }
    __syncthreads();
    }
    // the next kernel on the stream may start now: its weight fills no longer
    // compete with this kernel's activation loads
    pdl_launch_dependents();
    uint4 a[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = live ? *reinterpret_cast<const uint4 *>(act + 16 * (8 * j + (k ^ jj)))
                                            : make_uint4(0, 0, 0, 0);

    // ---- the row loop: two rows per team per iteration
    int hpos = 0;  // iterations of block values held since the last fold
    for (int it = 0; it < p.n_iter; ++it) {
        const int slot = it % p.D;
        const int64_t lA = (int64_t)it * 2 * p.nt + 2 * team;  // row index within the CTA's range
        const bool haveA = live && lA < count, hasB = live && lA + 1 < count;
        const uint8_t *rA = ring + ((int64_t)(slot * p.nt + team) * 2) * p.rec;
        const uint8_t *rB = rA + p.rec;
        float *vA = val + ((hpos * p.nt + team) * 2) * p.vstride;
        float *vB = vA + p.vstride;
        bool ok = true;
        if (haveA) ok = mbar_wait_bounded(bars + slot, (uint32_t)((it / p.D) & 1), p.fault);
        const bool go = haveA && ok;
        if (F == kQ8_0) {
            if (go) {
                half_q8_0(rA + 128 * j, rA + p.K + 8 * j, ascl + 4 * j, a, jj, vA + 4 * j);
                if (hasB) half_q8_0(rB + 128 * j, rB + p.K + 8 * j, ascl + 4 * j, a, jj, vB + 4 * j);
            }
        } else {
            // partial sums of my half for both rows; every lane then swaps one
            // pair with its partner (lane ^ 1, the other half of the block)
            int CA = 0, CB = 0, OA = 0, OB = 0;
            uint32_t dA = 0, dB = 0;
            if (go) {
                if (F == kQ4K) {
                    half_q4k(rA + 144 * sb, h, a, S[0], S[1], CA, OA, dA);
                    if (hasB) half_q4k(rB + 144 * sb, h, a, S[0], S[1], CB, OB, dB);
                } else {
                    CA = half_q6k(rA + 208 * sb, h, a, S);
                    dA = *reinterpret_cast<const uint16_t *>(rA + 208 * p.nb + 2 * sb);
                    if (hasB) {
                        CB = half_q6k(rB + 208 * sb, h, a, S);
                        dB = *reinterpret_cast<const uint16_t *>(rB + 208 * p.nb + 2 * sb);
                    }
                }
            }
            const int rC = __shfl_xor_sync(0xFFFFFFFFu, h ? CA : CB, 1);
            const int rO = (F == kQ4K) ? __shfl_xor_sync(0xFFFFFFFFu, h ? OA : OB, 1) : 0;
            if (go && (!h || hasB)) {
                float v;
                const int Cs = (h ? CB : CA) + rC, O = (h ? OB : OA) + rO;
                const int C = (F == kQ4K) ? (Cs >> 4) : Cs;  // Q4_K: the halves hold 16*C (exact shift)
                const uint32_t dd = h ? dB : dA;
                if (F == kQ4K) v = lane_value_fast<1>(C, O, dd & 0xFFFFu, dd >> 16, m0, e0);
                else v = lane_value_fast<0>(C, 0, dd, 0, m0, e0);
                (h ? vB : vA)[sb] = v;
            }
        }
        if (p.wfold) {
            // a single iteration: each warp folds its own teams' rows (lane r
            // folds line r of the warp) as soon as its lanes have written
            // them -- no CTA-wide barrier
            if (!__all_sync(0xFFFFFFFFu, ok)) return;  // a fill never completed: fault word raised
            __syncwarp();
            const int lane = tid & 31, line = 2 * (tid >> 5) * (32 / p.ts) + lane;
            if (lane < 2 * (32 / p.ts) && line < 2 * p.nt && line < count) {
                const float4 *v4 = reinterpret_cast<const float4 *>(val + line * p.vstride);
                float acc = 0.0f;
                const int n4 = p.nb >> 2;
                for (int q = 0; q < n4; ++q) {
                    const float4 x = v4[q];
                    acc = fadd_ftz(fadd_ftz(fadd_ftz(fadd_ftz(acc, x.x), x.y), x.z), x.w);
                }
                const float *vt = val + line * p.vstride;
                for (int b = 4 * n4; b < p.nb; ++b) acc = fadd_ftz(acc, vt[b]);
                if (acc != acc) acc = __uint_as_float(kEngineNaN);
                if constexpr (MULTI) *out_ptr(p.mt, 0, row0 + line) = acc;
                else p.out[row0 + line] = acc;
            }
            continue;
        }
        if (!__syncthreads_and(ok)) return;  // a fill never completed: fault word raised
        if (tid == 0 && it + p.D < p.n_iter) {
            fence_proxy_async_smem();
            issue_fill<MULTI>(p, ring, bars, it + p.D, row0, count);
        }
        // ---- fold H iterations' rows: one thread per row, blocks in order
        if (++hpos == p.H || it == p.n_iter - 1) {
            const int nline = hpos * p.nt * 2;
            if (tid < nline) {
                const int64_t l = (int64_t)(it + 1 - hpos) * 2 * p.nt + tid;  // row of the CTA's range
                if (l < count) {
                    const float4 *v4 = reinterpret_cast<const float4 *>(val + tid * p.vstride);
                    float acc = 0.0f;
                    const int n4 = p.nb >> 2;
                    int q = 0;
                    for (; q + 4 <= n4; q += 4) {
                        const float4 x0 = v4[q], x1 = v4[q + 1], x2 = v4[q + 2], x3 = v4[q + 3];
                        acc = fadd_ftz(fadd_ftz(fadd_ftz(fadd_ftz(acc, x0.x), x0.y), x0.z), x0.w);
                        acc = fadd_ftz(fadd_ftz(fadd_ftz(fadd_ftz(acc, x1.x), x1.y), x1.z), x1.w);
                        acc = fadd_ftz(fadd_ftz(fadd_ftz(fadd_ftz(acc, x2.x), x2.y), x2.z), x2.w);
                        acc = fadd_ftz(fadd_ftz(fadd_ftz(fadd_ftz(acc, x3.x), x3.y), x3.z), x3.w);
                    }
                    for (; q < n4; ++q) {
                        const float4 x = v4[q];
                        acc = fadd_ftz(fadd_ftz(fadd_ftz(fadd_ftz(acc, x.x), x.y), x.z), x.w);
                    }
                    const float *vt = val + tid * p.vstride;
                    for (int b = 4 * n4; b < p.nb; ++b) acc = fadd_ftz(acc, vt[b]);
                    if (acc != acc) acc = __uint_as_float(kEngineNaN);
                    if constexpr (MULTI) *out_ptr(p.mt, 0, row0 + l) = acc;
                    else p.out[row0 + l] = acc;
                }
            }
            hpos = 0;
            if (it != p.n_iter - 1) __syncthreads();  // before the history is overwritten
        }
    }
}

template <int F>
int launch_gemv2(const GemvArgs &a, cudaStream_t stream, const float *x = nullptr) {
    if (a.ncols != 1 || a.mode != 0 || a.K % 256 != 0) return QB_E_ARG;
    const int K = (int)a.K;
    const int ts = K / 128;
    if (ts > 512) return QB_E_ARG;
    Gemv2KM k;
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.rows = k.mt.start[k.mt.n];
    k.W = k.mt.W[0];
    k.out = k.mt.out[0];
    k.K = K;
    k.rec = (int)record_bytes(F, a.K);
    k.ts = ts;
    k.nb = K / fmt_block(F);
    k.vstride = (k.nb + 3) / 4 * 4;
    if (((k.vstride / 4) & 1) == 0) k.vstride += 4;  // odd number of 16-B units: conflict-free fold
    const int sms = num_sms();
    const int max_nt = std::max(1, 512 / ts);
    // one CTA per SM (fewer for a short matrix); teams per CTA: enough for all
    // of the CTA's rows in one iteration when that fits, else as many as leave
    // room for two ring slots
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, k.rows));
    const int64_t rpc = (k.rows + grid - 1) / grid;  // most rows any CTA owns
    const int64_t need = (rpc + 1) / 2;
    k.nt = (int)std::min<int64_t>(max_nt, std::max<int64_t>(1, need));
    const bool multi = k.nt < need;  // more than one iteration per CTA
    // Shared memory: a single-iteration product with a staged activation stays
    // under ~110 KB so the next launch's CTA fits beside it and streams early;
    // otherwise the whole 225 KB serves a two-slot ring with as many teams as fit.
    const int fixed = gemv2_smem(K, k.rec, 0, 0, 1, k.vstride).total + 8 * 2 * 20 * 4 * 16;
    const int budget = (x || multi) ? 225 * 1024 : 110 * 1024;
    if (multi) k.nt = std::min(k.nt, std::max(1, (budget - fixed) / (2 * 2 * k.rec)));
    // the in-kernel quantizer needs K/8 <= 4 * threads (nt >= 4); one 8-element
    // group a thread (nt >= 16) is fastest
    if (x) k.nt = std::max(k.nt, std::min(multi ? 4 : 16, max_nt));
    k.n_iter = (int)((rpc + 2LL * k.nt - 1) / (2LL * k.nt));
    k.wfold = (k.n_iter == 1 && 32 % ts == 0) ? 1 : 0;
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    const int slot = 2 * k.nt * k.rec;
    k.H = std::max(1, std::min({k.n_iter, 8, ts / 2}));  // one fold line per thread: H * 2 * nt <= nt * ts
    k.D = std::max(1, std::min({k.n_iter, 4, (budget - fixed) / std::max(1, slot)}));
    if (k.D < 2 && k.n_iter > 1) k.D = 2;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.x = x;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    Gemv2Smem L = gemv2_smem(K, k.rec, k.nt, k.D, k.H, k.vstride);
    while (L.total > 225 * 1024 && (k.D > 1 || k.H > 1)) {
        if (k.D > 1) --k.D; else --k.H;
        L = gemv2_smem(K, k.rec, k.nt, k.D, k.H, k.vstride);
    }
    if (L.total > 227 * 1024) return QB_E_ARG;
    const int threads = (k.nt * ts + 31) / 32 * 32;
    if (x && K / 8 > 4 * threads) return QB_E_ARG;  // the in-kernel quantizer holds at most 4 groups a thread
    auto set_attr = [&](const void *f) { return ensure_smem_limit(f, 227 * 1024) == QB_OK; };
    const Gemv2K &k1 = k;  // a one-matrix launch takes the plain parameters
    if (k.mt.n > 1) {
        auto kern = x ? gemv2_kernel<F, true, true> : gemv2_kernel<F, false, true>;
        if (!set_attr(reinterpret_cast<const void *>(kern))) return QB_E_CUDA;
        return launch_pdl(kern, dim3(grid), dim3(threads), (size_t)L.total, stream, k);
    }
    auto kern = x ? gemv2_kernel<F, true, false> : gemv2_kernel<F, false, false>;
    if (!set_attr(reinterpret_cast<const void *>(kern))) return QB_E_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(threads), (size_t)L.total, stream, k1);
}

}  // namespace qb
