// qb_sub32.cuh -- the product under ActScaling::Sub32 (the decode engine's
// numerics page: block_scale, quantize, ACT_BLOCK, GROUP, exact_sum, dot; the
// block-scale lane page: group).
//
// Every 32-element activation block carries its own scale m_s*2^e_s (m in
// 8..15).  A group is 256 elements: its value is the exact sum of all its
// sub-blocks' terms -- weight scale x activation scale x integer sum --
// rounded once to f32; a row is its groups' values added in order from +0
// (f32, round to nearest even, subnormal results flushed).
//
// Fast path.  With Emin the least exponent of a group's eight activation
// scales, m_s*2^e_s = M_s*2^Emin for the integer M_s = m_s << (e_s - Emin).
// While every M_s < 2^16 (exponents within 12 places), the sub-block sums
// times M_s add exactly in 64 bits and the group is a one- or two-term combine
// with the weight scales, as a PerBlock block is.  Q8_0 weight scales differ
// per sub-block: their exponents align at the group's least, which the fast
// path takes while they lie within 13 places.  Bounds (|a| <= 127):
//   Q4_K-like  sum over the group of sc*M*16*sum(q*a) < 8 * 2^22 * 2^20 = 2^45;
//              d*C < 2^11 * 2^41; sum mn*M*A < 2^37, dmin*O < 2^48;
//   Q6_K-like  M * sum over 32 of sc*(q-32)*a < 2^16 * 2^24; d*C < 2^11 * 2^43;
//   Q8_0       (d_s*M_s) * sum(q*a) < 2^27 * 2^19, shifted <= 13: 8 terms < 2^62.
// Anything else -- a wider spread, a multiplier past 16 bits -- takes an
// out-of-line routine that rebuilds the group's terms from the row record and
// the codes and sums them exactly in a 384-bit integer.  An activation block
// without a scale (m = 0) or an unreadable weight scale makes the group, and so
// the row, the engine's NaN.
//
// The streaming organisation is the multi-column kernel's (qb_gemv3.cuh):
// persistent CTAs over contiguous row ranges, weights through a ring of bulk
// copies completing on mbarriers, teams of K/128 threads owning 128-element
// half-slices (half a group) for CG columns, two rows per team per iteration
// with one swap of partial sums between the two halves of a group, and an
// in-order fold from shared memory.  Shapes that do not fit its shared memory
// take a plain kernel built on the exact routine.
#pragma once

#include <algorithm>
#include <climits>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_gemv3.cuh"
#include "qb_launch.h"

namespace qb {

// ------------------------------------------------------------------ exact routine

// exact_sum (numerics page) of n terms sig_k * 2^E_k (|sig_k| < 2^44), rounded
// once by round_to_f32's rule.  The terms add in a 384-bit two's-complement
// integer aligned at the least exponent of the n terms; a nonzero term 318 or
// more places above it lies outside that window and makes the result the
// engine's NaN (f16 weight scales with block_scale activation scales stay
// within 290 places).
static __device__ __noinline__ float exact_sum_terms(const long long *sig, const int *E, int n) {
    if (n == 0) return 0.0f;
    int lo = E[0];
    for (int k = 1; k < n; ++k) lo = min(lo, E[k]);
    unsigned long long acc[6] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
    for (int k = 0; k < n; ++k) {
        if (sig[k] == 0) continue;
        const int sh = E[k] - lo;
        if (sh >= 318) return __uint_as_float(kEngineNaN);
        const bool neg = sig[k] < 0;
        const unsigned long long mag = neg ? 0ull - (unsigned long long)sig[k] : (unsigned long long)sig[k];
        const int L = sh >> 6, b = sh & 63;
        const unsigned long long p0 = mag << b, p1 = b ? mag >> (64 - b) : 0ull;
        unsigned long long cy = 0ull;  // carry (add) or borrow (subtract)
        for (int i = L; i < 6; ++i) {
            const unsigned long long t = (i == L) ? p0 : (i == L + 1) ? p1 : 0ull;
            if (!neg) {
                const unsigned long long s1 = acc[i] + t, s2 = s1 + cy;
                cy = (unsigned long long)((s1 < t) | (s2 < cy));
                acc[i] = s2;
            } else {
                const unsigned long long d1 = acc[i] - t, d2 = d1 - cy;
                cy = (unsigned long long)((acc[i] < t) | (d1 < cy));
                acc[i] = d2;
            }
        }
    }
    const bool neg = (acc[5] >> 63) != 0;
    if (neg) {
        unsigned long long cy = 1ull;
        for (int i = 0; i < 6; ++i) {
            const unsigned long long v = ~acc[i] + cy;
            cy = (cy && v == 0ull) ? 1ull : 0ull;
            acc[i] = v;
        }
    }
    int top = 5;
    while (top >= 0 && acc[top] == 0ull) --top;
    if (top < 0) return 0.0f;  // an exact zero is +0
    const int p = 64 * top + 63 - __clzll((long long)acc[top]);  // leading place
    if (p <= 61) {
        const long long v = (long long)acc[0];
        return round_to_f32(neg ? -v : v, lo);
    }
    // the 62 places below and at p, the rest folded into a sticky bit
    const int q = p - 61, L0 = q >> 6, b0 = q & 63;
    unsigned long long w = acc[L0] >> b0;
    if (b0 && L0 + 1 < 6) w |= acc[L0 + 1] << (64 - b0);
    bool sticky = b0 ? (acc[L0] & ((1ull << b0) - 1ull)) != 0ull : false;
    for (int i = 0; i < L0; ++i) sticky |= acc[i] != 0ull;
    const long long v = (long long)(w | (sticky ? 1ull : 0ull));
    return round_to_f32(neg ? -v : v, lo + q);
}

// Code of element b of a column whose first 16-B unit is unit0 of `act`: the
// streaming kernels' staged layout (256-element formats: unit u at
// (u & ~7) | ((u & 7) ^ ((u >> 3) & 7))) when swz, else linear.
__device__ __forceinline__ int s32_code(const uint8_t *act, int64_t unit0, int b, bool swz) {
    const int64_t u = unit0 + (b >> 4);
    const int64_t pos = swz ? ((u & ~7ll) | ((u & 7) ^ ((u >> 3) & 7))) : u;
    return (int)(int8_t)act[16 * pos + (b & 15)];
}

// group (lane page) g of a row under Sub32, exactly: every sub-block's terms
// rebuilt from the row record and the column's codes (numerics page, CodedRow:
// weight = a*coef + b*offs), then exact_sum_terms.  gs: the group's eight
// activation scales (m | e << 16).
template <int F>
static __device__ __noinline__ float group_value_exact(const uint8_t *row, int K, int g, const uint8_t *act,
                                                       int64_t unit0, bool swz, const uint32_t *gs) {
    long long sig[16];
    int E[16];
    int n = 0;
    const int nb = K / 256;
    for (int s = 0; s < 8; ++s) {
        const uint32_t sw = gs[s];
        const int m = (int)(sw & 0xFFu), e = (int)(int16_t)(sw >> 16);
        if (m == 0) return __uint_as_float(kEngineNaN);
        const int b0 = 256 * g + 32 * s;
        long long C = 0, O = 0;
        uint32_t d1, d2 = 0;
        if (F == kQ8_0) {
            const int8_t *q = reinterpret_cast<const int8_t *>(row) + b0;
            for (int i = 0; i < 32; ++i) C += (int)q[i] * s32_code(act, unit0, b0 + i, swz);
            d1 = row[K + 2 * (8 * g + s)] | ((uint32_t)row[K + 2 * (8 * g + s) + 1] << 8);
        } else if (F == kQ4K) {
            const uint8_t *blk = row + 144 * g;
            unsigned long long sc48 = 0, mn48 = 0;
            for (int b = 0; b < 6; ++b) {
                sc48 |= (unsigned long long)blk[4 + b] << (8 * b);
                mn48 |= (unsigned long long)blk[10 + b] << (8 * b);
            }
            const int sc = (int)((sc48 >> (6 * s)) & 63u), mn = (int)((mn48 >> (6 * s)) & 63u);
            int cq = 0, asum = 0;
            for (int i = 0; i < 32; ++i) {
                const int a = s32_code(act, unit0, b0 + i, swz);
                const int q = (i < 16) ? (blk[16 + 16 * s + i] & 15) : (blk[16 + 16 * s + i - 16] >> 4);
                cq += q * a;
                asum += a;
            }
            C = (long long)sc * cq;
            O = (long long)mn * asum;
            d1 = blk[0] | ((uint32_t)blk[1] << 8);
            d2 = blk[2] | ((uint32_t)blk[3] << 8);
        } else {
            const uint8_t *blk = row + 208 * g;
            for (int i = 0; i < 32; ++i) {
                const int i2 = i & 15;
                const int lo = (blk[16 * s + i2] >> (i < 16 ? 0 : 4)) & 15;
                const int hi = (blk[128 + 8 * s + (i < 16 ? 0 : 4) + (i2 & 3)] >> (2 * (i2 >> 2))) & 3;
                const int sc = (int)(int8_t)blk[192 + 2 * s + (i >> 4)];
                C += (long long)sc * ((lo | (hi << 4)) - 32) * s32_code(act, unit0, b0 + i, swz);
            }
            d1 = row[208 * nb + 2 * g] | ((uint32_t)row[208 * nb + 2 * g + 1] << 8);
        }
        int sg, ex;
        if (!f16_scale(d1, sg, ex)) return __uint_as_float(kEngineNaN);
        sig[n] = (long long)sg * m * C;
        E[n] = ex + e;
        ++n;
        if (F == kQ4K) {
            if (!f16_scale(d2, sg, ex)) return __uint_as_float(kEngineNaN);
            sig[n] = -(long long)sg * m * O;
            E[n] = ex + e;
            ++n;
        }
    }
    return exact_sum_terms(sig, E, n);
}

// ------------------------------------------------------------------ fast path pieces

// The group's eight activation scales gs (m | e << 16): the least exponent,
// the mode (0 fast, 1 exact routine, 2 NaN: a block without a scale) and, in
// the fast mode, the multipliers M_s of sub-blocks 4h..4h+3 packed as 16-bit
// pairs.  The mode depends on all eight scales, so both halves of a group
// agree on it.
__device__ __forceinline__ void s32_group_scales(const uint32_t *gs, int h, uint32_t (&Mw)[2], int &emin, int &mode) {
    const uint4 s0 = *reinterpret_cast<const uint4 *>(gs), s1 = *reinterpret_cast<const uint4 *>(gs + 4);
    const uint32_t w[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    int lo = INT_MAX, hi = INT_MIN;
    bool zero = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = (int)(int16_t)(w[i] >> 16);
        zero |= (w[i] & 0xFFu) == 0u;
        lo = min(lo, e);
        hi = max(hi, e);
    }
    mode = zero ? 2 : (hi - lo > 12 ? 1 : 0);
    Mw[0] = Mw[1] = 0u;
    emin = lo;
    if (mode != 0) return;
    bool big = false;
    uint32_t Ms[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        Ms[i] = (w[i] & 0xFFu) << ((int)(int16_t)(w[i] >> 16) - lo);  // < 2^20
        big |= Ms[i] > 0xFFFFu;
    }
    if (big) { mode = 1; return; }
    Mw[0] = h ? (Ms[4] | (Ms[5] << 16)) : (Ms[0] | (Ms[1] << 16));
    Mw[1] = h ? (Ms[6] | (Ms[7] << 16)) : (Ms[2] | (Ms[3] << 16));
}

__device__ __forceinline__ int mul16(const uint32_t (&Mw)[2], int s) {
    return (int)((Mw[s >> 1] >> (16 * (s & 1))) & 0xFFFFu);
}

// Q4_K-like half block h for CG columns under Sub32: C[c] += 16 * sum over my
// sub-blocks of sc*M*sum(q*a), O[c] += sum of mn*(M*A) (AM holds M_s times the
// sub-block's code sum).
template <int CG>
__device__ __forceinline__ void half_q4k_s32(const uint8_t *blk, int h, const uint4 (&a)[CG][8],
                                             const uint32_t (&Mw)[CG][2], const int (&AM)[CG][4],
                                             long long (&C)[CG], long long (&O)[CG], uint32_t &dd) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    dd = meta.x;
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
    const uint32_t scm = (uint32_t)(sc48 >> (24 * h)), mnm = (uint32_t)(mn48 >> (24 * h));
    const uint8_t *qs = blk + 16 + 64 * h;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint4 w = *reinterpret_cast<const uint4 *>(qs + 16 * s);
        const uint32_t l0 = (w.x << 4) & 0xF0F0F0F0u, l1 = (w.y << 4) & 0xF0F0F0F0u;
        const uint32_t l2 = (w.z << 4) & 0xF0F0F0F0u, l3 = (w.w << 4) & 0xF0F0F0F0u;
        const uint32_t g0 = w.x & 0xF0F0F0F0u, g1 = w.y & 0xF0F0F0F0u, g2 = w.z & 0xF0F0F0F0u, g3 = w.w & 0xF0F0F0F0u;
        const int sc = (int)((scm >> (6 * s)) & 63u), mn = (int)((mnm >> (6 * s)) & 63u);
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            int p = dp4a_us(l0, a[c][2 * s].x, 0);
            p = dp4a_us(l1, a[c][2 * s].y, p);
            p = dp4a_us(l2, a[c][2 * s].z, p);
            p = dp4a_us(l3, a[c][2 * s].w, p);
            p = dp4a_us(g0, a[c][2 * s + 1].x, p);
            p = dp4a_us(g1, a[c][2 * s + 1].y, p);
            p = dp4a_us(g2, a[c][2 * s + 1].z, p);
            p = dp4a_us(g3, a[c][2 * s + 1].w, p);
            C[c] += (long long)(sc * mul16(Mw[c], s)) * p;
            O[c] += (long long)mn * AM[c][s];
        }
    }
}

// Q6_K-like half block h (32-element chunks 4h..4h+3) for CG columns under
// Sub32: C[c] += sum over my chunks of M * sum(sc*(q-32)*a).
template <int CG>
__device__ __forceinline__ void half_q6k_s32(const uint8_t *blk, int h, const uint4 (&a)[CG][8],
                                             const uint32_t (&S)[CG][4], const uint32_t (&Mw)[CG][2],
                                             long long (&C)[CG]) {
    const uint2 scw = *reinterpret_cast<const uint2 *>(blk + 192 + 8 * h);
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 64 * h + 16 * ch);
        const uint2 hb = *reinterpret_cast<const uint2 *>(blk + 128 + 32 * h + 8 * ch);
        const uint32_t wl[4] = {w.x, w.y, w.z, w.w};
        uint32_t ql[4], qh[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t hl = (k < 3) ? (hb.x << (4 - 2 * k)) : (hb.x >> 2);
            const uint32_t hh = (k < 3) ? (hb.y << (4 - 2 * k)) : (hb.y >> 2);
            ql[k] = (wl[k] & 0x0F0F0F0Fu) | (hl & 0x30303030u);
            qh[k] = ((wl[k] >> 4) & 0x0F0F0F0Fu) | (hh & 0x30303030u);
        }
        const uint32_t sw = (ch < 2) ? scw.x : scw.y;
        const int sc_lo = (int)(int8_t)((sw >> (16 * (ch & 1))) & 0xFFu);
        const int sc_hi = (int)(int8_t)((sw >> (16 * (ch & 1) + 8)) & 0xFFu);
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            int pl = dp4a_ss(ql[0], a[c][2 * ch].x, 0);
            pl = dp4a_ss(ql[1], a[c][2 * ch].y, pl);
            pl = dp4a_ss(ql[2], a[c][2 * ch].z, pl);
            pl = dp4a_ss(ql[3], a[c][2 * ch].w, pl);
            int ph = dp4a_ss(qh[0], a[c][2 * ch + 1].x, 0);
            ph = dp4a_ss(qh[1], a[c][2 * ch + 1].y, ph);
            ph = dp4a_ss(qh[2], a[c][2 * ch + 1].z, ph);
            ph = dp4a_ss(qh[3], a[c][2 * ch + 1].w, ph);
            const int cs = sc_lo * (pl - 32 * (int)(int16_t)(S[c][ch] & 0xFFFFu)) +
                           sc_hi * (ph - 32 * (int)(int16_t)(S[c][ch] >> 16));
            C[c] += (long long)mul16(Mw[c], ch) * cs;
        }
    }
}

// A Q8_0 group's eight weight scales (at dptr): the mode (0 fast, 1 exact
// routine: exponents more than 13 places apart, 2 NaN: an unreadable scale),
// the least exponent, and for blocks 4h..4h+3 the signed significand and its
// shift to the least exponent (0 outside the fast mode).  Both halves of the
// group read all eight and agree.
__device__ __forceinline__ void q8_group_scales(const uint8_t *dptr, int h, int (&sg)[4], int (&sh)[4], int &exmin,
                                                int &mode) {
    const uint4 dw = *reinterpret_cast<const uint4 *>(dptr);
    const uint32_t w[4] = {dw.x, dw.y, dw.z, dw.w};
    int lo = 64, hi = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t hb = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
        const int E5 = (int)((hb >> 10) & 31u);
        bad |= E5 == 31;
        lo = min(lo, max(E5, 1));
        hi = max(hi, max(E5, 1));
    }
    mode = bad ? 2 : (hi - lo > 13 ? 1 : 0);
    exmin = lo - 25;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint32_t hb = (w[2 * h + (t >> 1)] >> (16 * (t & 1))) & 0xFFFFu;
        const int E5 = (int)((hb >> 10) & 31u), f = (int)(hb & 1023u);
        const int s = E5 ? (f | 1024) : f;
        sg[t] = (hb & 0x8000u) ? -s : s;
        sh[t] = mode == 0 ? max(E5, 1) - lo : 0;
    }
}

template <typename T>
__device__ __forceinline__ T sel4(const T (&v)[4], int i) {
    return i == 0 ? v[0] : i == 1 ? v[1] : i == 2 ? v[2] : v[3];
}

// Q8_0 half-slice (blocks 4j..4j+3 = sub-blocks 4h..4h+3 of group j/2) for CG
// columns: t[c] = sum of (d_s*M_s * sum(q*a)) << shift_s.  Units visited in the
// order k ^ jj (a[c][k] holds unit 8j + (k ^ jj)).
template <int CG>
__device__ __forceinline__ void half_q8_0_s32(const uint8_t *q, const uint4 (&a)[CG][8], int jj,
                                              const uint32_t (&Mw)[CG][2], const int (&sg)[4], const int (&sh)[4],
                                              long long (&t)[CG]) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int u0 = (2 * kk) ^ jj, u1 = u0 ^ 1;
        const int i = u0 >> 1;
        const uint4 w0 = *reinterpret_cast<const uint4 *>(q + 16 * u0);
        const uint4 w1 = *reinterpret_cast<const uint4 *>(q + 16 * u1);
        const int sgi = sel4(sg, i), shi = sel4(sh, i);
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            int p = dp4a_ss(w0.x, a[c][2 * kk].x, 0);
            p = dp4a_ss(w0.y, a[c][2 * kk].y, p);
            p = dp4a_ss(w0.z, a[c][2 * kk].z, p);
            p = dp4a_ss(w0.w, a[c][2 * kk].w, p);
            p = dp4a_ss(w1.x, a[c][2 * kk + 1].x, p);
            p = dp4a_ss(w1.y, a[c][2 * kk + 1].y, p);
            p = dp4a_ss(w1.z, a[c][2 * kk + 1].z, p);
            p = dp4a_ss(w1.w, a[c][2 * kk + 1].w, p);
            t[c] += ((long long)(sgi * mul16(Mw[c], i)) * p) << shi;
        }
    }
}

// t1*2^e1 + t2*2^e2 rounded once (|t1| < 2^53, |t2| < 2^49, |e1 - e2| <= 29).
__device__ __forceinline__ float round_pair(long long t1, int e1, long long t2, int e2) {
    const int d = e1 - e2;
    if (d >= 0 && d <= 8) return round_fast((t1 << d) + t2, e2);
    if (d < 0 && d >= -12) return round_fast(t1 + (t2 << (-d)), e1);
    const __int128 w = d >= 0 ? ((__int128)t1 << d) + t2 : (__int128)t1 + ((__int128)t2 << (-d));
    return round_to_f32_wide(w, d >= 0 ? e2 : e1);
}

// ------------------------------------------------------------------ streaming kernel

struct S32K {
    const uint8_t *W;
    float *out;      // output at this launch's first column
    int64_t rows;
    int K;
    int rec;
    int nt;       // teams per CTA
    int ts;       // threads per column group = K / 128
    int ncg;      // column groups per team
    int ncols;    // real columns of this launch
    int D;        // ring slots
    int H;        // iterations of group values held before a fold
    int ng;       // groups per row
    int vstride;  // floats per value line (odd)
    int n_iter;
    int64_t base;
    int64_t rem;
    const int8_t *codes;  // column 0 of this launch
    const qb_scale *scales;
    const int16_t *sums16;
    const float *x;  // FUSED: the f32 activation, quantized in the prologue
    int *fault;
};

struct S32Smem {
    int bars, act, scl, sums, val, ring, total;
};

// sums: the unit sums the single-launch form quantizes into (fused only)
__host__ __device__ inline S32Smem s32_smem(int K, int ncols, int rec, int nt, int ncp, int D, int H, int vstride,
                                            bool fused = false) {
    S32Smem s;
    s.bars = 0;
    s.act = 128;                                          // the launch's codes
    s.scl = s.act + ((ncols * K + 127) & ~127);           // its scales, K/32 a column
    s.sums = s.scl + ((ncols * (K / 32) * 4 + 127) & ~127);
    s.val = s.sums + (fused ? ((K / 16 * 2 + 127) & ~127) : 0);
    s.ring = s.val + ((H * nt * 2 * ncp * vstride * 4 + 127) & ~127);
    s.total = s.ring + D * nt * 2 * rec;
    return s;
}

// FUSED (one column): the f32 activation p.x is quantized under Sub32 in the
// prologue (the quantize_act_sub32 arithmetic: a 32-element block on four
// lanes) while the first weight fills are in flight.
template <int F, int CG, bool FUSED = false>
__global__ void __launch_bounds__(gemv3_threads<CG>(), 1) s32_kernel(const S32K p) {
    static_assert(!FUSED || CG == 1, "the single-launch form takes one column");
    extern __shared__ __align__(128) uint8_t smem[];
    const int ncp = p.ncg * CG;
    const S32Smem L = s32_smem(p.K, p.ncols, p.rec, p.nt, ncp, p.D, p.H, p.vstride, FUSED);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint8_t *act = smem + L.act;
    uint32_t *ascl = reinterpret_cast<uint32_t *>(smem + L.scl);
    int16_t *asum = reinterpret_cast<int16_t *>(smem + L.sums);
    float *val = reinterpret_cast<float *>(smem + L.val);
    uint8_t *ring = smem + L.ring;

    const int tid = threadIdx.x;
    const int tpt = p.ncg * p.ts;
    const int team = tid / tpt, tr = tid - team * tpt;
    const int g = tr / p.ts, j = tr - g * p.ts;
    const bool live = team < p.nt;
    const int sb = j >> 1, h = j & 1, jj = j & 7;
    const int nsc = p.K / 32;  // scales a column

    const int64_t cta = blockIdx.x;
    const int64_t row0 = cta * p.base + (cta < p.rem ? cta : p.rem);
    const int64_t count = p.base + (cta < p.rem ? 1 : 0);
    const int64_t per_it = 2LL * p.nt;
    if (tid == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto fill = [&](int it) {
        const int slot = it % p.D;
        const int64_t first = (int64_t)it * per_it;
        const int64_t n = (count - first < per_it) ? count - first : per_it;
        const uint32_t bytes = n > 0 ? (uint32_t)(n * p.rec) : 0u;
        mbar_arrive_expect_tx(bars + slot, bytes);
        if (!bytes) return;
        bulk_g2s(ring + (int64_t)slot * per_it * p.rec, p.W + (row0 + first) * p.rec, bytes, bars + slot);
    };
    if (tid == 0)
        for (int it = 0; it < p.D && it < p.n_iter; ++it) fill(it);  // weights depend on no earlier kernel
    pdl_wait();

    // ---- the launch's codes (the multi-column kernel's staged layout) and
    // scales; the single-launch form quantizes x here instead: a thread takes
    // 8 consecutive elements (a 32-element block is 4 consecutive lanes),
    // up to four rounds of loads first, then the quantizer
    if constexpr (FUSED) {
        constexpr int kR = 4;
        const int G = p.K / 8;  // a multiple of 32: whole warps are in or out of a round
        for (int g0 = 0; g0 < G; g0 += kR * (int)blockDim.x) {
            float4 xv[2 * kR];
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const int g8 = g0 + tid + r * (int)blockDim.x;
                const bool in = g8 < G;
                xv[2 * r] = in ? ldg_f4_ordered(reinterpret_cast<const float4 *>(p.x) + 2 * g8) : make_float4(0, 0, 0, 0);
                xv[2 * r + 1] = in ? ldg_f4_ordered(reinterpret_cast<const float4 *>(p.x) + 2 * g8 + 1)
                                   : make_float4(0, 0, 0, 0);
            }
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                if (g0 + r * (int)blockDim.x >= G) break;  // uniform: whole warps are in or out
                const int g8 = g0 + tid + r * (int)blockDim.x;
                const uint32_t xb[8] = {__float_as_uint(xv[2 * r].x), __float_as_uint(xv[2 * r].y),
                                        __float_as_uint(xv[2 * r].z), __float_as_uint(xv[2 * r].w),
                                        __float_as_uint(xv[2 * r + 1].x), __float_as_uint(xv[2 * r + 1].y),
                                        __float_as_uint(xv[2 * r + 1].z), __float_as_uint(xv[2 * r + 1].w)};
                uint2 cq;
                int usum;
                uint32_t scale;
                quantize8<4, true>(xb, cq, usum, scale);
                if (g8 < G) {
                    const int u = g8 >> 1;
                    const int pos = (F == kQ8_0) ? u : ((u & ~7) | ((u & 7) ^ ((u >> 3) & 7)));
                    *reinterpret_cast<uint2 *>(act + 16 * pos + 8 * (g8 & 1)) = cq;
                    if ((g8 & 1) == 0) asum[u] = (int16_t)usum;
                    if ((g8 & 3) == 0) ascl[g8 >> 2] = scale;
                }
            }
        }
        __syncthreads();
    } else {
        const int nu = p.ncols * (p.K / 16);
        const uint4 *src = reinterpret_cast<const uint4 *>(p.codes);
        constexpr int kU = 4;
        for (int u0 = tid; u0 < nu; u0 += kU * (int)blockDim.x) {
            uint4 v[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int u = u0 + q * (int)blockDim.x;
                v[q] = u < nu ? ldg_v4_ordered(src + u) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int u = u0 + q * (int)blockDim.x;
                const int pos = (F == kQ8_0) ? u : ((u & ~7) | ((u & 7) ^ ((u >> 3) & 7)));
                if (u < nu) *reinterpret_cast<uint4 *>(act + 16 * pos) = v[q];
            }
        }
        const uint32_t *ssrc = reinterpret_cast<const uint32_t *>(p.scales);
        for (int i = tid; i < p.ncols * nsc; i += blockDim.x) ascl[i] = ldg_u32_ordered(ssrc + i);
    }
    // my columns' unit sums (global memory; small)
    uint32_t S[CG][4];
#pragma unroll
    for (int c = 0; c < CG; ++c) {
        const int col = g * CG + c;
        S[c][0] = S[c][1] = S[c][2] = S[c][3] = 0;
        if (F != kQ8_0 && live && col < p.ncols) {
            const uint4 sw = FUSED ? *reinterpret_cast<const uint4 *>(asum + 8 * j)
                                   : __ldg(reinterpret_cast<const uint4 *>(p.sums16 + (int64_t)col * (p.K / 16)) + j);
            S[c][0] = sw.x; S[c][1] = sw.y; S[c][2] = sw.z; S[c][3] = sw.w;
        }
    }
    __syncthreads();
    pdl_launch_dependents();

    uint4 a[CG][8];
    uint32_t Mw[CG][2];
    int emin[CG], amode[CG];
    int AM[CG][4];  // Q4_K-like: M_s times the code sum of my sub-block s
#pragma unroll
    for (int c = 0; c < CG; ++c) {
        const int col = g * CG + c;
        const bool in = live && col < p.ncols;
        const uint8_t *base = act + (int64_t)col * p.K + 128 * j;
        const int key = (F == kQ8_0) ? jj : ((col * p.ts + j) & 7);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            a[c][k] = in ? *reinterpret_cast<const uint4 *>(base + 16 * (k ^ key)) : make_uint4(0, 0, 0, 0);
        Mw[c][0] = Mw[c][1] = 0u;
        emin[c] = 0;
        amode[c] = 0;
        if (in) s32_group_scales(ascl + col * nsc + 8 * sb, h, Mw[c], emin[c], amode[c]);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int A = (int)(int16_t)(S[c][s] & 0xFFFFu) + (int)(int16_t)(S[c][s] >> 16);
            AM[c][s] = A * mul16(Mw[c], s);
        }
    }

    const int vcol = p.vstride;
    int hpos = 0;
    for (int it = 0; it < p.n_iter; ++it) {
        const int slot = it % p.D;
        const int64_t lA = (int64_t)it * per_it + 2 * team;
        const bool haveA = live && lA < count, hasB = live && lA + 1 < count;
        const uint8_t *rA = ring + ((int64_t)(slot * p.nt + team) * 2) * p.rec;
        const uint8_t *rB = rA + p.rec;
        float *vA = val + (((hpos * p.nt + team) * 2) * ncp + g * CG) * p.vstride;
        float *vB = vA + ncp * p.vstride;
        bool ok = true;
        if (haveA) ok = mbar_wait_bounded(bars + slot, (uint32_t)((it / p.D) & 1), p.fault);
        const bool go = haveA && ok;
        // partial sums of my half for both rows; each lane then swaps one per
        // column with its partner (lane ^ 1, the group's other half) and
        // finishes one row's group
        long long CA[CG], CB[CG], OA[CG], OB[CG];
#pragma unroll
        for (int c = 0; c < CG; ++c) { CA[c] = 0; CB[c] = 0; OA[c] = 0; OB[c] = 0; }
        uint32_t dA = 0, dB = 0;
        int wmA = 0, wmB = 0, exA = 0, exB = 0;  // Q8_0: weight-scale mode and least exponent
        if (go) {
            if (F == kQ4K) {
                half_q4k_s32<CG>(rA + 144 * sb, h, a, Mw, AM, CA, OA, dA);
                if (hasB) half_q4k_s32<CG>(rB + 144 * sb, h, a, Mw, AM, CB, OB, dB);
            } else if (F == kQ6K) {
                half_q6k_s32<CG>(rA + 208 * sb, h, a, S, Mw, CA);
                dA = *reinterpret_cast<const uint16_t *>(rA + 208 * p.ng + 2 * sb);
                if (hasB) {
                    half_q6k_s32<CG>(rB + 208 * sb, h, a, S, Mw, CB);
                    dB = *reinterpret_cast<const uint16_t *>(rB + 208 * p.ng + 2 * sb);
                }
            } else {
                int sg[4], sh[4];
                q8_group_scales(rA + p.K + 16 * sb, h, sg, sh, exA, wmA);
                half_q8_0_s32<CG>(rA + 128 * j, a, jj, Mw, sg, sh, CA);
                if (hasB) {
                    q8_group_scales(rB + p.K + 16 * sb, h, sg, sh, exB, wmB);
                    half_q8_0_s32<CG>(rB + 128 * j, a, jj, Mw, sg, sh, CB);
                }
            }
        }
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            const long long rC = __shfl_xor_sync(0xFFFFFFFFu, h ? CA[c] : CB[c], 1);
            const long long rO = (F == kQ4K) ? __shfl_xor_sync(0xFFFFFFFFu, h ? OA[c] : OB[c], 1) : 0ll;
            if (go && (!h || hasB)) {
                const int col = g * CG + c;
                const long long Ct = (h ? CB[c] : CA[c]) + rC;
                const int mode = max(amode[c], F == kQ8_0 ? (h ? wmB : wmA) : 0);
                float v;
                if (mode == 2) {
                    v = __uint_as_float(kEngineNaN);
                } else if (mode == 1) {
                    v = group_value_exact<F>(h ? rB : rA, p.K, sb, act, (int64_t)col * (p.K / 16), F != kQ8_0,
                                             ascl + col * nsc + 8 * sb);
                } else if (F == kQ8_0) {
                    v = round_fast(Ct, (h ? exB : exA) + emin[c]);
                } else {
                    const uint32_t dd = h ? dB : dA;
                    int sig1, ex1;
                    const bool ok1 = f16_scale(dd & 0xFFFFu, sig1, ex1);
                    if (F == kQ6K) {
                        v = ok1 ? round_fast((long long)sig1 * Ct, ex1 + emin[c]) : __uint_as_float(kEngineNaN);
                    } else {
                        int sig2, ex2;
                        const bool ok2 = f16_scale(dd >> 16, sig2, ex2);
                        const long long Ot = (h ? OB[c] : OA[c]) + rO;
                        v = (ok1 && ok2) ? round_pair((long long)sig1 * (Ct >> 4), ex1 + emin[c],
                                                      -(long long)sig2 * Ot, ex2 + emin[c])
                                         : __uint_as_float(kEngineNaN);
                    }
                }
                (h ? vB : vA)[c * vcol + sb] = v;
            }
        }
        if (!__syncthreads_and(ok)) return;  // a fill never completed: fault word raised
        if (tid == 0 && it + p.D < p.n_iter) {
            fence_proxy_async_smem();
            fill(it + p.D);
        }
        // ---- fold: one thread per (row, column) line, groups in order
        if (++hpos == p.H || it == p.n_iter - 1) {
            const int nline = hpos * p.nt * 2 * ncp;
            for (int f = tid; f < nline; f += blockDim.x) {
                const int c = f % ncp;
                const int64_t l = (int64_t)(it + 1 - hpos) * per_it + f / ncp;
                if (c < p.ncols && l < count) {
                    const float *vt = val + (int64_t)f * p.vstride;
                    float acc = 0.0f;
                    for (int b = 0; b < p.ng; ++b) acc = fadd_ftz(acc, vt[b]);
                    if (acc != acc) acc = __uint_as_float(kEngineNaN);
                    p.out[(int64_t)c * p.rows + row0 + l] = acc;
                }
            }
            hpos = 0;
            if (it != p.n_iter - 1) __syncthreads();
        }
    }
}

// ------------------------------------------------------------------ plain kernel

// One warp per (row, column): lane l takes groups l, l+32, ... through the
// exact routine, and the warp folds each 32 groups' values in order.
template <int F>
__global__ void __launch_bounds__(256) s32_plain_kernel(const uint8_t *__restrict__ W, int64_t rows, int K, int rec,
                                                        int ncols, const int8_t *__restrict__ codes,
                                                        const qb_scale *__restrict__ scales, float *__restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= rows * ncols) return;  // whole warps
    const int64_t r = wid / ncols;
    const int c = (int)(wid - r * ncols);
    const uint8_t *row = W + r * rec;
    const uint8_t *ac = reinterpret_cast<const uint8_t *>(codes + (int64_t)c * K);
    const uint32_t *sc = reinterpret_cast<const uint32_t *>(scales) + (int64_t)c * (K / 32);
    const int ng = K / 256;
    float acc = 0.0f;
    for (int g0 = 0; g0 < ng; g0 += 32) {
        const int gi = g0 + lane;
        const float v = gi < ng ? group_value_exact<F>(row, K, gi, ac, 0, false, sc + 8 * gi) : 0.0f;
        const int nv = min(32, ng - g0);
        for (int i = 0; i < nv; ++i) acc = fadd_ftz(acc, __shfl_sync(0xFFFFFFFFu, v, i));
    }
    if (lane == 0) out[(int64_t)c * rows + r] = (acc != acc) ? __uint_as_float(kEngineNaN) : acc;
}

// ------------------------------------------------------------------ launch

template <int F, int CG>
bool s32_shape(int64_t rows, int64_t K, int ncols, S32K &k, int &grid, int &threads, int &smem, bool fused = false) {
    constexpr int kThreads = gemv3_threads<CG>();
    const int ts = (int)(K / 128);
    const int ncg = (ncols + CG - 1) / CG, ncp = ncg * CG;
    const int tpt = ncg * ts;
    if (tpt > kThreads || ts < 2) return false;
    k.rows = rows;
    k.K = (int)K;
    k.rec = (int)record_bytes(F, K);
    k.ts = ts;
    k.ncg = ncg;
    k.ncols = ncols;
    k.ng = (int)(K / 256);
    k.vstride = (k.ng & 1) ? k.ng : k.ng + 1;
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), rows));
    const int64_t rpc = (rows + grid - 1) / grid;
    const int budget = 225 * 1024;
    k.nt = (int)std::min<int64_t>(kThreads / tpt, std::max<int64_t>(1, (rpc + 1) / 2));
    while (k.nt > 1 && s32_smem(k.K, ncols, k.rec, k.nt, ncp, 2, 1, k.vstride, fused).total > budget) --k.nt;
    if (s32_smem(k.K, ncols, k.rec, k.nt, ncp, 1, 1, k.vstride, fused).total > budget) return false;
    k.n_iter = (int)((rpc + 2LL * k.nt - 1) / (2LL * k.nt));
    k.base = rows / grid;
    k.rem = rows % grid;
    threads = (k.nt * tpt + 31) / 32 * 32;
    k.H = std::max(1, std::min({k.n_iter, 8, threads / (k.nt * 2 * ncp)}));
    const int hist = s32_smem(k.K, ncols, k.rec, k.nt, ncp, 0, k.H, k.vstride, fused).total;
    k.D = std::max(1, std::min({k.n_iter, 4, (budget - hist) / (2 * k.nt * k.rec)}));
    while (s32_smem(k.K, ncols, k.rec, k.nt, ncp, k.D, k.H, k.vstride, fused).total > budget && k.H > 1) --k.H;
    smem = s32_smem(k.K, ncols, k.rec, k.nt, ncp, k.D, k.H, k.vstride, fused).total;
    return smem <= 227 * 1024;
}

template <int F, int CG>
int launch_s32_cg(const GemvArgs &a, cudaStream_t stream, const float *x = nullptr) {
    const bool fused = x != nullptr;
    if (fused && (CG != 1 || a.ncols != 1)) return QB_E_ARG;
    const int ts = (int)(a.K / 128);
    const int per = (gemv3_threads<CG>() / ts) / CG * CG;
    if (per < 1) return QB_E_ARG;
    int *fault = fault_word();
    if (!fault) return QB_E_CUDA;
    for (int c0 = 0; c0 < a.ncols; c0 += per) {
        S32K k;
        int grid, threads, smem;
        if (!s32_shape<F, CG>(a.rows, a.K, std::min(per, a.ncols - c0), k, grid, threads, smem, fused)) return QB_E_ARG;
    }
    {
        const void *f = fused ? reinterpret_cast<const void *>(s32_kernel<F, CG, (CG == 1)>)
                              : reinterpret_cast<const void *>(s32_kernel<F, CG, false>);
        if (ensure_smem_limit(f, 227 * 1024) != QB_OK) return QB_E_CUDA;
    }
    for (int c0 = 0; c0 < a.ncols; c0 += per) {
        S32K k;
        int grid, threads, smem;
        s32_shape<F, CG>(a.rows, a.K, std::min(per, a.ncols - c0), k, grid, threads, smem, fused);
        k.W = static_cast<const uint8_t *>(a.W);
        k.out = a.out + (int64_t)c0 * a.rows;
        k.codes = fused ? nullptr : a.codes + (int64_t)c0 * a.K;
        k.scales = fused ? nullptr : a.scales + (int64_t)c0 * (a.K / 32);
        k.sums16 = (fused || !a.sums16) ? nullptr : a.sums16 + (int64_t)c0 * (a.K / 16);
        k.x = x;
        k.fault = fault;
        const int rc = fused ? launch_pdl(s32_kernel<F, CG, (CG == 1)>, dim3(grid), dim3(threads), (size_t)smem,
                                          stream, k)
                             : launch_pdl(s32_kernel<F, CG, false>, dim3(grid), dim3(threads), (size_t)smem, stream, k);
        if (rc) return rc;
    }
    return QB_OK;
}

// The Sub32 product: the streaming kernel (one column: groups of one; more:
// groups of two), else the plain kernel.
template <int F>
int launch_gemv_sub32(const GemvArgs &a, cudaStream_t stream) {
    if (a.rows < 1 || a.K < 256 || a.K % 256 != 0) return QB_E_ARG;
    const int rc = a.ncols == 1 ? launch_s32_cg<F, 1>(a, stream) : launch_s32_cg<F, 2>(a, stream);
    if (rc != QB_E_ARG) return rc;
    const int64_t warps = a.rows * a.ncols;
    const unsigned grid = (unsigned)((warps + 7) / 8);
    return launch_pdl(s32_plain_kernel<F>, dim3(grid), dim3(256), 0, stream, static_cast<const uint8_t *>(a.W), a.rows,
                      (int)a.K, (int)record_bytes(F, a.K), a.ncols, a.codes, a.scales, a.out);
}

// One column from the f32 activation in a single launch (the streaming
// kernel quantizing x in its prologue); QB_E_ARG where that kernel does not
// take the shape.
template <int F>
int launch_matvec_sub32(const GemvArgs &a, const float *x, cudaStream_t stream) {
    if (a.ncols != 1 || a.rows < 1 || a.K < 256 || a.K % 256 != 0) return QB_E_ARG;
    return launch_s32_cg<F, 1>(a, stream, x);
}

}  // namespace qb
