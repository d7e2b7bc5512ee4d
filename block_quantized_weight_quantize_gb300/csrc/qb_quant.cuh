// qb_quant.cuh -- the activation quantizer as device functions, shared by the
// quantize_act kernel and the single-launch product kernel.
//
// The decode engine's quantize_blocks under ActScaling::PerBlock (numerics
// page): per block, absmax (a denormal read as zero, NaN passed over),
// wide_scale (the least m*2^e, m in 128..255, with 127*m*2^e >= amax) and
// rne_div (the nearest integer of x/(m*2^e), ties to even, exactly).  The
// scale comes from the integer fields of amax; the division takes an f32
// path whose result is certain away from half-integers and an exact integer
// routine otherwise.  A thread holds 8 consecutive elements; a block of B
// elements spans B/8 consecutive lanes of a warp.
#pragma once

#include "qb_common.cuh"

namespace qb {

// wide_scale of amax = M * 2^(E8-150) (M the 24-bit significand): at
// e = E8-141 the least 8-bit significand is ceil(M / (127*2^9)), which lies in
// 130..259; past 255 the next exponent is taken.  m = 0 marks an infinity,
// an all-zero block gets 128 * 2^0.
__device__ __forceinline__ void wide_scale_bits(uint32_t amax, int &m, int &e) {
    if (amax == 0x7F800000u) { m = 0; e = 0; return; }
    if (amax == 0) { m = 128; e = 0; return; }
    const uint32_t E8 = amax >> 23, M = (amax & 0x7FFFFFu) | 0x800000u;
    uint32_t mm = (M + 65023u) / 65024u;
    int ee = (int)E8 - 141;
    if (mm > 255u) { mm = (M + 130047u) / 130048u; ++ee; }
    m = (int)mm;
    e = ee;
}

// block_scale (numerics page, ActScaling::Sub32): the same search with a 4-bit
// significand.  At e = E8-137 the least m is ceil(M / (127*2^13)), in 9..17;
// past 15 the next exponent gives ceil(M / (127*2^14)), 8 or 9.  m = 0 marks
// an infinity, an all-zero block gets 8 * 2^0.
__device__ __forceinline__ void block_scale_bits(uint32_t amax, int &m, int &e) {
    if (amax == 0x7F800000u) { m = 0; e = 0; return; }
    if (amax == 0) { m = 8; e = 0; return; }
    const uint32_t E8 = amax >> 23, M = (amax & 0x7FFFFFu) | 0x800000u;
    uint32_t mm = (M + 1040383u) / 1040384u;
    int ee = (int)E8 - 137;
    if (mm > 15u) { mm = (M + 2080767u) / 2080768u; ++ee; }
    m = (int)mm;
    e = ee;
}

// rne_div of one element, exactly, on the integer fields: |x| = mant *
// 2^(E8x-150), so x/s = mant / (m * 2^k) with k = e - (E8x-150).  Every
// |x| <= amax has |x/s| <= 127, which forces k >= 9 for m <= 255 and k >= 13
// for m <= 15; k >= 22 puts |x/s| below 1/2 for any m >= 8, code 0.
// Otherwise hi = mant >> k (< 2^15 for m >= 128, < 2^11 for m <= 15), and
// floor(hi / m) is (hi * ceil(2^24/m)) >> 24: the product overestimates hi/m
// by less than hi/2^24 < 1/m, so the floor is exact, and it fits 32 bits
// (hi * ceil(2^24/m) < 2^15 * 2^17 for m >= 128, < 2^11 * 2^21 for m >= 8).  With rem = hi - q*m and lo = mant mod 2^k, the remainder is
// R = rem*2^k + lo, and 2R - m*2^k = (2*rem - m)*2^k + 2*lo decides the
// rounding, ties to even.  A denormal, NaN or (m = 0) element gets code 0.
// Out of line: only the rare elements the fast path below cannot decide
// come here, and keeping it out of the hot code keeps that code short.
static __device__ __noinline__ int rne_div1_exact(uint32_t xbits, int m, int e) {
    const uint32_t a = xbits & 0x7FFFFFFFu;
    const int k = e - ((int)(a >> 23) - 150);
    const bool valid = (m != 0) & (a >= 0x00800000u) & (a < 0x7F800000u) & (k <= 21);
    const int kc = valid ? k : 9;
    const uint32_t mu = valid ? (uint32_t)m : 128u;
    const uint32_t magic = ((1u << 24) + mu - 1u) / mu;
    const uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
    const uint32_t hi = mant >> kc, lo = mant & ((1u << kc) - 1u), half = 1u << (kc - 1);
    const uint32_t qq = (hi * magic) >> 24;
    const int t2 = 2 * (int)(hi - qq * mu) - (int)mu;  // in [-m, m-2]
    const uint32_t thr = t2 == 0 ? 0u : half;           // t2 = 0: up iff lo > 0; t2 = -1: iff lo > half
    const bool up = (t2 >= 1) | ((t2 >= -1) & ((lo > thr) | ((lo == thr) & (qq & 1u))));
    const int c = valid ? (int)qq + (up ? 1 : 0) : 0;
    return (xbits & 0x80000000u) ? -c : c;
}

// Quantize the 8 elements xb of a block spanning L lanes: returns the codes
// packed in two words, the sum of the 16-element unit this lane pair forms,
// and the block's scale packed as m | e << 16 (identical on the L lanes).
// Every lane of the warp must call it (shuffles).
//
// absmax: max of |x| with denormal inputs flushed to zero (abs.ftz), NaN
// passed over (max returns the other operand), +inf kept.
// rne_div fast path in f32: c = RN(1/m) * 2^-e is exact (an exponent-field
// subtraction; a normal number for e in [-134, 118] when m is 128..255, in
// [-130, 122] when m is 8..15), and qf = RN(x * c) with
// denormal inputs and results flushed (both mean |x/s| < 1/2, code 0) is
// RN(x' * RN(1/m)) for x' = x * 2^-e, within |x/s| * 2^-23 (1 + 2^-23) <
// 2^-16 of x/s (|x/s| <= 127).  So unless qf lies within 2^-16 of a
// half-integer, x/s lies on the same side of every half-integer as qf and its
// nearest integer is that of qf, found by one add of 1.5*2^23 (all on the FMA
// pipe; no conversion instruction).  Elements in that band (exact ties among
// them), and blocks with e outside the range, take the exact routine.
// S32: the scale is block_scale (ActScaling::Sub32) instead of wide_scale.
template <int L, bool S32 = false>
__device__ __forceinline__ void quantize8(const uint32_t (&xb)[8], uint2 &codes, int &unit_sum, uint32_t &scale) {
    float ax[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) asm("abs.ftz.f32 %0, %1;" : "=f"(ax[i]) : "f"(__uint_as_float(xb[i])));
    // a tree of fmaxf (a NaN operand yields the other), then against +0: the
    // same maximum as folding from +0 in any order
    const float am = fmaxf(0.0f, fmaxf(fmaxf(fmaxf(ax[0], ax[1]), fmaxf(ax[2], ax[3])),
                                       fmaxf(fmaxf(ax[4], ax[5]), fmaxf(ax[6], ax[7]))));
    uint32_t amax = __float_as_uint(am);  // non-negative: ordered as an unsigned integer
    if (L == 32) {
        amax = __reduce_max_sync(0xFFFFFFFFu, amax);
    } else {
#pragma unroll
        for (int o = L / 2; o > 0; o >>= 1) {
            const uint32_t u = __shfl_xor_sync(0xFFFFFFFFu, amax, o);
            amax = u > amax ? u : amax;
        }
    }
    int m, e;
    if (S32) block_scale_bits(amax, m, e);
    else wide_scale_bits(amax, m, e);
    int q[8];  // byte 0 of each: the element's code
    if ((m != 0) & (e >= (S32 ? -130 : -134)) & (e <= (S32 ? 122 : 118))) {
        const float inv_m = __frcp_rn((float)m);
        const float c = __uint_as_float(__float_as_uint(inv_m) - ((uint32_t)e << 23));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float qf;
            asm("mul.rn.ftz.f32 %0, %1, %2;" : "=f"(qf) : "f"(__uint_as_float(xb[i])), "f"(c));
            // the nearest integer n of qf, ties to even, on the FMA pipe: |qf| <=
            // 127 + 2^-16, so qf + 1.5*2^23 rounds (to nearest even) to
            // 1.5*2^23 + n, an f32 whose bits are 0x4B400000 + n -- byte 0 is n
            // as an int8; d = qf - n is exact.  The band, and NaN (which fails
            // every comparison), take the exact routine.
            const float r = __fadd_rn(qf, 12582912.0f);
            const float d = __fsub_rn(qf, __fsub_rn(r, 12582912.0f));
            int v = (int)__float_as_uint(r);
            if (!(fabsf(d) < 0.5f - 0x1p-16f)) v = rne_div1_exact(xb[i], m, e);
            q[i] = v;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = rne_div1_exact(xb[i], m, e);
    }
    codes.x = __byte_perm(__byte_perm(q[0], q[1], 0x0040), __byte_perm(q[2], q[3], 0x0040), 0x5410);
    codes.y = __byte_perm(__byte_perm(q[4], q[5], 0x0040), __byte_perm(q[6], q[7], 0x0040), 0x5410);
    const int s = dp4a_ss(codes.y, 0x01010101u, dp4a_ss(codes.x, 0x01010101u, 0));
    unit_sum = s + __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    scale = (uint32_t)(m & 0xFF) | ((uint32_t)(uint16_t)(int16_t)e << 16);
}

}  // namespace qb
