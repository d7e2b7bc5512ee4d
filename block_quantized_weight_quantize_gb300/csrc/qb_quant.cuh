// qb_quant.cuh -- the activation quantizer as device functions, shared by the
// quantize_act kernel and the single-launch product kernel.
//
// The decode engine's quantize_blocks under ActScaling::PerBlock (numerics
// page): per block, absmax (a denormal read as zero, NaN passed over),
// wide_scale (the least m*2^e, m in 128..255, with 127*m*2^e >= amax) and
// rne_div (the nearest integer of x/(m*2^e), ties to even, exactly), all on
// the integer fields of the f32 values.  A thread holds 8 consecutive
// elements; a block of B elements spans B/8 consecutive lanes of a warp.
#pragma once

#include "qb_common.cuh"

namespace qb {

// |x| bits for absmax: a denormal reads as 0, NaN is passed over, +inf kept.
__device__ __forceinline__ uint32_t absmax_bits8(const uint32_t (&xb)[8]) {
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t a = xb[i] & 0x7FFFFFFFu;
        if (a < 0x00800000u || a > 0x7F800000u) a = 0;
        amax = a > amax ? a : amax;
    }
    return amax;
}

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

// rne_div for 8 elements under m*2^e.  |x| = mant * 2^(E8x-150), so
// x/s = mant / (m * 2^k) with k = e - (E8x-150) >= 9 for every |x| <= amax
// (|x/s| <= 127 forces it), hence hi = mant >> k < 2^15.  floor(hi / m) is
// (hi * ceil(2^24/m)) >> 24: the product overestimates hi/m by less than
// hi/2^24 < 2^-9 < 1/m, so the floor is exact for m < 512.  The remainder
// R = (hi - q*m)*2^k + lo against half the divisor decides the rounding,
// ties to even.  A denormal, NaN or (m = 0) element gets code 0.
__device__ __forceinline__ void rne_div8(const uint32_t (&xb)[8], int m, int e, int (&q)[8]) {
    const uint32_t magic = m ? (((1u << 24) + (uint32_t)m - 1u) / (uint32_t)m) : 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a = xb[i] & 0x7FFFFFFFu;
        int c = 0;
        if (m != 0 && a >= 0x00800000u && a < 0x7F800000u) {
            const uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
            const int k = e - ((int)(a >> 23) - 150);
            if (k < 32) {
                const uint32_t hi = mant >> k, lo = mant & ((1u << k) - 1u), half = 1u << (k - 1);
                const uint32_t qq = (uint32_t)(((unsigned long long)hi * magic) >> 24);
                const int t2 = 2 * (int)(hi - qq * (uint32_t)m) - m;  // 2R - m*2^k = t2*2^k + 2*lo
                bool up;
                if (t2 >= 1) up = true;
                else if (t2 <= -2) up = false;
                else if (t2 == -1) up = lo > half || (lo == half && (qq & 1u));
                else up = lo > 0 || (qq & 1u);
                c = (int)qq + (up ? 1 : 0);
            }
            if (xb[i] & 0x80000000u) c = -c;
        }
        q[i] = c;
    }
}

// Quantize the 8 elements xb of a block spanning L lanes: returns the codes
// packed in two words, the sum of the 16-element unit this lane pair forms,
// and the block's scale packed as m | e << 16 (identical on the L lanes).
// Every lane of the warp must call it (shuffles).
template <int L>
__device__ __forceinline__ void quantize8(const uint32_t (&xb)[8], uint2 &codes, int &unit_sum, uint32_t &scale) {
    uint32_t amax = absmax_bits8(xb);
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) {
        const uint32_t u = __shfl_xor_sync(0xFFFFFFFFu, amax, o);
        amax = u > amax ? u : amax;
    }
    int m, e;
    wide_scale_bits(amax, m, e);
    int q[8];
    rne_div8(xb, m, e, q);
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += q[i];
    unit_sum = s + __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    codes.x = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) | ((uint32_t)(q[2] & 0xFF) << 16) |
              ((uint32_t)(q[3] & 0xFF) << 24);
    codes.y = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) | ((uint32_t)(q[6] & 0xFF) << 16) |
              ((uint32_t)(q[7] & 0xFF) << 24);
    scale = (uint32_t)(m & 0xFF) | ((uint32_t)(uint16_t)(int16_t)e << 16);
}

}  // namespace qb
