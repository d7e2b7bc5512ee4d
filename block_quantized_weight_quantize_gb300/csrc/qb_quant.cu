// qb_quant.cu -- activation quantization kernels.
//
// quantize_act: the decode engine's quantize_blocks under ActScaling::PerBlock
// (numerics page): per block, absmax (a denormal read as zero, NaN passed
// over), wide_scale (the least m*2^e, m in 128..255, with 127*m*2^e >= amax)
// and rne_div (the nearest integer of x/(m*2^e), ties to even, exactly) --
// all in integer arithmetic on the f32 bit fields.  It also writes the sum of
// the codes of every 16-element unit (the activation side's unit sums of the
// block-scale lane page).
//
// quantize_act_f16: f32_to_f16 (numerics page) by the hardware conversion
// cvt.rn.f16.f32, NaN canonicalised.
#include <cuda_fp16.h>

#include "qb_common.cuh"
#include "qb_launch.h"

namespace qb {

// One thread per 8 consecutive elements; a block of B elements spans B/8
// consecutive lanes of one warp (4 lanes for B = 32, 32 lanes for B = 256).
template <int B>
__global__ void __launch_bounds__(256) quantize_act_kernel(const float *__restrict__ x, int64_t n8, int K,
                                                           int8_t *__restrict__ codes, qb_scale *__restrict__ scales,
                                                           int16_t *__restrict__ sums16) {
    constexpr int L = B / 8;  // lanes per block
    pdl_launch_dependents();
    pdl_wait();  // x may come from the previous kernel; codes may still be read by it
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const bool live = t < n8;
    uint32_t xb[8];
    if (live) {
        const float4 *p = reinterpret_cast<const float4 *>(x + t * 8);
        const float4 v0 = __ldg(p), v1 = __ldg(p + 1);
        xb[0] = __float_as_uint(v0.x); xb[1] = __float_as_uint(v0.y);
        xb[2] = __float_as_uint(v0.z); xb[3] = __float_as_uint(v0.w);
        xb[4] = __float_as_uint(v1.x); xb[5] = __float_as_uint(v1.y);
        xb[6] = __float_as_uint(v1.z); xb[7] = __float_as_uint(v1.w);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xb[i] = 0;
    }
    // absmax on magnitudes' bits: denormal -> 0, NaN skipped, +inf kept
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t a = xb[i] & 0x7FFFFFFFu;
        if (a < 0x00800000u || a > 0x7F800000u) a = 0;
        amax = a > amax ? a : amax;
    }
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) {
        const uint32_t u = __shfl_xor_sync(0xFFFFFFFFu, amax, o);
        amax = u > amax ? u : amax;
    }
    // wide_scale on amax = M * 2^(E8-150): the least 8-bit significand at
    // e = E8-141 is ceil(M / (127*2^9)); past 255 the next exponent is taken.
    int m, e;
    if (amax == 0x7F800000u) {
        m = 0; e = 0;  // an infinity: no scale
    } else if (amax == 0) {
        m = 128; e = 0;
    } else {
        const uint32_t E8 = amax >> 23, M = (amax & 0x7FFFFFu) | 0x800000u;
        uint32_t mm = (M + 65023u) / 65024u;
        int ee = (int)E8 - 141;
        if (mm > 255u) { mm = (M + 130047u) / 130048u; ++ee; }
        m = (int)mm; e = ee;
    }
    // rne_div per element: |x| = mant * 2^(E8x-150); x/s = mant / (m * 2^k), k = e - (E8x-150) >= 9
    int q[8];
    int usum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t a = xb[i] & 0x7FFFFFFFu;
        int c = 0;
        if (m != 0 && a >= 0x00800000u && a < 0x7F800000u) {
            const uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
            const int k = e - ((int)(a >> 23) - 150);
            if (k < 32) {
                const uint32_t hi = mant >> k, lo = mant & ((1u << k) - 1u), half = 1u << (k - 1);
                const uint32_t qq = hi / (uint32_t)m;
                const int t2 = 2 * (int)(hi - qq * (uint32_t)m) - m;  // (2R - m*2^k) = t2*2^k + 2*lo
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
        usum += c;
    }
    // unit sums: two lanes (16 elements) per unit
    usum += __shfl_xor_sync(0xFFFFFFFFu, usum, 1);
    if (live) {
        const uint32_t w0 = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
                            ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
        const uint32_t w1 = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) |
                            ((uint32_t)(q[6] & 0xFF) << 16) | ((uint32_t)(q[7] & 0xFF) << 24);
        *reinterpret_cast<uint2 *>(codes + t * 8) = make_uint2(w0, w1);
        if ((t & 1) == 0) sums16[t >> 1] = (int16_t)usum;
        if ((t & (L - 1)) == 0) {
            qb_scale s;
            s.m = (uint8_t)m; s._pad = 0; s.e = (int16_t)e;
            scales[t / L] = s;
        }
    }
}

__global__ void __launch_bounds__(256) quantize_f16_kernel(const float *__restrict__ x, int64_t n,
                                                           uint16_t *__restrict__ x16) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n) return;
    const float v = __ldg(x + t);
    uint16_t h = __half_as_ushort(__float2half_rn(v));
    if ((h & 0x7C00u) == 0x7C00u && (h & 0x03FFu)) h = 0x7E00u;  // canonical quiet NaN
    x16[t] = h;
}

int launch_quantize_act(int block, const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales,
                        int16_t *sums16, cudaStream_t stream) {
    const int64_t n8 = K * ncols / 8;
    const unsigned grid = (unsigned)((n8 + 255) / 256);
    // every grid's blocks begin at a multiple of the block's lanes (K % block == 0)
    if (block == 32)
        return launch_pdl(quantize_act_kernel<32>, grid, 256, 0, stream, x, n8, (int)K, codes, scales, sums16);
    return launch_pdl(quantize_act_kernel<256>, grid, 256, 0, stream, x, n8, (int)K, codes, scales, sums16);
}

int launch_quantize_f16(const float *x, int64_t n, uint16_t *x16, cudaStream_t stream) {
    const unsigned grid = (unsigned)((n + 255) / 256);
    return launch_pdl(quantize_f16_kernel, grid, 256, 0, stream, x, n, x16);
}

}  // namespace qb
