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
// quantize_act_sub32: quantize under ActScaling::Sub32 (numerics page): per
// ACT_BLOCK = 32 elements, block_scale (the least m*2^e, m in 8..15, with
// 127*m*2^e >= amax), then rne_div as above; the same unit sums.
//
// quantize_act_f16: f32_to_f16 (numerics page) by the hardware conversion
// cvt.rn.f16.f32, NaN canonicalised.
#include <cuda_fp16.h>

#include "qb_common.cuh"
#include "qb_launch.h"
#include "qb_quant.cuh"

namespace qb {

// One thread per 8 consecutive elements; a block of B elements spans B/8
// consecutive lanes of one warp (4 lanes for B = 32, 32 lanes for B = 256).
template <int B, bool S32>
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
    uint2 c;
    int usum;
    uint32_t scale;
    quantize8<L, S32>(xb, c, usum, scale);
    if (live) {
        *reinterpret_cast<uint2 *>(codes + t * 8) = c;
        if ((t & 1) == 0) sums16[t >> 1] = (int16_t)usum;
        if ((t & (L - 1)) == 0) reinterpret_cast<uint32_t *>(scales)[t / L] = scale;
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
        return launch_pdl(quantize_act_kernel<32, false>, grid, 256, 0, stream, x, n8, (int)K, codes, scales, sums16);
    return launch_pdl(quantize_act_kernel<256, false>, grid, 256, 0, stream, x, n8, (int)K, codes, scales, sums16);
}

int launch_quantize_sub32(const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales, int16_t *sums16,
                          cudaStream_t stream) {
    const int64_t n8 = K * ncols / 8;
    const unsigned grid = (unsigned)((n8 + 255) / 256);
    return launch_pdl(quantize_act_kernel<32, true>, grid, 256, 0, stream, x, n8, (int)K, codes, scales, sums16);
}

int launch_quantize_f16(const float *x, int64_t n, uint16_t *x16, cudaStream_t stream) {
    const unsigned grid = (unsigned)((n + 255) / 256);
    return launch_pdl(quantize_f16_kernel, grid, 256, 0, stream, x, n, x16);
}

}  // namespace qb
