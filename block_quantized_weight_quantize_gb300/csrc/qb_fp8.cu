// qb_fp8.cu -- FP8 E4M3 weights with 128x128 block scales against an f32
// activation (colizig OPS page, FP8: e4m3ToF32, dequantRow, matmulFp8).
//
// A weight is its E4M3 byte decoded ([s:1][e:4][m:3], bias 7, subnormals,
// S.1111.111 NaN, no infinity) times the f32 scale of its 128x128 block; a
// row's dot with each activation column is taken in f32.  This is a float
// path on the page (checked there against "dequantize then f32 matmul"); its
// result is held to the f32 summation bound (K + 4) * 2^-24 * sum |x_i*w_i|
// around the exact dot of the dequantized weights.
//
// Decode in registers (the page's S = 1 form, no weight buffer): the
// hardware's exact e4m3x2 -> f16x2 conversion on both half words of a 32-bit
// weight word, then f16 -> f32.  One warp
// takes a row at a time; lane l owns the 16-byte chunks l, l + 32, ... (16
// weights each, all in one scale block), so a warp's loads are 512 contiguous
// bytes; per chunk the 16 products are summed by an FMA chain and added into
// the row's sum times the chunk's block scale; the 32 lanes fold by shuffles.
// The activation is staged in shared memory in the order the lanes read it
// (lane l's float4 q of chunk j at (4j + q) * 32 + l), so the reads are
// conflict-free.
#include <cuda_fp16.h>

#include <algorithm>

#include "qb_common.cuh"
#include "qb_launch.h"

namespace qb {

// four E4M3 bytes (byte i of the word is weight i) to f32, exactly: the
// hardware's e4m3x2 -> f16x2 conversion on each half word, then f16 -> f32
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t four, float &w0, float &w1, float &w2, float &w3) {
    uint32_t h01, h23;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.rn.f16x2.e4m3x2 %0, lo; cvt.rn.f16x2.e4m3x2 %1, hi; }"
        : "=r"(h01), "=r"(h23) : "r"(four));
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
    w0 = a.x; w1 = a.y; w2 = b.x; w3 = b.y;
}

struct Fp8K {
    const uint8_t *W;
    const float *scales;
    int64_t rows;
    int K;
    int kb;     // scale blocks along K
    int nc;     // columns of this launch
    const float *x;  // column 0 of this launch [nc][K]
    float *out;      // column 0 of this launch (out[c * rows + r])
};

// RPW rows a warp at a time (two for four or more columns: each staged
// activation read then serves both rows).  The first batch of a warp's
// weights is loaded before the programmatic-dependent-launch wait and the
// activation staging (weights depend on no earlier kernel).  FULL: K a
// multiple of 4096 (a lane's 16-byte chunks come in whole batches of 8 rounds
// of 32), so no chunk needs a bounds test.
template <int NC, int RPW, bool FULL>
__global__ void __launch_bounds__(256) gemv_fp8_kernel(const Fp8K p) {
    extern __shared__ __align__(16) float4 xs[];  // [NC][128 * nj] in lane order
    const int lane = threadIdx.x & 31;
    const int nch = p.K / 16;        // 16-byte chunks a row
    const int nj = (nch + 31) / 32;  // chunks a lane (the last partial)
    const int cs = 128 * nj;         // float4 a column in shared memory (whole rounds of 32 chunks)
    const int nf = p.K / 4;          // float4 a column in x
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t r0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW;

    uint4 w[RPW][8];
    float s[RPW][8];
    auto load = [&](int64_t r, int j0) {
#pragma unroll
        for (int q = 0; q < RPW; ++q) {
            const bool rin = r + q < p.rows;
            const uint8_t *wr = p.W + (r + q) * p.K;
            const float *sr = p.scales + ((r + q) / 128) * p.kb;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int ch = lane + 32 * (j0 + u);
                const bool in = rin && (FULL || (j0 + u < nj && ch < nch));
                w[q][u] = in ? __ldg(reinterpret_cast<const uint4 *>(wr) + ch) : make_uint4(0, 0, 0, 0);
                s[q][u] = in ? __ldg(sr + (ch >> 3)) : 0.0f;
            }
        }
    };
    if (r0 < p.rows) load(r0, 0);

    pdl_launch_dependents();
    pdl_wait();
#pragma unroll
    for (int c = 0; c < NC; ++c)
        for (int f = threadIdx.x; f < nf; f += blockDim.x) {
            const int ch = f >> 2, q = f & 3, l = ch & 31, j = ch >> 5;
            xs[c * cs + (4 * j + q) * 32 + l] =
                c < p.nc ? __ldg(reinterpret_cast<const float4 *>(p.x + (int64_t)c * p.K) + f) : make_float4(0, 0, 0, 0);
        }
    __syncthreads();
    bool first = true;
    for (int64_t r = r0; r < p.rows; r += nw * RPW) {
        float acc[RPW][NC];
#pragma unroll
        for (int q = 0; q < RPW; ++q)
#pragma unroll
            for (int c = 0; c < NC; ++c) acc[q][c] = 0.0f;
        for (int j0 = 0; j0 < nj; j0 += 8) {
            if (!first) load(r, j0);
            first = false;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                if (!FULL && (j >= nj || lane + 32 * j >= nch)) break;
                float wf[RPW][16];
#pragma unroll
                for (int q = 0; q < RPW; ++q) {
                    const uint32_t wv[4] = {w[q][u].x, w[q][u].y, w[q][u].z, w[q][u].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        e4m3x4_to_f32(wv[k], wf[q][4 * k], wf[q][4 * k + 1], wf[q][4 * k + 2], wf[q][4 * k + 3]);
                }
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const float4 *xc = xs + c * cs + (4 * j) * 32 + lane;
                    float t[RPW];
#pragma unroll
                    for (int q = 0; q < RPW; ++q) t[q] = 0.0f;
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const float4 xv = xc[32 * k4];
#pragma unroll
                        for (int q = 0; q < RPW; ++q) {
                            t[q] = fmaf(wf[q][4 * k4], xv.x, t[q]);
                            t[q] = fmaf(wf[q][4 * k4 + 1], xv.y, t[q]);
                            t[q] = fmaf(wf[q][4 * k4 + 2], xv.z, t[q]);
                            t[q] = fmaf(wf[q][4 * k4 + 3], xv.w, t[q]);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < RPW; ++q) acc[q][c] = fmaf(t[q], s[q][u], acc[q][c]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < RPW; ++q)
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float v = acc[q][c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                if (lane == 0 && c < p.nc && r + q < p.rows)
                    p.out[(int64_t)c * p.rows + r + q] = (v != v) ? __uint_as_float(kEngineNaN) : v;
            }
    }
}

__host__ __device__ inline size_t fp8_smem(int NC, int64_t K) { return (size_t)NC * ((K / 16 + 31) / 32) * 2048; }

// Two rows a warp for every column count: at one row a warp, 4096 rows took
// 512 CTAs of 256 threads, more than the register file holds at once (three
// a SM at 78 registers), so the last CTAs ran as a second wave.  The grid is
// clamped to what is resident at once (the occupancy calculator); the rows
// past it loop within the warps.
template <int NC>
static int launch_fp8_nc(const Fp8K &k, cudaStream_t stream) {
    constexpr int RPW = 2;
    const size_t smem = fp8_smem(NC, k.K);
    const bool full = k.K % 4096 == 0;  // a lane's chunks come in whole batches of 8 rounds of 32
    {
        const void *f = full ? reinterpret_cast<const void *>(gemv_fp8_kernel<NC, RPW, true>)
                             : reinterpret_cast<const void *>(gemv_fp8_kernel<NC, RPW, false>);
        if (ensure_smem_limit(f, 200 * 1024) != QB_OK) return QB_E_CUDA;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm,
            full ? reinterpret_cast<const void *>(gemv_fp8_kernel<NC, RPW, true>)
                 : reinterpret_cast<const void *>(gemv_fp8_kernel<NC, RPW, false>),
            256, smem) != cudaSuccess)
        return QB_E_CUDA;
    per_sm = std::max(1, per_sm);
    const int64_t blocks = (k.rows + 8 * RPW - 1) / (8 * RPW);
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)num_sms() * per_sm));
    return full ? launch_pdl(gemv_fp8_kernel<NC, RPW, true>, dim3(grid), dim3(256), smem, stream, k)
                : launch_pdl(gemv_fp8_kernel<NC, RPW, false>, dim3(grid), dim3(256), smem, stream, k);
}

// Columns in launches of at most 16 (a power of two) that fit 200 KB of
// staged activation.
int launch_gemv_fp8(const uint8_t *W, const float *scales, int64_t rows, int64_t K, const float *x, int ncols,
                    float *out, cudaStream_t stream) {
    int cmax = 16;
    while (cmax > 1 && fp8_smem(cmax, K) > 200 * 1024) cmax >>= 1;
    if (fp8_smem(cmax, K) > 200 * 1024) return QB_E_ARG;
    for (int c0 = 0; c0 < ncols; c0 += cmax) {
        Fp8K k;
        k.W = W;
        k.scales = scales;
        k.rows = rows;
        k.K = (int)K;
        k.kb = (int)((K + 127) / 128);
        k.nc = std::min(cmax, ncols - c0);
        k.x = x + (int64_t)c0 * K;
        k.out = out + (int64_t)c0 * rows;
        int rc;
        if (k.nc == 1) rc = launch_fp8_nc<1>(k, stream);
        else if (k.nc == 2) rc = launch_fp8_nc<2>(k, stream);
        else if (k.nc <= 4) rc = launch_fp8_nc<4>(k, stream);
        else if (k.nc <= 8) rc = launch_fp8_nc<8>(k, stream);
        else rc = launch_fp8_nc<16>(k, stream);
        if (rc) return rc;
    }
    return QB_OK;
}

}  // namespace qb
