// qb_gemv_f16.cu -- F16 weights against an f16-rounded activation (numerics
// page, fdot / tree / f32_to_f16).
//
// Each thread owns one row and keeps its 8 lane accumulators in registers:
// element i's product -- exact in f32, since two binary16 values multiply to
// at most 22 significant bits -- is added to lane i mod 8 in index order from
// +0, and the lanes fold as ((l0+l1)+(l2+l3))+((l4+l5)+(l6+l7)).  An FMA of an
// exact product rounds exactly as the separate multiply and add do.  The
// activation, widened to f32 (exactly), sits in shared memory and is read as
// broadcasts; the row streams through 16-byte non-coherent loads, four in
// flight per thread.
#include <cuda_fp16.h>

#include "qb_common.cuh"
#include "qb_launch.h"

namespace qb {

__device__ __forceinline__ uint4 ldg_nc16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void widen8(const uint4 w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&u[k]));
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
}

template <int NC>
__global__ void __launch_bounds__(128) gemv_f16_kernel(const uint16_t *__restrict__ W, int64_t rows, int K,
                                                       const uint16_t *__restrict__ x16, float *__restrict__ out) {
    extern __shared__ __align__(16) float xs[];  // [NC][K], exact widening of x16
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint4 *wp = reinterpret_cast<const uint4 *>(W + row * (int64_t)K);
    const int n8 = K / 8;
    // the first weights need nothing from earlier kernels
    uint4 pre = make_uint4(0, 0, 0, 0);
    if (row < rows) pre = ldg_nc16(wp);
    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i < NC * K; i += blockDim.x) xs[i] = __half2float(__ushort_as_half(x16[i]));
    __syncthreads();
    if (row >= rows) return;
    float l[NC][8];
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) l[c][j] = 0.0f;
    uint4 cur = pre;
    for (int j = 0; j < n8; ++j) {
        const uint4 nxt = (j + 1 < n8) ? ldg_nc16(wp + j + 1) : make_uint4(0, 0, 0, 0);
        float wf[8];
        widen8(cur, wf);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const float4 x0 = *reinterpret_cast<const float4 *>(xs + c * K + 8 * j);
            const float4 x1 = *reinterpret_cast<const float4 *>(xs + c * K + 8 * j + 4);
            l[c][0] = fmaf(wf[0], x0.x, l[c][0]);
            l[c][1] = fmaf(wf[1], x0.y, l[c][1]);
            l[c][2] = fmaf(wf[2], x0.z, l[c][2]);
            l[c][3] = fmaf(wf[3], x0.w, l[c][3]);
            l[c][4] = fmaf(wf[4], x1.x, l[c][4]);
            l[c][5] = fmaf(wf[5], x1.y, l[c][5]);
            l[c][6] = fmaf(wf[6], x1.z, l[c][6]);
            l[c][7] = fmaf(wf[7], x1.w, l[c][7]);
        }
        cur = nxt;
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const float t = __fadd_rn(__fadd_rn(l[c][0], l[c][1]), __fadd_rn(l[c][2], l[c][3]));
        const float u = __fadd_rn(__fadd_rn(l[c][4], l[c][5]), __fadd_rn(l[c][6], l[c][7]));
        float r = __fadd_rn(t, u);
        if (r != r) r = __uint_as_float(kEngineNaN);
        out[(int64_t)c * rows + row] = r;
    }
}

template <int NC>
static int launch_f16_nc(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, float *out,
                         cudaStream_t stream) {
    const size_t smem = (size_t)NC * K * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(gemv_f16_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
            cudaSuccess)
            return QB_E_CUDA;
        attr_set = true;
    }
    const unsigned grid = (unsigned)((rows + 127) / 128);
    return launch_pdl(gemv_f16_kernel<NC>, dim3(grid), dim3(128), smem, stream, W, rows, (int)K, x16, out);
}

int launch_gemv_f16(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, int ncols, float *out,
                    cudaStream_t stream) {
    if ((int64_t)ncols * K * 4 > 227 * 1024) return QB_E_ARG;
    switch (ncols) {
#define QB_CASE(N) \
    case N: return launch_f16_nc<N>(W, rows, K, x16, out, stream);
        QB_CASE(1) QB_CASE(2) QB_CASE(3) QB_CASE(4) QB_CASE(5) QB_CASE(6) QB_CASE(7) QB_CASE(8)
        QB_CASE(9) QB_CASE(10) QB_CASE(11) QB_CASE(12) QB_CASE(13) QB_CASE(14) QB_CASE(15) QB_CASE(16)
#undef QB_CASE
    }
    return QB_E_ARG;
}

}  // namespace qb
