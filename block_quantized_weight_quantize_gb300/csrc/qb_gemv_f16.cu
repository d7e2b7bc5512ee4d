// qb_gemv_f16.cu -- F16 weights against an f16-rounded activation (numerics
// page: fdot, tree, f32_to_f16).
//
// Element i's product -- exact in f32, since two binary16 values multiply to at
// most 22 significant bits -- goes to lane i mod 8, each lane adding in index
// order from +0; the lanes fold as ((l0+l1)+(l2+l3))+((l4+l5)+(l6+l7)).  An FMA
// of an exact product rounds exactly as the separate multiply and add do.
//
// Streaming organisation (persistent CTAs, one per SM):
//   * a CTA owns a contiguous range of rows; they reach shared memory through
//     a ring of D slots of R rows, one bulk asynchronous copy per row (the TMA
//     engine) into a row pitch padded to an odd number of 16-B units, so the
//     threads reading consecutive rows hit different banks; the first fills
//     are issued before the programmatic-dependent-launch wait;
//   * four threads per row: thread p owns lanes 2p and 2p+1 for every column
//     and walks the row's 16-byte chunks in order (chunk c holds elements
//     8c..8c+7, one per lane), so each lane's sum keeps index order;
//   * the tree is finished with two shuffles: (l0+l1) + (l2+l3) on the pair of
//     threads 0,1, (l4+l5) + (l6+l7) on 2,3, then the two halves.
#include <cuda_fp16.h>

#include <algorithm>

#include "qb_common.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"

namespace qb {

struct F16K {
    MatTable mt;   // the matrix (or matrices sharing x16) as one range of rows
    int64_t rows;  // rows of the whole range
    int K;
    int pitch;     // bytes per row in shared memory (2K padded)
    int R;         // rows per ring slot
    int D;         // ring slots
    int n_iter;    // slots a CTA consumes
    int64_t base;  // rows per CTA, and how many CTAs own one more
    int64_t rem;
    const uint16_t *x16;
    int *fault;
};

__host__ __device__ inline int f16_xs_bytes(int K, int nc) { return (nc * K * 4 + 127) & ~127; }

// rows of iteration `it` into slot it % D: one bulk copy per row
__device__ __forceinline__ void f16_fill(const F16K &p, uint8_t *ring, uint64_t *bars, int it, int64_t row0,
                                         int64_t count, int lane) {
    const int slot = it % p.D;
    const int64_t first = (int64_t)it * p.R;
    const int n = (int)((count - first < p.R) ? count - first : (int64_t)p.R);
    if (lane == 0) mbar_arrive_expect_tx(bars + slot, n > 0 ? (uint32_t)n * (uint32_t)(2 * p.K) : 0u);
    __syncwarp();
    for (int r = lane; r < n; r += 32)
        bulk_g2s(ring + ((int64_t)slot * p.R + r) * p.pitch, row_ptr(p.mt, row0 + first + r, 2 * p.K),
                 (uint32_t)(2 * p.K), bars + slot);
}

template <int NC>
__global__ void __launch_bounds__(256) gemv_f16_kernel(const F16K p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    float *xs = reinterpret_cast<float *>(smem + 128);  // [NC][K], exact widening of x16
    uint8_t *ring = smem + 128 + f16_xs_bytes(p.K, NC);

    const int tid = threadIdx.x, lane = tid & 31;
    const int rr = tid >> 2, pp = tid & 3;  // row within the slot, lane pair
    const int64_t c = blockIdx.x;
    const int64_t row0 = c * p.base + (c < p.rem ? c : p.rem);
    const int64_t count = p.base + (c < p.rem ? 1 : 0);

    if (tid == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid < 32)
        for (int it = 0; it < p.D && it < p.n_iter; ++it) f16_fill(p, ring, bars, it, row0, count, lane);
    pdl_wait();
    for (int i = tid; i < NC * p.K; i += blockDim.x) xs[i] = __half2float(__ushort_as_half(p.x16[i]));
    __syncthreads();
    pdl_launch_dependents();

    const int n8 = p.K / 8;
    for (int it = 0; it < p.n_iter; ++it) {
        const int slot = it % p.D;
        const int64_t l = (int64_t)it * p.R + rr;  // row within the CTA's range
        const bool have = l < count;
        bool ok = true;
        if (have) ok = mbar_wait_bounded(bars + slot, (uint32_t)((it / p.D) & 1), p.fault);
        float acc0[NC], acc1[NC];
#pragma unroll
        for (int q = 0; q < NC; ++q) { acc0[q] = 0.0f; acc1[q] = 0.0f; }
        if (have && ok) {
            const uint32_t *wr = reinterpret_cast<const uint32_t *>(ring + ((int64_t)slot * p.R + rr) * p.pitch) + pp;
#pragma unroll 4
            for (int k = 0; k < n8; ++k) {
                const uint32_t w2 = wr[4 * k];  // elements 8k+2pp, 8k+2pp+1: lanes 2pp, 2pp+1
                const float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&w2));
#pragma unroll
                for (int q = 0; q < NC; ++q) {
                    const float2 xv = *reinterpret_cast<const float2 *>(xs + q * p.K + 8 * k + 2 * pp);
                    acc0[q] = fmaf(wf.x, xv.x, acc0[q]);
                    acc1[q] = fmaf(wf.y, xv.y, acc1[q]);
                }
            }
        }
        // tree: thread pp holds lanes (2pp, 2pp+1)
#pragma unroll
        for (int q = 0; q < NC; ++q) {
            const float pair = __fadd_rn(acc0[q], acc1[q]);              // (l0+l1), (l2+l3), (l4+l5), (l6+l7)
            const float quad = __fadd_rn(pair, __shfl_xor_sync(0xFFFFFFFFu, pair, 1));  // on even pp
            const float all = __fadd_rn(quad, __shfl_xor_sync(0xFFFFFFFFu, quad, 2));   // on pp == 0
            if (have && ok && pp == 0) {
                float r = all;
                if (r != r) r = __uint_as_float(kEngineNaN);
                *out_ptr(p.mt, q, row0 + l) = r;
            }
        }
        if (!__syncthreads_and(ok)) return;  // a fill never completed: fault word raised
        if (tid < 32 && it + p.D < p.n_iter) {
            if (tid == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            f16_fill(p, ring, bars, it + p.D, row0, count, lane);
        }
    }
}

// ------------------------------------------------------------------ warp rings
// The same arithmetic with every warp streaming its own groups of 8 rows
// through D slots of its own: a slot is refilled as soon as its warp has used
// it (a bulk copy per row into the padded pitch, completing on the warp's
// slot mbarrier), so no warp waits at a CTA-wide barrier for a refill.  The
// CTA's rows are contiguous; warp w takes its 8-row groups w, w + nw, ...
// FUSED: the activation is rounded to f16 here (f32_to_f16, as
// quantize_act_f16 does) and widened to f32 in shared memory.
struct F16WK {
    MatTable mt;
    int64_t rows;
    int K;
    int pitch;  // bytes per row in a slot (2K padded to an odd number of 16-B units)
    int D;      // slots a warp
    int nw;     // warps a CTA
    int64_t base;
    int64_t rem;
    const uint16_t *x16;
    const float *x32;  // FUSED: the f32 activation
    int *fault;
};

__host__ __device__ inline int f16w_smem(int K, int nc, int pitch, int D, int nw) {
    return 256 + f16_xs_bytes(K, nc) + nw * D * 8 * pitch;
}

template <int NC, bool FUSED>
__global__ void __launch_bounds__(256) gemv_f16w_kernel(const F16WK p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int rr = lane >> 2, pp = lane & 3;  // row of the group, lane pair
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem) + w * p.D;
    float *xs = reinterpret_cast<float *>(smem + 256);
    uint8_t *ring = smem + 256 + f16_xs_bytes(p.K, NC) + (int64_t)w * p.D * 8 * p.pitch;
    const int64_t c = blockIdx.x;
    const int64_t row0 = c * p.base + (c < p.rem ? c : p.rem);
    const int64_t count = p.base + (c < p.rem ? 1 : 0);
    const int64_t ngroups = (count + 7) / 8;
    const uint32_t rowb = (uint32_t)(2 * p.K);

    if (lane == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // the fill of this warp's j-th group into slot j % D
    auto fill = [&](int j) {
        const int64_t gi = w + (int64_t)j * p.nw;
        if (gi >= ngroups) return;
        const int slot = j % p.D;
        const int n = (int)(count - 8 * gi < 8 ? count - 8 * gi : 8);
        if (lane == 0) mbar_arrive_expect_tx(bars + slot, (uint32_t)n * rowb);
        __syncwarp();
        if (lane < n)
            bulk_g2s(ring + ((int64_t)slot * 8 + lane) * p.pitch, row_ptr(p.mt, row0 + 8 * gi + lane, rowb), rowb,
                     bars + slot);
    };
    for (int j = 0; j < p.D; ++j) fill(j);  // weights depend on no earlier kernel
    pdl_wait();
    if (FUSED) {
        for (int i = tid; i < NC * p.K; i += blockDim.x) xs[i] = __half2float(__float2half_rn(__ldg(p.x32 + i)));
    } else {
        for (int i = tid; i < NC * p.K; i += blockDim.x) xs[i] = __half2float(__ushort_as_half(p.x16[i]));
    }
    __syncthreads();
    pdl_launch_dependents();

    const int n8 = p.K / 8;
    for (int j = 0;; ++j) {
        const int64_t gi = w + (int64_t)j * p.nw;
        if (gi >= ngroups) break;
        const int slot = j % p.D;
        const bool ok = mbar_wait_bounded(bars + slot, (uint32_t)((j / p.D) & 1), p.fault);
        if (!__all_sync(0xFFFFFFFFu, ok)) return;  // a fill never completed: fault word raised
        const int64_t l = 8 * gi + rr;              // row within the CTA's range
        const bool have = l < count;
        float acc0[NC], acc1[NC];
#pragma unroll
        for (int q = 0; q < NC; ++q) { acc0[q] = 0.0f; acc1[q] = 0.0f; }
        if (have) {
            const uint32_t *wr = reinterpret_cast<const uint32_t *>(ring + ((int64_t)slot * 8 + rr) * p.pitch) + pp;
#pragma unroll 4
            for (int k = 0; k < n8; ++k) {
                const uint32_t w2 = wr[4 * k];  // elements 8k+2pp, 8k+2pp+1: lanes 2pp, 2pp+1
                const float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&w2));
#pragma unroll
                for (int q = 0; q < NC; ++q) {
                    const float2 xv = *reinterpret_cast<const float2 *>(xs + q * p.K + 8 * k + 2 * pp);
                    acc0[q] = fmaf(wf.x, xv.x, acc0[q]);
                    acc1[q] = fmaf(wf.y, xv.y, acc1[q]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < NC; ++q) {
            const float pair = __fadd_rn(acc0[q], acc1[q]);                             // (l0+l1) .. (l6+l7)
            const float quad = __fadd_rn(pair, __shfl_xor_sync(0xFFFFFFFFu, pair, 1));  // on even pp
            const float all = __fadd_rn(quad, __shfl_xor_sync(0xFFFFFFFFu, quad, 2));   // on pp == 0
            if (have && pp == 0) {
                float r = all;
                if (r != r) r = __uint_as_float(kEngineNaN);
                *out_ptr(p.mt, q, row0 + l) = r;
            }
        }
        __syncwarp();  // every lane has read the slot
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        fill(j + p.D);
    }
}

template <int NC>
static int launch_f16w_nc(const F16WK &k, int smem, unsigned grid, bool fused, cudaStream_t stream) {
    const void *f = fused ? reinterpret_cast<const void *>(gemv_f16w_kernel<NC, true>)
                          : reinterpret_cast<const void *>(gemv_f16w_kernel<NC, false>);
    if (ensure_smem_limit(f, 227 * 1024) != QB_OK) return QB_E_CUDA;
    return fused ? launch_pdl(gemv_f16w_kernel<NC, true>, dim3(grid), dim3(32 * k.nw), (size_t)smem, stream, k)
                 : launch_pdl(gemv_f16w_kernel<NC, false>, dim3(grid), dim3(32 * k.nw), (size_t)smem, stream, k);
}

// The warp-ring kernel over a table of matrices: 8 warps a CTA (or as many
// as fit with two slots each, at least 4), up to 3 slots a warp; QB_E_ARG
// when fewer than 4 warps fit.
static int launch_f16w_table(const MatTable &t, int64_t K, const uint16_t *x16, const float *x32, int ncols,
                             cudaStream_t stream) {
    F16WK k;
    k.mt = t;
    k.rows = t.start[t.n];
    k.K = (int)K;
    const int units = (int)(K / 8);
    k.pitch = 16 * (units + ((units & 1) ? 2 : 1));  // odd number of 16-B units
    const int budget = 227 * 1024 - 1024;
    k.nw = 8;
    while (k.nw > 4 && f16w_smem(k.K, ncols, k.pitch, 2, k.nw) > budget) --k.nw;
    if (f16w_smem(k.K, ncols, k.pitch, 2, k.nw) > budget) return QB_E_ARG;
    k.D = 2;
    while (k.D < 3 && f16w_smem(k.K, ncols, k.pitch, k.D + 1, k.nw) <= budget) ++k.D;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), (k.rows + 8 * k.nw - 1) / (8 * k.nw)));
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    k.x16 = x16;
    k.x32 = x32;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    const int smem = f16w_smem(k.K, ncols, k.pitch, k.D, k.nw);
    const bool fused = x32 != nullptr;
    switch (ncols) {
#define QB_CASE(N) \
    case N: return launch_f16w_nc<N>(k, smem, (unsigned)grid, fused, stream);
        QB_CASE(1) QB_CASE(2) QB_CASE(3) QB_CASE(4) QB_CASE(5) QB_CASE(6) QB_CASE(7) QB_CASE(8)
        QB_CASE(9) QB_CASE(10) QB_CASE(11) QB_CASE(12) QB_CASE(13) QB_CASE(14) QB_CASE(15) QB_CASE(16)
#undef QB_CASE
    }
    return QB_E_ARG;
}

// Rows longer than the streaming kernel's shared-memory ring allows: one
// thread per row, the row read straight from global memory in 16-byte chunks.
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
__global__ void __launch_bounds__(128) gemv_f16_rowthread_kernel(const uint16_t *__restrict__ W, int64_t rows, int K,
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
static int launch_f16_rowthread(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, float *out,
                                cudaStream_t stream) {
    const size_t smem = (size_t)NC * K * sizeof(float);
    if (ensure_smem_limit(reinterpret_cast<const void *>(gemv_f16_rowthread_kernel<NC>), 227 * 1024) != QB_OK)
        return QB_E_CUDA;
    const unsigned grid = (unsigned)((rows + 127) / 128);
    return launch_pdl(gemv_f16_rowthread_kernel<NC>, dim3(grid), dim3(128), smem, stream, W, rows, (int)K, x16, out);
}

template <int NC>
static int launch_f16_nc(const F16K &k, int smem, unsigned grid, int threads, cudaStream_t stream) {
    if (ensure_smem_limit(reinterpret_cast<const void *>(gemv_f16_kernel<NC>), 227 * 1024) != QB_OK)
        return QB_E_CUDA;
    return launch_pdl(gemv_f16_kernel<NC>, dim3(grid), dim3(threads), (size_t)smem, stream, k);
}

// The streaming kernel over a table of matrices; QB_E_ARG when a slot of 8
// rows does not fit (then only the row-per-thread kernel takes the shape).
static int launch_f16_table(const MatTable &t, int64_t K, const uint16_t *x16, int ncols, cudaStream_t stream) {
    F16K k;
    k.mt = t;
    k.rows = t.start[t.n];
    const int64_t rows = k.rows;
    k.K = (int)K;
    const int units = (int)(K / 8);  // 16-B units per row
    k.pitch = 16 * (units + ((units & 1) ? 2 : 1));  // odd number of units
    const int sms = num_sms();
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, (rows + 31) / 32));
    k.base = rows / grid;
    k.rem = rows % grid;
    const int64_t rpc = (rows + grid - 1) / grid;
    const int xsb = f16_xs_bytes((int)K, ncols);
    const int budget = 200 * 1024 - 128 - xsb;
    if (budget < 8 * k.pitch) return QB_E_ARG;
    // rows per slot: a multiple of 8 (whole warps), at most 64, at least two slots
    k.R = (int)std::min<int64_t>(64, std::max<int64_t>(8, (rpc + 7) / 8 * 8));
    while (k.R > 8 && 2 * k.R * k.pitch > budget) k.R -= 8;
    k.n_iter = (int)((rpc + k.R - 1) / k.R);
    k.D = std::max(1, std::min(k.n_iter, std::min(4, budget / (k.R * k.pitch))));
    k.x16 = x16;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    const int smem = 128 + xsb + k.D * k.R * k.pitch;
    const int threads = 4 * k.R;
    switch (ncols) {
#define QB_CASE(N) \
    case N: return launch_f16_nc<N>(k, smem, (unsigned)grid, threads, stream);
        QB_CASE(1) QB_CASE(2) QB_CASE(3) QB_CASE(4) QB_CASE(5) QB_CASE(6) QB_CASE(7) QB_CASE(8)
        QB_CASE(9) QB_CASE(10) QB_CASE(11) QB_CASE(12) QB_CASE(13) QB_CASE(14) QB_CASE(15) QB_CASE(16)
#undef QB_CASE
    }
    return QB_E_ARG;
}

int launch_gemv_f16(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, int ncols, float *out,
                    cudaStream_t stream) {
    int rc = launch_f16w_table(single_table(W, rows, out), K, x16, nullptr, ncols, stream);
    if (rc != QB_E_ARG) return rc;
    rc = launch_f16_table(single_table(W, rows, out), K, x16, ncols, stream);
    if (rc != QB_E_ARG) return rc;
    switch (ncols) {  // a slot of 8 rows does not fit: the row-per-thread kernel
#define QB_CASE(N) \
    case N: return launch_f16_rowthread<N>(W, rows, K, x16, out, stream);
        QB_CASE(1) QB_CASE(2) QB_CASE(3) QB_CASE(4) QB_CASE(5) QB_CASE(6) QB_CASE(7) QB_CASE(8)
        QB_CASE(9) QB_CASE(10) QB_CASE(11) QB_CASE(12) QB_CASE(13) QB_CASE(14) QB_CASE(15) QB_CASE(16)
#undef QB_CASE
    }
    return QB_E_ARG;
}

int launch_gemv_f16_many(const MatTable &t, int64_t K, const uint16_t *x16, int ncols, cudaStream_t stream) {
    const int rc = launch_f16w_table(t, K, x16, nullptr, ncols, stream);
    return rc != QB_E_ARG ? rc : launch_f16_table(t, K, x16, ncols, stream);
}

int launch_matvec_f16(const MatTable &t, int64_t K, const float *x, int ncols, cudaStream_t stream) {
    return launch_f16w_table(t, K, nullptr, x, ncols, stream);
}

}  // namespace qb
