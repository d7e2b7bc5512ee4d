// qb_gemv6.cuh -- the one-column product of the 256-element formats at
// K = 4096 with a ring per warp.
//
// The arithmetic is the other streaming kernels' (the lane's exact block sums
// from the same half-block routines, the exact combine rounded once, the row
// folded in block order from +0).  The organisation differs: at K = 4096 a
// team (K/128 threads, one 128-element half-slice each) is exactly one warp,
// so every warp streams its own pairs of rows through D slots of its own --
// one bulk copy of the two (contiguous) rows into a slot, completing on the
// warp's slot mbarrier -- and refills a slot as soon as it has used it.  The
// two halves of a block swap one partial through a shuffle, and each row's 16
// block values are folded in order by one lane through shuffles: no
// CTA-wide barrier after the prologue, so no warp waits for a slower one's
// refill.  Warp w of a CTA takes the CTA's row pairs w, w + 16, ...
#pragma once

#include <algorithm>
#include <type_traits>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_gemv3.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"
#include "qb_quant.cuh"

namespace qb {

struct Gemv6K {
    MatTable mt;   // the matrix (or matrices sharing the activation) as one row range
    int64_t rows;  // rows of the whole range
    int rec;       // bytes per row record
    int D;         // slots a warp (two rows each)
    int64_t base;  // rows per CTA, and how many CTAs own one more
    int64_t rem;
    const int8_t *codes;  // the quantized activation (not FUSED)
    const qb_scale *scales;
    const int16_t *sums16;
    const float *x;  // FUSED: the f32 activation, quantized in the prologue
    int *fault;
};

constexpr int kG6K = 4096;     // K this kernel takes
constexpr int kG6Warps = 16;   // warps a CTA

// shared memory: D mbarriers per warp, the staged activation (codes, unit
// sums, block scales), each warp's 32 block values for the row fold, then the
// warps' rings
__host__ __device__ inline int gemv6_fold_offset() { return 1024 + kG6K + (kG6K / 16) * 2 + (kG6K / 256) * 4 + 128; }
__host__ __device__ inline int gemv6_ring_offset() { return gemv6_fold_offset() + kG6Warps * 32 * 4; }
__host__ __device__ inline int gemv6_smem(int rec, int D) { return gemv6_ring_offset() + kG6Warps * D * 2 * rec; }

template <int F, bool FUSED>
__global__ void __launch_bounds__(512, 1) gemv6_kernel(const Gemv6K p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int j = lane, sb = j >> 1, h = j & 1, jj = j & 7;  // half-slice j of K
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem) + w * p.D;
    uint8_t *act = smem + 1024;
    int16_t *asum = reinterpret_cast<int16_t *>(smem + 1024 + kG6K);
    uint32_t *ascl = reinterpret_cast<uint32_t *>(smem + 1024 + kG6K + (kG6K / 16) * 2);
    uint8_t *ring = smem + gemv6_ring_offset() + (int64_t)w * p.D * 2 * p.rec;
    float *fv = reinterpret_cast<float *>(smem + gemv6_fold_offset()) + 32 * w;

    const int64_t c = blockIdx.x;
    const int64_t row0 = c * p.base + (c < p.rem ? c : p.rem);
    const int64_t count = p.base + (c < p.rem ? 1 : 0);
    const int64_t npairs = (count + 1) / 2;

    if (lane == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // the fill of this warp's k-th pair (range pair w + 16k) into slot k % D
    auto fill = [&](int k) {
        const int64_t pi = w + (int64_t)k * kG6Warps;
        if (pi >= npairs || lane != 0) return;
        const int slot = k % p.D;
        const int64_t n = count - 2 * pi < 2 ? count - 2 * pi : 2;
        mbar_arrive_expect_tx(bars + slot, (uint32_t)(n * p.rec));
        fill_rows(p.mt, ring + (int64_t)slot * 2 * p.rec, row0 + 2 * pi, n, p.rec, bars + slot);
    };
    for (int k = 0; k < p.D; ++k) fill(k);  // weights depend on no earlier kernel
    // the next launch may be scheduled now: it reads nothing this one writes
    // before its own pdl_wait, which returns once this grid has finished
    pdl_launch_dependents();
    pdl_wait();

    // ---- the activation, once per CTA: codes in the multi-column kernel's
    // swizzled layout (16-B unit u at (u & ~7) | ((u & 7) ^ ((u >> 3) & 7))),
    // unit sums and block scales; the single-launch form quantizes x here (a
    // thread per 8 consecutive elements, a 256-element block on one warp)
    if constexpr (FUSED) {
        const int g8 = tid;  // K/8 = 512 groups: one a thread
        const float4 *xp = reinterpret_cast<const float4 *>(p.x) + 2 * g8;
        const float4 v0 = ldg_f4_ordered(xp), v1 = ldg_f4_ordered(xp + 1);
        const uint32_t xb[8] = {__float_as_uint(v0.x), __float_as_uint(v0.y), __float_as_uint(v0.z),
                                __float_as_uint(v0.w), __float_as_uint(v1.x), __float_as_uint(v1.y),
                                __float_as_uint(v1.z), __float_as_uint(v1.w)};
        uint2 cd;
        int usum;
        uint32_t scale;
        quantize8<32>(xb, cd, usum, scale);
        const int u = g8 >> 1;
        const int pos = (u & ~7) | ((u & 7) ^ ((u >> 3) & 7));
        *reinterpret_cast<uint2 *>(act + 16 * pos + 8 * (g8 & 1)) = cd;
        if ((g8 & 1) == 0) asum[u] = (int16_t)usum;
        if ((g8 & 31) == 0) ascl[g8 / 32] = scale;
    } else {
        if (tid < kG6K / 16) {  // 256 units of 16 codes
            const int u = tid;
            const uint4 v = ldg_v4_ordered(reinterpret_cast<const uint4 *>(p.codes) + u);
            const int pos = (u & ~7) | ((u & 7) ^ ((u >> 3) & 7));
            *reinterpret_cast<uint4 *>(act + 16 * pos) = v;
        } else if (tid < kG6K / 16 + kG6K / 32) {  // 128 words of unit sums (256 int16)
            const int i = tid - kG6K / 16;
            reinterpret_cast<uint32_t *>(asum)[i] = ldg_u32_ordered(reinterpret_cast<const uint32_t *>(p.sums16) + i);
        } else if (tid < kG6K / 16 + kG6K / 32 + kG6K / 256) {  // 16 block scales
            const int i = tid - kG6K / 16 - kG6K / 32;
            ascl[i] = ldg_u32_ordered(reinterpret_cast<const uint32_t *>(p.scales) + i);
        }
    }
    __syncthreads();
    // my half-slice's codes, unit sums and block scale
    uint4 a[1][8];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[0][k] = *reinterpret_cast<const uint4 *>(act + 128 * j + 16 * (k ^ jj));
    uint32_t S[1][4] = {{0, 0, 0, 0}};
    {
        const uint4 sw = *reinterpret_cast<const uint4 *>(asum + 8 * j);
        const uint32_t pw[4] = {sw.x, sw.y, sw.z, sw.w};
        if (F == kQ4K) {  // per-32 sums of my four sub-blocks from the per-16 ones
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                const int Sv = (int)(int16_t)(pw[s2] & 0xFFFFu) + (int)(int16_t)(pw[s2] >> 16);
                S[0][s2 >> 1] |= ((uint32_t)Sv & 0xFFFFu) << (16 * (s2 & 1));
            }
        } else {
            S[0][0] = pw[0]; S[0][1] = pw[1]; S[0][2] = pw[2]; S[0][3] = pw[3];
        }
    }
    const uint32_t sv = ascl[sb];
    const int m0 = (int)(sv & 0xFFu), e0 = (int)(int16_t)(sv >> 16);

    // ---- this warp's row pairs
    for (int k = 0;; ++k) {
        const int64_t pi = w + (int64_t)k * kG6Warps;
        if (pi >= npairs) break;
        const int slot = k % p.D;
        const bool ok = mbar_wait_bounded(bars + slot, (uint32_t)((k / p.D) & 1), p.fault);
        if (!__all_sync(0xFFFFFFFFu, ok)) return;  // a fill never completed: fault word raised
        const uint8_t *rA = ring + (int64_t)slot * 2 * p.rec, *rB = rA + p.rec;
        const bool hasB = 2 * pi + 1 < count;
        int CA[1] = {0}, CB[1] = {0}, OA[1] = {0}, OB[1] = {0};
        uint32_t dA = 0, dB = 0;
        if (F == kQ4K) {
            half_q4k_cg<1>(rA + 144 * sb, h, a, S, CA, OA, dA);
            if (hasB) half_q4k_cg<1>(rB + 144 * sb, h, a, S, CB, OB, dB);
        } else {
            half_q6k_cg<1>(rA + 208 * sb, h, a, S, CA);
            dA = *reinterpret_cast<const uint16_t *>(rA + 208 * 16 + 2 * sb);
            if (hasB) {
                half_q6k_cg<1>(rB + 208 * sb, h, a, S, CB);
                dB = *reinterpret_cast<const uint16_t *>(rB + 208 * 16 + 2 * sb);
            }
        }
        __syncwarp();  // every lane has read the slot
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        fill(k + p.D);
        // partner lane (the block's other half) swaps one partial: lane h = 0
        // finishes block sb of row A, lane h = 1 of row B
        const int rC = __shfl_xor_sync(0xFFFFFFFFu, h ? CA[0] : CB[0], 1);
        const int rO = (F == kQ4K) ? __shfl_xor_sync(0xFFFFFFFFu, h ? OA[0] : OB[0], 1) : 0;
        float v = 0.0f;
        if (!h || hasB) {
            const int Cs = (h ? CB[0] : CA[0]) + rC, O = (h ? OB[0] : OA[0]) + rO;
            const int C = (F == kQ4K) ? (Cs >> 4) : Cs;  // Q4_K: the halves hold 16*C (exact shift)
            const uint32_t dd = h ? dB : dA;
            v = (F == kQ4K) ? lane_value_fast<1>(C, O, dd & 0xFFFFu, dd >> 16, m0, e0)
                            : lane_value_fast<0>(C, 0, dd, 0, m0, e0);
        }
        // fold: the block values go to the warp's strip, row A's 16 (lanes 0,
        // 2, ..., 30) then row B's; lane 0 adds row A's in block order from
        // +0, lane 1 row B's
        fv[16 * h + sb] = v;
        __syncwarp();
        if (lane < 2 && (lane == 0 || hasB)) {
            const float4 *q4 = reinterpret_cast<const float4 *>(fv + 16 * lane);
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 t = q4[i];
                acc = fadd_ftz(acc, t.x);
                acc = fadd_ftz(acc, t.y);
                acc = fadd_ftz(acc, t.z);
                acc = fadd_ftz(acc, t.w);
            }
            if (acc != acc) acc = __uint_as_float(kEngineNaN);
            *out_ptr(p.mt, 0, row0 + 2 * pi + lane) = acc;
        }
        __syncwarp();  // the strip is read before the next pair writes it
    }
}

// The kernel for one column of a Q4_K-like or Q6_K-like matrix (or a table of
// them) at K = 4096: every Q6_K-like shape, and Q4_K-like ones up to 48 rows a
// CTA, where it measured faster than the other streaming kernels (single
// launch: Q4_K-like 4096 rows 3.95 -> 3.84 us, 6144 rows 5.50 -> 5.23 us;
// Q6_K-like 4096 rows 4.70 -> 4.56 us, 128256 rows 82.0 -> 65.7 us); the
// one-column gemv3 form stayed faster for Q4_K-like at 14336 and 28672 rows
// (7.9 against 8.6 us, 13.3 against 14.0 us).  x given: the single-launch
// form.  QB_E_ARG otherwise.
template <int F>
int launch_gemv6(const GemvArgs &a, cudaStream_t stream, const float *x) {
    if ((F != kQ4K && F != kQ6K) || a.ncols != 1 || a.mode != 0 || a.K != kG6K) return QB_E_ARG;
    Gemv6K k;
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.rows = k.mt.start[k.mt.n];
    if (k.rows < 1) return QB_E_ARG;
    {
        const int64_t g = std::max<int64_t>(1, std::min<int64_t>(num_sms(), (k.rows + 1) / 2));
        if (F == kQ4K && (k.rows + g - 1) / g > 3 * kG6Warps) return QB_E_ARG;  // more than 48 rows a CTA
    }
    k.rec = (int)record_bytes(F, kG6K);
    const int budget = 225 * 1024;
    k.D = 1;
    while (k.D < 4 && gemv6_smem(k.rec, k.D + 1) <= budget) ++k.D;
    if (k.D < 2) return QB_E_ARG;  // two slots a warp at least (Q4_K-like: 3, Q6_K-like: 2)
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), (k.rows + 1) / 2));
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.x = x;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    const int smem = gemv6_smem(k.rec, k.D);
    const bool fused = x != nullptr;
    {
        const void *f = fused ? reinterpret_cast<const void *>(gemv6_kernel<F, true>)
                              : reinterpret_cast<const void *>(gemv6_kernel<F, false>);
        if (ensure_smem_limit(f, 227 * 1024) != QB_OK) return QB_E_CUDA;
    }
    return fused ? launch_pdl(gemv6_kernel<F, true>, dim3(grid), dim3(512), (size_t)smem, stream, k)
                 : launch_pdl(gemv6_kernel<F, false>, dim3(grid), dim3(512), (size_t)smem, stream, k);
}

}  // namespace qb
