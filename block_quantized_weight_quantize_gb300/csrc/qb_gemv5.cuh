// qb_gemv5.cuh -- the Q4_K-like product for 11..16 activation columns with
// the sub-block dot products on the tensor cores (below 11 columns the dp4a
// streaming kernel measures faster: the MMA's 16 column slots are then
// mostly padding).
//
// Per block the lane's sums are C = sum_s sc_s * sum_{i in s} q_i a_i and
// O = sum_s mn_s * S_s (lane page: block_sums).  C is a dense contraction of
// the weights' coefficients sc_s*q_i (integers 0..945) with the activation
// codes a (integers -127..127) -- and both are exact in f16, and every
// partial sum over a 128-element half block is an integer of magnitude at
// most 945 * 127 * 128 < 2^24, exact in f32.  So an f16 tensor-core product
// with f32 accumulation (mma.sync m16n8k16) gives each half block's C
// exactly, in any order of accumulation; the two halves are added as
// integers.  O stays on the integer pipeline (dp2a over packed 16-bit
// sub-block sums), and the combine, rounding and row fold are those of the
// other kernels, so every value is the bits the one-column product gives.
//
// Roles in the MMA: A = activation, 16 columns x 16 k (column m = fragment
// row); B = weights, 16 k x 8 rows; D = 16 columns x 8 rows.  The order of
// k inside one MMA is free as long as A and B agree; it is chosen to match
// the nibble layout: thread (g = lane/4, t = lane%4) holds, for a 16-element
// chunk, k-slots (2t, 2t+1) = elements (4t, 4t+2) and slots (2t+8, 2t+9) =
// elements (4t+1, 4t+3) -- so one 32-bit word of a sub-block's nibbles
// (bytes 4t..4t+3) yields both of its B registers for the low-nibble chunk
// and both for the high-nibble chunk.
//
// Nibble to f16: the half word 0x6400 | n is 1024 + n; one fused multiply-add
// (1024 + n)*sc - 1024*sc = n*sc rounds once, so the result (an integer
// <= 945) is exact.  High nibbles sit at bit 4 (1024 + 16 n), scaled by
// sc/16 and offset by -64 sc.  Activation codes a: 0x6400 | (a ^ 0x80) is
// 1152 + a, and one subtraction leaves a exactly.
//
// Organisation: persistent CTAs of 16 warps over contiguous row ranges;
// rows arrive by bulk copies into a ring of chunks of R rows (R a multiple
// of 8).  Warp w takes blocks w, w+16, ... (K <= 4096: at most one), keeps
// that block's activation fragments (16 k-steps x 4 registers) in
// registers, and for each 8-row tile of the chunk runs 16 MMAs (8 sub-blocks
// x low/high nibbles) into two accumulators (the block's halves), then the
// exact combine for its (row, column) pairs.  Block values go to shared
// memory and one thread per (row, column) folds them in block order.
#pragma once

#include <algorithm>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"

namespace qb {

struct Gemv5K {
    MatTable mt;   // the matrix (or matrices sharing the activation)
    int64_t rows;  // rows of the whole range
    int K;
    int rec;
    int pitch;    // bytes between rows in a ring slot: rec padded to an odd number of 16-B units
    int nb;       // blocks per row (<= 16)
    int ncols;    // 11..16 real columns
    int R;        // rows per chunk (multiple of 8)
    int D;        // ring slots
    int vstride;  // floats per (row, column) line of block values (odd)
    int n_iter;
    int64_t base;
    int64_t rem;
    const int8_t *codes;
    const qb_scale *scales;
    const int16_t *sums16;
    int *fault;
};

struct Gemv5Smem {
    int bars, act, val, ring, total;
};

// act: the activation codes, 16 columns x K bytes at a column stride of
// K + 16 (fragment reads land on distinct banks); val: block values of a
// chunk; ring: D slots of R rows at the padded pitch.
__host__ __device__ inline Gemv5Smem gemv5_smem(int K, int pitch, int R, int D, int vstride) {
    Gemv5Smem s;
    s.bars = 0;
    s.act = 128;
    s.val = s.act + 16 * (K + 16);
    s.ring = s.val + ((R * 16 * vstride * 4 + 127) & ~127);
    s.total = s.ring + D * R * pitch;
    return s;
}

__host__ __device__ inline int gemv5_pitch(int rec) { return ((rec / 16) & 1) ? rec : rec + 16; }

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hadd2_u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// f16x2 constants (bit patterns)
constexpr uint32_t kH2Magic = 0x64006400u;     // (1024, 1024)
constexpr uint32_t kH2M1024 = 0xE400E400u;     // (-1024, -1024)
constexpr uint32_t kH2M1152 = 0xE480E480u;     // (-1152, -1152)
constexpr uint32_t kH2Sixteenth = 0x2C002C00u; // (1/16, 1/16)
constexpr uint32_t kH2M64 = 0xD400D400u;       // (-64, -64)

// Activation fragment registers of one 16-element chunk for columns g and
// g+8: a[0] = (x_g[4t], x_g[4t+2]), a[1] = the same for column g+8,
// a[2] = (x_g[4t+1], x_g[4t+3]), a[3] = column g+8.  w0, w1: the four codes
// x[4t..4t+3] of the two columns as words.
__device__ __forceinline__ void act_frag(uint32_t w0, uint32_t w1, uint32_t (&a)[4]) {
    w0 ^= 0x80808080u;
    w1 ^= 0x80808080u;
    a[0] = hadd2_u(__byte_perm(w0, 0x64646464u, 0x4240), kH2M1152);
    a[2] = hadd2_u(__byte_perm(w0, 0x64646464u, 0x4341), kH2M1152);
    a[1] = hadd2_u(__byte_perm(w1, 0x64646464u, 0x4240), kH2M1152);
    a[3] = hadd2_u(__byte_perm(w1, 0x64646464u, 0x4341), kH2M1152);
}

// The combine for a row whose scales are unreadable or whose two scale
// exponents are too far apart for the 64-bit form (out of line: rare).
static __device__ __noinline__ float lane_value_cold(int C, int O, uint32_t dd, int m, int e) {
    return lane_value<1>(C, O, dd & 0xFFFFu, dd >> 16, m, e);
}

// Per-row part of the combine: the decoded block scales of a row and how
// the two terms align (numerics page: exact_sum; lane page: lane).
struct RowScale {
    int sig1, sig2, sh1, sh2, E;  // value = (sig1*m*C << sh1) - (sig2*m*O << sh2) at 2^(E+e)
    bool fast;                    // both scales readable and the spread fits the 64-bit form
};
__device__ __forceinline__ RowScale row_scale(uint32_t dd) {
    RowScale r;
    int ex1, ex2;
    const bool ok = f16_scale(dd & 0xFFFFu, r.sig1, ex1) & f16_scale(dd >> 16, r.sig2, ex2);
    const int d = ex1 - ex2;
    r.fast = ok & (d >= -21) & (d <= 17);
    r.sh1 = d > 0 ? d : 0;
    r.sh2 = d < 0 ? -d : 0;
    r.E = d >= 0 ? ex2 : ex1;
    return r;
}
// |sig*m| < 2^19, |C| < 2^25, |O| < 2^21: t1 << sh1 and t2 << sh2 stay below 2^61.
__device__ __forceinline__ float combine_fast(const RowScale &r, uint32_t dd, int C, int O, int m, int e) {
    if (!r.fast || m == 0) return m == 0 ? __uint_as_float(kEngineNaN) : lane_value_cold(C, O, dd, m, e);
    const long long t1 = (long long)(r.sig1 * m) * (long long)C;
    const long long t2 = -(long long)(r.sig2 * m) * (long long)O;
    return round_fast((t1 << r.sh1) + (t2 << r.sh2), r.E + e);
}

template <int F>
__global__ void __launch_bounds__(512, 1) gemv5_kernel(const Gemv5K p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const Gemv5Smem L = gemv5_smem(p.K, p.pitch, p.R, p.D, p.vstride);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint8_t *act = smem + L.act;
    float *val = reinterpret_cast<float *>(smem + L.val);
    uint8_t *ring = smem + L.ring;

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int64_t cta = blockIdx.x;
    const int64_t row0 = cta * p.base + (cta < p.rem ? cta : p.rem);
    const int64_t count = p.base + (cta < p.rem ? 1 : 0);

    if (tid == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // the fill of chunk `it` by warp 0: one bulk copy per row (lane i: rows
    // i, i+32, ...) into the padded pitch, all on the slot's mbarrier
    auto fill = [&](int it) {
        const int slot = it % p.D;
        const int64_t first = (int64_t)it * p.R;
        const int64_t n = count - first < p.R ? count - first : (int64_t)p.R;
        if (lane == 0) mbar_arrive_expect_tx(bars + slot, n > 0 ? (uint32_t)(n * p.rec) : 0u);
        __syncwarp();
        for (int64_t r = lane; r < n; r += 32)
            bulk_g2s(ring + ((int64_t)slot * p.R + r) * p.pitch, row_ptr(p.mt, row0 + first + r, p.rec),
                     (uint32_t)p.rec, bars + slot);
    };
    if (w == 0)
        for (int it = 0; it < p.D && it < p.n_iter; ++it) fill(it);  // weights depend on no earlier kernel
    pdl_wait();
    pdl_launch_dependents();  // a following kernel waits for this grid before it writes anything read here

    // ---- the activation codes of all columns into shared memory (zeros past
    // ncols), 16-B loads
    {
        const int upc = p.K / 16;  // 16-B units per column
        constexpr int kU = 8;      // loads in flight per thread
        for (int u0 = tid; u0 < 16 * upc; u0 += kU * (int)blockDim.x) {
            uint4 v[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int u = u0 + q * (int)blockDim.x, c = u / upc, uu = u - c * upc;
                v[q] = (u < 16 * upc && c < p.ncols)
                           ? ldg_v4_ordered(reinterpret_cast<const uint4 *>(p.codes + (int64_t)c * p.K) + uu)
                           : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int u = u0 + q * (int)blockDim.x, c = u / upc, uu = u - c * upc;
                if (u < 16 * upc) *reinterpret_cast<uint4 *>(act + c * (p.K + 16) + 16 * uu) = v[q];
            }
        }
    }
    // this warp's block: sub-block sums and scales of columns g and g+8
    const int b = w;
    const bool has_block = b < p.nb;
    const int c0 = g, c1 = g + 8;
    const bool in0 = c0 < p.ncols, in1 = c1 < p.ncols;
    uint32_t S0[4] = {0, 0, 0, 0}, S1[4] = {0, 0, 0, 0};  // sub-block sums (16-bit pairs), columns c0, c1
    int m0a = 128, e0a = 0, m0b = 128, e0b = 0;
    if (has_block && in0) {
        // per-16 unit sums u_0..u_15 of the block; S_s = u_{2s} + u_{2s+1}
        const uint4 *su = reinterpret_cast<const uint4 *>(p.sums16 + (int64_t)c0 * (p.K / 16) + 16 * b);
        const uint4 s0 = __ldg(su), s1 = __ldg(su + 1);
        const uint32_t pw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int Sv = (int)(int16_t)(pw[q] & 0xFFFFu) + (int)(int16_t)(pw[q] >> 16);
            S0[q >> 1] |= ((uint32_t)Sv & 0xFFFFu) << (16 * (q & 1));
        }
        const uint32_t sv = __ldg(reinterpret_cast<const uint32_t *>(p.scales) + (int64_t)c0 * p.nb + b);
        m0a = (int)(sv & 0xFFu);
        e0a = (int)(int16_t)(sv >> 16);
    }
    if (has_block && in1) {
        const uint4 *su = reinterpret_cast<const uint4 *>(p.sums16 + (int64_t)c1 * (p.K / 16) + 16 * b);
        const uint4 s0 = __ldg(su), s1 = __ldg(su + 1);
        const uint32_t pw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int Sv = (int)(int16_t)(pw[q] & 0xFFFFu) + (int)(int16_t)(pw[q] >> 16);
            S1[q >> 1] |= ((uint32_t)Sv & 0xFFFFu) << (16 * (q & 1));
        }
        const uint32_t sv = __ldg(reinterpret_cast<const uint32_t *>(p.scales) + (int64_t)c1 * p.nb + b);
        m0b = (int)(sv & 0xFFu);
        e0b = (int)(int16_t)(sv >> 16);
    }
    __syncthreads();
    // activation fragments of the block: chunk kk = elements 16kk.. of the
    // block, my word t (column stride K + 16: lanes (g, t) hit bank 4g + t + const)
    uint32_t A[16][4];
    if (has_block) {
        const uint8_t *x0 = act + c0 * (p.K + 16) + 256 * b + 4 * t, *x1 = act + c1 * (p.K + 16) + 256 * b + 4 * t;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            act_frag(*reinterpret_cast<const uint32_t *>(x0 + 16 * kk), *reinterpret_cast<const uint32_t *>(x1 + 16 * kk),
                     A[kk]);
    } else {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) A[kk][0] = A[kk][1] = A[kk][2] = A[kk][3] = 0u;
    }

    for (int it = 0; it < p.n_iter; ++it) {
        const int slot = it % p.D;
        const int64_t first = (int64_t)it * p.R;
        const int64_t nrow = count - first < p.R ? count - first : (int64_t)p.R;
        bool ok = true;
        if (nrow > 0) ok = mbar_wait_bounded(bars + slot, (uint32_t)((it / p.D) & 1), p.fault);
        const uint8_t *sl = ring + (int64_t)slot * p.R * p.pitch;
        if (has_block && ok) {
            for (int tile = 0; 8 * tile < nrow; ++tile) {
                // ---- B operand: row g of the tile, 8 sub-blocks
                const uint8_t *blk = sl + (int64_t)(8 * tile + g) * p.pitch + 144 * b;
                const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
                const unsigned long long sc48 =
                    (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
                float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
                // B registers of sub-block s: low-nibble chunk (blo0, blo1), high (bhi0, bhi1)
                auto bprep = [&](int s, uint32_t &blo0, uint32_t &blo1, uint32_t &bhi0, uint32_t &bhi1) {
                    const uint32_t sc = (uint32_t)(sc48 >> (6 * s)) & 63u;
                    const uint32_t SC = hadd2_u((sc * 0x00010001u) | kH2Magic, kH2M1024);  // (sc, sc)
                    const uint32_t NSC = hmul2_u(SC, kH2M1024);                             // -1024 sc
                    const uint32_t SC16 = hmul2_u(SC, kH2Sixteenth);                        // sc / 16
                    const uint32_t N64 = hmul2_u(SC, kH2M64);                               // -64 sc
                    const uint32_t qw = *reinterpret_cast<const uint32_t *>(blk + 16 + 16 * s + 4 * t);
                    const uint32_t q8 = qw >> 8;
                    blo0 = hfma2_u((qw & 0x000F000Fu) | kH2Magic, SC, NSC);
                    blo1 = hfma2_u((q8 & 0x000F000Fu) | kH2Magic, SC, NSC);
                    bhi0 = hfma2_u((qw & 0x00F000F0u) | kH2Magic, SC16, N64);
                    bhi1 = hfma2_u((q8 & 0x00F000F0u) | kH2Magic, SC16, N64);
                };
#pragma unroll
                for (int s = 0; s < 4; ++s) {  // the two halves' chains interleaved
                    uint32_t l0, l1, h0, h1, L0, L1, H0, H1;
                    bprep(s, l0, l1, h0, h1);
                    bprep(s + 4, L0, L1, H0, H1);
                    mma_f16_16816(acc0, A[2 * s], l0, l1);
                    mma_f16_16816(acc1, A[2 * s + 8], L0, L1);
                    mma_f16_16816(acc0, A[2 * s + 1], h0, h1);
                    mma_f16_16816(acc1, A[2 * s + 9], H0, H1);
                }
                // ---- my pairs: columns c0 (acc[0], acc[1]) and c1 (acc[2], acc[3]),
                // rows 2t and 2t+1 of the tile
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const int rr = 8 * tile + 2 * t + r;  // row within the chunk
                    const uint8_t *rb = sl + (int64_t)rr * p.pitch + 144 * b;
                    const uint4 mt = *reinterpret_cast<const uint4 *>(rb);
                    const unsigned long long mn48 =
                        (unsigned long long)(mt.z >> 16) | ((unsigned long long)mt.w << 16);
                    const uint32_t mlo = spread6((uint32_t)mn48), mhi = spread6((uint32_t)(mn48 >> 24));
                    const RowScale rs = row_scale(mt.x);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (!(h ? in1 : in0)) continue;  // a padding column
                        const int C = __float2int_rn(acc0[2 * h + r]) + __float2int_rn(acc1[2 * h + r]);
                        const uint32_t(&S)[4] = h ? S1 : S0;
                        const int O = dp2a_hi_su(S[3], mhi, dp2a_lo_su(S[2], mhi, dp2a_hi_su(S[1], mlo,
                                                                                       dp2a_lo_su(S[0], mlo, 0))));
                        val[(rr * 16 + (h ? c1 : c0)) * p.vstride + b] =
                            combine_fast(rs, mt.x, C, O, h ? m0b : m0a, h ? e0b : e0a);
                    }
                }
            }
        }
        if (!__syncthreads_and(ok)) return;  // a fill never completed: fault word raised
        if (w == 0 && it + p.D < p.n_iter) {
            fence_proxy_async_smem();
            fill(it + p.D);
        }
        // ---- fold: one thread per (row, column), blocks in order
        for (int f = tid; f < p.R * 16; f += blockDim.x) {
            const int rr = f >> 4, c = f & 15;
            if (c < p.ncols && rr < nrow) {
                const float *vt = val + f * p.vstride;
                float acc = 0.0f;
                for (int bb = 0; bb < p.nb; ++bb) acc = fadd_ftz(acc, vt[bb]);
                if (acc != acc) acc = __uint_as_float(kEngineNaN);
                *out_ptr(p.mt, c, row0 + first + rr) = acc;
            }
        }
        if (it != p.n_iter - 1) __syncthreads();  // the fold has read the values before they are overwritten
    }
}

// Launch shape; QB_E_ARG when the kernel does not apply (Q4_K-like, 11..16
// columns, K % 256 == 0 and K <= 4096).
template <int F>
int launch_gemv5(const GemvArgs &a, cudaStream_t stream) {
    if (F != kQ4K || a.ncols < 11 || a.ncols > 16 || a.mode != 0 || a.K % 256 != 0 || a.K > 4096 ||
        (!a.mats && a.rows < 1))
        return QB_E_ARG;
    Gemv5K k;
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.rows = k.mt.start[k.mt.n];
    k.K = (int)a.K;
    k.rec = (int)record_bytes(F, a.K);
    k.pitch = gemv5_pitch(k.rec);
    k.nb = (int)(a.K / 256);
    k.ncols = a.ncols;
    k.vstride = (k.nb & 1) ? k.nb : k.nb + 1;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), k.rows));
    const int64_t rpc = (k.rows + grid - 1) / grid;
    const int budget = 225 * 1024;
    // a chunk of R rows: all of a CTA's rows when they fit one slot, else the
    // largest multiple of 8 (<= 32) that leaves room for two slots
    const int64_t all = (rpc + 7) / 8 * 8;
    if (all <= 32 && gemv5_smem(k.K, k.pitch, (int)all, 1, k.vstride).total <= budget) {
        k.R = (int)all;
        k.D = 1;
    } else {
        k.R = 32;
        while (k.R > 8 && gemv5_smem(k.K, k.pitch, k.R, 2, k.vstride).total > budget) k.R -= 8;
        k.D = gemv5_smem(k.K, k.pitch, k.R, 2, k.vstride).total <= budget ? 2 : 1;
    }
    if (gemv5_smem(k.K, k.pitch, k.R, k.D, k.vstride).total > budget) return QB_E_ARG;
    k.n_iter = (int)((rpc + k.R - 1) / k.R);
    if (k.n_iter > 1 && k.D < 2) k.D = std::min(k.n_iter, 2);
    if (gemv5_smem(k.K, k.pitch, k.R, k.D, k.vstride).total > budget) return QB_E_ARG;
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    const int smem = gemv5_smem(k.K, k.pitch, k.R, k.D, k.vstride).total;
    if (ensure_smem_limit(reinterpret_cast<const void *>(gemv5_kernel<F>), 227 * 1024) != QB_OK) return QB_E_CUDA;
    return launch_pdl(gemv5_kernel<F>, dim3(grid), dim3(512), (size_t)smem, stream, k);
}

}  // namespace qb
