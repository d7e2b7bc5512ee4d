// qb_gemv7.cuh -- the one-column product at K = 4096 with a warp per weight
// block and a lane per row.
//
// The arithmetic is the other kernels' (the lane page's exact block sums, the
// exact combine rounded once, each row folded in block order from +0); the
// organisation is chosen for the batch-1 step, whose time after the
// dependency wait is spent moving the activation and the weights through
// shared memory and issuing the block arithmetic:
//   * warp w owns block w of K (16 warps at K = 4096) and quantizes only that
//     block of the activation (8 elements a lane, the block's absmax by
//     shuffles), so the codes are written once and read as broadcasts;
//   * lane r owns row r of the CTA's rows (up to 32, or 64 as two a lane) and
//     forms its whole block w -- C, O and the rounded value -- alone: no
//     partial sums cross lanes;
//   * the CTA's rows arrive by one bulk copy each (the TMA engine) into a
//     pitch of rec + 16 bytes, an odd number of 16-B units, so the eight lanes
//     of a shared-memory phase read eight different bank groups;
//   * the whole slab is requested before the dependency wait, and with at
//     most ~72 KB a CTA two CTAs fit a SM: the next launch's CTAs are
//     resident, their weights in flight, while this launch's compute;
//   * block values go to a [row][17] table and one thread per row folds its
//     16 values in block order after one CTA barrier.
#pragma once

#include <algorithm>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"
#include "qb_quant.cuh"

namespace qb {

struct Gemv7K {
    MatTable mt;   // the matrix (or matrices sharing the activation) as one row range
    int64_t rows;  // rows of the whole range
    int rec;       // bytes per row record
    int pitch;     // bytes per row in shared memory (rec + 16)
    int64_t base;  // rows per CTA, and how many CTAs own one more
    int64_t rem;
    const int8_t *codes;  // the quantized activation (not FUSED)
    const qb_scale *scales;
    const int16_t *sums16;
    const float *x;  // FUSED: the f32 activation, quantized in the prologue
    int *fault;
};

constexpr int kG7K = 4096;             // K this kernel takes
constexpr int kG7Warps = kG7K / 256;   // a warp per 256-element block
constexpr int kG7MaxRows = 64;         // rows a CTA (two a lane at most)
constexpr int kG7VStride = kG7Warps + 1;  // floats per row of the block-value table

// shared memory: the mbarrier, each warp's 256 codes and 16 int16 sums, the
// block-value table, then the rows
constexpr int kG7Act = 128;
constexpr int kG7Sums = kG7Act + kG7K;
constexpr int kG7Vals = kG7Sums + kG7Warps * 32;
constexpr int kG7Slab = kG7Vals + ((kG7MaxRows * kG7VStride * 4 + 127) & ~127);
__host__ __device__ inline int gemv7_smem(int rows, int pitch) { return kG7Slab + rows * pitch; }

// Q4_K-like block at blk against the warp's codes a (256, natural order) and
// sub-block sums S (8 int16): C is returned as 16*C (each sub-block's sum as
// 16*(sum lo*a) + (sum 16*hi*a), hi read in place: |16*C| < 2^31), and O.
template <int UNR>
__device__ __forceinline__ void block_q4k(const uint8_t *blk, const uint8_t *a, const int16_t *S, int &C16, int &O,
                                          uint32_t &dd) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    dd = meta.x;
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
    int c = 0;
#pragma unroll UNR
    for (int s = 0; s < 8; ++s) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * s);
        const uint4 al = *reinterpret_cast<const uint4 *>(a + 32 * s);       // elements 32s .. 32s+15
        const uint4 ah = *reinterpret_cast<const uint4 *>(a + 32 * s + 16);  // elements 32s+16 .. 32s+31
        int pl = dp4a_ss(w.x & 0x0F0F0F0Fu, al.x, 0);
        pl = dp4a_ss(w.y & 0x0F0F0F0Fu, al.y, pl);
        pl = dp4a_ss(w.z & 0x0F0F0F0Fu, al.z, pl);
        pl = dp4a_ss(w.w & 0x0F0F0F0Fu, al.w, pl);
        int ph = dp4a_us(w.x & 0xF0F0F0F0u, ah.x, 0);
        ph = dp4a_us(w.y & 0xF0F0F0F0u, ah.y, ph);
        ph = dp4a_us(w.z & 0xF0F0F0F0u, ah.z, ph);
        ph = dp4a_us(w.w & 0xF0F0F0F0u, ah.w, ph);
        c += (int)((sc48 >> (6 * s)) & 63u) * (16 * pl + ph);
    }
    C16 = c;
    const uint4 sw = *reinterpret_cast<const uint4 *>(S);  // (S0,S1), (S2,S3), (S4,S5), (S6,S7)
    const uint32_t mb0 = spread6((uint32_t)mn48 & 0xFFFFFFu), mb1 = spread6((uint32_t)(mn48 >> 24));
    O = dp2a_hi_su(sw.w, mb1, dp2a_lo_su(sw.z, mb1, dp2a_hi_su(sw.y, mb0, dp2a_lo_su(sw.x, mb0, 0))));
}

// block_q4k for NC activation columns (codes at a + c*stride, sums at
// S + c*sstride): the weights read and unpacked once for all of them.
template <int NC, int UNR = 2>
__device__ __forceinline__ void block_q4k_cols(const uint8_t *blk, const uint8_t *a, int stride, const int16_t *S,
                                               int sstride, int (&C)[NC], int (&O)[NC], uint32_t &dd) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    dd = meta.x;
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
#pragma unroll
    for (int c = 0; c < NC; ++c) C[c] = 0;
#pragma unroll UNR
    for (int s = 0; s < 8; ++s) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * s);
        const uint32_t l0 = w.x & 0x0F0F0F0Fu, l1 = w.y & 0x0F0F0F0Fu, l2 = w.z & 0x0F0F0F0Fu, l3 = w.w & 0x0F0F0F0Fu;
        const uint32_t g0 = w.x & 0xF0F0F0F0u, g1 = w.y & 0xF0F0F0F0u, g2 = w.z & 0xF0F0F0F0u, g3 = w.w & 0xF0F0F0F0u;
        const int sc = (int)((sc48 >> (6 * s)) & 63u);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 al = *reinterpret_cast<const uint4 *>(a + c * stride + 32 * s);
            const uint4 ah = *reinterpret_cast<const uint4 *>(a + c * stride + 32 * s + 16);
            int pl = dp4a_ss(l0, al.x, 0);
            pl = dp4a_ss(l1, al.y, pl);
            pl = dp4a_ss(l2, al.z, pl);
            pl = dp4a_ss(l3, al.w, pl);
            int ph = dp4a_us(g0, ah.x, 0);
            ph = dp4a_us(g1, ah.y, ph);
            ph = dp4a_us(g2, ah.z, ph);
            ph = dp4a_us(g3, ah.w, ph);
            C[c] += sc * (16 * pl + ph);
        }
    }
    const uint32_t mb0 = spread6((uint32_t)mn48 & 0xFFFFFFu), mb1 = spread6((uint32_t)(mn48 >> 24));
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 sw = *reinterpret_cast<const uint4 *>(S + c * sstride);
        O[c] = dp2a_hi_su(sw.w, mb1, dp2a_lo_su(sw.z, mb1, dp2a_hi_su(sw.y, mb0, dp2a_lo_su(sw.x, mb0, 0))));
    }
}

// Q6_K-like block at blk (ql, qh, 16 int8 sub-scales) against the warp's codes a
// and unit sums S (16 int16): C = sum over the 16 units of sc_u * sum (q - 32)*a.
template <int UNR>
__device__ __forceinline__ int block_q6k(const uint8_t *blk, const uint8_t *a, const int16_t *S) {
    const uint4 scv = *reinterpret_cast<const uint4 *>(blk + 192);
    const uint32_t scw[4] = {scv.x, scv.y, scv.z, scv.w};
    const uint4 s0 = *reinterpret_cast<const uint4 *>(S), s1 = *reinterpret_cast<const uint4 *>(S + 8);
    const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    int c = 0;
#pragma unroll UNR
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 16 * ch);
        const uint2 hb = *reinterpret_cast<const uint2 *>(blk + 128 + 8 * ch);
        const uint4 al = *reinterpret_cast<const uint4 *>(a + 32 * ch);
        const uint4 ah = *reinterpret_cast<const uint4 *>(a + 32 * ch + 16);
        const uint32_t wl[4] = {w.x, w.y, w.z, w.w};
        const uint32_t alv[4] = {al.x, al.y, al.z, al.w};
        const uint32_t ahv[4] = {ah.x, ah.y, ah.z, ah.w};
        int pl = 0, ph = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t hl = (k < 3) ? (hb.x << (4 - 2 * k)) : (hb.x >> 2);
            const uint32_t hh = (k < 3) ? (hb.y << (4 - 2 * k)) : (hb.y >> 2);
            pl = dp4a_ss((wl[k] & 0x0F0F0F0Fu) | (hl & 0x30303030u), alv[k], pl);
            ph = dp4a_ss(((wl[k] >> 4) & 0x0F0F0F0Fu) | (hh & 0x30303030u), ahv[k], ph);
        }
        const uint32_t scp = scw[ch >> 1] >> (16 * (ch & 1));  // sub-scales of units 2ch, 2ch+1
        const int sc_lo = (int)(int8_t)(scp & 0xFFu), sc_hi = (int)(int8_t)((scp >> 8) & 0xFFu);
        // sum over a unit of (q - 32) * a = sum q*a - 32 * S_u
        c += sc_lo * (pl - 32 * (int)(int16_t)(sw[ch] & 0xFFFFu)) + sc_hi * (ph - 32 * (int)(int16_t)(sw[ch] >> 16));
    }
    return c;
}

// A Q4_K-like block held in registers: the 128 bytes of nibbles, the packed
// d/dmin pair, and the eight 6-bit sc and mn fields spread to bytes.
struct BlkQ4 {
    uint4 q[8];
    uint32_t dd, sc0, sc1, mn0, mn1;
};

__device__ __forceinline__ void load_q4k(const uint8_t *blk, BlkQ4 &b) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    b.dd = meta.x;
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
    b.sc0 = spread6((uint32_t)sc48 & 0xFFFFFFu);
    b.sc1 = spread6((uint32_t)(sc48 >> 24));
    b.mn0 = spread6((uint32_t)mn48 & 0xFFFFFFu);
    b.mn1 = spread6((uint32_t)(mn48 >> 24));
#pragma unroll
    for (int s = 0; s < 8; ++s) b.q[s] = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * s);
}

// block_q4k's sums for a block held in registers.
__device__ __forceinline__ void dot_q4k(const BlkQ4 &b, const uint8_t *a, const int16_t *S, int &C16, int &O) {
    int c = 0;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint4 w = b.q[s];
        const uint4 al = *reinterpret_cast<const uint4 *>(a + 32 * s);
        const uint4 ah = *reinterpret_cast<const uint4 *>(a + 32 * s + 16);
        int pl = dp4a_ss(w.x & 0x0F0F0F0Fu, al.x, 0);
        pl = dp4a_ss(w.y & 0x0F0F0F0Fu, al.y, pl);
        pl = dp4a_ss(w.z & 0x0F0F0F0Fu, al.z, pl);
        pl = dp4a_ss(w.w & 0x0F0F0F0Fu, al.w, pl);
        int ph = dp4a_us(w.x & 0xF0F0F0F0u, ah.x, 0);
        ph = dp4a_us(w.y & 0xF0F0F0F0u, ah.y, ph);
        ph = dp4a_us(w.z & 0xF0F0F0F0u, ah.z, ph);
        ph = dp4a_us(w.w & 0xF0F0F0F0u, ah.w, ph);
        const uint32_t scb = s < 4 ? b.sc0 : b.sc1;
        c += (int)((scb >> (8 * (s & 3))) & 0xFFu) * (16 * pl + ph);
    }
    C16 = c;
    const uint4 sw = *reinterpret_cast<const uint4 *>(S);
    O = dp2a_hi_su(sw.w, b.mn1, dp2a_lo_su(sw.z, b.mn1, dp2a_hi_su(sw.y, b.mn0, dp2a_lo_su(sw.x, b.mn0, 0))));
}

// UNR: sub-blocks (chunks) of a block in flight at once -- the register
// budget of MINB CTAs a SM.  PRE (Q4_K-like, at most 32 rows a CTA): the
// CTA waits for its rows before the dependency wait and each lane holds its
// row's block in registers, scales decoded, so that after the wait only the
// activation's work remains.
template <int F, bool FUSED, int MINB, int UNR, bool PRE>
__global__ void __launch_bounds__(kG7Warps * 32, MINB) gemv7_kernel(const Gemv7K p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint8_t *aw = smem + kG7Act + 256 * w;
    int16_t *Sw = reinterpret_cast<int16_t *>(smem + kG7Sums + 32 * w);
    float *vals = reinterpret_cast<float *>(smem + kG7Vals);
    uint8_t *slab = smem + kG7Slab;

    const int64_t c = blockIdx.x;
    const int64_t row0 = c * p.base + (c < p.rem ? c : p.rem);
    const int count = (int)(p.base + (c < p.rem ? 1 : 0));

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(count * p.rec));
    }
    __syncthreads();
    // the CTA's rows (weights depend on no earlier kernel)
    if (w == 0)
        for (int r = lane; r < count; r += 32)
            bulk_g2s(slab + r * p.pitch, row_ptr(p.mt, row0 + r, p.rec), (uint32_t)p.rec, bar);
    // the next launch may be scheduled now: it reads nothing this one writes
    // before its own pdl_wait, which returns once this grid has finished
    pdl_launch_dependents();
    BlkQ4 mine;
    if constexpr (PRE) {
        const bool ok = mbar_wait_bounded(bar, 0, p.fault);
        if (!__syncthreads_and(ok)) return;  // the slab never completed: fault word raised
        if (lane < count) load_q4k(slab + lane * p.pitch + 144 * w, mine);
    }
    pdl_wait();

    // ---- block w of the activation: codes (natural order), the sums the
    // format needs (Q4_K-like: per 32-element sub-block; Q6_K-like: per
    // 16-element unit) and the block's scale
    uint32_t scale;
    if constexpr (FUSED) {
        const float4 *xp = reinterpret_cast<const float4 *>(p.x + 256 * w + 8 * lane);
        const float4 v0 = ldg_f4_ordered(xp), v1 = ldg_f4_ordered(xp + 1);
        const uint32_t xb[8] = {__float_as_uint(v0.x), __float_as_uint(v0.y), __float_as_uint(v0.z),
                                __float_as_uint(v0.w), __float_as_uint(v1.x), __float_as_uint(v1.y),
                                __float_as_uint(v1.z), __float_as_uint(v1.w)};
        uint2 cd;
        int usum;  // the sum of the 16-element unit of this lane pair
        quantize8<32>(xb, cd, usum, scale);
        *reinterpret_cast<uint2 *>(aw + 8 * lane) = cd;
        if (F == kQ4K) {
            const int s2 = usum + __shfl_down_sync(0xFFFFFFFFu, usum, 2);
            if ((lane & 3) == 0) Sw[lane >> 2] = (int16_t)s2;
        } else {
            if ((lane & 1) == 0) Sw[lane >> 1] = (int16_t)usum;
        }
    } else {
        const uint2 cd = *reinterpret_cast<const uint2 *>(p.codes + 256 * w + 8 * lane);
        *reinterpret_cast<uint2 *>(aw + 8 * lane) = cd;
        const int us = lane < 16 ? (int)p.sums16[16 * w + lane] : 0;
        if (F == kQ4K) {
            const int s2 = us + __shfl_down_sync(0xFFFFFFFFu, us, 1);
            if (lane < 16 && (lane & 1) == 0) Sw[lane >> 1] = (int16_t)s2;
        } else {
            if (lane < 16) Sw[lane] = (int16_t)us;
        }
        scale = reinterpret_cast<const uint32_t *>(p.scales)[w];
    }
    __syncwarp();
    const int m0 = (int)(scale & 0xFFu), e0 = (int)(int16_t)(scale >> 16);

    // ---- block w of each of my rows
    if constexpr (PRE) {
        if (lane < count) {
            int C16, O;
            dot_q4k(mine, aw, Sw, C16, O);
            vals[lane * kG7VStride + w] =
                lane_value_fast<1>(C16 >> 4, O, mine.dd & 0xFFFFu, mine.dd >> 16, m0, e0);  // 16*C: exact shift
        }
    } else {
    const bool ok = mbar_wait_bounded(bar, 0, p.fault);
    if (!__syncthreads_and(ok)) return;  // the slab never completed: fault word raised
    for (int r = lane; r < count; r += 32) {
        const uint8_t *row = slab + r * p.pitch;
        float v;
        if (F == kQ4K) {
            int C16, O;
            uint32_t dd;
            block_q4k<UNR>(row + 144 * w, aw, Sw, C16, O, dd);
            v = lane_value_fast<1>(C16 >> 4, O, dd & 0xFFFFu, dd >> 16, m0, e0);  // 16*C: exact shift
        } else {
            const int C = block_q6k<UNR>(row + 208 * w, aw, Sw);
            const uint32_t d = *reinterpret_cast<const uint16_t *>(row + 208 * kG7Warps + 2 * w);
            v = lane_value_fast<0>(C, 0, d, 0, m0, e0);
        }
        vals[r * kG7VStride + w] = v;
    }
    }
    __syncthreads();
    // ---- fold: thread r adds row r's 16 block values in block order from +0
    if (tid < count) {
        const float *vr = vals + tid * kG7VStride;
        float acc = 0.0f;
#pragma unroll
        for (int b = 0; b < kG7Warps; ++b) acc = fadd_ftz(acc, vr[b]);
        if (acc != acc) acc = __uint_as_float(kEngineNaN);
        *out_ptr(p.mt, 0, row0 + tid) = acc;
    }
}

// One column of a Q4_K-like or Q6_K-like matrix (or a table of them) at
// K = 4096 with at most 64 rows a CTA and MINB CTAs a SM.  QB_E_ARG when the
// shape does not fit.
template <int F, int MINB, int UNR, bool PRE>
int launch_gemv7(const GemvArgs &a, cudaStream_t stream, const float *x) {
    if ((F != kQ4K && F != kQ6K) || a.ncols != 1 || a.mode != 0 || a.K != kG7K) return QB_E_ARG;
    Gemv7K k;
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.rows = k.mt.start[k.mt.n];
    if (k.rows < 1) return QB_E_ARG;
    int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), k.rows));
    int64_t per_cta = (k.rows + grid - 1) / grid;
    if (PRE && per_cta > 32 && per_cta <= 48) {
        // 33..48 rows a SM: CTAs of at most 32 rows (two on some SMs) keep every
        // lane's block in registers from before the dependency wait (6144 x 4096:
        // 3.96 -> 3.47 us a step)
        grid = (int)((k.rows + 31) / 32);
        per_cta = (k.rows + grid - 1) / grid;
    }
    if (per_cta > (PRE ? 32 : kG7MaxRows) || (PRE && F != kQ4K)) return QB_E_ARG;
    k.rec = (int)record_bytes(F, kG7K);
    k.pitch = k.rec + 16;
    const int smem = gemv7_smem((int)per_cta, k.pitch);
    if (smem > (228 * 1024) / MINB - 1024 - 256) return QB_E_ARG;
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.x = x;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    auto kern = x ? gemv7_kernel<F, true, MINB, UNR, PRE> : gemv7_kernel<F, false, MINB, UNR, PRE>;
    if (ensure_smem_limit(reinterpret_cast<const void *>(kern), smem) != QB_OK) return QB_E_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(kG7Warps * 32), (size_t)smem, stream, k);
}

// shared memory for NC columns: the mbarrier, each column's block scales,
// codes (each warp's 256) and int16 sums (each warp's 16), the block-value table ([row][column][17],
// its row stride made odd so the lanes of a warp -- one row each -- write
// different banks), then the rows
__host__ __device__ constexpr int gemv7m_vs(int nc) { return (nc * 17) | 1; }
struct Gemv7MSmem {
    int scl, act, sums, vals, slab;
};
__host__ __device__ inline Gemv7MSmem gemv7m_layout(int nc) {
    Gemv7MSmem s;
    s.scl = 128;  // nc x 16 block scales
    s.act = s.scl + ((nc * kG7Warps * 4 + 127) & ~127);
    s.sums = s.act + nc * kG7K;
    s.vals = s.sums + nc * kG7Warps * 32;
    s.slab = s.vals + ((kG7MaxRows * gemv7m_vs(nc) * 4 + 127) & ~127);
    return s;
}
__host__ __device__ inline int gemv7m_smem(int nc, int rows, int pitch) { return gemv7m_layout(nc).slab + rows * pitch; }

// NC activation columns (2..4) in one launch: each warp prepares block w of
// every column (quantizing it in the single-launch form), each lane forms its
// rows' block w for every column from the one copy of the weights in shared
// memory (Q4_K-like: the weights unpacked once for all the columns;
// Q6_K-like: column by column).
template <int F, bool FUSED, int MINB, int UNR, int NC>
__global__ void __launch_bounds__(kG7Warps * 32, MINB) gemv7m_kernel(const Gemv7K p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const Gemv7MSmem Lo = gemv7m_layout(NC);
    constexpr int VS = gemv7m_vs(NC);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint32_t *sclw = reinterpret_cast<uint32_t *>(smem + Lo.scl) + w;  // column c at + c * 16
    uint8_t *aw = smem + Lo.act + 256 * w;                             // column c at + c * K
    int16_t *Sw = reinterpret_cast<int16_t *>(smem + Lo.sums + 32 * w);  // column c at + c * 256
    float *vals = reinterpret_cast<float *>(smem + Lo.vals);
    uint8_t *slab = smem + Lo.slab;

    const int64_t c = blockIdx.x;
    const int64_t row0 = c * p.base + (c < p.rem ? c : p.rem);
    const int count = (int)(p.base + (c < p.rem ? 1 : 0));

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(count * p.rec));
    }
    __syncthreads();
    // the CTA's rows (weights depend on no earlier kernel)
    if (w == 0)
        for (int r = lane; r < count; r += 32)
            bulk_g2s(slab + r * p.pitch, row_ptr(p.mt, row0 + r, p.rec), (uint32_t)p.rec, bar);
    // the next launch may be scheduled now: it reads nothing this one writes
    // before its own pdl_wait, which returns once this grid has finished
    pdl_launch_dependents();
    pdl_wait();

    // ---- block w of the activation, each column: codes (natural order), the
    // sums the format needs (Q4_K-like: per 32-element sub-block; Q6_K-like:
    // per 16-element unit) and the block's scale
    // every column's elements requested before the first is quantized (the
    // quantizer's shuffles would otherwise hold each load behind the last)
    float4 xv[FUSED ? 2 * NC : 1];
    if constexpr (FUSED) {
#pragma unroll
        for (int col = 0; col < NC; ++col) {
            const float4 *xp = reinterpret_cast<const float4 *>(p.x + (int64_t)col * kG7K + 256 * w + 8 * lane);
            xv[2 * col] = ldg_f4_ordered(xp);
            xv[2 * col + 1] = ldg_f4_ordered(xp + 1);
        }
    }
#pragma unroll
    for (int col = 0; col < NC; ++col) {
        uint32_t scale;
        uint8_t *ac = aw + col * kG7K;
        int16_t *Sc = Sw + col * (kG7Warps * 16);
        if constexpr (FUSED) {
            const float4 v0 = xv[2 * col], v1 = xv[2 * col + 1];
            const uint32_t xb[8] = {__float_as_uint(v0.x), __float_as_uint(v0.y), __float_as_uint(v0.z),
                                    __float_as_uint(v0.w), __float_as_uint(v1.x), __float_as_uint(v1.y),
                                    __float_as_uint(v1.z), __float_as_uint(v1.w)};
            uint2 cd;
            int usum;  // the sum of the 16-element unit of this lane pair
            quantize8<32>(xb, cd, usum, scale);
            *reinterpret_cast<uint2 *>(ac + 8 * lane) = cd;
            if (F == kQ4K) {
                const int s2 = usum + __shfl_down_sync(0xFFFFFFFFu, usum, 2);
                if ((lane & 3) == 0) Sc[lane >> 2] = (int16_t)s2;
            } else {
                if ((lane & 1) == 0) Sc[lane >> 1] = (int16_t)usum;
            }
        } else {
            const uint2 cd = *reinterpret_cast<const uint2 *>(p.codes + (int64_t)col * kG7K + 256 * w + 8 * lane);
            *reinterpret_cast<uint2 *>(ac + 8 * lane) = cd;
            const int us = lane < 16 ? (int)p.sums16[(int64_t)col * (kG7K / 16) + 16 * w + lane] : 0;
            if (F == kQ4K) {
                const int s2 = us + __shfl_down_sync(0xFFFFFFFFu, us, 1);
                if (lane < 16 && (lane & 1) == 0) Sc[lane >> 1] = (int16_t)s2;
            } else {
                if (lane < 16) Sc[lane] = (int16_t)us;
            }
            scale = reinterpret_cast<const uint32_t *>(p.scales)[col * kG7Warps + w];
        }
        if (lane == 0) sclw[col * kG7Warps] = scale;
    }
    __syncwarp();

    // ---- block w of each of my rows, each column
    {
        const bool ok = mbar_wait_bounded(bar, 0, p.fault);
        if (!__syncthreads_and(ok)) return;  // the slab never completed: fault word raised
        for (int r = lane; r < count; r += 32) {
            const uint8_t *row = slab + r * p.pitch;
            int col = 0;
            if (F == kQ4K) {  // every column at once: the weights unpacked once
                int C[NC], O[NC];
                uint32_t dd;
                block_q4k_cols<NC>(row + 144 * w, aw, kG7K, Sw, kG7Warps * 16, C, O, dd);
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) {
                    const uint32_t sv = sclw[cc * kG7Warps];
                    vals[r * VS + cc * 17 + w] = lane_value_fast<1>(C[cc] >> 4, O[cc], dd & 0xFFFFu, dd >> 16,
                                                                    (int)(sv & 0xFFu), (int)(int16_t)(sv >> 16));
                }
                col = NC;
            }
#pragma unroll 1
            for (; col < NC; ++col) {
                const uint8_t *ac = aw + col * kG7K;
                const int16_t *Sc = Sw + col * (kG7Warps * 16);
                const uint32_t sv = sclw[col * kG7Warps];
                const int m0 = (int)(sv & 0xFFu), e0 = (int)(int16_t)(sv >> 16);
                float v;
                if (F == kQ4K) {
                    int C16, O;
                    uint32_t dd;
                    block_q4k<UNR>(row + 144 * w, ac, Sc, C16, O, dd);
                    v = lane_value_fast<1>(C16 >> 4, O, dd & 0xFFFFu, dd >> 16, m0, e0);  // 16*C: exact shift
                } else {
                    const int C = block_q6k<UNR>(row + 208 * w, ac, Sc);
                    const uint32_t d = *reinterpret_cast<const uint16_t *>(row + 208 * kG7Warps + 2 * w);
                    v = lane_value_fast<0>(C, 0, d, 0, m0, e0);
                }
                vals[r * VS + col * 17 + w] = v;
            }
        }
    }
    __syncthreads();
    // ---- fold: thread (r, col) adds row r's 16 block values of that column in
    // block order from +0
    for (int t = tid; t < count * NC; t += kG7Warps * 32) {
        const int r = t / NC, col = t - r * NC;
        const float *vr = vals + r * VS + col * 17;
        float acc = 0.0f;
#pragma unroll
        for (int b = 0; b < kG7Warps; ++b) acc = fadd_ftz(acc, vr[b]);
        if (acc != acc) acc = __uint_as_float(kEngineNaN);
        *out_ptr(p.mt, col, row0 + r) = acc;
    }
}

// NC columns (2..4) of a Q4_K-like or Q6_K-like matrix (or a table of them)
// at K = 4096 with at most 64 rows a CTA and MINB CTAs a SM.  QB_E_ARG when
// the shape does not fit.
template <int F, int MINB, int UNR, int NC>
int launch_gemv7m(const GemvArgs &a, cudaStream_t stream, const float *x) {
    if ((F != kQ4K && F != kQ6K) || a.ncols != NC || a.mode != 0 || a.K != kG7K) return QB_E_ARG;
    Gemv7K k;
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.rows = k.mt.start[k.mt.n];
    if (k.rows < 1) return QB_E_ARG;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), k.rows));
    const int64_t per_cta = (k.rows + grid - 1) / grid;
    if (per_cta > kG7MaxRows) return QB_E_ARG;
    k.rec = (int)record_bytes(F, kG7K);
    k.pitch = k.rec + 16;
    const int smem = gemv7m_smem(NC, (int)per_cta, k.pitch);
    if (smem > (228 * 1024) / MINB - 1024 - 256) return QB_E_ARG;
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.x = x;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    auto kern = x ? gemv7m_kernel<F, true, MINB, UNR, NC> : gemv7m_kernel<F, false, MINB, UNR, NC>;
    if (ensure_smem_limit(reinterpret_cast<const void *>(kern), smem) != QB_OK) return QB_E_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(kG7Warps * 32), (size_t)smem, stream, k);
}

// ---------------------------------------------------------------- ring form
// Q4_K-like, 2..4 columns, more rows than one slab holds or a longer K: the
// CTA's rows stream through a ring of two tiles, a tile being 32 rows by one
// chunk of NW blocks (K = 256 * NW * chunks; chunks of a row tile in order).
// Compute warps 0..NW-1 form block k*NW + w of every row of the tile in chunk
// k (a lane a row) for every column, the weights unpacked once.  A producer
// warp issues each tile's row copies and folds each computed tile into its
// rows' running sums (block order: the chunks in order, blocks in order within
// each), so that neither the copy issue (which stalls while the copy engine is
// busy) nor the fold delays the arithmetic.  The roles hand over through
// mbarriers only:
//   full[s]   the copies of the tile in slot s have landed (transaction count)
//   done[b]   the compute warps have read the tile in slot b and written its
//             block values into value buffer b
//   vfree[b]  the producer has folded value buffer b (it may be rewritten)
// Tile t (row tile t / chunks, chunk t % chunks) uses slot and buffer t & 1;
// each barrier completes once per tile that uses it, so tile t waits for phase
// (t >> 1) & 1.
constexpr int kG7RTile = 32;   // rows a tile (a lane a row)
constexpr int kG7RUnr = 2;     // sub-blocks unrolled (the register budget of one CTA a SM)

struct Gemv7RSmem {
    int scl, act, sums, vals, slab, vbuf, total;
};
// nc columns, K, nw blocks a chunk, pitch: bytes a row of a tile in shared memory
__host__ __device__ inline Gemv7RSmem gemv7r_layout(int nc, int K, int nw, int pitch) {
    const int nb = K / 256;
    Gemv7RSmem s;
    s.scl = 128;  // 6 mbarriers at 0
    s.act = s.scl + ((nc * nb * 4 + 127) & ~127);
    s.sums = s.act + nc * K;
    s.vals = s.sums + ((nc * nb * 32 + 127) & ~127);
    s.vbuf = (kG7RTile * ((nc * (nw + 1)) | 1) * 4 + 127) & ~127;
    s.slab = s.vals + 2 * s.vbuf;
    s.total = s.slab + 2 * kG7RTile * pitch;
    return s;
}

template <bool FUSED, int NC, int NW, int NCH>
__global__ void __launch_bounds__((NW + 1) * 32, 1) gemv7r_kernel(const Gemv7K p, int pitch) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    constexpr int nch = NCH, nb = NW * NCH, K = 256 * nb;  // chunks, blocks and elements a row
    const int cbytes = NW * 144;               // bytes of a row's chunk
    const Gemv7RSmem Lo = gemv7r_layout(NC, K, NW, pitch);
    constexpr int VS = (NC * (NW + 1)) | 1;    // floats a row of a value buffer (odd: rows in distinct banks)
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *done = full + 2;
    uint64_t *vfree = done + 2;
    uint32_t *scl = reinterpret_cast<uint32_t *>(smem + Lo.scl);  // [col][block]
    uint8_t *act = smem + Lo.act;                                              // [col][K]
    int16_t *sums = reinterpret_cast<int16_t *>(smem + Lo.sums);               // [col][block][16]
    uint8_t *slab = smem + Lo.slab;

    const int64_t c = blockIdx.x;
    const int64_t row0 = c * p.base + (c < p.rem ? c : p.rem);
    const int count = (int)(p.base + (c < p.rem ? 1 : 0));
    const int ntiles = ((count + kG7RTile - 1) / kG7RTile) * nch;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(full + s, 1);
            mbar_init(done + s, NW);
            mbar_init(vfree + s, 1);
        }
        fence_mbar_init();
    }
    __syncthreads();  // the last CTA-wide barrier: the roles part here

    if (w == NW) {
        // ---- producer: tile t into slot t & 1, a copy a row by the lanes
        auto fill = [&](int t) {
            const int rt = t / nch, k = t - rt * nch;
            const int n = min(kG7RTile, count - rt * kG7RTile);
            uint64_t *bar = full + (t & 1);
            if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(n * cbytes));
            __syncwarp();
            uint8_t *dst = slab + (t & 1) * (kG7RTile * pitch);
            if (lane < n)
                bulk_g2s(dst + lane * pitch,
                         row_ptr(p.mt, row0 + (int64_t)rt * kG7RTile + lane, p.rec) + (int64_t)k * cbytes,
                         (uint32_t)cbytes, bar);
        };
        // the first tiles (weights depend on no earlier kernel)
        for (int t = 0; t < 2 && t < ntiles; ++t) fill(t);
        pdl_launch_dependents();
        pdl_wait();  // the outputs this warp writes: after the previous kernel
        float acc[NC];  // lane = row of the row tile: its running sums
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) acc[cc] = 0.0f;
        for (int t = 0; t < ntiles; ++t) {
            const int b = t & 1;
            if (!mbar_wait_bounded(done + b, (uint32_t)((t >> 1) & 1), p.fault)) return;
            if (t + 2 < ntiles) {
                fence_proxy_async_smem();  // the compute warps' reads of the slot before the copies into it
                fill(t + 2);
            }
            // fold chunk k of row tile rt: block values in block order
            const int rt = t / nch, k = t - rt * nch;
            const int n = min(kG7RTile, count - rt * kG7RTile);
            const float *vr = reinterpret_cast<const float *>(smem + Lo.vals + b * Lo.vbuf) + lane * VS;
#pragma unroll
            for (int cc = 0; cc < NC; ++cc)
#pragma unroll
                for (int q = 0; q < NW; ++q) acc[cc] = fadd_ftz(acc[cc], vr[cc * (NW + 1) + q]);
            __syncwarp();
            if (lane == 0) mbar_arrive(vfree + b);
            if (k == nch - 1) {
                if (lane < n)
#pragma unroll
                    for (int cc = 0; cc < NC; ++cc) {
                        const float v = acc[cc] != acc[cc] ? __uint_as_float(kEngineNaN) : acc[cc];
                        *out_ptr(p.mt, cc, row0 + (int64_t)rt * kG7RTile + lane) = v;
                    }
#pragma unroll
                for (int cc = 0; cc < NC; ++cc) acc[cc] = 0.0f;
            }
        }
        return;
    }

    // ---- compute warps
    pdl_launch_dependents();
    pdl_wait();
    // blocks w, NW + w, 2*NW + w, ... of the activation, each column: codes
    // (natural order), the per-32 sums and the block's scale
    for (int k = 0; k < nch; ++k) {
        const int blk = k * NW + w;
        float4 xv[FUSED ? 2 * NC : 1];
        if constexpr (FUSED) {  // every column's elements requested first
#pragma unroll
            for (int col = 0; col < NC; ++col) {
                const float4 *xp = reinterpret_cast<const float4 *>(p.x + (int64_t)col * K + 256 * blk + 8 * lane);
                xv[2 * col] = ldg_f4_ordered(xp);
                xv[2 * col + 1] = ldg_f4_ordered(xp + 1);
            }
        }
#pragma unroll
        for (int col = 0; col < NC; ++col) {
            uint32_t scale;
            uint8_t *ac = act + col * K + 256 * blk;
            int16_t *Sc = sums + (col * nb + blk) * 16;
            if constexpr (FUSED) {
                const float4 v0 = xv[2 * col], v1 = xv[2 * col + 1];
                const uint32_t xb[8] = {__float_as_uint(v0.x), __float_as_uint(v0.y), __float_as_uint(v0.z),
                                        __float_as_uint(v0.w), __float_as_uint(v1.x), __float_as_uint(v1.y),
                                        __float_as_uint(v1.z), __float_as_uint(v1.w)};
                uint2 cd;
                int usum;  // the sum of the 16-element unit of this lane pair
                quantize8<32>(xb, cd, usum, scale);
                *reinterpret_cast<uint2 *>(ac + 8 * lane) = cd;
                const int s2 = usum + __shfl_down_sync(0xFFFFFFFFu, usum, 2);
                if ((lane & 3) == 0) Sc[lane >> 2] = (int16_t)s2;
            } else {
                const uint2 cd = *reinterpret_cast<const uint2 *>(p.codes + (int64_t)col * K + 256 * blk + 8 * lane);
                *reinterpret_cast<uint2 *>(ac + 8 * lane) = cd;
                const int us = lane < 16 ? (int)p.sums16[(int64_t)col * (K / 16) + 16 * blk + lane] : 0;
                const int s2 = us + __shfl_down_sync(0xFFFFFFFFu, us, 1);
                if (lane < 16 && (lane & 1) == 0) Sc[lane >> 1] = (int16_t)s2;
                scale = reinterpret_cast<const uint32_t *>(p.scales)[(int64_t)col * nb + blk];
            }
            if (lane == 0) scl[col * nb + blk] = scale;
        }
    }
    __syncwarp();
    uint32_t sv1[NC];  // one chunk: the scales of my block held in registers
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) sv1[cc] = scl[cc * nb + w];

    for (int t = 0; t < ntiles; ++t) {
        const int b = t & 1;
        const uint32_t ph = (uint32_t)((t >> 1) & 1);
        const int rt = t / nch, k = t - rt * nch;
        const int blk = k * NW + w;
        if (!mbar_wait_bounded(full + b, ph, p.fault)) return;              // the tile landed
        if (t >= 2 && !mbar_wait_bounded(vfree + b, ph ^ 1u, p.fault)) return;  // tile t-2 folded
        const int n = min(kG7RTile, count - rt * kG7RTile);
        float *vb = reinterpret_cast<float *>(smem + Lo.vals + b * Lo.vbuf);
        if (lane < n) {
            const uint8_t *row = slab + b * (kG7RTile * pitch) + lane * pitch + 144 * w;
            int C[NC], O[NC];
            uint32_t dd;
            block_q4k_cols<NC, kG7RUnr>(row, act + 256 * blk, K, sums + blk * 16, nb * 16, C, O, dd);
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                const uint32_t sv = NCH == 1 ? sv1[cc] : scl[cc * nb + blk];
                vb[lane * VS + cc * (NW + 1) + w] = lane_value_fast<1>(C[cc] >> 4, O[cc], dd & 0xFFFFu, dd >> 16,
                                                                       (int)(sv & 0xFFu), (int)(int16_t)(sv >> 16));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(done + b);
    }
}

// The ring form for NC columns (2..4) of a Q4_K-like matrix (or a table of
// them) at K = 256 * NW * NCH; QB_E_ARG when the shape does not fit.
// min_rows: take it only past this many rows a CTA.
template <int NC, int NW, int NCH>
int launch_gemv7r(const GemvArgs &a, cudaStream_t stream, const float *x, int64_t min_rows) {
    if (a.ncols != NC || a.mode != 0 || a.K != 256 * NW * NCH) return QB_E_ARG;
    Gemv7K k;
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.rows = k.mt.start[k.mt.n];
    if (k.rows < 1) return QB_E_ARG;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), k.rows));
    const int64_t per_cta = (k.rows + grid - 1) / grid;
    if (per_cta <= min_rows) return QB_E_ARG;
    k.rec = (int)record_bytes(kQ4K, a.K);
    k.pitch = NW * 144 + 16;  // a row's chunk, offset by 16 B a row: the lanes of a phase in distinct banks
    const int smem = gemv7r_layout(NC, (int)a.K, NW, k.pitch).total;
    if (smem > 227 * 1024) return QB_E_ARG;
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.x = x;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    auto kern = x ? gemv7r_kernel<true, NC, NW, NCH> : gemv7r_kernel<false, NC, NW, NCH>;
    if (ensure_smem_limit(reinterpret_cast<const void *>(kern), smem) != QB_OK) return QB_E_CUDA;
    return launch_pdl(kern, dim3(grid), dim3((NW + 1) * 32), (size_t)smem, stream, k, k.pitch);
}

// The ring form for a.ncols (2..4) columns at K = 4096 (one chunk of 16
// blocks), 8192 (two) or 14336 (four chunks of 14).
template <int NC>
int launch_gemv7r_k(const GemvArgs &a, cudaStream_t stream, const float *x, int64_t min_rows) {
    switch (a.K) {
    case 4096: return launch_gemv7r<NC, 16, 1>(a, stream, x, min_rows);
    case 8192: return launch_gemv7r<NC, 16, 2>(a, stream, x, min_rows);
    case 14336: return launch_gemv7r<NC, 14, 4>(a, stream, x, min_rows);
    default: return QB_E_ARG;
    }
}
inline int launch_gemv7r_cols(const GemvArgs &a, cudaStream_t stream, const float *x, int64_t min_rows) {
    switch (a.ncols) {
    case 2: return launch_gemv7r_k<2>(a, stream, x, min_rows);
    case 3: return launch_gemv7r_k<3>(a, stream, x, min_rows);
    case 4: return launch_gemv7r_k<4>(a, stream, x, min_rows);
    default: return QB_E_ARG;
    }
}

// 2..4 columns at K = 4096 (the multi-column form above); QB_E_ARG where it
// does not apply.
template <int F>
int launch_gemv7_cols(const GemvArgs &a, cudaStream_t stream, const float *x) {
    constexpr int U = F == kQ4K ? 2 : 4;
    // 3..4 columns past 32 rows a CTA: one CTA a SM (twice the registers) beat
    // two (Q4_K-like 6144 x 4096 at 4 columns: 8.24 -> 7.68 us)
    const int64_t g = std::max<int64_t>(1, std::min<int64_t>(num_sms(), a.mats ? a.mats->start[a.mats->n] : a.rows));
    const bool one = ((a.mats ? a.mats->start[a.mats->n] : a.rows) + g - 1) / g > 32;
    int r = QB_E_ARG;
    switch (a.ncols) {
    case 2: r = launch_gemv7m<F, 2, U, 2>(a, stream, x); break;
    case 3: r = one ? launch_gemv7m<F, 1, U, 3>(a, stream, x) : launch_gemv7m<F, 2, U, 3>(a, stream, x); break;
    case 4: r = one ? launch_gemv7m<F, 1, U, 4>(a, stream, x) : launch_gemv7m<F, 2, U, 4>(a, stream, x); break;
    default: return QB_E_ARG;
    }
    if (r != QB_E_ARG || F != kQ4K) return r;
    // more rows a CTA (K = 4096), or a longer K: the ring form
    return launch_gemv7r_cols(a, stream, x, a.K == kG7K ? kG7MaxRows : 0);
}

}  // namespace qb
