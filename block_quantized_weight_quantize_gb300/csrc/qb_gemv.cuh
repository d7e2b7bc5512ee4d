// qb_gemv.cuh -- the block-quantized product kernel for sm_103a.
//
// Computes the decode engine's dot under ActScaling::PerBlock (numerics page,
// dot; block-scale lane page, block_sums / lane) for a tile of R consecutive
// rows per CTA and up to 16 activation columns:
//   1. one thread issues a single bulk asynchronous copy (cp.async.bulk, the
//      TMA engine) of the tile's R row records -- contiguous in memory -- into
//      shared memory, BEFORE the programmatic-dependent-launch wait, so the
//      weight stream starts while the previous kernel drains;
//   2. after griddepcontrol.wait the CTA stages the activation codes (XOR-
//      swizzled so that threads reading different blocks hit different banks),
//      unit sums and scales into shared memory;
//   3. every (row, weight block) item is one thread: it unpacks the block's
//      codes in registers, forms the exact integer sums with dp4a, multiplies
//      by the sub-block scales, and combines with the block scales and the
//      activation scale exactly in 64-bit integers (128-bit for a wide scale
//      exponent spread), rounding once to f32 (lane_value);
//   4. one thread per (column, row) adds the row's rounded block values in
//      block order from +0 (f32, ftz) and writes out[c*rows + r].
// Consecutive threads take consecutive blocks of a row: the 144-B (Q4_K) and
// 208-B (Q6_K) block strides are odd multiples of 16 B, so their shared-memory
// reads are free of bank conflicts.
#pragma once

#include <algorithm>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_launch.h"

namespace qb {

struct GemvK {
    const uint8_t *W;
    int64_t rows;
    int K;
    int nb;        // weight blocks per row
    int rec;       // bytes per row record
    int R;         // rows per CTA tile
    int kcb;       // weight blocks per staged activation chunk
    int vstride;   // floats per (column, row) line of block values
    const int8_t *codes;
    const qb_scale *scales;
    const int16_t *sums16;
    float *out;
    int32_t *dbgC;
    int32_t *dbgO;
    float *dbgV;
    int *fault;    // the library's device fault word
};

// Shared memory carve-up, identical on host and device.
struct GemvSmem {
    int tile, act, sums, scl, val, total;
};

__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }

// Per-column strides of the staged activation chunk, whole 128-B lines so the
// swizzle never leaves a column's region.
template <int F>
__host__ __device__ inline int act_col_bytes(int kcb) { return align128(kcb * fmt_block(F)); }
template <int F>
__host__ __device__ inline int sums_col_bytes(int kcb) {
    return F == kQ4K ? align128(kcb * 8 * 2) : F == kQ6K ? align128(kcb * 16 * 2) : 0;
}

template <int F>
__host__ __device__ inline GemvSmem gemv_smem(int R, int rec, int kcb, int nc, int vstride, int mode) {
    constexpr int blk = fmt_block(F);
    GemvSmem s;
    s.tile = 128;
    s.act = s.tile + align128(R * rec);
    s.sums = s.act + nc * act_col_bytes<F>(kcb);
    s.scl = s.sums + nc * sums_col_bytes<F>(kcb);
    s.val = s.scl + align128(nc * kcb * 4);
    s.total = s.val + (mode == 0 ? align128(nc * R * vstride * 4) : 0);
    return s;
}

// 16-B unit u of a column's staged activation codes, XOR-swizzled within its
// 128-B line.  256-element blocks: a thread on block b reads units 16b..16b+15
// and the swizzle key is b & 7.  32-element blocks (Q8_0): units 2b, 2b+1, key
// = line & 7.
template <int F>
__device__ __forceinline__ int act_phys(int u) {
    const int line = u >> 3, pos = u & 7;
    const int key = (F == kQ8_0) ? (line & 7) : ((line >> 1) & 7);
    return (line << 3) | (pos ^ key);
}

template <int F, int NC>
__device__ __forceinline__ uint4 act_unit(const uint8_t *act, int chunk_bytes, int c, int u) {
    return *reinterpret_cast<const uint4 *>(act + c * chunk_bytes + act_phys<F>(u) * 16);
}

// ----------------------------------------------------------------- per-format block sums

// Q4_K-like block: C_c = sum_s sc_s * sum_{i in s} q_i a_i, O_c = sum_s mn_s * S_s.
template <int NC>
__device__ __forceinline__ void block_q4k(const uint8_t *blk, const uint8_t *act, int cb, const int16_t *s32,
                                          int s32_stride, int bl, int (&C)[NC], int (&O)[NC], uint32_t &s1,
                                          uint32_t &s2) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    s1 = meta.x & 0xFFFFu;
    s2 = meta.x >> 16;
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
#pragma unroll
    for (int c = 0; c < NC; ++c) { C[c] = 0; O[c] = 0; }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * s);
        const uint32_t l0 = w.x & 0x0F0F0F0Fu, l1 = w.y & 0x0F0F0F0Fu, l2 = w.z & 0x0F0F0F0Fu,
                       l3 = w.w & 0x0F0F0F0Fu;
        const uint32_t h0 = w.x & 0xF0F0F0F0u, h1 = w.y & 0xF0F0F0F0u, h2 = w.z & 0xF0F0F0F0u,
                       h3 = w.w & 0xF0F0F0F0u;
        const int sc = (int)((sc48 >> (6 * s)) & 63u);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 a0 = act_unit<kQ4K, NC>(act, cb, c, 16 * bl + 2 * s);
            const uint4 a1 = act_unit<kQ4K, NC>(act, cb, c, 16 * bl + 2 * s + 1);
            int pl = dp4a_ss(l0, a0.x, 0);
            pl = dp4a_ss(l1, a0.y, pl);
            pl = dp4a_ss(l2, a0.z, pl);
            pl = dp4a_ss(l3, a0.w, pl);
            int ph = dp4a_us(h0, a1.x, 0);  // 16*q against a: a multiple of 16
            ph = dp4a_us(h1, a1.y, ph);
            ph = dp4a_us(h2, a1.z, ph);
            ph = dp4a_us(h3, a1.w, ph);
            C[c] += sc * (pl + (ph >> 4));
        }
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 sv = *reinterpret_cast<const uint4 *>(s32 + c * s32_stride + 8 * bl);
        const uint32_t wv[4] = {sv.x, sv.y, sv.z, sv.w};
        int o = 0;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int S = (int)(int16_t)((wv[s >> 1] >> (16 * (s & 1))) & 0xFFFFu);
            o += (int)((mn48 >> (6 * s)) & 63u) * S;
        }
        O[c] = o;
    }
}

// Q6_K-like block: C_c = sum_u sc_u * sum_{i in u} (q_i - 32) a_i.
template <int NC>
__device__ __forceinline__ void block_q6k(const uint8_t *blk, const uint8_t *act, int cb, const int16_t *s16,
                                          int s16_stride, int bl, int (&C)[NC]) {
    const uint4 scw = *reinterpret_cast<const uint4 *>(blk + 192);
    const uint32_t scv[4] = {scw.x, scw.y, scw.z, scw.w};
#pragma unroll
    for (int c = 0; c < NC; ++c) C[c] = 0;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 16 * ch);
        const uint2 h = *reinterpret_cast<const uint2 *>(blk + 128 + 8 * ch);
        const uint32_t wl[4] = {w.x, w.y, w.z, w.w};
        uint32_t qlo[4], qhi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t hl = (k < 3) ? (h.x << (4 - 2 * k)) : (h.x >> 2);
            const uint32_t hh = (k < 3) ? (h.y << (4 - 2 * k)) : (h.y >> 2);
            qlo[k] = (wl[k] & 0x0F0F0F0Fu) | (hl & 0x30303030u);
            qhi[k] = ((wl[k] >> 4) & 0x0F0F0F0Fu) | (hh & 0x30303030u);
        }
        const int sc_lo = (int)(int8_t)((scv[ch >> 1] >> (16 * (ch & 1))) & 0xFFu);
        const int sc_hi = (int)(int8_t)((scv[ch >> 1] >> (16 * (ch & 1) + 8)) & 0xFFu);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const uint4 a0 = act_unit<kQ6K, NC>(act, cb, c, 16 * bl + 2 * ch);
            const uint4 a1 = act_unit<kQ6K, NC>(act, cb, c, 16 * bl + 2 * ch + 1);
            int pl = dp4a_ss(qlo[0], a0.x, 0);
            pl = dp4a_ss(qlo[1], a0.y, pl);
            pl = dp4a_ss(qlo[2], a0.z, pl);
            pl = dp4a_ss(qlo[3], a0.w, pl);
            int ph = dp4a_ss(qhi[0], a1.x, 0);
            ph = dp4a_ss(qhi[1], a1.y, ph);
            ph = dp4a_ss(qhi[2], a1.z, ph);
            ph = dp4a_ss(qhi[3], a1.w, ph);
            C[c] += sc_lo * pl + sc_hi * ph;
        }
    }
    // the -32 offset of every code: minus 32 * sum_u sc_u * S_u
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int16_t *sp = s16 + c * s16_stride;
        const int u0 = act_phys<kQ8_0>(2 * bl), u1 = act_phys<kQ8_0>(2 * bl + 1);
        const uint4 sa = *reinterpret_cast<const uint4 *>(sp + 8 * u0);
        const uint4 sb = *reinterpret_cast<const uint4 *>(sp + 8 * u1);
        const uint32_t sw[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
        int t = 0;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int S = (int)(int16_t)((sw[u >> 1] >> (16 * (u & 1))) & 0xFFFFu);
            const int sc = (int)(int8_t)((scv[u >> 2] >> (8 * (u & 3))) & 0xFFu);
            t += sc * S;
        }
        C[c] -= 32 * t;
    }
}

// Q8_0 block of 32: C_c = sum q_i a_i.
template <int NC>
__device__ __forceinline__ void block_q8_0(const uint8_t *q, const uint8_t *act, int cb, int bl, int (&C)[NC]) {
    const uint4 w0 = *reinterpret_cast<const uint4 *>(q);
    const uint4 w1 = *reinterpret_cast<const uint4 *>(q + 16);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 a0 = act_unit<kQ8_0, NC>(act, cb, c, 2 * bl);
        const uint4 a1 = act_unit<kQ8_0, NC>(act, cb, c, 2 * bl + 1);
        int p = dp4a_ss(w0.x, a0.x, 0);
        p = dp4a_ss(w0.y, a0.y, p);
        p = dp4a_ss(w0.z, a0.z, p);
        p = dp4a_ss(w0.w, a0.w, p);
        p = dp4a_ss(w1.x, a1.x, p);
        p = dp4a_ss(w1.y, a1.y, p);
        p = dp4a_ss(w1.z, a1.z, p);
        p = dp4a_ss(w1.w, a1.w, p);
        C[c] = p;
    }
}

// ----------------------------------------------------------------- the kernel

template <int F, int NC, int MODE>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvK p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int blk = fmt_block(F);
    const GemvSmem L = gemv_smem<F>(p.R, p.rec, p.kcb, NC, p.vstride, MODE);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    uint8_t *tile = smem + L.tile;
    uint8_t *act = smem + L.act;
    int16_t *sums = reinterpret_cast<int16_t *>(smem + L.sums);
    uint32_t *scl = reinterpret_cast<uint32_t *>(smem + L.scl);
    float *val = reinterpret_cast<float *>(smem + L.val);

    const int tid = threadIdx.x, T = blockDim.x;
    const int64_t row0 = (int64_t)blockIdx.x * p.R;
    const int nrows = (int)min((int64_t)p.R, p.rows - row0);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)nrows * (uint32_t)p.rec;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(tile, p.W + row0 * p.rec, bytes, bar);  // weights do not depend on earlier kernels
    }
    pdl_launch_dependents();
    pdl_wait();

    const int cb = act_col_bytes<F>(p.kcb);          // bytes per column of staged codes
    const int sb = sums_col_bytes<F>(p.kcb) / 2;     // int16 per column of staged sums
    bool first = true;
    for (int kc0 = 0; kc0 < p.nb; kc0 += p.kcb) {
        const int kcn = min(p.kcb, p.nb - kc0);
        // ---- stage the activation chunk: codes (swizzled), sums, scales
        const int units = kcn * blk / 16;
        for (int i = tid; i < NC * units; i += T) {
            const int c = i / units, u = i - c * units;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.codes + (int64_t)c * p.K +
                                                                  (int64_t)kc0 * blk) + u);
            *reinterpret_cast<uint4 *>(act + c * cb + act_phys<F>(u) * 16) = v;
        }
        if (F == kQ4K) {  // per-32 sums: S_s = sum16[2s] + sum16[2s+1]
            const int n32 = kcn * 8;
            for (int i = tid; i < NC * n32; i += T) {
                const int c = i / n32, s = i - c * n32;
                const int32_t pr = __ldg(reinterpret_cast<const int32_t *>(p.sums16 + (int64_t)c * (p.K / 16) +
                                                                           (int64_t)kc0 * 16) + s);
                sums[c * sb + s] = (int16_t)((int16_t)(pr & 0xFFFF) + (int16_t)(pr >> 16));
            }
        }
        if (F == kQ6K) {  // per-16 sums, 16-B units swizzled by line & 7
            const int n16u = kcn * 2;
            for (int i = tid; i < NC * n16u; i += T) {
                const int c = i / n16u, u = i - c * n16u;
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.sums16 + (int64_t)c * (p.K / 16) +
                                                                      (int64_t)kc0 * 16) + u);
                *reinterpret_cast<uint4 *>(sums + c * sb + act_phys<kQ8_0>(u) * 8) = v;
            }
        }
        for (int i = tid; i < NC * kcn; i += T) {
            const int c = i / kcn, b = i - c * kcn;
            scl[c * p.kcb + b] = __ldg(reinterpret_cast<const uint32_t *>(p.scales) + (int64_t)c * p.nb + kc0 + b);
        }
        __syncthreads();
        if (first) {
            const bool ok = __syncthreads_and(mbar_wait_bounded(bar, 0, p.fault));
            if (!ok) return;  // fault word raised; the copy never completed
            first = false;
        }
        // ---- items: consecutive threads take consecutive blocks of a row
        const int items = nrows * kcn;
        for (int i = tid; i < items; i += T) {
            const int r = i / kcn, bl = i - r * kcn, b = kc0 + bl;
            const uint8_t *rowp = tile + (int64_t)r * p.rec;
            int C[NC], O[NC];
            uint32_t s1, s2 = 0;
            if (F == kQ4K) {
                block_q4k<NC>(rowp + 144 * b, act, cb, sums, sb, bl, C, O, s1, s2);
            } else if (F == kQ6K) {
                block_q6k<NC>(rowp + 208 * b, act, cb, sums, sb, bl, C);
                s1 = *reinterpret_cast<const uint16_t *>(rowp + 208 * p.nb + 2 * b);
            } else {
                block_q8_0<NC>(rowp + 32 * b, act, cb, bl, C);
                s1 = *reinterpret_cast<const uint16_t *>(rowp + p.K + 2 * b);
            }
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const uint32_t sw = scl[c * p.kcb + bl];
                const int m = (int)(sw & 0xFFu), e = (int)(int16_t)(sw >> 16);
                float v;
                if (F == kQ4K) v = lane_value<1>(C[c], O[c], s1, s2, m, e);
                else v = lane_value<0>(C[c], 0, s1, 0, m, e);
                if (MODE == 0) {
                    val[(c * p.R + r) * p.vstride + b] = v;
                } else {
                    const int64_t o = ((int64_t)c * p.rows + row0 + r) * p.nb + b;
                    if (p.dbgC) p.dbgC[o] = C[c];
                    if (p.dbgO) p.dbgO[o] = (F == kQ4K) ? O[c] : 0;
                    if (p.dbgV) p.dbgV[o] = v;
                }
            }
        }
        __syncthreads();
    }
    if (MODE != 0) return;
    // ---- the row fold: block order from +0, f32 round-to-nearest-even, ftz
    for (int j = tid; j < NC * nrows; j += T) {
        const int c = j / nrows, r = j - c * nrows;
        const float *vr = val + (c * p.R + r) * p.vstride;
        float acc = 0.0f;
        for (int b = 0; b < p.nb; ++b) acc = fadd_ftz(acc, vr[b]);
        if (acc != acc) acc = __uint_as_float(kEngineNaN);
        p.out[(int64_t)c * p.rows + row0 + r] = acc;
    }
}

// ----------------------------------------------------------------- host launcher

template <int F, int NC, int MODE>
int launch_gemv_nc(const GemvK &k, int threads, int smem, unsigned grid, cudaStream_t stream) {
    if (ensure_smem_limit(reinterpret_cast<const void *>(gemv_kernel<F, NC, MODE>), 227 * 1024) != QB_OK)
        return QB_E_CUDA;
    return launch_pdl(gemv_kernel<F, NC, MODE>, dim3(grid), dim3(threads), (size_t)smem, stream, k);
}

// Columns 1..8 are instantiated in the format's own translation unit, 9..16
// in a second one (qb_gemv_<fmt>_hi.cu), so the two halves compile in parallel.
template <int F, int LO, int HI>
int dispatch_range(int nc, const GemvK &k, int threads, int smem, unsigned grid, cudaStream_t s) {
    if constexpr (LO > HI) {
        return QB_E_ARG;
    } else {
        if (nc == LO) return launch_gemv_nc<F, LO, 0>(k, threads, smem, grid, s);
        return dispatch_range<F, LO + 1, HI>(nc, k, threads, smem, grid, s);
    }
}
template <int F>
int dispatch_hi(int nc, const GemvK &k, int threads, int smem, unsigned grid, cudaStream_t s);
// The streaming kernel for 2..16 columns (qb_gemv3.cuh, instantiated in
// qb_skinny_*.cu); QB_E_ARG when it does not apply to the shape.
template <int F>
int launch_skinny(const GemvArgs &a, cudaStream_t stream);
// One column through the multi-column kernel's organisation where it is the
// faster one (qb_gemv3.cuh, launch_gemv3_one); QB_E_ARG where it does not apply.
template <int F>
int launch_one_col3(const GemvArgs &a, cudaStream_t stream, const float *x);

inline int gcd_int(int a, int b) { while (b) { int t = a % b; a = b; b = t; } return a; }

// Tile and launch shape: a tile of R rows (about 24 KB of weights, fewer rows
// when the matrix would not fill every SM), R*blocks a multiple of 32 where
// possible; activation chunks of at most 64 KB of codes.
template <int F>
int launch_gemv_fmt(const GemvArgs &a, cudaStream_t stream) {
    constexpr int blk = fmt_block(F);
    if (a.mode == 0 && a.ncols == 1) {  // the streaming kernels, where they apply
        int rc = launch_one_col3<F>(a, stream, nullptr);
        if (rc != QB_E_ARG) return rc;
        rc = launch_gemv2<F>(a, stream);
        if (rc != QB_E_ARG) return rc;
    }
    if (a.mode == 0 && a.ncols >= 2) {
        const int rc = launch_skinny<F>(a, stream);
        if (rc != QB_E_ARG) return rc;
    }
    if (a.mats) return QB_E_ARG;  // a table of matrices: the streaming kernels only (the caller falls back)
    GemvK k;
    k.W = static_cast<const uint8_t *>(a.W);
    k.rows = a.rows;
    k.K = (int)a.K;
    k.nb = (int)(a.K / blk);
    k.rec = (int)record_bytes(F, a.K);
    const int64_t sms = num_sms();
    int R = std::max(1, 24576 / k.rec);
    R = (int)std::min<int64_t>(R, std::max<int64_t>(1, (a.rows + sms - 1) / sms));
    R = std::min(R, 64);
    const int g = 32 / gcd_int(k.nb, 32);
    if (R > g) R = R / g * g;
    k.R = R;
    k.kcb = std::min(k.nb, std::max(1, 65536 / (a.ncols * blk)));
    k.vstride = (k.nb & 1) ? k.nb : k.nb + 1;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.out = a.out;
    k.dbgC = a.dbgC;
    k.dbgO = a.dbgO;
    k.dbgV = a.dbgV;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    const GemvSmem L = gemv_smem<F>(R, k.rec, k.kcb, a.ncols, k.vstride, a.mode);
    if (L.total > 227 * 1024) return QB_E_ARG;
    const int threads = (int)std::min<int64_t>(256, (int64_t)(R * std::min(k.nb, k.kcb) + 31) / 32 * 32);
    const unsigned grid = (unsigned)((a.rows + R - 1) / R);
    if (a.mode == 0) {
        if (a.ncols <= 8) return dispatch_range<F, 1, 8>(a.ncols, k, threads, L.total, grid, stream);
        return dispatch_hi<F>(a.ncols, k, threads, L.total, grid, stream);
    }
    // per-block results (testing): one single-column launch per column
    for (int c = 0; c < a.ncols; ++c) {
        GemvK kc = k;
        kc.codes = a.codes + (int64_t)c * a.K;
        kc.scales = a.scales + (int64_t)c * k.nb;
        kc.sums16 = a.sums16 ? a.sums16 + (int64_t)c * (a.K / 16) : nullptr;
        const int64_t o = (int64_t)c * a.rows * k.nb;
        kc.dbgC = a.dbgC ? a.dbgC + o : nullptr;
        kc.dbgO = a.dbgO ? a.dbgO + o : nullptr;
        kc.dbgV = a.dbgV ? a.dbgV + o : nullptr;
        const GemvSmem L1 = gemv_smem<F>(R, k.rec, k.kcb, 1, k.vstride, 1);
        const int rc = launch_gemv_nc<F, 1, 1>(kc, threads, L1.total, grid, stream);
        if (rc) return rc;
    }
    return QB_OK;
}

}  // namespace qb
