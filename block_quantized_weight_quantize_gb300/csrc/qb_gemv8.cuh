// qb_gemv8.cuh -- 1..16 activation columns of a Q4_K-like or Q6_K-like matrix
// (or a table of them) at K = 256 * NB, NB <= 16: a warp per weight block, a
// lane per row, rows streamed in chunks of 32.
//
// The arithmetic is the other kernels' (the lane page's exact block sums, the
// exact combine rounded once, each row folded in block order from +0, every
// column by itself).  The organisation reads each weight once and unpacks it
// once for all the columns of a launch:
//   * the CTA's rows arrive in chunks of 32 by one bulk copy a row (the TMA
//     engine) into a pitch of rec + 16 bytes (an odd number of 16-B units,
//     so the eight lanes of a shared-memory phase read eight bank groups),
//     through a ring of one or two chunk slots;
//   * lane r of warp w moves block w of the chunk's row r into registers, the
//     slot is released for the next fill, and the lane forms the block's sums
//     and rounded value for each column in turn, reading that column's codes
//     of block w as broadcasts;
//   * block values go to a [row][column][17] table, and after a CTA barrier
//     one thread per (row, column) folds its row's values in block order.
#pragma once

#include <algorithm>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_gemv7.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"

namespace qb {

struct Gemv8K {
    MatTable mt;   // the matrix (or matrices sharing the activation) as one row range
    int64_t rows;  // rows of the whole range
    int rec;       // bytes per row record
    int pitch;     // bytes per row in a slot (rec + 16)
    int nb;        // weight blocks per row (= warps a CTA)
    int D;         // chunk slots (1 or 2)
    int64_t base;  // rows per CTA, and how many CTAs own one more
    int64_t rem;
    const int8_t *codes;  // the quantized activation: NC columns
    const qb_scale *scales;
    const int16_t *sums16;
    int *fault;
};

constexpr int kG8Chunk = 32;  // rows a chunk: a lane each

// The value table's stride per row: NC columns of 17 floats, made odd so the
// lanes of a warp (one row each) write different banks.
__host__ __device__ constexpr int gemv8_rs(int nc) { return (nc * 17) | 1; }

struct Gemv8Smem {
    int bars, codes, sums, scl, vals, slots, total;
};
__host__ __device__ inline Gemv8Smem gemv8_smem(int nc, int nb, int pitch, int D) {
    Gemv8Smem s;
    s.bars = 0;
    s.codes = 128;                                                  // nc x 256*nb codes
    s.sums = s.codes + nc * 256 * nb;                               // nc x nb x 16 int16
    s.scl = s.sums + nc * nb * 32;                                  // nc x nb scales
    s.vals = s.scl + ((nc * nb * 4 + 127) & ~127);                  // 32 rows x gemv8_rs(nc)
    s.slots = s.vals + ((kG8Chunk * gemv8_rs(nc) * 4 + 127) & ~127);
    s.total = s.slots + D * kG8Chunk * pitch;
    return s;
}

// A Q6_K-like block held in registers: ql (8 x 16 B), qh (8 x 8 B), the 16
// sub-scales, and the row's f16 scale of this block.
struct BlkQ6 {
    uint4 ql[8];
    uint2 qh[8];
    uint4 sc;
    uint32_t d;
};

__device__ __forceinline__ void load_q6k(const uint8_t *blk, const uint8_t *dptr, BlkQ6 &b) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        b.ql[ch] = *reinterpret_cast<const uint4 *>(blk + 16 * ch);
        b.qh[ch] = *reinterpret_cast<const uint2 *>(blk + 128 + 8 * ch);
    }
    b.sc = *reinterpret_cast<const uint4 *>(blk + 192);
    b.d = *reinterpret_cast<const uint16_t *>(dptr);
}

// block_q6k's sum for a block held in registers.
__device__ __forceinline__ int dot_q6k(const BlkQ6 &b, const uint8_t *a, const int16_t *S) {
    const uint32_t scw[4] = {b.sc.x, b.sc.y, b.sc.z, b.sc.w};
    const uint4 s0 = *reinterpret_cast<const uint4 *>(S), s1 = *reinterpret_cast<const uint4 *>(S + 8);
    const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    int c = 0;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = b.ql[ch];
        const uint2 hb = b.qh[ch];
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
        c += sc_lo * (pl - 32 * (int)(int16_t)(sw[ch] & 0xFFFFu)) + sc_hi * (ph - 32 * (int)(int16_t)(sw[ch] >> 16));
    }
    return c;
}

template <int F, int NC>
__global__ void __launch_bounds__(512, 1) gemv8_kernel(const Gemv8K p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nb = p.nb, K = 256 * nb, nthreads = 32 * nb;
    const Gemv8Smem L = gemv8_smem(NC, nb, p.pitch, p.D);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint8_t *codes = smem + L.codes;                                 // [NC][K]
    int16_t *sums = reinterpret_cast<int16_t *>(smem + L.sums);      // [NC][nb][16]
    uint32_t *scl = reinterpret_cast<uint32_t *>(smem + L.scl);      // [NC][nb]
    float *vals = reinterpret_cast<float *>(smem + L.vals);          // [32][gemv8_rs(NC)]
    uint8_t *slots = smem + L.slots;
    constexpr int RS = gemv8_rs(NC);

    const int64_t c0 = blockIdx.x;
    const int64_t row0 = c0 * p.base + (c0 < p.rem ? c0 : p.rem);
    const int count = (int)(p.base + (c0 < p.rem ? 1 : 0));
    const int nchunk = (count + kG8Chunk - 1) / kG8Chunk;

    if (tid == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // chunk i's rows into slot i % D, one bulk copy a row from the lanes of warp 0
    auto fill = [&](int i) {
        if (w != 0 || i >= nchunk) return;
        const int n = min(kG8Chunk, count - kG8Chunk * i);
        uint64_t *bar = bars + (i % p.D);
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(n * p.rec));
        __syncwarp();
        if (lane < n)
            bulk_g2s(slots + (i % p.D) * kG8Chunk * p.pitch + lane * p.pitch,
                     row_ptr(p.mt, row0 + kG8Chunk * i + lane, p.rec), (uint32_t)p.rec, bar);
    };
    for (int i = 0; i < p.D; ++i) fill(i);  // weights depend on no earlier kernel
    pdl_launch_dependents();
    pdl_wait();

    // ---- the activation: codes of every column, each block's sub-block (Q4_K)
    // or unit (Q6_K) sums, the block scales
    for (int t = tid; t < NC * K / 16; t += nthreads)
        reinterpret_cast<uint4 *>(codes)[t] = ldg_v4_ordered(reinterpret_cast<const uint4 *>(p.codes) + t);
    for (int t = tid; t < NC * nb * 16; t += nthreads) {  // (column, block, unit)
        const int cb = t >> 4, u = t & 15;
        if (F == kQ4K) {
            if (u < 8) {
                const int16_t *src = p.sums16 + (int64_t)cb * 16 + 2 * u;
                sums[cb * 16 + u] = (int16_t)((int)src[0] + (int)src[1]);
            }
        } else {
            sums[cb * 16 + u] = p.sums16[(int64_t)cb * 16 + u];
        }
    }
    for (int t = tid; t < NC * nb; t += nthreads) scl[t] = reinterpret_cast<const uint32_t *>(p.scales)[t];
    __syncthreads();

    for (int i = 0; i < nchunk; ++i) {
        const int slot = i % p.D;
        const int n = min(kG8Chunk, count - kG8Chunk * i);
        const bool ok = mbar_wait_bounded(bars + slot, (uint32_t)((i / p.D) & 1), p.fault);
        if (!__syncthreads_and(ok)) return;  // a fill never completed: fault word raised
        const uint8_t *row = slots + slot * kG8Chunk * p.pitch + lane * p.pitch;
        BlkQ4 b4;
        BlkQ6 b6;
        if (lane < n) {
            if (F == kQ4K) load_q4k(row + 144 * w, b4);
            else load_q6k(row + 208 * w, row + 208 * nb + 2 * w, b6);
        }
        __syncthreads();  // every warp has its blocks of the slot; the last fold has read the table
        if (w == 0 && i + p.D < nchunk) {
            if (lane == 0) fence_proxy_async_smem();
            __syncwarp();
            fill(i + p.D);
        }
        if (lane < n) {
#pragma unroll 1
            for (int c = 0; c < NC; ++c) {
                const uint8_t *a = codes + c * K + 256 * w;
                const int16_t *S = sums + (c * nb + w) * 16;
                const uint32_t sv = scl[c * nb + w];
                const int m0 = (int)(sv & 0xFFu), e0 = (int)(int16_t)(sv >> 16);
                float v;
                if (F == kQ4K) {
                    int C16, O;
                    dot_q4k(b4, a, S, C16, O);
                    v = lane_value_fast<1>(C16 >> 4, O, b4.dd & 0xFFFFu, b4.dd >> 16, m0, e0);  // 16*C: exact shift
                } else {
                    v = lane_value_fast<0>(dot_q6k(b6, a, S), 0, b6.d, 0, m0, e0);
                }
                vals[lane * RS + c * 17 + w] = v;
            }
        }
        __syncthreads();
        // ---- fold: thread (r, c) adds row r's block values of column c in order
        for (int t = tid; t < kG8Chunk * NC; t += nthreads) {
            const int r = t / NC, c = t - r * NC;
            if (r < n) {
                const float *vr = vals + r * RS + c * 17;
                float acc = 0.0f;
                for (int bk = 0; bk < nb; ++bk) acc = fadd_ftz(acc, vr[bk]);
                if (acc != acc) acc = __uint_as_float(kEngineNaN);
                *out_ptr(p.mt, c, row0 + kG8Chunk * i + r) = acc;
            }
        }
    }
}

// NC columns of a Q4_K-like or Q6_K-like matrix (or a table of them) at
// K = 256 * nb, nb <= 16, from a quantized activation.  QB_E_ARG when the
// shape does not fit.
template <int F, int NC>
int launch_gemv8_nc(const GemvArgs &a, cudaStream_t stream) {
    if ((F != kQ4K && F != kQ6K) || a.mode != 0 || a.K % 256 != 0 || a.K > 4096 || a.K < 256) return QB_E_ARG;
    Gemv8K k;
    k.mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    k.rows = k.mt.start[k.mt.n];
    if (k.rows < 1) return QB_E_ARG;
    k.nb = (int)(a.K / 256);
    k.rec = (int)record_bytes(F, a.K);
    k.pitch = k.rec + 16;
    k.D = 2;
    if (gemv8_smem(NC, k.nb, k.pitch, 2).total > 227 * 1024) k.D = 1;
    const int smem = gemv8_smem(NC, k.nb, k.pitch, k.D).total;
    if (smem > 227 * 1024) return QB_E_ARG;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), k.rows));
    k.base = k.rows / grid;
    k.rem = k.rows % grid;
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    auto kern = gemv8_kernel<F, NC>;
    if (ensure_smem_limit(reinterpret_cast<const void *>(kern), smem) != QB_OK) return QB_E_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(32 * k.nb), (size_t)smem, stream, k);
}

}  // namespace qb
