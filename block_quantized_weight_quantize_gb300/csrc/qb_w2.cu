// qb_w2.cu -- the product with activation codes that cross in two words
// (lane page, opening description and WordSums; numerics page, Words): a
// 16-bit code a = 256*hi + lo, hi its signed high byte and lo its unsigned
// low byte.
//
// The array takes a code word by word, so here each unit's dots are formed
// per word with dp4a -- the weights against the signed high bytes and against
// the unsigned low bytes -- and joined as 256*(high) + (low); the block sums
// C = sum coef*a and O = sum offs*a reach 2^36 in magnitude, so they are
// accumulated in 64 bits and combined with the block's scales and the
// activation scale in 128 bits, rounded once (the same rounding as every other
// path), and each row's values are added in block order from +0.
//
// Organisation: a warp per row (grid-stride over rows), lanes over the row's
// blocks; a lane holds its block's weights in registers while it forms the
// block's value for each column of a chunk, the values go to a per-warp
// shared strip [column][block], and one lane per column folds them in order.
#include <algorithm>

#include "qb_common.cuh"
#include "qb_launch.h"

namespace qb {

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four 16-bit codes (two 32-bit words) as their high bytes (signed) and low
// bytes (unsigned), each packed four to a word in element order.
__device__ __forceinline__ void split_words(uint2 w, uint32_t &hi, uint32_t &lo) {
    uint32_t h, l;
    asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(h) : "r"(w.x), "r"(w.y));
    asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(l) : "r"(w.x), "r"(w.y));
    hi = h;
    lo = l;
}

// sum over 4 elements of q*a for four weight bytes q (signed if QS) and four
// 16-bit codes: 256*(q . hi) + (q . lo)
template <bool QS>
__device__ __forceinline__ int dot4_w2(uint32_t q, uint2 w) {
    uint32_t hi, lo;
    split_words(w, hi, lo);
    const int ph = QS ? dp4a_ss(q, hi, 0) : dp4a_us(q, hi, 0);
    const int pl = QS ? dp4a_su(q, lo, 0) : dp4a_uu(q, lo, 0);
    return 256 * ph + pl;
}
// sum of four 16-bit codes
__device__ __forceinline__ int sum4_w2(uint2 w) {
    uint32_t hi, lo;
    split_words(w, hi, lo);
    return 256 * dp4a_ss(0x01010101u, hi, 0) + dp4a_uu(0x01010101u, lo, 0);
}

// m*2^e*(s1*C - s2*O) (kind 1) or m*2^e*s1*C (kind 0) with 64-bit sums,
// rounded once (lane page, lane); the engine's NaN for an unreadable scale or
// an activation block without one.
__device__ __noinline__ float lane_value_w2(long long C, long long O, uint32_t s1, uint32_t s2, int kind, int m,
                                            int e) {
    int sig1, ex1, sig2 = 0, ex2 = 0;
    bool ok = f16_scale(s1, sig1, ex1) && m != 0;
    if (kind) ok = f16_scale(s2, sig2, ex2) && ok;
    if (!ok) return __uint_as_float(kEngineNaN);
    const __int128 t1 = (__int128)((long long)sig1 * m) * C;  // |t1| < 2^19 * 2^37
    if (!kind) return round_to_f32_wide(t1, ex1 + e);
    const __int128 t2 = -(__int128)((long long)sig2 * m) * O;
    const int lo = ex1 < ex2 ? ex1 : ex2;
    return round_to_f32_wide((t1 << (ex1 - lo)) + (t2 << (ex2 - lo)), lo + e);  // < 2^56 shifted <= 29 places
}

struct W2K {
    const uint8_t *W;
    int64_t rows, K;
    int64_t rec;
    int nb;     // blocks a row
    int ncols;  // columns
    int ncc;    // columns a chunk (the strip holds ncc x nb values)
    const int16_t *codes;
    const qb_scale *scales;
    float *out;
};

constexpr int kW2Warps = 8;

template <int F>
__global__ void __launch_bounds__(kW2Warps * 32) w2_kernel(const W2K p) {
    extern __shared__ __align__(16) float strip[];  // [warp][ncc][nb]
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float *vs = strip + (size_t)w * p.ncc * p.nb;
    pdl_wait();  // the codes may come from the previous kernel; out may be read by it
    for (int64_t r = (int64_t)blockIdx.x * kW2Warps + w; r < p.rows; r += (int64_t)gridDim.x * kW2Warps) {
        const uint8_t *row = p.W + r * p.rec;
        for (int c0 = 0; c0 < p.ncols; c0 += p.ncc) {
            const int nc = min(p.ncc, p.ncols - c0);
            for (int b = lane; b < p.nb; b += 32) {
                if (F == kQ8_0) {
                    uint32_t q[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) q[i] = reinterpret_cast<const uint32_t *>(row + 32 * b)[i];
                    const uint32_t d = *reinterpret_cast<const uint16_t *>(row + p.K + 2 * b);
                    for (int c = 0; c < nc; ++c) {
                        const int16_t *a = p.codes + (int64_t)(c0 + c) * p.K + 32 * b;
                        int s = 0;  // |sum| <= 127 * 32768 * 32 < 2^31
#pragma unroll
                        for (int i = 0; i < 8; ++i) s += dot4_w2<true>(q[i], reinterpret_cast<const uint2 *>(a)[i]);
                        const uint32_t sc = reinterpret_cast<const uint32_t *>(p.scales)[(int64_t)(c0 + c) * p.nb + b];
                        vs[c * p.nb + b] = lane_value_w2(s, 0, d, 0, 0, (int)(sc & 0xFFu), (int)(int16_t)(sc >> 16));
                    }
                } else if (F == kQ4K) {
                    const uint8_t *blk = row + 144 * b;
                    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
                    const unsigned long long sc48 =
                        (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
                    const unsigned long long mn48 =
                        (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
                    uint4 qs[8];
#pragma unroll
                    for (int s = 0; s < 8; ++s) qs[s] = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * s);
                    for (int c = 0; c < nc; ++c) {
                        const int16_t *a = p.codes + (int64_t)(c0 + c) * p.K + 256 * b;
                        long long C = 0, O = 0;
#pragma unroll
                        for (int s = 0; s < 8; ++s) {
                            const uint32_t wq[4] = {qs[s].x, qs[s].y, qs[s].z, qs[s].w};
                            const uint2 *al = reinterpret_cast<const uint2 *>(a + 32 * s);       // elements 0..15
                            const uint2 *ah = reinterpret_cast<const uint2 *>(a + 32 * s + 16);  // elements 16..31
                            int dsum = 0, asum = 0;  // |dsum| <= 15 * 32768 * 32 < 2^24
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                // byte j of the 16: element j (low nibble) and element 16 + j (high nibble)
                                dsum += dot4_w2<false>(wq[k] & 0x0F0F0F0Fu, al[k]);
                                dsum += dot4_w2<false>((wq[k] >> 4) & 0x0F0F0F0Fu, ah[k]);
                                asum += sum4_w2(al[k]) + sum4_w2(ah[k]);
                            }
                            C += (long long)((sc48 >> (6 * s)) & 63u) * dsum;
                            O += (long long)((mn48 >> (6 * s)) & 63u) * asum;
                        }
                        const uint32_t sc = reinterpret_cast<const uint32_t *>(p.scales)[(int64_t)(c0 + c) * p.nb + b];
                        vs[c * p.nb + b] = lane_value_w2(C, O, meta.x & 0xFFFFu, meta.x >> 16, 1, (int)(sc & 0xFFu),
                                                         (int)(int16_t)(sc >> 16));
                    }
                } else {
                    const uint8_t *blk = row + 208 * b;
                    const uint32_t d = *reinterpret_cast<const uint16_t *>(row + 208 * p.nb + 2 * b);
                    for (int c = 0; c < nc; ++c) {
                        const int16_t *a = p.codes + (int64_t)(c0 + c) * p.K + 256 * b;
                        long long C = 0;
#pragma unroll 2
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint4 w = *reinterpret_cast<const uint4 *>(blk + 16 * ch);
                            const uint2 hb = *reinterpret_cast<const uint2 *>(blk + 128 + 8 * ch);
                            const uint32_t wl[4] = {w.x, w.y, w.z, w.w};
                            const uint2 *al = reinterpret_cast<const uint2 *>(a + 32 * ch);
                            const uint2 *ah = reinterpret_cast<const uint2 *>(a + 32 * ch + 16);
                            int pl = 0, ph = 0;  // the chunk's two units: sum (q - 32)*a, |.| <= 32 * 32768 * 16
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint32_t hl = (k < 3) ? (hb.x << (4 - 2 * k)) : (hb.x >> 2);
                                const uint32_t hh = (k < 3) ? (hb.y << (4 - 2 * k)) : (hb.y >> 2);
                                // q - 32 for four bytes: q in 0..63, as signed bytes (q ^ 0x20) - 0x20 per byte
                                const uint32_t ql = (wl[k] & 0x0F0F0F0Fu) | (hl & 0x30303030u);
                                const uint32_t qh = ((wl[k] >> 4) & 0x0F0F0F0Fu) | (hh & 0x30303030u);
                                pl += dot4_w2<true>(__vsub4(ql, 0x20202020u), al[k]);
                                ph += dot4_w2<true>(__vsub4(qh, 0x20202020u), ah[k]);
                            }
                            const uint32_t scp = *reinterpret_cast<const uint16_t *>(blk + 192 + 2 * ch);
                            C += (long long)(int8_t)(scp & 0xFFu) * pl + (long long)(int8_t)(scp >> 8) * ph;
                        }
                        const uint32_t sc = reinterpret_cast<const uint32_t *>(p.scales)[(int64_t)(c0 + c) * p.nb + b];
                        vs[c * p.nb + b] = lane_value_w2(C, 0, d, 0, 0, (int)(sc & 0xFFu), (int)(int16_t)(sc >> 16));
                    }
                }
            }
            __syncwarp();
            // fold: lane c adds column c's values in block order from +0
            for (int c = lane; c < nc; c += 32) {
                float acc = 0.0f;
                for (int b = 0; b < p.nb; ++b) acc = fadd_ftz(acc, vs[c * p.nb + b]);
                if (acc != acc) acc = __uint_as_float(kEngineNaN);
                p.out[(int64_t)(c0 + c) * p.rows + r] = acc;
            }
            __syncwarp();
        }
    }
}

int launch_gemv_w2(int f, const void *W, int64_t rows, int64_t K, const int16_t *codes, const qb_scale *scales,
                   int ncols, float *out, cudaStream_t stream) {
    W2K k;
    k.W = static_cast<const uint8_t *>(W);
    k.rows = rows;
    k.K = K;
    k.rec = record_bytes(f, K);
    k.nb = (int)(K / fmt_block(f));
    k.ncols = ncols;
    const int budget = 96 * 1024;  // the strip of all warps
    k.ncc = std::max(1, std::min(ncols, budget / (kW2Warps * 4 * k.nb)));
    if ((int64_t)kW2Warps * 4 * k.nb * k.ncc > 227 * 1024) return QB_E_ARG;  // a row longer than the strip
    k.codes = codes;
    k.scales = scales;
    k.out = out;
    const int smem = kW2Warps * 4 * k.nb * k.ncc;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + kW2Warps - 1) / kW2Warps,
                                                                 (int64_t)num_sms() * 8));
    auto kern = f == kQ8_0 ? w2_kernel<kQ8_0> : f == kQ4K ? w2_kernel<kQ4K> : w2_kernel<kQ6K>;
    if (ensure_smem_limit(reinterpret_cast<const void *>(kern), smem) != QB_OK) return QB_E_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(kW2Warps * 32), (size_t)smem, stream, k);
}

}  // namespace qb
