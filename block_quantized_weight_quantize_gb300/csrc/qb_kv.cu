// qb_kv.cu -- the int8 cache's score path (the decode engine's numerics page:
// cache_row, int8_codes, INV_127, quantize_head, int8_score).
//
// kv_cache_rows: a cache row is stored as int8 codes under one f16 scale:
//   amax = absmax(row) (a denormal read as zero, NaN passed over), the scale
//   f32_to_f16(amax * INV_127) (an f32 product, flushed), the codes
//   int8_codes of the row under the reciprocal of that scale: x*inv (f32,
//   flushed) to the nearest integer, ties to even, within +-127, a NaN product
//   0, all codes 0 when the reciprocal is infinite (a scale that rounded to
//   zero).  The reciprocal is the correctly rounded f32 1/s (the page's recip
//   seeds Newton steps from a table it does not print).
// kv_quantize_heads: quantize_head -- per 32 elements with the head padded by
//   zeros to a whole number of groups (ActScaling::Sub32), or the whole head
//   one block under wide_scale (ActScaling::PerBlock).
// kv_scores: int8_score of every query head against every cached key row of
//   its key head: per query block b, D_b = sum of q_i*k_i; the terms
//   sig(ks)*m_b*D_b at exponent exp(ks)+e_b summed exactly and rounded once;
//   then the f32 product with the attention scale (flushed).
//
// The score kernel puts the block dots on the tensor cores: one
// mma.sync.m16n8k32 (int8 x int8 -> int32) is 16 key rows by 8 query heads by
// exactly one 32-element block, so its accumulators are the D_b themselves.
// Each thread loads 8 contiguous bytes of a row's block (rows g and g+8) as
// its A registers and the same 8 bytes of its query head as its B registers:
// thread t's A and B fragments cover the same logical k slots, so any
// physical-to-logical map that depends only on t gives the same dot.  The
// block sums are then made exact as in the Sub32 product: with Emin the least
// exponent of a head's blocks, M_b = m_b << (e_b - Emin) < 2^16 while the
// exponents lie within 12 places, and sum_b M_b*D_b is exact in 64 bits
// (|D_b| < 2^19, at most 32 blocks); one rounding per score.  A head whose
// scales spread wider takes an out-of-line exact routine per score.
#include <cuda_fp16.h>

#include <algorithm>
#include <climits>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_launch.h"
#include "qb_quant.cuh"
#include "qb_sub32.cuh"

namespace qb {

constexpr uint32_t kInv127Bits = 0x3C010204u;  // INV_127: 1/127 rounded to f32

__device__ __forceinline__ float fmul_ftz(float a, float b) {
    float d;
    asm("mul.rn.ftz.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ float abs_ftz(float a) {
    float d;
    asm("abs.ftz.f32 %0, %1;" : "=f"(d) : "f"(a));
    return d;
}

// int8_codes of one element under inv (zero: the reciprocal is infinite).
__device__ __forceinline__ int int8_code(float x, float inv, bool zero) {
    const float p = fmul_ftz(x, inv);
    if (zero) return 0;
    if (p >= 127.0f) return 127;
    if (p <= -127.0f) return -127;
    return __float2int_rn(p);  // ties to even; NaN gives 0
}

// ------------------------------------------------------------------ cache_row

// One warp per row; d % 4 == 0.
__global__ void __launch_bounds__(256) kv_cache_rows_kernel(const float *__restrict__ x, int64_t n, int d,
                                                            int8_t *__restrict__ codes,
                                                            uint16_t *__restrict__ scales) {
    // no early launch_dependents: the score kernel reads key rows before its
    // own pdl_wait, so the kernel after this one starts when it has finished
    pdl_wait();
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= n) return;  // whole warps
    const float4 *xr = reinterpret_cast<const float4 *>(x + row * d);
    const int n4 = d / 4;
    float am = 0.0f;
    for (int i = lane; i < n4; i += 32) {
        const float4 v = __ldg(xr + i);
        am = fmaxf(fmaxf(fmaxf(fmaxf(am, abs_ftz(v.x)), abs_ftz(v.y)), abs_ftz(v.z)), abs_ftz(v.w));
    }
    uint32_t ab = __float_as_uint(am);  // non-negative: the integer order is the value order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ab = max(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, o));
    const __half hs = __float2half_rn(fmul_ftz(__uint_as_float(ab), __uint_as_float(kInv127Bits)));
    const float inv = __frcp_rn(__half2float(hs));
    const bool zero = isinf(inv);
    char4 *cr = reinterpret_cast<char4 *>(codes + row * d);
    for (int i = lane; i < n4; i += 32) {
        const float4 v = __ldg(xr + i);
        cr[i] = make_char4((signed char)int8_code(v.x, inv, zero), (signed char)int8_code(v.y, inv, zero),
                           (signed char)int8_code(v.z, inv, zero), (signed char)int8_code(v.w, inv, zero));
    }
    if (lane == 0) scales[row] = __half_as_ushort(hs);
}

// ------------------------------------------------------------------ quantize_head

// Sub32: one thread per 8 elements of the padded heads [nh][dp]; a 32-element
// block is 4 consecutive lanes.  Elements past d are zeros.
__global__ void __launch_bounds__(256) kv_heads_sub32_kernel(const float *__restrict__ q, int nh, int d, int dp,
                                                             int8_t *__restrict__ codes,
                                                             qb_scale *__restrict__ scales) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n8 = (int64_t)nh * dp / 8;
    const bool live = t < n8;
    const int64_t h = live ? (t * 8) / dp : 0;
    const int i0 = live ? (int)(t * 8 - h * dp) : 0;
    uint32_t xb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xb[i] = (live && i0 + i < d) ? __float_as_uint(__ldg(q + h * d + i0 + i)) : 0u;
    uint2 c;
    int usum;
    uint32_t scale;
    quantize8<4, true>(xb, c, usum, scale);
    if (live) {
        *reinterpret_cast<uint2 *>(codes + t * 8) = c;
        if ((t & 3) == 0) reinterpret_cast<uint32_t *>(scales)[t / 4] = scale;
    }
}

// PerBlock: one CTA per head, the whole head one block under wide_scale; the
// codes by the exact integer routine (a head is a few hundred elements).
__global__ void __launch_bounds__(256) kv_heads_perblock_kernel(const float *__restrict__ q, int d,
                                                                int8_t *__restrict__ codes,
                                                                qb_scale *__restrict__ scales) {
    __shared__ uint32_t red[8];
    pdl_launch_dependents();
    pdl_wait();
    const int h = blockIdx.x;
    const float *qh = q + (int64_t)h * d;
    float am = 0.0f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) am = fmaxf(am, abs_ftz(__ldg(qh + i)));
    uint32_t ab = __float_as_uint(am);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ab = max(ab, __shfl_xor_sync(0xFFFFFFFFu, ab, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ab;
    __syncthreads();
    ab = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) ab = max(ab, red[w]);
    int m, e;
    wide_scale_bits(ab, m, e);
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        codes[(int64_t)h * d + i] = (int8_t)rne_div1_exact(__float_as_uint(__ldg(qh + i)), m, e);
    if (threadIdx.x == 0) reinterpret_cast<uint32_t *>(scales)[h] = (uint32_t)(m & 0xFF) | ((uint32_t)(uint16_t)(int16_t)e << 16);
}

// ------------------------------------------------------------------ int8_score

// One score exactly: the query head's nbq blocks of blk codes (scales qs),
// the key row's d codes and f16 scale bits ksb, summed by exact_sum_terms.
static __device__ __noinline__ float kv_score_exact(const int8_t *q, const qb_scale *qs, int nbq, int blk, int d,
                                                    const int8_t *k, uint32_t ksb) {
    int sg, ex;
    if (!f16_scale(ksb, sg, ex)) return __uint_as_float(kEngineNaN);
    long long sig[32];
    int E[32];
    for (int b = 0; b < nbq; ++b) {
        const uint32_t sw = reinterpret_cast<const uint32_t *>(qs)[b];
        const int m = (int)(sw & 0xFFu), e = (int)(int16_t)(sw >> 16);
        if (m == 0) return __uint_as_float(kEngineNaN);
        long long D = 0;
        for (int i = b * blk; i < (b + 1) * blk && i < d; ++i) D += (int)q[i] * (int)k[i];
        sig[b] = (long long)sg * m * D;
        E[b] = ex + e;
    }
    return exact_sum_terms(sig, E, nbq);
}

struct KvK {
    const int8_t *qc;
    const qb_scale *qs;
    int nh, d, dp, nbq, G, nchunk;
    const int8_t *kc;
    const uint16_t *ks;
    int64_t L, lcap, ntr, ntiles;
    int nkv;
    float scale;
    float *out;
};

__device__ __forceinline__ void mma_s8_16832(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float finish_score(float v, float scale) {
    v = fmul_ftz(v, scale);
    return (v != v) ? __uint_as_float(kEngineNaN) : v;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int NB>
constexpr int kv_ring_depth() { return NB >= 8 ? 2 : 4; }
// Shared memory of a score CTA: the head table, then each warp's ring of
// tiles (16 rows at a pitch of d + 32 bytes, so that the fragment reads of a
// half warp -- 4 rows x 4 eight-byte slots -- fall in 16 distinct bank pairs).
template <int NB>
__host__ __device__ inline int kv_smem_bytes(int nh) {
    return ((nh * (2 + NB) * 4 + 15) & ~15) + 8 * kv_ring_depth<NB>() * 16 * (32 * NB + 32);
}

// Per query head, in shared memory: [mode, emin, M_0 .. M_{NB-1}] (mode 0
// fast, 1 exact routine, 2 NaN).  Tiles are 16 key rows x 8 query heads (of
// one key head), ordered key head, head chunk, row tile; each warp takes a
// contiguous range of them (consecutive tiles are consecutive 16*d bytes of
// the cache) and streams them through its own ring of asynchronous copies,
// several tiles ahead; the query fragments and multipliers stay in registers
// while the key head and chunk are the same.  NB = d / 32 blocks a key row.
template <bool S32, int NB>
__global__ void __launch_bounds__(256, 2) kv_scores_kernel(const KvK p) {
    extern __shared__ __align__(16) int hsm[];
    constexpr int kW = 2 + NB, kD = kv_ring_depth<NB>(), kPitch = 32 * NB + 32, kTile = 16 * kPitch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    uint8_t *ring = reinterpret_cast<uint8_t *>(hsm) + ((p.nh * kW * 4 + 15) & ~15) + warp * kD * kTile;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t wid = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
    const int64_t t_begin = wid * p.ntiles / nw, t_end = (wid + 1) * p.ntiles / nw;
    const bool any = t_begin < t_end;
    const int ntr = (int)p.ntr;

    // this lane's copies within a tile: chunk ci = lane + 32q is row ci / (2NB),
    // 16-byte column ci % (2NB)
    int crow[NB], csrc[NB], cdst[NB];
#pragma unroll
    for (int q = 0; q < NB; ++q) {
        const int ci = lane + 32 * q, r = ci / (2 * NB), c = ci % (2 * NB);
        crow[q] = r;
        csrc[q] = r * p.d + 16 * c;
        cdst[q] = r * kPitch + 16 * c;
    }
    // tile coordinates, advanced without division: key head, head chunk, row tile
    struct Pos { int kvh, chunk, rt; };
    auto advance = [&](Pos &x) {
        if (++x.rt == ntr) {
            x.rt = 0;
            if (++x.chunk == p.nchunk) { x.chunk = 0; ++x.kvh; }
        }
    };
    Pos cur;
    {
        const int64_t kc0 = t_begin / ntr;
        cur.rt = (int)(t_begin - kc0 * ntr);
        cur.kvh = (int)(kc0 / p.nchunk);
        cur.chunk = (int)(kc0 - (int64_t)cur.kvh * p.nchunk);
    }
    // the copies kD tiles ahead: one commit group per call, empty past the range
    Pos ip = cur;
    int64_t itile = t_begin;
    int islot = 0;
    auto issue = [&]() {
        if (itile < t_end) {
            uint8_t *dst = ring + islot * kTile;
            const int64_t left = p.L - (int64_t)ip.rt * 16;
            const int rows_left = left < 16 ? (int)left : 16;
            const int8_t *src = p.kc + ((int64_t)ip.kvh * p.lcap + (int64_t)ip.rt * 16) * p.d;
#pragma unroll
            for (int q = 0; q < NB; ++q) {
                const bool ok = crow[q] < rows_left;
                cp_async16(dst + cdst[q], ok ? src + csrc[q] : src, ok ? 16u : 0u);
            }
            advance(ip);
        }
        cp_async_commit();
        ++itile;
        islot = (islot + 1 == kD) ? 0 : islot + 1;
    };
    // the key cache depends on no earlier kernel (kv_cache_rows, which writes
    // it, lets its successor start only when it has finished): the first kD
    // tiles and key scales are requested before the wait
    if (any) {
#pragma unroll
        for (int i = 0; i < kD; ++i) issue();
    }

    // key scales of a tile's rows g and g + 8 (0 past L; never read there)
    auto ks_load = [&](const Pos &x, uint32_t &a, uint32_t &b) {
        const int64_t r = (int64_t)x.rt * 16 + g;
        const uint16_t *base = p.ks + (int64_t)x.kvh * p.lcap + r;
        a = r < p.L ? __ldg(base) : 0u;
        b = r + 8 < p.L ? __ldg(base + 8) : 0u;
    };
    uint32_t ks0 = 0, ks1 = 0;
    if (any) ks_load(cur, ks0, ks1);

    pdl_launch_dependents();
    pdl_wait();
    // per query head, the block multipliers (after the wait: the query scales
    // are the previous kernel's output)

    for (int h = threadIdx.x; h < p.nh; h += blockDim.x) {
        const uint32_t *qs = reinterpret_cast<const uint32_t *>(p.qs) + (int64_t)h * p.nbq;
        int *w = hsm + h * kW;
        if (!S32) {
            const uint32_t sw = qs[0];
            w[0] = (sw & 0xFFu) == 0u ? 2 : 0;
            w[1] = (int)(int16_t)(sw >> 16);
            for (int b = 0; b < NB; ++b) w[2 + b] = (int)(sw & 0xFFu);
        } else {
            bool zero = false;
            int lo = INT_MAX, hi = INT_MIN;
            for (int b = 0; b < p.nbq; ++b) {
                const uint32_t sw = qs[b];
                zero |= (sw & 0xFFu) == 0u;
                if (b < NB) {
                    const int e = (int)(int16_t)(sw >> 16);
                    lo = min(lo, e);
                    hi = max(hi, e);
                }
            }
            int mode = zero ? 2 : (hi - lo > 12 ? 1 : 0);
            for (int b = 0; b < NB; ++b) {
                const uint32_t sw = qs[b];
                const uint32_t M = mode == 0 ? (sw & 0xFFu) << ((int)(int16_t)(sw >> 16) - lo) : 0u;
                if (M > 0xFFFFu) mode = 1;
                w[2 + b] = (int)M;
            }
            w[0] = mode;
            w[1] = lo;
        }
    }
    __syncthreads();

    if (!any) return;  // after the barrier: every thread takes part in the table
    int held = -1;  // key head * nchunk + chunk of the fragments held
    uint2 B[NB];
    int M0[NB], M1[NB];
    int mode0 = 0, mode1 = 0, emin0 = 0, emin1 = 0, h0 = 0;
    bool hv0 = false, hv1 = false;
    float *out0 = p.out, *out1 = p.out;
    int slot = 0;
    for (int64_t tile = t_begin; tile < t_end; ++tile) {
        Pos nxt = cur;
        advance(nxt);
        uint32_t kn0 = 0, kn1 = 0;
        if (tile + 1 < t_end) ks_load(nxt, kn0, kn1);  // early: used one tile later
        const int kc_ = cur.kvh * p.nchunk + cur.chunk;
        if (kc_ != held) {
            held = kc_;
            const int jb = cur.chunk * 8 + g;
            const bool bin = jb < p.G;
            const int8_t *qb = p.qc + (int64_t)(cur.kvh * p.G + (bin ? jb : 0)) * p.dp + 8 * t;
#pragma unroll
            for (int b = 0; b < NB; ++b)
                B[b] = bin ? __ldg(reinterpret_cast<const uint2 *>(qb + 32 * b)) : make_uint2(0, 0);
            const int j0 = cur.chunk * 8 + 2 * t;
            hv0 = j0 < p.G;
            hv1 = j0 + 1 < p.G;
            h0 = cur.kvh * p.G + j0;
            const int *w0 = hsm + (hv0 ? h0 : 0) * kW, *w1 = hsm + (hv1 ? h0 + 1 : 0) * kW;
            mode0 = w0[0]; emin0 = w0[1];
            mode1 = w1[0]; emin1 = w1[1];
#pragma unroll
            for (int b = 0; b < NB; ++b) { M0[b] = w0[2 + b]; M1[b] = w1[2 + b]; }
            out0 = p.out + (int64_t)h0 * p.L;
            out1 = out0 + p.L;
        }
        cp_async_wait<kD - 1>();  // this tile's group has landed (this lane's copies)
        __syncwarp();             // ... and every lane's
        const uint8_t *sl = ring + slot * kTile;
        long long acc[4] = {0, 0, 0, 0};
        int c[4] = {0, 0, 0, 0};
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint2 a0 = *reinterpret_cast<const uint2 *>(sl + g * kPitch + 32 * b + 8 * t);
            const uint2 a1 = *reinterpret_cast<const uint2 *>(sl + (g + 8) * kPitch + 32 * b + 8 * t);
            if (S32) { c[0] = c[1] = c[2] = c[3] = 0; }
            mma_s8_16832(c, a0.x, a1.x, a0.y, a1.y, B[b].x, B[b].y);
            if (S32) {
                acc[0] += (long long)M0[b] * c[0];
                acc[1] += (long long)M1[b] * c[1];
                acc[2] += (long long)M0[b] * c[2];
                acc[3] += (long long)M1[b] * c[3];
            }
        }
        __syncwarp();  // every lane has read the slot
        issue();       // refill it kD tiles ahead
        slot = (slot + 1 == kD) ? 0 : slot + 1;
        if (!S32) {
            acc[0] = (long long)M0[0] * c[0];
            acc[1] = (long long)M1[0] * c[1];
            acc[2] = (long long)M0[0] * c[2];
            acc[3] = (long long)M1[0] * c[3];
        }
        // epilogue: (row, head) pairs (pA, h0) (pA, h0+1) (pB, h0) (pB, h0+1)
        const int64_t pA = (int64_t)cur.rt * 16 + g, pB = pA + 8;
        const bool rA = pA < p.L, rB = pB < p.L;
        int sgA, exA, sgB, exB;
        const bool okA = f16_scale(ks0, sgA, exA), okB = f16_scale(ks1, sgB, exB);
        if ((mode0 | mode1) == 0 && okA && okB) {
            if (rA) {
                if (hv0) out0[pA] = finish_score(round_fast((long long)sgA * acc[0], exA + emin0), p.scale);
                if (hv1) out1[pA] = finish_score(round_fast((long long)sgA * acc[1], exA + emin1), p.scale);
            }
            if (rB) {
                if (hv0) out0[pB] = finish_score(round_fast((long long)sgB * acc[2], exB + emin0), p.scale);
                if (hv1) out1[pB] = finish_score(round_fast((long long)sgB * acc[3], exB + emin1), p.scale);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool rowok = (i < 2) ? rA : rB;
                const bool hok = (i & 1) ? hv1 : hv0;
                if (!rowok || !hok) continue;
                const int64_t pr = (i < 2) ? pA : pB;
                const int h = h0 + (i & 1);
                const int mode = (i & 1) ? mode1 : mode0;
                const uint32_t ksb = (i < 2) ? ks0 : ks1;
                float v;
                if (mode == 2) {
                    v = __uint_as_float(kEngineNaN);
                } else if (mode == 1) {
                    v = kv_score_exact(p.qc + (int64_t)h * p.dp, p.qs + (int64_t)h * p.nbq, p.nbq, S32 ? 32 : p.d,
                                       p.d, p.kc + ((int64_t)cur.kvh * p.lcap + pr) * p.d, ksb);
                } else {
                    const bool ok = (i < 2) ? okA : okB;
                    v = ok ? round_fast((long long)((i < 2) ? sgA : sgB) * acc[i],
                                        ((i < 2) ? exA : exB) + ((i & 1) ? emin1 : emin0))
                           : __uint_as_float(kEngineNaN);
                }
                ((i & 1) ? out1 : out0)[pr] = finish_score(v, p.scale);
            }
        }
        cur = nxt;
        ks0 = kn0;
        ks1 = kn1;
    }
    cp_async_wait<0>();  // no copy outlives the warp
}

// Any d (% 16 == 0, <= 1024): one thread per score through the exact routine.
__global__ void __launch_bounds__(256) kv_scores_plain_kernel(const KvK p, int blk) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t n = (int64_t)p.nh * p.L;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int h = (int)(i / p.L);
        const int64_t pr = i - (int64_t)h * p.L;
        const int64_t krow = (int64_t)(h / p.G) * p.lcap + pr;
        const float v = kv_score_exact(p.qc + (int64_t)h * p.dp, p.qs + (int64_t)h * p.nbq, p.nbq, blk, p.d,
                                       p.kc + krow * p.d, __ldg(p.ks + krow));
        p.out[i] = finish_score(v, p.scale);
    }
}

// ------------------------------------------------------------------ launchers

int launch_kv_cache_rows(const float *x, int64_t n, int d, int8_t *codes, uint16_t *scales, cudaStream_t stream) {
    const unsigned grid = (unsigned)((n + 7) / 8);
    return launch_pdl(kv_cache_rows_kernel, dim3(grid), dim3(256), 0, stream, x, n, d, codes, scales);
}

int launch_kv_quantize_heads(int scaling, const float *q, int nh, int d, int8_t *codes, qb_scale *scales,
                             cudaStream_t stream) {
    if (scaling == 1) {
        const int dp = (d + 255) / 256 * 256;
        const int64_t n8 = (int64_t)nh * dp / 8;
        return launch_pdl(kv_heads_sub32_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0, stream, q, nh, d,
                          dp, codes, scales);
    }
    return launch_pdl(kv_heads_perblock_kernel, dim3((unsigned)nh), dim3(256), 0, stream, q, d, codes, scales);
}

template <bool S32, int NB>
static int launch_scores_nb(const KvK &k, cudaStream_t stream) {
    const int smem = kv_smem_bytes<NB>(k.nh);
    if (smem > 113 * 1024) return QB_E_ARG;
    if (ensure_smem_limit(reinterpret_cast<const void *>(kv_scores_kernel<S32, NB>), 113 * 1024) != QB_OK)
        return QB_E_CUDA;
    // persistent: two CTAs of 8 warps a SM, each warp a contiguous range of tiles
    const int64_t blocks = (k.ntiles + 7) / 8;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)num_sms() * 2));
    return launch_pdl(kv_scores_kernel<S32, NB>, dim3(grid), dim3(256), (size_t)smem, stream, k);
}

int launch_kv_scores(int scaling, const int8_t *qc, const qb_scale *qs, int nh, int d, const int8_t *kc,
                     const uint16_t *ks, int64_t L, int64_t lcap, int nkv, float scale, float *out,
                     cudaStream_t stream) {
    KvK k = {};
    k.qc = qc;
    k.qs = qs;
    k.nh = nh;
    k.d = d;
    k.dp = scaling == 1 ? (d + 255) / 256 * 256 : d;
    k.nbq = scaling == 1 ? k.dp / 32 : 1;
    k.G = nh / nkv;
    k.nchunk = (k.G + 7) / 8;
    k.kc = kc;
    k.ks = ks;
    k.L = L;
    k.lcap = lcap;
    k.ntr = (L + 15) / 16;
    k.nkv = nkv;
    k.ntiles = (int64_t)nkv * k.ntr * k.nchunk;
    k.scale = scale;
    k.out = out;
    if (d % 32 == 0) {
        int rc = QB_E_ARG;
        const bool s = scaling == 1;
        switch (d / 32) {
        case 2: rc = s ? launch_scores_nb<true, 2>(k, stream) : launch_scores_nb<false, 2>(k, stream); break;
        case 4: rc = s ? launch_scores_nb<true, 4>(k, stream) : launch_scores_nb<false, 4>(k, stream); break;
        case 8: rc = s ? launch_scores_nb<true, 8>(k, stream) : launch_scores_nb<false, 8>(k, stream); break;
        default: break;
        }
        if (rc != QB_E_ARG) return rc;
    }
    const int64_t n = (int64_t)nh * L;
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 8));
    return launch_pdl(kv_scores_plain_kernel, dim3(grid), dim3(256), 0, stream, k, scaling == 1 ? 32 : d);
}

}  // namespace qb
