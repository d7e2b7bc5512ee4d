// qb_gemv3.cuh -- the streaming product kernel for 2..16 activation columns.
//
// The organisation of the one-column streaming kernel (qb_gemv2.cuh:
// persistent CTAs over contiguous row ranges, teams of K/128 threads owning
// 128-element half-slices of K, weights through a ring of bulk-copy slots,
// two rows per team per iteration, in-order fold from shared memory), with the
// columns split into groups of CG: a team is NCG groups of K/128 threads, and
// thread (g, j) keeps the activation codes of columns CG*g .. CG*g+CG-1 over
// half-slice j in registers (staged once per CTA through shared memory) and
// reads each weight once for its CG columns.  Columns past the launch's count
// (padding of the last group) run on zeros and are never written.  Per column
// every block value and every row are the bits the one-column product gives:
// the same integer sums, the same exact combine, the same fold order.
//
// A launch covers as many column groups as fit in one CTA; more columns take
// further launches over the same weights (the weights then stream again; at
// these column counts the integer work, not the weight stream, bounds the
// product).
#pragma once

#include <algorithm>
#include <type_traits>

#include "qb_common.cuh"
#include "qb_gemv2.cuh"
#include "qb_launch.h"
#include "qb_mats.cuh"

namespace qb {

struct Gemv3K {
    const uint8_t *W;  // the matrix (one-matrix launches)
    float *out;        // its output at this launch's first column (one-matrix launches)
    int64_t rows;      // rows of the whole range
    int K;
    int rec;
    int nt;     // teams per CTA
    int ts;     // threads per group = K / 128 (one half-slice each)
    int ncg;    // column groups per team
    int ncols;  // real columns of this launch
    int D;      // ring slots
    int H;      // iterations of block values held before a fold
    int nb;     // blocks per row
    int vstride;
    int n_iter;
    int64_t base;
    int64_t rem;
    const int8_t *codes;  // column 0 of this launch
    const qb_scale *scales;
    const int16_t *sums16;
    const float *x;  // one-column single-launch form: the f32 activation, quantized in the kernel
    int *fault;
};
// A launch over several matrices sharing the activation: the table, outputs
// at this launch's first column (W and out unused).
struct Gemv3KM : Gemv3K {
    MatTable mt;
};

struct Gemv3Smem {
    int bars, act, sums, scl, val, ring, total;
};

// act: the launch's activation codes (ncols * K bytes); sums, scl: the unit
// sums and scales the single-launch form quantizes into (fused only); val:
// the block values of H iterations; ring: D slots of 2*nt weight rows.
__host__ __device__ inline Gemv3Smem gemv3_smem(int K, int ncols, int rec, int nt, int ncp, int D, int H,
                                                int vstride, bool fused = false) {
    Gemv3Smem s;
    s.bars = 0;
    s.act = 128;
    s.sums = s.act + ((ncols * K + 127) & ~127);
    s.scl = s.sums + (fused ? ((K / 16 * 2 + 127) & ~127) : 0);
    s.val = s.scl + (fused ? ((K / 32 * 4 + 127) & ~127) : 0);
    s.ring = s.val + ((H * nt * 2 * ncp * vstride * 4 + 127) & ~127);
    s.total = s.ring + D * nt * 2 * rec;
    return s;
}

// Q4_K-like half block h for CG columns: 16*C[c] and O[c] over sub-blocks
// 4h..4h+3.  a[c][k] holds unit 8j+k of column c; S[c][0] the unit-pair sums
// of sub-blocks 4h, 4h+1 as 16-bit halves, S[c][1] those of 4h+2, 4h+3.
template <int CG>
__device__ __forceinline__ void half_q4k_cg(const uint8_t *blk, int h, const uint4 (&a)[CG][8],
                                            const uint32_t (&S)[CG][4], int (&C)[CG], int (&O)[CG], uint32_t &dd) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    dd = meta.x;
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
    const uint32_t scm = (uint32_t)(sc48 >> (24 * h)), mnm = (uint32_t)(mn48 >> (24 * h));
    const uint8_t *qs = blk + 16 + 64 * h;
#pragma unroll
    for (int c = 0; c < CG; ++c) C[c] = 0;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint4 w = *reinterpret_cast<const uint4 *>(qs + 16 * s);
        // the low nibbles as q, the high ones as 16*q (masked in place): two
        // chains of four dp4a, 16 * (the sub-block's sum) = 16 * pl + ph, so
        // C is returned as 16*C (|16*C| <= 16 * 63 * 15 * 127 * 256 < 2^31)
        const uint32_t l0 = w.x & 0x0F0F0F0Fu, l1 = w.y & 0x0F0F0F0Fu, l2 = w.z & 0x0F0F0F0Fu, l3 = w.w & 0x0F0F0F0Fu;
        const uint32_t g0 = w.x & 0xF0F0F0F0u, g1 = w.y & 0xF0F0F0F0u, g2 = w.z & 0xF0F0F0F0u, g3 = w.w & 0xF0F0F0F0u;
        const int sc = (int)((scm >> (6 * s)) & 63u);
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            int pl = dp4a_ss(l0, a[c][2 * s].x, 0);
            pl = dp4a_ss(l1, a[c][2 * s].y, pl);
            pl = dp4a_ss(l2, a[c][2 * s].z, pl);
            pl = dp4a_ss(l3, a[c][2 * s].w, pl);
            int ph = dp4a_us(g0, a[c][2 * s + 1].x, 0);
            ph = dp4a_us(g1, a[c][2 * s + 1].y, ph);
            ph = dp4a_us(g2, a[c][2 * s + 1].z, ph);
            ph = dp4a_us(g3, a[c][2 * s + 1].w, ph);
            C[c] += sc * (16 * pl + ph);
        }
    }
    // O = sum over the four sub-blocks of mn * (the sub-block's activation sum)
    const uint32_t mnb = spread6(mnm);
#pragma unroll
    for (int c = 0; c < CG; ++c) O[c] = dp2a_hi_su(S[c][1], mnb, dp2a_lo_su(S[c][0], mnb, 0));
}

// Q6_K-like half block h (32-element chunks 4h..4h+3) for CG columns.
template <int CG>
__device__ __forceinline__ void half_q6k_cg(const uint8_t *blk, int h, const uint4 (&a)[CG][8],
                                            const uint32_t (&S)[CG][4], int (&C)[CG]) {
    const uint2 scw = *reinterpret_cast<const uint2 *>(blk + 192 + 8 * h);
#pragma unroll
    for (int c = 0; c < CG; ++c) C[c] = 0;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 64 * h + 16 * ch);
        const uint2 hb = *reinterpret_cast<const uint2 *>(blk + 128 + 32 * h + 8 * ch);
        const uint32_t wl[4] = {w.x, w.y, w.z, w.w};
        uint32_t ql[4], qh[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t hl = (k < 3) ? (hb.x << (4 - 2 * k)) : (hb.x >> 2);
            const uint32_t hh = (k < 3) ? (hb.y << (4 - 2 * k)) : (hb.y >> 2);
            ql[k] = (wl[k] & 0x0F0F0F0Fu) | (hl & 0x30303030u);
            qh[k] = ((wl[k] >> 4) & 0x0F0F0F0Fu) | (hh & 0x30303030u);
        }
        const uint32_t sw = (ch < 2) ? scw.x : scw.y;
        const int sc_lo = (int)(int8_t)((sw >> (16 * (ch & 1))) & 0xFFu);
        const int sc_hi = (int)(int8_t)((sw >> (16 * (ch & 1) + 8)) & 0xFFu);
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            int pl = dp4a_ss(ql[0], a[c][2 * ch].x, 0);
            pl = dp4a_ss(ql[1], a[c][2 * ch].y, pl);
            pl = dp4a_ss(ql[2], a[c][2 * ch].z, pl);
            pl = dp4a_ss(ql[3], a[c][2 * ch].w, pl);
            int ph = dp4a_ss(qh[0], a[c][2 * ch + 1].x, 0);
            ph = dp4a_ss(qh[1], a[c][2 * ch + 1].y, ph);
            ph = dp4a_ss(qh[2], a[c][2 * ch + 1].z, ph);
            ph = dp4a_ss(qh[3], a[c][2 * ch + 1].w, ph);
            // sum over a unit of (q - 32) * a = sum q*a - 32 * S_u
            C[c] += sc_lo * (pl - 32 * (int)(int16_t)(S[c][ch] & 0xFFFFu)) +
                    sc_hi * (ph - 32 * (int)(int16_t)(S[c][ch] >> 16));
        }
    }
}

// Q8_0 half-slice (blocks 4j..4j+3) for CG columns.  The thread visits its
// eight 16-B weight units in the order k ^ jj, so the eight lanes of a
// shared-memory phase hit eight banks; a[c][k] holds unit 8j + (k ^ jj) of
// column c to match.  Block i's value for column c goes to vl[c*vcol + i].
template <int CG>
__device__ __forceinline__ void half_q8_0_cg(const uint8_t *q, const uint8_t *dptr, const uint4 (&scl)[CG],
                                             const uint4 (&a)[CG][8], int jj, float *vl, int vcol) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const int u0 = (2 * kk) ^ jj, u1 = u0 ^ 1;
        const int i = u0 >> 1;
        const uint4 w0 = *reinterpret_cast<const uint4 *>(q + 16 * u0);
        const uint4 w1 = *reinterpret_cast<const uint4 *>(q + 16 * u1);
        const uint32_t d = *reinterpret_cast<const uint16_t *>(dptr + 2 * i);
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            int p = dp4a_ss(w0.x, a[c][2 * kk].x, 0);
            p = dp4a_ss(w0.y, a[c][2 * kk].y, p);
            p = dp4a_ss(w0.z, a[c][2 * kk].z, p);
            p = dp4a_ss(w0.w, a[c][2 * kk].w, p);
            p = dp4a_ss(w1.x, a[c][2 * kk + 1].x, p);
            p = dp4a_ss(w1.y, a[c][2 * kk + 1].y, p);
            p = dp4a_ss(w1.z, a[c][2 * kk + 1].z, p);
            p = dp4a_ss(w1.w, a[c][2 * kk + 1].w, p);
            const uint32_t sw = i == 0 ? scl[c].x : i == 1 ? scl[c].y : i == 2 ? scl[c].z : scl[c].w;
            vl[c * vcol + i] = lane_value_fast<0>(p, 0, d, 0, (int)(sw & 0xFFu), (int)(int16_t)(sw >> 16));
        }
    }
}

// Threads a CTA: two columns of codes (64 registers) fit 512 threads at the
// 128-register bound; four would need 256 threads.
template <int CG>
constexpr int gemv3_threads() { return CG >= 4 ? 256 : 512; }

// FUSED (one column, CG = 1): the f32 activation p.x is quantized in the
// prologue (quantize_blocks, as the one-column kernel's single-launch form
// does) while the first weight fills are in flight.
template <int F, int CG, bool MULTI, bool FUSED = false>
__global__ void __launch_bounds__(gemv3_threads<CG>(), 1)
    gemv3_kernel(const typename std::conditional<MULTI, Gemv3KM, Gemv3K>::type p) {
    static_assert(!FUSED || CG == 1, "the single-launch form takes one column");
    extern __shared__ __align__(128) uint8_t smem[];
    const int ncp = p.ncg * CG;  // padded columns
    const Gemv3Smem L = gemv3_smem(p.K, p.ncols, p.rec, p.nt, ncp, p.D, p.H, p.vstride, FUSED);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint8_t *act = smem + L.act;
    int16_t *asum = reinterpret_cast<int16_t *>(smem + L.sums);
    uint32_t *ascl = reinterpret_cast<uint32_t *>(smem + L.scl);
    float *val = reinterpret_cast<float *>(smem + L.val);
    uint8_t *ring = smem + L.ring;

    const int tid = threadIdx.x;
    const int tpt = p.ncg * p.ts;  // threads per team
    const int team = tid / tpt, tr = tid - team * tpt;
    const int g = tr / p.ts, j = tr - g * p.ts;
    const bool live = team < p.nt;
    const int sb = j >> 1, h = j & 1, jj = j & 7;

    const int64_t cta = blockIdx.x;
    const int64_t row0 = cta * p.base + (cta < p.rem ? cta : p.rem);
    const int64_t count = p.base + (cta < p.rem ? 1 : 0);
    const int64_t per_it = 2LL * p.nt;
    if (tid == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // the fill of iteration `it`: its rows are contiguous, one bulk copy into slot it % D
    auto fill = [&](int it) {
        const int slot = it % p.D;
        const int64_t first = (int64_t)it * per_it;
        const int64_t n = (count - first < per_it) ? count - first : per_it;
        const uint32_t bytes = n > 0 ? (uint32_t)(n * p.rec) : 0u;
        mbar_arrive_expect_tx(bars + slot, bytes);
        if (!bytes) return;
        uint8_t *dst = ring + (int64_t)slot * per_it * p.rec;
        if constexpr (MULTI) fill_rows(p.mt, dst, row0 + first, n, p.rec, bars + slot);
        else bulk_g2s(dst, p.W + (row0 + first) * p.rec, bytes, bars + slot);
    };
    // weights depend on no earlier kernel.  One column: only the first slot
    // ahead of the activation, whose loads would otherwise queue behind the
    // whole ring's fills; the rest once it is staged
    const int pre = CG == 1 ? 1 : p.D;
    if (tid == 0)
        for (int it = 0; it < pre && it < p.n_iter; ++it) fill(it);
    // the next launch may be scheduled now: it reads nothing this one writes
    // before its own pdl_wait, which returns once this grid has finished
    pdl_launch_dependents();
    pdl_wait();

    // ---- the activation codes of every column, once per CTA: coalesced
    // loads, stored in shared memory with 16-B unit u of the launch's codes at
    // (u & ~7) | ((u & 7) ^ ((u >> 3) & 7)) (Q8_0: at u), so that the register
    // loads below hit eight banks per phase.  The single-launch form quantizes
    // x here instead: a thread takes 8 consecutive elements, a block of B
    // elements is B/8 consecutive lanes; all loads first, then the quantizer.
    if constexpr (FUSED) {
        constexpr int kB = fmt_block(F), kL = kB / 8, kMaxG = 4;  // groups per thread: K/8 <= 4 * blockDim
        const int G = p.K / 8;
        float4 xv[2 * kMaxG];
#pragma unroll
        for (int r = 0; r < kMaxG; ++r) {
            const int g8 = tid + r * (int)blockDim.x;
            const bool in = g8 < G;
            xv[2 * r] = in ? ldg_f4_ordered(reinterpret_cast<const float4 *>(p.x) + 2 * g8) : make_float4(0, 0, 0, 0);
            xv[2 * r + 1] = in ? ldg_f4_ordered(reinterpret_cast<const float4 *>(p.x) + 2 * g8 + 1)
                               : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int r = 0; r < kMaxG; ++r) {
            if (r * (int)blockDim.x >= G) break;  // uniform: whole warps are in or out (G % 32 == 0)
            const int g8 = tid + r * (int)blockDim.x;
            const uint32_t xb[8] = {__float_as_uint(xv[2 * r].x), __float_as_uint(xv[2 * r].y),
                                    __float_as_uint(xv[2 * r].z), __float_as_uint(xv[2 * r].w),
                                    __float_as_uint(xv[2 * r + 1].x), __float_as_uint(xv[2 * r + 1].y),
                                    __float_as_uint(xv[2 * r + 1].z), __float_as_uint(xv[2 * r + 1].w)};
            uint2 c;
            int usum;
            uint32_t scale;
            quantize8<kL>(xb, c, usum, scale);
            if (g8 < G) {
                const int u = g8 >> 1;
                const int pos = (F == kQ8_0) ? u : ((u & ~7) | ((u & 7) ^ ((u >> 3) & 7)));
                *reinterpret_cast<uint2 *>(act + 16 * pos + 8 * (g8 & 1)) = c;
                if ((g8 & 1) == 0) asum[u] = (int16_t)usum;
                if ((g8 & (kL - 1)) == 0) ascl[g8 / kL] = scale;
            }
        }
        __syncthreads();
    } else {
        const int nu = p.ncols * (p.K / 16);
        const uint4 *src = reinterpret_cast<const uint4 *>(p.codes);
        constexpr int kU = 4;
        for (int u0 = tid; u0 < nu; u0 += kU * (int)blockDim.x) {
            uint4 v[kU];
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int u = u0 + q * (int)blockDim.x;
                v[q] = u < nu ? ldg_v4_ordered(src + u) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int u = u0 + q * (int)blockDim.x;
                const int pos = (F == kQ8_0) ? u : ((u & ~7) | ((u & 7) ^ ((u >> 3) & 7)));
                if (u < nu) *reinterpret_cast<uint4 *>(act + 16 * pos) = v[q];
            }
        }
    }
    // my columns' unit sums and scales (global memory, small; the single-launch
    // form's own, in shared memory)
    uint4 a[CG][8];
    uint32_t S[CG][4];
    uint4 scl[CG];  // Q8_0: the scales of blocks 4j..4j+3
    int m0[CG], e0[CG];
#pragma unroll
    for (int c = 0; c < CG; ++c) {
        const int col = g * CG + c;
        const bool in = live && col < p.ncols;
        S[c][0] = S[c][1] = S[c][2] = S[c][3] = 0;
        scl[c] = make_uint4(128, 128, 128, 128);
        m0[c] = 128;
        e0[c] = 0;
        if (in && F == kQ8_0) {
            scl[c] = FUSED ? *reinterpret_cast<const uint4 *>(ascl + 4 * j)
                           : __ldg(reinterpret_cast<const uint4 *>(p.scales + (int64_t)col * (p.K / 32)) + j);
        } else if (in) {
            const uint4 sw = FUSED ? *reinterpret_cast<const uint4 *>(asum + 8 * j)
                                   : __ldg(reinterpret_cast<const uint4 *>(p.sums16 + (int64_t)col * (p.K / 16)) + j);
            const uint32_t pw[4] = {sw.x, sw.y, sw.z, sw.w};
            if (F == kQ4K) {  // per-32 sums of my four sub-blocks from the per-16 ones
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2) {
                    const int Sv = (int)(int16_t)(pw[s2] & 0xFFFFu) + (int)(int16_t)(pw[s2] >> 16);
                    S[c][s2 >> 1] |= ((uint32_t)Sv & 0xFFFFu) << (16 * (s2 & 1));
                }
            } else {
                S[c][0] = pw[0]; S[c][1] = pw[1]; S[c][2] = pw[2]; S[c][3] = pw[3];
            }
            const uint32_t sv = FUSED ? ascl[sb]
                                      : __ldg(reinterpret_cast<const uint32_t *>(p.scales) + (int64_t)col * (p.K / 256) + sb);
            m0[c] = (int)(sv & 0xFFu);
            e0[c] = (int)(int16_t)(sv >> 16);
        }
    }
    __syncthreads();
    if (tid == 0)
        for (int it = pre; it < p.D && it < p.n_iter; ++it) fill(it);
    // codes of half-slice j (Q4_K/Q6_K: a[c][k] = unit 8j+k; Q8_0: unit 8j + (k ^ jj))
#pragma unroll
    for (int c = 0; c < CG; ++c) {
        const int col = g * CG + c;
        const bool in = live && col < p.ncols;
        const uint8_t *base = act + (int64_t)col * p.K + 128 * j;
        const int key = (F == kQ8_0) ? jj : ((col * p.ts + j) & 7);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            a[c][k] = in ? *reinterpret_cast<const uint4 *>(base + 16 * (k ^ key)) : make_uint4(0, 0, 0, 0);
    }

    // value lines: [history][team][row A/B][padded column][vstride]
    const int vcol = p.vstride;
    int hpos = 0;
    for (int it = 0; it < p.n_iter; ++it) {
        const int slot = it % p.D;
        const int64_t lA = (int64_t)it * per_it + 2 * team;  // row index within the CTA's range
        const bool haveA = live && lA < count, hasB = live && lA + 1 < count;
        const uint8_t *rA = ring + ((int64_t)(slot * p.nt + team) * 2) * p.rec;
        const uint8_t *rB = rA + p.rec;
        float *vA = val + (((hpos * p.nt + team) * 2) * ncp + g * CG) * p.vstride;
        float *vB = vA + ncp * p.vstride;
        bool ok = true;
        if (haveA) ok = mbar_wait_bounded(bars + slot, (uint32_t)((it / p.D) & 1), p.fault);
        const bool go = haveA && ok;
        if (F == kQ8_0) {
            if (go) {
                half_q8_0_cg<CG>(rA + 128 * j, rA + p.K + 8 * j, scl, a, jj, vA + 4 * j, vcol);
                if (hasB) half_q8_0_cg<CG>(rB + 128 * j, rB + p.K + 8 * j, scl, a, jj, vB + 4 * j, vcol);
            }
        } else {
            // partial sums of my half for both rows; each lane then swaps one
            // pair per column with its partner (lane ^ 1, the block's other half)
            int CA[CG], CB[CG], OA[CG], OB[CG];
            uint32_t dA = 0, dB = 0;
#pragma unroll
            for (int c = 0; c < CG; ++c) { CA[c] = 0; CB[c] = 0; OA[c] = 0; OB[c] = 0; }
            if (go) {
                if (F == kQ4K) {
                    half_q4k_cg<CG>(rA + 144 * sb, h, a, S, CA, OA, dA);
                    if (hasB) half_q4k_cg<CG>(rB + 144 * sb, h, a, S, CB, OB, dB);
                } else {
                    half_q6k_cg<CG>(rA + 208 * sb, h, a, S, CA);
                    dA = *reinterpret_cast<const uint16_t *>(rA + 208 * p.nb + 2 * sb);
                    if (hasB) {
                        half_q6k_cg<CG>(rB + 208 * sb, h, a, S, CB);
                        dB = *reinterpret_cast<const uint16_t *>(rB + 208 * p.nb + 2 * sb);
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < CG; ++c) {
                const int rC = __shfl_xor_sync(0xFFFFFFFFu, h ? CA[c] : CB[c], 1);
                const int rO = (F == kQ4K) ? __shfl_xor_sync(0xFFFFFFFFu, h ? OA[c] : OB[c], 1) : 0;
                if (go && (!h || hasB)) {
                    const int Cs = (h ? CB[c] : CA[c]) + rC, O = (h ? OB[c] : OA[c]) + rO;
                    const int C = (F == kQ4K) ? (Cs >> 4) : Cs;  // Q4_K: the halves hold 16*C (exact shift)
                    const uint32_t dd = h ? dB : dA;
                    float v;
                    if (F == kQ4K) v = lane_value_fast<1>(C, O, dd & 0xFFFFu, dd >> 16, m0[c], e0[c]);
                    else v = lane_value_fast<0>(C, 0, dd, 0, m0[c], e0[c]);
                    (h ? vB : vA)[c * vcol + sb] = v;
                }
            }
        }
        if (!__syncthreads_and(ok)) return;  // a fill never completed: fault word raised
        if (tid == 0 && it + p.D < p.n_iter) {
            fence_proxy_async_smem();
            fill(it + p.D);
        }
        // ---- fold: one thread per (row, column) line, blocks in order
        if (++hpos == p.H || it == p.n_iter - 1) {
            const int nline = hpos * p.nt * 2 * ncp;
            for (int f = tid; f < nline; f += blockDim.x) {
                const int c = f % ncp;
                const int64_t l = (int64_t)(it + 1 - hpos) * per_it + f / ncp;  // row of the CTA's range
                if (c < p.ncols && l < count) {
                    const float *vt = val + (int64_t)f * p.vstride;
                    float acc = 0.0f;
                    for (int b = 0; b < p.nb; ++b) acc = fadd_ftz(acc, vt[b]);
                    if (acc != acc) acc = __uint_as_float(kEngineNaN);
                    if constexpr (MULTI) *out_ptr(p.mt, c, row0 + l) = acc;
                    else p.out[(int64_t)c * p.rows + row0 + l] = acc;
                }
            }
            hpos = 0;
            if (it != p.n_iter - 1) __syncthreads();  // before the history is overwritten
        }
    }
}

// The shape of one launch over `ncols` columns; false when it does not fit.
// fused: the one-column single-launch form (its quantizer holds at most four
// 8-element groups a thread, so at least K/32 threads).
template <int F, int CG>
bool gemv3_shape(int64_t rows, int64_t K, int ncols, Gemv3K &k, int &grid, int &threads, int &smem,
                 bool fused = false) {
    constexpr int kThreads = gemv3_threads<CG>();
    const int ts = (int)(K / 128);
    const int ncg = (ncols + CG - 1) / CG, ncp = ncg * CG;
    const int tpt = ncg * ts;
    if (tpt > kThreads) return false;
    k.rows = rows;
    k.K = (int)K;
    k.rec = (int)record_bytes(F, K);
    k.ts = ts;
    k.ncg = ncg;
    k.ncols = ncols;
    k.nb = (int)(K / fmt_block(F));
    k.vstride = (k.nb & 1) ? k.nb : k.nb + 1;  // odd: the fold's lines fall in distinct banks
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), rows));
    const int64_t rpc = (rows + grid - 1) / grid;  // most rows any CTA owns
    const int budget = 225 * 1024;
    k.nt = (int)std::min<int64_t>(kThreads / tpt, std::max<int64_t>(1, (rpc + 1) / 2));
    if (fused) k.nt = std::max(k.nt, std::min(4, kThreads / tpt));
    auto L = [&](int D, int H) { return gemv3_smem(k.K, ncols, k.rec, k.nt, ncp, D, H, k.vstride, fused).total; };
    // room for two ring slots and one history step
    while (k.nt > 1 && L(2, 1) > budget) --k.nt;
    if (L(1, 1) > budget) return false;
    k.n_iter = (int)((rpc + 2LL * k.nt - 1) / (2LL * k.nt));
    k.base = rows / grid;
    k.rem = rows % grid;
    threads = (k.nt * tpt + 31) / 32 * 32;
    if (fused && K / 8 > 4 * threads) return false;
    k.H = std::max(1, std::min({k.n_iter, 8, threads / (k.nt * 2 * ncp)}));  // about one fold line a thread
    const int hist = L(0, k.H);
    // one column: two slots in flight.  With more, every slot of every CTA is
    // requested at once and they land together near the end of the stream,
    // leaving all the arithmetic for after it (Q4_K-like 4096 x 14336: 8.43 ->
    // 7.83 us with two)
    k.D = std::max(1, std::min({k.n_iter, CG == 1 ? 2 : 4, (budget - hist) / (2 * k.nt * k.rec)}));
    while (L(k.D, k.H) > budget && k.H > 1) --k.H;
    smem = L(k.D, k.H);
    return smem <= 227 * 1024;
}

// One column in groups of one (CG = 1), the activation quantized beforehand
// or, with x, in the prologue (one launch).  Taken for the 256-element
// formats where the one-column kernel (qb_gemv2.cuh) would need more than one
// ring iteration per CTA -- there this organisation measured faster (Q6_K-like
// 14336x4096: 9.46 against 11.5 us; Q4_K-like 14336x4096: 8.0 against 8.3);
// QB_E_ARG otherwise, or when the shape does not fit.
template <int F>
int launch_gemv3_one(const GemvArgs &a, cudaStream_t stream, const float *x) {
    if (F == kQ8_0 || a.ncols != 1 || a.mode != 0 || a.K % 256 != 0) return QB_E_ARG;
    const MatTable mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    const int64_t rows = mt.start[mt.n];
    const int ts = (int)(a.K / 128);
    if (rows < 1 || ts > 512) return QB_E_ARG;
    const int64_t g1 = std::max<int64_t>(1, std::min<int64_t>(num_sms(), rows));
    if (((rows + g1 - 1) / g1 + 1) / 2 <= 512 / ts) return QB_E_ARG;  // one iteration: the one-column kernel
    Gemv3KM k;
    int grid, threads, smem;
    const bool fused = x != nullptr;
    if (!gemv3_shape<F, 1>(rows, a.K, 1, k, grid, threads, smem, fused)) return QB_E_ARG;
    int *fault = fault_word();
    if (!fault) return QB_E_CUDA;
    k.mt = mt;
    k.W = mt.W[0];
    k.out = mt.out[0];
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.x = x;
    k.fault = fault;
    const bool multi = mt.n > 1;
    const void *f = multi ? (fused ? reinterpret_cast<const void *>(gemv3_kernel<F, 1, true, true>)
                                   : reinterpret_cast<const void *>(gemv3_kernel<F, 1, true, false>))
                          : (fused ? reinterpret_cast<const void *>(gemv3_kernel<F, 1, false, true>)
                                   : reinterpret_cast<const void *>(gemv3_kernel<F, 1, false, false>));
    if (ensure_smem_limit(f, 227 * 1024) != QB_OK) return QB_E_CUDA;
    const Gemv3K &k1 = k;
    if (multi)
        return fused ? launch_pdl(gemv3_kernel<F, 1, true, true>, dim3(grid), dim3(threads), (size_t)smem, stream, k)
                     : launch_pdl(gemv3_kernel<F, 1, true, false>, dim3(grid), dim3(threads), (size_t)smem, stream, k);
    return fused ? launch_pdl(gemv3_kernel<F, 1, false, true>, dim3(grid), dim3(threads), (size_t)smem, stream, k1)
                 : launch_pdl(gemv3_kernel<F, 1, false, false>, dim3(grid), dim3(threads), (size_t)smem, stream, k1);
}

// The product for 2..16 columns: as many columns a launch as one CTA holds,
// launches in column order.  QB_E_ARG (nothing launched) when the kernel does
// not apply to the shape.
template <int F, int CG>
int launch_gemv3_cg(const GemvArgs &a, cudaStream_t stream) {
    constexpr int blk = fmt_block(F);
    const int ts = (int)(a.K / 128);
    const int per = (gemv3_threads<CG>() / ts) / CG * CG;  // columns one launch holds
    if (per < 1) return QB_E_ARG;
    int *fault = fault_word();
    if (!fault) return QB_E_CUDA;
    const MatTable mt = a.mats ? *a.mats : single_table(a.W, a.rows, a.out);
    const int64_t rows = mt.start[mt.n];
    for (int c0 = 0; c0 < a.ncols; c0 += per) {  // every launch's shape fits before the first is issued
        Gemv3K k;
        int grid, threads, smem;
        if (!gemv3_shape<F, CG>(rows, a.K, std::min(per, a.ncols - c0), k, grid, threads, smem)) return QB_E_ARG;
    }
    const bool multi = mt.n > 1;
    {
        const void *f = multi ? reinterpret_cast<const void *>(gemv3_kernel<F, CG, true>)
                              : reinterpret_cast<const void *>(gemv3_kernel<F, CG, false>);
        if (ensure_smem_limit(f, 227 * 1024) != QB_OK) return QB_E_CUDA;
    }
    for (int c0 = 0; c0 < a.ncols; c0 += per) {
        Gemv3KM k;
        int grid, threads, smem;
        gemv3_shape<F, CG>(rows, a.K, std::min(per, a.ncols - c0), k, grid, threads, smem);
        k.mt = mt;  // outputs from column c0: each matrix's own column stride is its row count
        for (int i = 0; i < mt.n; ++i) k.mt.out[i] = mt.out[i] + (int64_t)c0 * (mt.start[i + 1] - mt.start[i]);
        k.W = k.mt.W[0];
        k.out = k.mt.out[0];
        k.codes = a.codes + (int64_t)c0 * a.K;
        k.scales = a.scales + (int64_t)c0 * (a.K / blk);
        k.sums16 = a.sums16 ? a.sums16 + (int64_t)c0 * (a.K / 16) : nullptr;
        k.x = nullptr;
        k.fault = fault;
        const Gemv3K &k1 = k;
        const int rc = multi ? launch_pdl(gemv3_kernel<F, CG, true>, dim3(grid), dim3(threads), (size_t)smem, stream, k)
                             : launch_pdl(gemv3_kernel<F, CG, false>, dim3(grid), dim3(threads), (size_t)smem, stream,
                                          k1);
        if (rc) return rc;
    }
    return QB_OK;
}

template <int F>
int launch_gemv3(const GemvArgs &a, cudaStream_t stream) {
    if (a.ncols < 2 || a.ncols > 16 || a.mode != 0 || a.K % 256 != 0 || (!a.mats && a.rows < 1)) return QB_E_ARG;
    // two-column groups at 512 threads measure faster than four-column groups
    // at 256 (more warps to hide the integer pipeline's latency) at 2..16 columns
    return launch_gemv3_cg<F, 2>(a, stream);
}

}  // namespace qb
