// qb_gemv2.cuh -- the streaming product kernel (one activation column).
//
// Same arithmetic as qb_gemv.cuh (the decode engine's dot under PerBlock:
// exact block sums, exact two-term combine, one rounding per block, in-order
// row fold), organised for throughput:
//   * persistent CTAs, one "team" of K/256 threads per row in flight: thread j
//     of a team owns the 256-element slice j of K for every row the team
//     visits, and holds that slice's activation codes, unit sums and scale in
//     registers, loaded once per kernel;
//   * rows reach shared memory through a ring of D slots; every slot holds one
//     row record per team and is filled by bulk asynchronous copies (the TMA
//     engine) completing on the slot's mbarrier.  The first D fills are issued
//     before the programmatic-dependent-launch wait, so a launch streams its
//     weights while the previous kernel finishes;
//   * rows are dealt to teams round-robin across all CTAs (team t of CTA c has
//     global index t*gridDim.x + c), which balances rows per SM to within one;
//   * the rounded block values of H iterations are kept in shared memory and
//     folded (block order, from +0, f32 round-to-nearest-even with ftz) by one
//     thread per row, H*teams rows at a time.
// Shared-memory reads of a row are conflict-free: consecutive threads read
// consecutive blocks, whose strides (144 B, 208 B) are odd multiples of 16 B;
// the staged activation is XOR-swizzled per slice for the same reason.
#pragma once

#include <algorithm>

#include "qb_common.cuh"
#include "qb_launch.h"

namespace qb {

struct Gemv2K {
    const uint8_t *W;
    int64_t rows;
    int K;
    int rec;       // bytes per row record
    int nt;        // teams per CTA
    int ts;        // threads per team = K / 256
    int D;         // ring slots
    int H;         // iterations of block values kept before a fold
    int nb;        // weight blocks per row
    int vstride;   // floats per (iteration, team) line of block values
    int n_iter;    // ceil(rows / (teams in the grid))
    const int8_t *codes;
    const qb_scale *scales;
    const int16_t *sums16;
    float *out;
    int *fault;
};

struct Gemv2Smem {
    int bars, act, scl, val, ring, total;
};

__host__ __device__ inline Gemv2Smem gemv2_smem(int K, int rec, int nt, int D, int H, int vstride) {
    Gemv2Smem s;
    s.bars = 0;                                            // D mbarriers
    s.act = 128;                                           // K codes
    s.scl = s.act + ((K + 127) & ~127);                    // K/32 activation scales (Q8_0)
    s.val = s.scl + ((K / 32 * 4 + 127) & ~127);           // H * nt * vstride floats
    s.ring = s.val + ((H * nt * vstride * 4 + 127) & ~127);
    s.total = s.ring + D * nt * rec;
    return s;
}

// The slice-local 16-B unit k of slice j sits at unit 16j + (k ^ (j & 7)).
__device__ __forceinline__ int slice_unit(int j, int k) { return 16 * j + (k ^ (j & 7)); }

// ------------------------------------------------------------------ per-slice block math
// Activation of one 256-element slice in registers: a[2s] holds elements
// 32s..32s+15, a[2s+1] elements 32s+16..32s+31 (as four packed int8 words).

// Q4_K-like: one block per slice.
__device__ __forceinline__ float slice_q4k(const uint8_t *blk, const uint4 (&a)[16], const uint32_t (&S)[4], int m,
                                           int e) {
    const uint4 meta = *reinterpret_cast<const uint4 *>(blk);
    const unsigned long long sc48 = (unsigned long long)meta.y | ((unsigned long long)(meta.z & 0xFFFFu) << 32);
    const unsigned long long mn48 = (unsigned long long)(meta.z >> 16) | ((unsigned long long)meta.w << 16);
    uint4 w[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) w[s] = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * s);
    int C = 0, O = 0;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        int pl = dp4a_ss(w[s].x & 0x0F0F0F0Fu, a[2 * s].x, 0);
        pl = dp4a_ss(w[s].y & 0x0F0F0F0Fu, a[2 * s].y, pl);
        pl = dp4a_ss(w[s].z & 0x0F0F0F0Fu, a[2 * s].z, pl);
        pl = dp4a_ss(w[s].w & 0x0F0F0F0Fu, a[2 * s].w, pl);
        int ph = dp4a_us(w[s].x & 0xF0F0F0F0u, a[2 * s + 1].x, 0);  // 16*q against a
        ph = dp4a_us(w[s].y & 0xF0F0F0F0u, a[2 * s + 1].y, ph);
        ph = dp4a_us(w[s].z & 0xF0F0F0F0u, a[2 * s + 1].z, ph);
        ph = dp4a_us(w[s].w & 0xF0F0F0F0u, a[2 * s + 1].w, ph);
        C += (int)((sc48 >> (6 * s)) & 63u) * (pl + (ph >> 4));
        const int Ss = (int)(int16_t)((S[s >> 1] >> (16 * (s & 1))) & 0xFFFFu);
        O += (int)((mn48 >> (6 * s)) & 63u) * Ss;
    }
    return lane_value<1>(C, O, meta.x & 0xFFFFu, meta.x >> 16, m, e);
}

// Q6_K-like: one block per slice; d stored apart from the block.
__device__ __forceinline__ float slice_q6k(const uint8_t *blk, uint32_t d, const uint4 (&a)[16],
                                           const uint32_t (&S)[8], int m, int e) {
    const uint4 scw = *reinterpret_cast<const uint4 *>(blk + 192);
    const uint32_t scv[4] = {scw.x, scw.y, scw.z, scw.w};
    int C = 0;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4 *>(blk + 16 * ch);
        const uint2 h = *reinterpret_cast<const uint2 *>(blk + 128 + 8 * ch);
        const uint32_t wl[4] = {w.x, w.y, w.z, w.w};
        const uint32_t al[4] = {a[2 * ch].x, a[2 * ch].y, a[2 * ch].z, a[2 * ch].w};
        const uint32_t ah[4] = {a[2 * ch + 1].x, a[2 * ch + 1].y, a[2 * ch + 1].z, a[2 * ch + 1].w};
        int pl = 0, ph = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t hl = (k < 3) ? (h.x << (4 - 2 * k)) : (h.x >> 2);
            const uint32_t hh = (k < 3) ? (h.y << (4 - 2 * k)) : (h.y >> 2);
            pl = dp4a_ss((wl[k] & 0x0F0F0F0Fu) | (hl & 0x30303030u), al[k], pl);
            ph = dp4a_ss(((wl[k] >> 4) & 0x0F0F0F0Fu) | (hh & 0x30303030u), ah[k], ph);
        }
        const int sc_lo = (int)(int8_t)((scv[ch >> 1] >> (16 * (ch & 1))) & 0xFFu);
        const int sc_hi = (int)(int8_t)((scv[ch >> 1] >> (16 * (ch & 1) + 8)) & 0xFFu);
        // sum over the unit of (q - 32) * a = sum q*a - 32 * S_u
        const int Slo = (int)(int16_t)(S[ch] & 0xFFFFu), Shi = (int)(int16_t)(S[ch] >> 16);
        C += sc_lo * (pl - 32 * Slo) + sc_hi * (ph - 32 * Shi);
    }
    return lane_value<0>(C, 0, d, 0, m, e);
}

// Q8_0: eight blocks of 32 per slice.  Lane j visits the slice's 16-B units in
// the order u ^ (j & 7) (a[u] holds activation unit u ^ (j & 7)), so the eight
// lanes of a shared-memory phase read eight different banks; block i's value
// goes to vl[i].
__device__ __forceinline__ void slice_q8_0(const uint8_t *q, const uint8_t *dptr, const uint32_t *scl,
                                           const uint4 (&a)[16], int jj, float *vl) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const int u0 = (2 * kk) ^ jj, u1 = u0 ^ 1;
        const int i = u0 >> 1;  // the block these two units belong to
        const uint4 w0 = *reinterpret_cast<const uint4 *>(q + 16 * u0);
        const uint4 w1 = *reinterpret_cast<const uint4 *>(q + 16 * u1);
        int p = dp4a_ss(w0.x, a[2 * kk].x, 0);
        p = dp4a_ss(w0.y, a[2 * kk].y, p);
        p = dp4a_ss(w0.z, a[2 * kk].z, p);
        p = dp4a_ss(w0.w, a[2 * kk].w, p);
        p = dp4a_ss(w1.x, a[2 * kk + 1].x, p);
        p = dp4a_ss(w1.y, a[2 * kk + 1].y, p);
        p = dp4a_ss(w1.z, a[2 * kk + 1].z, p);
        p = dp4a_ss(w1.w, a[2 * kk + 1].w, p);
        const uint32_t d = *reinterpret_cast<const uint16_t *>(dptr + 2 * i);
        const uint32_t sw = scl[i];
        vl[i] = lane_value<0>(p, 0, d, 0, (int)(sw & 0xFFu), (int)(int16_t)(sw >> 16));
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Issue the fills of iteration `it` into ring slot it % D: one bulk copy per
// team whose row exists, all completing on that slot's mbarrier.
__device__ __forceinline__ void issue_fill(const Gemv2K &p, uint8_t *ring, uint64_t *bars, int it) {
    const int slot = it % p.D;
    const int64_t nteams = (int64_t)gridDim.x * p.nt;
    int have = 0;
    for (int t = 0; t < p.nt; ++t) have += ((int64_t)t * gridDim.x + blockIdx.x + (int64_t)it * nteams) < p.rows;
    mbar_arrive_expect_tx(bars + slot, (uint32_t)have * (uint32_t)p.rec);
    for (int t = 0; t < p.nt; ++t) {
        const int64_t row = (int64_t)t * gridDim.x + blockIdx.x + (int64_t)it * nteams;
        if (row < p.rows)
            bulk_g2s(ring + ((int64_t)slot * p.nt + t) * p.rec, p.W + row * p.rec, (uint32_t)p.rec, bars + slot);
    }
}

template <int F>
__global__ void __launch_bounds__(256, 2) gemv2_kernel(const Gemv2K p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const Gemv2Smem L = gemv2_smem(p.K, p.rec, p.nt, p.D, p.H, p.vstride);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint8_t *act = smem + L.act;
    uint32_t *ascl = reinterpret_cast<uint32_t *>(smem + L.scl);
    float *val = reinterpret_cast<float *>(smem + L.val);
    uint8_t *ring = smem + L.ring;

    const int tid = threadIdx.x;
    const int team = tid / p.ts, j = tid - team * p.ts;
    const bool live = team < p.nt;
    const int64_t nteams = (int64_t)gridDim.x * p.nt;
    const int64_t gk = (int64_t)team * gridDim.x + blockIdx.x;

    if (tid == 0) {
        for (int s = 0; s < p.D; ++s) mbar_init(bars + s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
        for (int it = 0; it < p.D && it < p.n_iter; ++it) issue_fill(p, ring, bars, it);  // weights: no dependency
    pdl_launch_dependents();
    pdl_wait();

    // ---- this slice's activation: codes staged in shared memory (XOR-swizzled
    // per slice for Q4_K/Q6_K, whose lanes read unit k at step k; linear for
    // Q8_0, whose lanes read unit k ^ (j & 7)), then copied to registers.
    for (int u = tid; u < p.K / 16; u += blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p.codes) + u);
        const int pos = (F == kQ8_0) ? u : slice_unit(u >> 4, u & 15);
        *reinterpret_cast<uint4 *>(act + 16 * pos) = v;
    }
    if (F == kQ8_0)
        for (int b = tid; b < p.K / 32; b += blockDim.x) ascl[b] = __ldg(reinterpret_cast<const uint32_t *>(p.scales) + b);
    uint32_t S4[4] = {0, 0, 0, 0}, S8[8] = {0, 0, 0, 0, 0, 0, 0, 0}, scl0 = 0;
    if (live) {
        if (F == kQ4K) {  // per-32 sums from the per-16 ones
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t pr = __ldg(reinterpret_cast<const uint32_t *>(p.sums16) + 8 * j + s);
                const int S = (int)(int16_t)(pr & 0xFFFFu) + (int)(int16_t)(pr >> 16);
                S4[s >> 1] |= ((uint32_t)S & 0xFFFFu) << (16 * (s & 1));
            }
            scl0 = __ldg(reinterpret_cast<const uint32_t *>(p.scales) + j);
        } else if (F == kQ6K) {
            const uint4 s0 = __ldg(reinterpret_cast<const uint4 *>(p.sums16) + 2 * j);
            const uint4 s1 = __ldg(reinterpret_cast<const uint4 *>(p.sums16) + 2 * j + 1);
            S8[0] = s0.x; S8[1] = s0.y; S8[2] = s0.z; S8[3] = s0.w;
            S8[4] = s1.x; S8[5] = s1.y; S8[6] = s1.z; S8[7] = s1.w;
            scl0 = __ldg(reinterpret_cast<const uint32_t *>(p.scales) + j);
        }
    }
    __syncthreads();
    const int jj = j & 7;
    uint4 a[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int pos = (F == kQ8_0) ? 16 * j + (k ^ jj) : slice_unit(j, k);
        a[k] = live ? *reinterpret_cast<const uint4 *>(act + 16 * pos) : make_uint4(0, 0, 0, 0);
    }
    const int m0 = (int)(scl0 & 0xFFu), e0 = (int)(int16_t)(scl0 >> 16);

    // ---- the row loop
    for (int it = 0; it < p.n_iter; ++it) {
        const int slot = it % p.D;
        const int64_t row = gk + (int64_t)it * nteams;
        bool ok = true;
        if (live && row < p.rows) {
            ok = mbar_wait_bounded(bars + slot, (uint32_t)((it / p.D) & 1), p.fault);
            if (ok) {
                const uint8_t *rp = ring + ((int64_t)slot * p.nt + team) * p.rec;
                float *vl = val + ((it % p.H) * p.nt + team) * p.vstride;
                if (F == kQ4K) {
                    vl[j] = slice_q4k(rp + 144 * j, a, S4, m0, e0);
                } else if (F == kQ6K) {
                    const uint32_t d = *reinterpret_cast<const uint16_t *>(rp + 208 * p.nb + 2 * j);
                    vl[j] = slice_q6k(rp + 208 * j, d, a, S8, m0, e0);
                } else {
                    slice_q8_0(rp + 256 * j, rp + p.K + 16 * j, ascl + 8 * j, a, jj, vl + 8 * j);
                }
            }
        }
        if (!__syncthreads_and(ok)) return;  // a fill never completed: fault word raised
        if (tid == 0 && it + p.D < p.n_iter) {
            fence_proxy_async_smem();
            issue_fill(p, ring, bars, it + p.D);
        }
        // ---- fold H iterations' rows: one thread per row, blocks in order
        if ((it % p.H) == p.H - 1 || it == p.n_iter - 1) {
            const int h0 = it - (it % p.H);
            const int nrow = (it - h0 + 1) * p.nt;
            for (int f = tid; f < nrow; f += blockDim.x) {
                const int hi = f / p.nt, t = f - hi * p.nt;
                const int64_t r = (int64_t)t * gridDim.x + blockIdx.x + (int64_t)(h0 + hi) * nteams;
                if (r < p.rows) {
                    const float *vr = val + (hi * p.nt + t) * p.vstride;
                    float acc = 0.0f;
                    for (int b = 0; b < p.nb; ++b) acc = fadd_ftz(acc, vr[b]);
                    if (acc != acc) acc = __uint_as_float(kEngineNaN);
                    p.out[r] = acc;
                }
            }
            __syncthreads();  // before the history is overwritten
        }
    }
}

// Host: the launch shape.  Returns QB_E_ARG when the streaming kernel does not
// apply (the caller then uses the general kernel).
template <int F>
int launch_gemv2(const GemvArgs &a, cudaStream_t stream) {
    if (a.ncols != 1 || a.mode != 0 || a.K % 256 != 0) return QB_E_ARG;
    const int K = (int)a.K;
    const int ts = K / 256;
    if (ts > 256) return QB_E_ARG;
    Gemv2K k;
    k.W = static_cast<const uint8_t *>(a.W);
    k.rows = a.rows;
    k.K = K;
    k.rec = (int)record_bytes(F, a.K);
    k.ts = ts;
    k.nt = std::max(1, 256 / ts);
    k.nb = K / fmt_block(F);
    k.vstride = (k.nb & 1) ? k.nb : k.nb + 1;
    const int sms = num_sms();
    const int64_t per_iter_rows = (int64_t)sms * k.nt;
    // grid: one CTA per SM, fewer when the matrix has fewer rows than teams
    int grid = sms;
    if (a.rows < per_iter_rows) grid = (int)std::max<int64_t>(1, (a.rows + k.nt - 1) / k.nt);
    k.n_iter = (int)((a.rows + (int64_t)grid * k.nt - 1) / ((int64_t)grid * k.nt));
    // ring: at most ~96 KB, so a following launch's CTA fits beside this one
    const int slot = k.nt * k.rec;
    k.D = std::max(1, std::min(k.n_iter, 98304 / std::max(1, slot)));
    if (k.D < 2 && k.n_iter > 1) k.D = 2;
    k.H = std::max(1, std::min(k.n_iter, 8));
    k.codes = a.codes;
    k.scales = a.scales;
    k.sums16 = a.sums16;
    k.out = a.out;
    k.fault = fault_word();
    if (!k.fault) return QB_E_CUDA;
    Gemv2Smem L = gemv2_smem(K, k.rec, k.nt, k.D, k.H, k.vstride);
    while (L.total > 200 * 1024 && k.D > 1) {
        --k.D;
        L = gemv2_smem(K, k.rec, k.nt, k.D, k.H, k.vstride);
    }
    if (L.total > 227 * 1024) return QB_E_ARG;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(gemv2_kernel<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
            cudaSuccess)
            return QB_E_CUDA;
        attr_set = true;
    }
    const int threads = (k.nt * ts + 31) / 32 * 32;
    return launch_pdl(gemv2_kernel<F>, dim3(grid), dim3(threads), (size_t)L.total, stream, k);
}

}  // namespace qb
