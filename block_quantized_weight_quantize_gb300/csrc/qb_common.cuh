// qb_common.cuh -- device helpers shared by the sm_103a kernels of this library:
// inline-PTX wrappers (mbarrier, bulk async copy, programmatic dependent
// launch, dp4a), the exact decode of an f16 block scale, and the exact
// two-term combine of a block rounded once to f32.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qgemv.h"

namespace qb {

// ---------------------------------------------------------------- formats

enum Fmt : int { kQ8_0 = 0, kQ4K = 1, kQ6K = 2 };

__host__ __device__ constexpr int fmt_block(int f) { return f == kQ8_0 ? 32 : 256; }

// Bytes of one row record (see qgemv.h for the layouts).
__host__ __device__ inline int64_t record_bytes(int f, int64_t K) {
    if (f == kQ8_0) return (K + 2 * (K / 32) + 15) / 16 * 16;
    if (f == kQ4K) return 144 * (K / 256);
    return (210 * (K / 256) + 15) / 16 * 16;
}

// Bit set in the library's device fault word (a __device__ int in qb_api.cu,
// passed to kernels by address) when a kernel gives up a bounded wait.
constexpr int kFaultMbarTimeout = 1;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` for at most ~`limit_cycles` SM cycles.
// Returns false (and raises the device fault word) if the wait ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int *fault,
                                                  long long limit_cycles = 4000000000LL) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit_cycles) {
            atomicOr(fault, kFaultMbarTimeout);
            return false;
        }
    }
    return true;
}

// One bulk asynchronous copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on `bar`.  src, dst 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start, and
// wait for the previous one (no-ops when the launch did not opt in).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// a: four unsigned bytes, b: four signed bytes
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// a: two signed 16-bit halves, b: four unsigned bytes; lo: a.h0*b.b0 + a.h1*b.b1
// + c, hi: a.h0*b.b2 + a.h1*b.b3 + c
__device__ __forceinline__ int dp2a_lo_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Four 6-bit fields f[i] = (v >> 6i) & 63 spread to the four bytes of a word.
__device__ __forceinline__ uint32_t spread6(uint32_t v) {
    return (v & 0x3Fu) | ((v << 2) & 0x3F00u) | ((v << 4) & 0x3F0000u) | ((v << 6) & 0x3F000000u);
}

__device__ __forceinline__ float fadd_ftz(float a, float b) {
    float d;
    asm("add.rn.ftz.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// ---------------------------------------------------------------- exact arithmetic

// A stored f16 scale as sig*2^ex exactly (numerics page, struct Scale).
// Returns false for inf/NaN (numerics page, Unreadable).
__device__ __forceinline__ bool f16_scale(uint32_t h, int &sig, int &ex) {
    const int E = (h >> 10) & 31, f = h & 1023;
    sig = E ? (f | 1024) : f;
    ex = (E ? E : 1) - 25;
    if (h & 0x8000) sig = -sig;
    return E != 31;
}

constexpr uint32_t kEngineNaN = 0x7FC00000u;  // numerics page, NAN

// Round the exact value n * 2^E (n != 0 fits 63 bits) once to f32: nearest
// even on the f32 grid (quantum 2^(x-23) at a normal leading place x, 2^-149
// below 2^-126), a subnormal result then flushed to a zero of its sign, past
// the top infinite (numerics page, scaled_to_f32 / ldexp).
__device__ __forceinline__ float round_to_f32(long long n, int E) {
    if (n == 0) return 0.0f;
    const uint32_t sign = n < 0 ? 0x80000000u : 0u;
    const unsigned long long a = n < 0 ? 0ull - (unsigned long long)n : (unsigned long long)n;
    const int p = 63 - __clzll((long long)a);  // leading place of a
    int x = p + E;
    if (x >= -126) {
        const int sh = p - 23;  // places dropped
        unsigned long long mant;
        if (sh <= 0) {
            mant = a << (-sh);
        } else {
            mant = a >> sh;
            const unsigned long long rem = a & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
            if (rem > half || (rem == half && (mant & 1ull))) ++mant;
            if (mant == (1ull << 24)) { mant >>= 1; ++x; }
        }
        if (x > 127) return __uint_as_float(sign | 0x7F800000u);
        return __uint_as_float(sign | ((uint32_t)(x + 127) << 23) | ((uint32_t)mant & 0x7FFFFFu));
    }
    // below the least normal: round to a multiple of 2^-149, keep only 2^-126
    const int sh = -149 - E;  // places dropped to reach the 2^-149 quantum
    if (sh <= 0 || sh >= 64) return __uint_as_float(sign);  // exact subnormal, or far below half a quantum
    unsigned long long r = a >> sh;
    const unsigned long long rem = a & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (r & 1ull))) ++r;
    return __uint_as_float(sign | (r == (1ull << 23) ? 0x00800000u : 0u));
}

// The same for a 128-bit n: shift it into 62 bits, folding the dropped bits
// into a sticky bit (keeps >= 2 places below any rounding position).
static __device__ __noinline__ float round_to_f32_wide(__int128 n, int E) {
    if (n == 0) return 0.0f;
    const bool neg = n < 0;
    unsigned __int128 a = neg ? (unsigned __int128)(-n) : (unsigned __int128)n;
    int s = 0;
    while ((a >> 62) != 0) {
        const unsigned __int128 sticky = a & 1u;
        a = (a >> 1) | sticky;
        ++s;
    }
    const long long v = (long long)(unsigned long long)a;
    return round_to_f32(neg ? -v : v, E + s);
}

// lane (lane page): a block's value s_a*(s1*C + s2sign*s2*O), summed exactly and
// rounded once.  kind 0: s_a*s1*C.  kind 1: s_a*(s1*C - s2*O).
// m == 0 (activation block without a scale) or an inf/NaN scale: the engine's NaN.
template <int KIND>
__device__ __forceinline__ float lane_value(int C, int O, uint32_t s1, uint32_t s2, int m, int e) {
    int sig1, ex1;
    bool ok = f16_scale(s1, sig1, ex1) && m != 0;
    if (KIND == 0) {
        if (!ok) return __uint_as_float(kEngineNaN);
        return round_to_f32((long long)(sig1 * m) * (long long)C, ex1 + e);  // < 2^19 * 2^28
    } else {
        int sig2, ex2;
        ok = f16_scale(s2, sig2, ex2) && ok;
        if (!ok) return __uint_as_float(kEngineNaN);
        const long long t1 = (long long)(sig1 * m) * (long long)C;   // |t1| < 2^44
        const long long t2 = -(long long)(sig2 * m) * (long long)O;  // |t2| < 2^40
        const int d = ex1 - ex2;
        if (d >= 0 && d <= 17) return round_to_f32((t1 << d) + t2, ex2 + e);
        if (d < 0 && d >= -21) return round_to_f32(t1 + (t2 << (-d)), ex1 + e);
        // wide exponent spread (up to 29 places): exact in 128 bits
        const __int128 w = d >= 0 ? ((__int128)t1 << d) + t2 : (__int128)t1 + ((__int128)t2 << (-d));
        return round_to_f32_wide(w, (d >= 0 ? ex2 : ex1) + e);
    }
}

}  // namespace qb
