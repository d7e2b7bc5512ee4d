// qb_api.cu -- the extern "C" entry points declared in include/qgemv.h:
// argument checks on the host, then one launch per call on the caller's
// stream.  Also the weight-scale scan (numerics page, reads / Unreadable) and
// the device fault word.
#include <cstdint>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "qb_common.cuh"
#include "qb_launch.h"

namespace qb {

__device__ int g_fault = 0;
__device__ int g_unreadable = 0;

// Per-device caches: each entry is written once per device with the same
// value by whichever thread gets there first, so relaxed atomics suffice.
int *fault_word() {
    static std::atomic<int *> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int *p = cache[dev].load(std::memory_order_relaxed);
    if (!p) {
        void *q = nullptr;
        if (cudaGetSymbolAddress(&q, g_fault) != cudaSuccess) return nullptr;
        p = static_cast<int *>(q);
        cache[dev].store(p, std::memory_order_relaxed);
    }
    return p;
}

int num_sms() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// The dynamic shared-memory limit is a property of a kernel in one device's
// context: raise it on the current device the first time a launch there needs
// it.  The record is per (kernel, device) under a mutex, so host threads that
// drive one or several devices may launch concurrently.
int ensure_smem_limit(const void *kernel, int bytes) {
    if (bytes <= 48 * 1024) return QB_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QB_E_CUDA;
    struct Entry { const void *k; int dev; int bytes; };
    static std::mutex mu;
    static std::vector<Entry> done;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &e : done)
        if (e.k == kernel && e.dev == dev && e.bytes >= bytes) return QB_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return QB_E_CUDA;
    for (Entry &e : done)
        if (e.k == kernel && e.dev == dev) { e.bytes = bytes; return QB_OK; }
    done.push_back({kernel, dev, bytes});
    return QB_OK;
}

// One thread per weight block: an f16 scale with exponent field 31 (inf/NaN).
__global__ void check_weights_kernel(const uint8_t *__restrict__ W, int64_t rows, int64_t nb, int64_t rec,
                                     int fmt, int64_t K) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t n = rows * nb;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / nb, b = i - r * nb;
        const uint8_t *rp = W + r * rec;
        uint32_t bad = 0;
        if (fmt == kQ8_0) {
            const uint32_t h = rp[K + 2 * b] | (rp[K + 2 * b + 1] << 8);
            bad = ((h >> 10) & 31) == 31;
        } else if (fmt == kQ4K) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(rp + 144 * b);
            bad = (((w >> 10) & 31) == 31) | (((w >> 26) & 31) == 31);
        } else {
            const uint32_t h = rp[208 * nb + 2 * b] | (rp[208 * nb + 2 * b + 1] << 8);
            bad = ((h >> 10) & 31) == 31;
        }
        if (bad) atomicOr(&g_unreadable, 1);
    }
}

int launch_check_weights(int fmt, const void *W, int64_t rows, int64_t K, int *flag, cudaStream_t stream) {
    const int64_t nb = K / fmt_block(fmt), rec = record_bytes(fmt, K);
    const int64_t n = rows * nb;
    const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 8);
    int zero = 0;
    if (cudaMemcpyToSymbolAsync(g_unreadable, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return QB_E_CUDA;
    int rc = launch_pdl(check_weights_kernel, dim3(grid), dim3(256), 0, stream, static_cast<const uint8_t *>(W),
                        rows, nb, rec, fmt, K);
    if (rc) return rc;
    if (cudaMemcpyFromSymbolAsync(flag, g_unreadable, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return QB_E_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return QB_E_CUDA;
    return QB_OK;
}

static int fmt_index(qb_fmt f) {
    switch (f) {
    case QB_Q8_0: return kQ8_0;
    case QB_Q4K: return kQ4K;
    case QB_Q6K: return kQ6K;
    default: return -1;
    }
}

static bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

constexpr int64_t kMaxK = int64_t(1) << 18;  // a row's record must fit a CTA tile in shared memory

}  // namespace qb

using namespace qb;

extern "C" {

int quantize_act(int block, const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales, int16_t *sums16,
                 void *stream) {
    if (block != 32 && block != 256) return QB_E_BLOCK;
    if (!x || !codes || !scales || !sums16) return QB_E_ARG;
    if (K < 0 || K % block != 0 || K > (int64_t(1) << 24) || ncols < 1 || ncols > 16) return QB_E_ARG;
    if (misaligned(x) || misaligned(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) ||
        (reinterpret_cast<uintptr_t>(sums16) & 3u))
        return QB_E_ARG;
    if (K == 0) return QB_OK;
    return launch_quantize_act(block, x, K, ncols, codes, scales, sums16, static_cast<cudaStream_t>(stream));
}

static int check_gemv_args(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols,
                           const void *out) {
    const int f = fmt_index(fmt);
    if (f < 0) return QB_E_FORMAT;
    if (!W || !act || !out || !act->codes || !act->scales) return QB_E_ARG;
    if (f != kQ8_0 && !act->sums16) return QB_E_ARG;
    if (act->block != fmt_block(f)) return QB_E_BLOCK;
    if (rows < 0 || K < 0 || K % fmt_block(f) != 0 || K > kMaxK || ncols < 1 || ncols > 16) return QB_E_ARG;
    if (rows > (int64_t(1) << 31)) return QB_E_ARG;
    if (misaligned(W) || misaligned(act->codes) || (act->sums16 && misaligned(act->sums16)) ||
        (reinterpret_cast<uintptr_t>(act->scales) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u))
        return QB_E_ARG;
    return QB_OK;
}

static int gemv_common(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols, float *out,
                       int32_t *C, int32_t *O, float *v, int mode, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemvArgs a = {};
    a.W = W;
    a.rows = rows;
    a.K = K;
    a.codes = act->codes;
    a.scales = act->scales;
    a.sums16 = act->sums16;
    a.ncols = ncols;
    a.out = out;
    a.dbgC = C;
    a.dbgO = O;
    a.dbgV = v;
    a.mode = mode;
    switch (fmt_index(fmt)) {
    case kQ8_0: return launch_gemv_q8_0(a, s);
    case kQ4K: return launch_gemv_q4k(a, s);
    default: return launch_gemv_q6k(a, s);
    }
}

int q_gemv(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols, float *out,
           void *stream) {
    const int rc = check_gemv_args(fmt, W, rows, K, act, ncols, out);
    if (rc) return rc;
    if (rows == 0) return QB_OK;
    if (K == 0) {  // rows of no blocks: the fold of no terms is +0
        return cudaMemsetAsync(out, 0, (size_t)ncols * rows * sizeof(float), static_cast<cudaStream_t>(stream)) ==
                       cudaSuccess
                   ? QB_OK
                   : QB_E_CUDA;
    }
    return gemv_common(fmt, W, rows, K, act, ncols, out, nullptr, nullptr, nullptr, 0, stream);
}

int q_gemv_w2(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act16 *act, int ncols, float *out,
              void *stream) {
    const int f = fmt_index(fmt);
    if (f < 0) return QB_E_FORMAT;
    if (!W || !act || !out || !act->codes || !act->scales) return QB_E_ARG;
    if (act->block != fmt_block(f)) return QB_E_BLOCK;
    if (rows < 0 || K < 0 || K % fmt_block(f) != 0 || K > kMaxK || ncols < 1 || ncols > 16) return QB_E_ARG;
    if (rows > (int64_t(1) << 31)) return QB_E_ARG;
    if (misaligned(W) || misaligned(act->codes) || (reinterpret_cast<uintptr_t>(act->scales) & 3u) ||
        (reinterpret_cast<uintptr_t>(out) & 3u))
        return QB_E_ARG;
    if (rows == 0) return QB_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)  // rows of no blocks: the fold of no terms is +0
        return cudaMemsetAsync(out, 0, (size_t)ncols * rows * sizeof(float), s) == cudaSuccess ? QB_OK : QB_E_CUDA;
    return launch_gemv_w2(f, W, rows, K, act->codes, act->scales, ncols, out, s);
}

int q_block_values(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols, int32_t *C,
                   int32_t *O, float *v, void *stream) {
    const void *any = C ? (const void *)C : O ? (const void *)O : (const void *)v;
    if (!any) return QB_E_ARG;
    const int rc = check_gemv_args(fmt, W, rows, K, act, ncols, any);
    if (rc) return rc;
    if (rows == 0 || K == 0) return QB_OK;
    return gemv_common(fmt, W, rows, K, act, ncols, nullptr, C, O, v, 1, stream);
}

int quantize_act_f16(const float *x, int64_t K, int ncols, uint16_t *x16, void *stream) {
    if (!x || !x16) return QB_E_ARG;
    if (K < 0 || ncols < 1 || ncols > 16 || K > (int64_t(1) << 24)) return QB_E_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(x16) & 1u)) return QB_E_ARG;
    if (K == 0) return QB_OK;
    return launch_quantize_f16(x, K * ncols, x16, static_cast<cudaStream_t>(stream));
}

int q_gemv_f16(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, int ncols, float *out, void *stream) {
    if (!W || !x16 || !out) return QB_E_ARG;
    if (rows < 0 || K < 0 || K % 8 != 0 || ncols < 1 || ncols > 16 || rows > (int64_t(1) << 31)) return QB_E_ARG;
    if ((int64_t)ncols * K * 4 > 227 * 1024) return QB_E_ARG;
    if (misaligned(W) || (reinterpret_cast<uintptr_t>(x16) & 1u) || (reinterpret_cast<uintptr_t>(out) & 3u))
        return QB_E_ARG;
    if (rows == 0) return QB_OK;
    if (K == 0)
        return cudaMemsetAsync(out, 0, (size_t)ncols * rows * sizeof(float), static_cast<cudaStream_t>(stream)) ==
                       cudaSuccess
                   ? QB_OK
                   : QB_E_CUDA;
    return launch_gemv_f16(W, rows, K, x16, ncols, out, static_cast<cudaStream_t>(stream));
}

int q_check_weights(qb_fmt fmt, const void *W, int64_t rows, int64_t K, void *stream) {
    const int f = fmt_index(fmt);
    if (fmt == QB_F16) return QB_OK;  // no block scales
    if (f < 0) return QB_E_FORMAT;
    if (!W || rows < 0 || K < 0 || K % fmt_block(f) != 0 || K > kMaxK || misaligned(W)) return QB_E_ARG;
    if (rows == 0 || K == 0) return QB_OK;
    int flag = 0;
    const int rc = launch_check_weights(f, W, rows, K, &flag, static_cast<cudaStream_t>(stream));
    if (rc) return rc;
    return flag ? QB_E_UNREADABLE : QB_OK;
}

int64_t q_weight_bytes(qb_fmt fmt, int64_t rows, int64_t K) {
    if (rows < 0 || K < 0) return QB_E_ARG;
    if (fmt == QB_F16) return K % 8 ? QB_E_ARG : rows * K * 2;
    const int f = fmt_index(fmt);
    if (f < 0) return QB_E_FORMAT;
    if (K % fmt_block(f) != 0) return QB_E_ARG;
    return rows * record_bytes(f, K);
}

int q_device_status(void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&h, g_fault, sizeof(int), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QB_E_CUDA;
    if (cudaMemcpyToSymbolAsync(g_fault, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QB_E_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QB_E_CUDA;
    return h ? QB_E_DEVICE : QB_OK;
}

static int64_t align16(int64_t n) { return (n + 15) / 16 * 16; }

int64_t q_matvec_workspace_bytes(qb_fmt fmt, int64_t K, int ncols) {
    if (K < 0 || ncols < 1 || ncols > 16) return QB_E_ARG;
    if (fmt == QB_F16) return K % 8 ? QB_E_ARG : align16(2 * K * ncols);
    const int f = fmt_index(fmt);
    if (f < 0) return QB_E_FORMAT;
    const int blk = fmt_block(f);
    if (K % blk) return QB_E_ARG;
    return align16(K * ncols) + align16(4 * (K / blk) * ncols) + align16(2 * (K / 16) * ncols);
}

int q_matvec(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x, int ncols, float *out,
             void *workspace, size_t workspace_bytes, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!x || !out || !W) return QB_E_ARG;
    if (misaligned(x)) return QB_E_ARG;
    const int64_t need = q_matvec_workspace_bytes(fmt, K, ncols);
    if (need < 0) return (int)need;
    if (fmt != QB_F16) {
        const int f = fmt_index(fmt);
        // argument checks of the product itself (with a stand-in activation)
        qb_act probe = {fmt_block(f), reinterpret_cast<const int8_t *>(x), reinterpret_cast<const qb_scale *>(x),
                        reinterpret_cast<const int16_t *>(x)};
        const int rc = check_gemv_args(fmt, W, rows, K, &probe, ncols, out);
        if (rc) return rc;
        if (rows == 0) return QB_OK;
        if (K == 0)
            return cudaMemsetAsync(out, 0, (size_t)ncols * rows * sizeof(float), s) == cudaSuccess ? QB_OK : QB_E_CUDA;
        // Q4_K-like rows of K >= 12288 with a workspace at hand: quantize_act and
        // the product as two launches measured faster than quantizing the long
        // activation inside every CTA of the single-launch kernel (4096 x 14336:
        // 10.7 against 12.0 us; Q6_K-like there, and every K = 4096 shape, the
        // other way round).
        const bool two = f == kQ4K && K >= 12288 && workspace && (int64_t)workspace_bytes >= need &&
                         !misaligned(workspace);
        // one launch: a single column, or 2..4 columns of the 256-element
        // formats at K = 4096 (each warp quantizes its block of every column)
        if ((ncols == 1 || (ncols <= 4 && K == 4096 && f != kQ8_0)) && !two) {
            GemvArgs a = {};
            a.W = W; a.rows = rows; a.K = K; a.ncols = ncols; a.out = out; a.mode = 0;
            const int r = f == kQ8_0 ? launch_matvec_q8_0(a, x, s)
                        : f == kQ4K  ? launch_matvec_q4k(a, x, s)
                                     : launch_matvec_q6k(a, x, s);
            if (r != QB_E_ARG) return r;  // QB_E_ARG: the single-launch kernel does not take this shape
        }
    }
    if (fmt == QB_F16) {  // one launch where the warp-ring kernel takes the shape (f16 rounding in its prologue)
        if (rows < 0 || K < 0 || K % 8 != 0 || ncols < 1 || ncols > 16 || rows > (int64_t(1) << 31) ||
            misaligned(W) || (reinterpret_cast<uintptr_t>(out) & 3u))
            return QB_E_ARG;
        if (rows == 0) return QB_OK;
        if (K == 0)
            return cudaMemsetAsync(out, 0, (size_t)ncols * rows * sizeof(float), s) == cudaSuccess ? QB_OK : QB_E_CUDA;
        if ((int64_t)ncols * K * 4 <= 227 * 1024) {
            const int r = launch_matvec_f16(single_table(W, rows, out), K, x, ncols, s);
            if (r != QB_E_ARG) return r;
        }
    }
    if (!workspace || (int64_t)workspace_bytes < need || misaligned(workspace)) return QB_E_ARG;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (fmt == QB_F16) {
        uint16_t *x16 = reinterpret_cast<uint16_t *>(ws);
        int rc = quantize_act_f16(x, K, ncols, x16, stream);
        if (rc) return rc;
        return q_gemv_f16(static_cast<const uint16_t *>(W), rows, K, x16, ncols, out, stream);
    }
    const int blk = fmt_block(fmt_index(fmt));
    qb_act act;
    act.block = blk;
    act.codes = reinterpret_cast<const int8_t *>(ws);
    act.scales = reinterpret_cast<const qb_scale *>(ws + align16(K * ncols));
    act.sums16 = reinterpret_cast<const int16_t *>(ws + align16(K * ncols) + align16(4 * (K / blk) * ncols));
    int rc = quantize_act(blk, x, K, ncols, const_cast<int8_t *>(act.codes), const_cast<qb_scale *>(act.scales),
                          const_cast<int16_t *>(act.sums16), stream);
    if (rc) return rc;
    return q_gemv(fmt, W, rows, K, &act, ncols, out, stream);
}

// ---------------------------------------------------------------- several matrices, one activation

// The host arrays of a grouped call as a matrix table; QB_E_ARG for a bad
// count or null arrays.  Per-matrix arguments are checked by the caller.
static int make_table(int nmat, const void *const *W, const int64_t *rows, float *const *out, MatTable &t) {
    if (nmat < 1 || nmat > QB_MAX_MATS || !W || !rows || !out) return QB_E_ARG;
    t = MatTable{};
    t.n = nmat;
    t.start[0] = 0;
    for (int i = 0; i < nmat; ++i) {
        t.W[i] = static_cast<const uint8_t *>(W[i]);
        t.out[i] = out[i];
        t.start[i + 1] = t.start[i] + rows[i];
    }
    if (t.start[nmat] > (int64_t(1) << 31)) return QB_E_ARG;
    return QB_OK;
}

int q_gemv_many(qb_fmt fmt, int nmat, const void *const *W, const int64_t *rows, int64_t K, const qb_act *act,
                int ncols, float *const *out, void *stream) {
    MatTable t;
    int rc = make_table(nmat, W, rows, out, t);
    if (rc) return rc;
    for (int i = 0; i < nmat; ++i)
        if ((rc = check_gemv_args(fmt, W[i], rows[i], K, act, ncols, out[i])) != QB_OK) return rc;
    if (t.start[nmat] > 0 && K > 0) {
        GemvArgs a = {};
        a.mats = &t;
        a.K = K;
        a.codes = act->codes;
        a.scales = act->scales;
        a.sums16 = act->sums16;
        a.ncols = ncols;
        a.mode = 0;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        const int f = fmt_index(fmt);
        rc = f == kQ8_0 ? launch_gemv_q8_0(a, s) : f == kQ4K ? launch_gemv_q4k(a, s) : launch_gemv_q6k(a, s);
        if (rc != QB_E_ARG) return rc;
    }
    for (int i = 0; i < nmat; ++i)  // shapes the streaming kernels do not take: one launch per matrix
        if ((rc = q_gemv(fmt, W[i], rows[i], K, act, ncols, out[i], stream)) != QB_OK) return rc;
    return QB_OK;
}

int q_gemv_f16_many(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t K, const uint16_t *x16,
                    int ncols, float *const *out, void *stream) {
    MatTable t;
    int rc = make_table(nmat, reinterpret_cast<const void *const *>(W), rows, out, t);
    if (rc) return rc;
    if (!x16 || K < 0 || K % 8 != 0 || ncols < 1 || ncols > 16 || (int64_t)ncols * K * 4 > 227 * 1024) return QB_E_ARG;
    for (int i = 0; i < nmat; ++i)
        if (!W[i] || !out[i] || rows[i] < 0 || misaligned(W[i]) || (reinterpret_cast<uintptr_t>(out[i]) & 3u))
            return QB_E_ARG;
    if ((reinterpret_cast<uintptr_t>(x16) & 1u)) return QB_E_ARG;
    if (t.start[nmat] > 0 && K > 0) {
        rc = launch_gemv_f16_many(t, K, x16, ncols, static_cast<cudaStream_t>(stream));
        if (rc != QB_E_ARG) return rc;
    }
    for (int i = 0; i < nmat; ++i)
        if ((rc = q_gemv_f16(W[i], rows[i], K, x16, ncols, out[i], stream)) != QB_OK) return rc;
    return QB_OK;
}

int q_matvec_many(qb_fmt fmt, int nmat, const void *const *W, const int64_t *rows, int64_t K, const float *x,
                  int ncols, float *const *out, void *workspace, size_t workspace_bytes, void *stream) {
    MatTable t;
    int rc = make_table(nmat, W, rows, out, t);
    if (rc) return rc;
    if (!x || misaligned(x)) return QB_E_ARG;
    const int64_t need = q_matvec_workspace_bytes(fmt, K, ncols);
    if (need < 0) return (int)need;
    if (fmt != QB_F16) {
        const int f = fmt_index(fmt);
        qb_act probe = {fmt_block(f), reinterpret_cast<const int8_t *>(x), reinterpret_cast<const qb_scale *>(x),
                        reinterpret_cast<const int16_t *>(x)};
        for (int i = 0; i < nmat; ++i)
            if ((rc = check_gemv_args(fmt, W[i], rows[i], K, &probe, ncols, out[i])) != QB_OK) return rc;
        if (t.start[nmat] == 0) return QB_OK;
        if (K == 0) {  // rows of no blocks: +0
            for (int i = 0; i < nmat; ++i)
                if (rows[i] > 0 && cudaMemsetAsync(out[i], 0, (size_t)ncols * rows[i] * sizeof(float),
                                                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
                    return QB_E_CUDA;
            return QB_OK;
        }
        if (ncols == 1) {  // one launch: quantized inside the product kernel
            GemvArgs a = {};
            a.mats = &t;
            a.K = K;
            a.ncols = 1;
            a.mode = 0;
            cudaStream_t s = static_cast<cudaStream_t>(stream);
            rc = f == kQ8_0 ? launch_matvec_q8_0(a, x, s) : f == kQ4K ? launch_matvec_q4k(a, x, s)
                                                                      : launch_matvec_q6k(a, x, s);
            if (rc != QB_E_ARG) return rc;
        }
    }
    if (fmt == QB_F16 && t.start[nmat] > 0 && K > 0 && K % 8 == 0 && ncols >= 1 && ncols <= 16 &&
        (int64_t)ncols * K * 4 <= 227 * 1024) {  // one launch for the group
        bool okp = true;
        for (int i = 0; i < nmat; ++i)
            okp = okp && W[i] && out[i] && rows[i] >= 0 && !misaligned(W[i]) &&
                  !(reinterpret_cast<uintptr_t>(out[i]) & 3u);
        if (okp) {
            rc = launch_matvec_f16(t, K, x, ncols, static_cast<cudaStream_t>(stream));
            if (rc != QB_E_ARG) return rc;
        }
    }
    if (!workspace || (int64_t)workspace_bytes < need || misaligned(workspace)) return QB_E_ARG;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (fmt == QB_F16) {
        uint16_t *x16 = reinterpret_cast<uint16_t *>(ws);
        if ((rc = quantize_act_f16(x, K, ncols, x16, stream)) != QB_OK) return rc;
        return q_gemv_f16_many(nmat, reinterpret_cast<const uint16_t *const *>(W), rows, K, x16, ncols, out, stream);
    }
    const int blk = fmt_block(fmt_index(fmt));
    qb_act act;
    act.block = blk;
    act.codes = reinterpret_cast<const int8_t *>(ws);
    act.scales = reinterpret_cast<const qb_scale *>(ws + align16(K * ncols));
    act.sums16 = reinterpret_cast<const int16_t *>(ws + align16(K * ncols) + align16(4 * (K / blk) * ncols));
    rc = quantize_act(blk, x, K, ncols, const_cast<int8_t *>(act.codes), const_cast<qb_scale *>(act.scales),
                      const_cast<int16_t *>(act.sums16), stream);
    if (rc) return rc;
    return q_gemv_many(fmt, nmat, W, rows, K, &act, ncols, out, stream);
}

// ---------------------------------------------------------------- ActScaling::Sub32

int quantize_act_sub32(const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales, int16_t *sums16,
                       void *stream) {
    if (!x || !codes || !scales || !sums16) return QB_E_ARG;
    if (K < 0 || K % 256 != 0 || K > (int64_t(1) << 24) || ncols < 1 || ncols > 16) return QB_E_ARG;
    if (misaligned(x) || misaligned(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) ||
        (reinterpret_cast<uintptr_t>(sums16) & 3u))
        return QB_E_ARG;
    if (K == 0) return QB_OK;
    return launch_quantize_sub32(x, K, ncols, codes, scales, sums16, static_cast<cudaStream_t>(stream));
}

static int check_sub32_args(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols,
                            const void *out) {
    const int f = fmt_index(fmt);
    if (f < 0) return QB_E_FORMAT;
    if (!W || !act || !out || !act->codes || !act->scales) return QB_E_ARG;
    if (f != kQ8_0 && !act->sums16) return QB_E_ARG;
    if (act->block != 32) return QB_E_BLOCK;
    if (rows < 0 || K < 0 || K % 256 != 0 || K > kMaxK || ncols < 1 || ncols > 16) return QB_E_ARG;
    if (rows > (int64_t(1) << 31)) return QB_E_ARG;
    if (misaligned(W) || misaligned(act->codes) || (act->sums16 && misaligned(act->sums16)) ||
        misaligned(act->scales) || (reinterpret_cast<uintptr_t>(out) & 3u))
        return QB_E_ARG;
    return QB_OK;
}

int q_gemv_sub32(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const qb_act *act, int ncols, float *out,
                 void *stream) {
    const int rc = check_sub32_args(fmt, W, rows, K, act, ncols, out);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rows == 0) return QB_OK;
    if (K == 0)
        return cudaMemsetAsync(out, 0, (size_t)ncols * rows * sizeof(float), s) == cudaSuccess ? QB_OK : QB_E_CUDA;
    GemvArgs a = {};
    a.W = W;
    a.rows = rows;
    a.K = K;
    a.codes = act->codes;
    a.scales = act->scales;
    a.sums16 = act->sums16;
    a.ncols = ncols;
    a.out = out;
    switch (fmt_index(fmt)) {
    case kQ8_0: return launch_gemv_sub32_q8_0(a, s);
    case kQ4K: return launch_gemv_sub32_q4k(a, s);
    default: return launch_gemv_sub32_q6k(a, s);
    }
}

int64_t q_matvec_sub32_workspace_bytes(int64_t K, int ncols) {
    if (K < 0 || K % 256 != 0 || ncols < 1 || ncols > 16) return QB_E_ARG;
    return align16(K * ncols) + align16(4 * (K / 32) * ncols) + align16(2 * (K / 16) * ncols);
}

int q_matvec_sub32(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x, int ncols, float *out,
                   void *workspace, size_t workspace_bytes, void *stream) {
    if (!x || misaligned(x)) return QB_E_ARG;
    const int64_t need = q_matvec_sub32_workspace_bytes(K, ncols);
    if (need < 0) return (int)need;
    if (ncols == 1) {  // one launch where the streaming kernel takes the shape (x quantized in its prologue)
        const qb_act probe = {32, reinterpret_cast<const int8_t *>(x), reinterpret_cast<const qb_scale *>(x),
                              reinterpret_cast<const int16_t *>(x)};
        const int rc = check_sub32_args(fmt, W, rows, K, &probe, ncols, out);
        if (rc) return rc;
        if (rows == 0) return QB_OK;
        if (K > 0) {
            GemvArgs a = {};
            a.W = W; a.rows = rows; a.K = K; a.ncols = 1; a.out = out; a.mode = 0;
            cudaStream_t s = static_cast<cudaStream_t>(stream);
            const int f = fmt_index(fmt);
            const int r = f == kQ8_0 ? launch_matvec_sub32_q8_0(a, x, s)
                        : f == kQ4K  ? launch_matvec_sub32_q4k(a, x, s)
                                     : launch_matvec_sub32_q6k(a, x, s);
            if (r != QB_E_ARG) return r;
        }
    }
    if (!workspace || (int64_t)workspace_bytes < need || misaligned(workspace)) return QB_E_ARG;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    qb_act act;
    act.block = 32;
    act.codes = reinterpret_cast<const int8_t *>(ws);
    act.scales = reinterpret_cast<const qb_scale *>(ws + align16(K * ncols));
    act.sums16 = reinterpret_cast<const int16_t *>(ws + align16(K * ncols) + align16(4 * (K / 32) * ncols));
    int rc = check_sub32_args(fmt, W, rows, K, &act, ncols, out);
    if (rc) return rc;
    if (rows == 0) return QB_OK;
    rc = quantize_act_sub32(x, K, ncols, const_cast<int8_t *>(act.codes), const_cast<qb_scale *>(act.scales),
                            const_cast<int16_t *>(act.sums16), stream);
    if (rc) return rc;
    return q_gemv_sub32(fmt, W, rows, K, &act, ncols, out, stream);
}

// ---------------------------------------------------------------- host buffers in, host buffers out

int64_t q_matvec_host_workspace_bytes(int scaling, qb_fmt fmt, int64_t rows, int64_t K, int ncols) {
    if ((scaling != QB_PERBLOCK && scaling != QB_SUB32) || rows < 0 || K < 0 || ncols < 1 || ncols > 16)
        return QB_E_ARG;
    if (scaling == QB_SUB32 && fmt == QB_F16) return QB_E_FORMAT;
    const int64_t inner =
        scaling == QB_SUB32 ? q_matvec_sub32_workspace_bytes(K, ncols) : q_matvec_workspace_bytes(fmt, K, ncols);
    if (inner < 0) return inner;
    return align16(4 * K * ncols) + align16(4 * rows * ncols) + inner;
}

int q_matvec_host(int scaling, qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x_host, int ncols,
                  float *out_host, void *workspace, size_t workspace_bytes, void *stream) {
    if (!x_host || !out_host || !W || !workspace || misaligned(workspace)) return QB_E_ARG;
    const int64_t need = q_matvec_host_workspace_bytes(scaling, fmt, rows, K, ncols);
    if (need < 0) return (int)need;
    if ((int64_t)workspace_bytes < need) return QB_E_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *xd = reinterpret_cast<float *>(ws);
    float *od = reinterpret_cast<float *>(ws + align16(4 * K * ncols));
    uint8_t *inner = ws + align16(4 * K * ncols) + align16(4 * rows * ncols);
    const size_t inner_bytes = (size_t)(need - (inner - ws));
    if (rows == 0) return QB_OK;
    if (K > 0 && cudaMemcpyAsync(xd, x_host, (size_t)(4 * K * ncols), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QB_E_CUDA;
    const int rc = scaling == QB_SUB32 ? q_matvec_sub32(fmt, W, rows, K, xd, ncols, od, inner, inner_bytes, stream)
                                       : q_matvec(fmt, W, rows, K, xd, ncols, od, inner, inner_bytes, stream);
    if (rc) return rc;
    if (cudaMemcpyAsync(out_host, od, (size_t)(4 * rows * ncols), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QB_E_CUDA;
    return QB_OK;
}

// ---------------------------------------------------------------- FP8 E4M3, 128x128 block scales

int q_gemv_fp8(const uint8_t *W, const float *scales, int64_t rows, int64_t K, const float *x, int ncols, float *out,
               void *stream) {
    if (!W || !scales || !x || !out) return QB_E_ARG;
    if (rows < 0 || rows > (int64_t(1) << 31) || K < 16 || K > 32768 || K % 16 != 0 || ncols < 1 || ncols > 16)
        return QB_E_ARG;
    if (misaligned(W) || misaligned(x) || (reinterpret_cast<uintptr_t>(scales) & 3u) ||
        (reinterpret_cast<uintptr_t>(out) & 3u))
        return QB_E_ARG;
    if (rows == 0) return QB_OK;
    return launch_gemv_fp8(W, scales, rows, K, x, ncols, out, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------- the int8 cache's score path

int kv_head_codes(int scaling, int d) {
    if ((scaling != QB_PERBLOCK && scaling != QB_SUB32) || d < 16 || d > 1024 || d % 16 != 0) return QB_E_ARG;
    return scaling == QB_SUB32 ? (d + 255) / 256 * 256 : d;
}

int kv_cache_rows(const float *x, int64_t n, int d, int8_t *codes, uint16_t *scales, void *stream) {
    if (!x || !codes || !scales) return QB_E_ARG;
    if (n < 0 || d < 16 || d > 1024 || d % 16 != 0) return QB_E_ARG;
    if (misaligned(x) || misaligned(codes) || (reinterpret_cast<uintptr_t>(scales) & 1u)) return QB_E_ARG;
    if (n == 0) return QB_OK;
    return launch_kv_cache_rows(x, n, d, codes, scales, static_cast<cudaStream_t>(stream));
}

int kv_quantize_heads(int scaling, const float *q, int nh, int d, int8_t *codes, qb_scale *scales, void *stream) {
    if (kv_head_codes(scaling, d) < 0 || !q || !codes || !scales || nh < 1 || nh > 4096) return QB_E_ARG;
    if (misaligned(q) || misaligned(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u)) return QB_E_ARG;
    return launch_kv_quantize_heads(scaling, q, nh, d, codes, scales, static_cast<cudaStream_t>(stream));
}

int kv_scores(int scaling, const int8_t *qcodes, const qb_scale *qscales, int nh, int d, const int8_t *kcodes,
              const uint16_t *kscales, int64_t L, int64_t lcap, int nkv, float scale, float *out, void *stream) {
    if (kv_head_codes(scaling, d) < 0) return QB_E_ARG;
    if (!qcodes || !qscales || !kcodes || !kscales || !out) return QB_E_ARG;
    if (nh < 1 || nh > 4096 || nkv < 1 || nh % nkv != 0 || L < 0 || lcap < L) return QB_E_ARG;
    if (misaligned(qcodes) || misaligned(kcodes) || (reinterpret_cast<uintptr_t>(qscales) & 3u) ||
        (reinterpret_cast<uintptr_t>(kscales) & 1u) || (reinterpret_cast<uintptr_t>(out) & 3u))
        return QB_E_ARG;
    if (L == 0) return QB_OK;
    return launch_kv_scores(scaling, qcodes, qscales, nh, d, kcodes, kscales, L, lcap, nkv, scale, out,
                            static_cast<cudaStream_t>(stream));
}

const char *q_strerror(int status) {
    switch (status) {
    case QB_OK: return "ok";
    case QB_E_ARG: return "invalid argument (null or misaligned pointer, size out of range)";
    case QB_E_FORMAT: return "weight format not read by this library";
    case QB_E_BLOCK: return "activation block differs from the weight format's block";
    case QB_E_CUDA: return "CUDA call or launch failed";
    case QB_E_UNREADABLE: return "weights hold an infinite or NaN block scale";
    case QB_E_DEVICE: return "a kernel gave up a bounded wait";
    case QB_E_SCRATCH: return "request needs more than the library's static scratch (QB_STATIC_SCRATCH_BYTES)";
    default: return "unknown status";
    }
}

}  // extern "C"
