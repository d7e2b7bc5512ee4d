// qb_static.cu -- q_matvec_static: the product from an f32 activation for
// callers that cannot allocate device memory.
//
// q_matvec needs a workspace for the quantized activation whenever it runs as
// two launches (quantize, then multiply), and the caller must allocate it.
// Some callers cannot: a serving process that has handed all device memory to
// its own pool at start-up and forbids allocations afterwards, or code on a
// latency-critical path that must not call cudaMalloc (which can synchronize
// the device and take a global lock).  This entry point keeps that workspace
// in a fixed array inside the library instead, so a call allocates nothing.
//
// The array is a file-scope __device__ variable of kStaticScratchBytes
// (QB_STATIC_SCRATCH_BYTES): every GPU that loads the library holds it until
// the process exits.  Host code cannot use the array's name as a device
// address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.
#include <atomic>
#include <cstdint>

#include "qb_common.cuh"
#include "qb_launch.h"

namespace {

constexpr int64_t kStaticScratchBytes = QB_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device; the lookup runs
// once per device and is cached (an entry is only ever set to the one address
// the device's module gives, so relaxed atomics suffice between host
// threads).  Returns nullptr on a CUDA error.
void *static_scratch_address() {
    static std::atomic<void *> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    void *p = cache[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return nullptr;
        cache[dev].store(p, std::memory_order_relaxed);
    }
    return p;
}

bool misaligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace

extern "C" int q_matvec_static(qb_fmt fmt, const void *W, int64_t rows, int64_t K, const float *x, int ncols,
                               float *out, void *stream) {
    const int64_t need = q_matvec_workspace_bytes(fmt, K, ncols);
    if (need < 0) return (int)need;
    if (need > kStaticScratchBytes) return QB_E_SCRATCH;
    if (!W || !x || !out || misaligned16(W) || misaligned16(x) || (reinterpret_cast<uintptr_t>(out) & 3u))
        return QB_E_ARG;
    if (rows < 0 || rows > (int64_t(1) << 31)) return QB_E_ARG;
    if (fmt == QB_F16) {
        if ((int64_t)ncols * K * 4 > 227 * 1024) return QB_E_ARG;
    } else if (K > (int64_t(1) << 18)) {
        return QB_E_ARG;
    }
    // no rows, or rows of no blocks: as q_matvec, nothing to launch, or an
    // output of +0 (the fold of no terms)
    if (rows == 0) return QB_OK;
    if (K == 0)
        return cudaMemsetAsync(out, 0, (size_t)ncols * rows * sizeof(float), static_cast<cudaStream_t>(stream)) ==
                       cudaSuccess
                   ? QB_OK
                   : QB_E_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(static_scratch_address());
    if (!ws) return QB_E_CUDA;
    if (fmt == QB_F16) {
        uint16_t *x16 = reinterpret_cast<uint16_t *>(ws);
        int rc = quantize_act_f16(x, K, ncols, x16, stream);
        if (rc) return rc;
        return q_gemv_f16(static_cast<const uint16_t *>(W), rows, K, x16, ncols, out, stream);
    }
    // the quantized activation's three parts, each 16-byte aligned, as q_matvec lays out its workspace
    const int blk = fmt == QB_Q8_0 ? 32 : 256;
    const int64_t codes_bytes = (K * ncols + 15) / 16 * 16;
    const int64_t scale_bytes = (4 * (K / blk) * ncols + 15) / 16 * 16;
    int8_t *codes = reinterpret_cast<int8_t *>(ws);
    qb_scale *scales = reinterpret_cast<qb_scale *>(ws + codes_bytes);
    int16_t *sums16 = reinterpret_cast<int16_t *>(ws + codes_bytes + scale_bytes);
    int rc = quantize_act(blk, x, K, ncols, codes, scales, sums16, stream);
    if (rc) return rc;
    qb_act act;
    act.block = blk;
    act.codes = codes;
    act.scales = scales;
    act.sums16 = sums16;
    return q_gemv(fmt, W, rows, K, &act, ncols, out, stream);
}
