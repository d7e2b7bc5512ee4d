// qb_launch.h -- host-side launch helper and the internal launcher prototypes.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qgemv.h"

namespace qb {

// Launch with programmatic dependent launch allowed (the kernel may begin
// while the previous kernel on the stream drains; each kernel here calls
// griddepcontrol.wait before touching data a predecessor may produce).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      Args... args) {
    if (grid.x == 0) return QB_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    return err == cudaSuccess ? QB_OK : QB_E_CUDA;
}

int launch_quantize_act(int block, const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales,
                        int16_t *sums16, cudaStream_t stream);
int launch_quantize_sub32(const float *x, int64_t K, int ncols, int8_t *codes, qb_scale *scales, int16_t *sums16,
                          cudaStream_t stream);
int launch_quantize_f16(const float *x, int64_t n, uint16_t *x16, cudaStream_t stream);

// Matrices that share one activation (the same K and format), seen by a
// kernel as one range of rows: matrix i holds rows [start[i], start[i+1]) of
// the range, reads its records from W[i] and writes its own output out[i]
// (out[i][c*rows_i + r]).  A single matrix is the table of one.
constexpr int kMaxMats = QB_MAX_MATS;
struct MatTable {
    int n;
    const uint8_t *W[kMaxMats];
    float *out[kMaxMats];
    int64_t start[kMaxMats + 1];
};
inline MatTable single_table(const void *W, int64_t rows, float *out) {
    MatTable t = {};
    t.n = 1;
    t.W[0] = static_cast<const uint8_t *>(W);
    t.out[0] = out;
    t.start[0] = 0;
    t.start[1] = rows;
    return t;
}

// The per-format product launchers (qb_gemv_*.cu).  mode 0: rows folded into
// out; mode 1: per-block C, O, v written instead (testing).  mats, when not
// null, replaces W / rows / out by a table of matrices (streaming kernels).
struct GemvArgs {
    const void *W;
    int64_t rows;
    int64_t K;
    const int8_t *codes;
    const qb_scale *scales;
    const int16_t *sums16;
    int ncols;
    float *out;
    int32_t *dbgC;
    int32_t *dbgO;
    float *dbgV;
    int mode;
    const MatTable *mats;
};
int launch_gemv_q8_0(const GemvArgs &a, cudaStream_t stream);
int launch_gemv_q4k(const GemvArgs &a, cudaStream_t stream);
int launch_gemv_q6k(const GemvArgs &a, cudaStream_t stream);
// The product under ActScaling::Sub32 (activation scales per 32 elements,
// one rounding per 256-element group).
int launch_gemv_sub32_q8_0(const GemvArgs &a, cudaStream_t stream);
int launch_gemv_sub32_q4k(const GemvArgs &a, cudaStream_t stream);
int launch_gemv_sub32_q6k(const GemvArgs &a, cudaStream_t stream);
// one column of Sub32 from the f32 activation in one launch; QB_E_ARG where the kernel does not take it
int launch_matvec_sub32_q8_0(const GemvArgs &a, const float *x, cudaStream_t stream);
int launch_matvec_sub32_q4k(const GemvArgs &a, const float *x, cudaStream_t stream);
int launch_matvec_sub32_q6k(const GemvArgs &a, const float *x, cudaStream_t stream);
// The single-launch product (activation quantized inside the kernel); returns
// QB_E_ARG when that kernel does not apply to the shape.
int launch_matvec_q8_0(const GemvArgs &a, const float *x, cudaStream_t stream);
int launch_matvec_q4k(const GemvArgs &a, const float *x, cudaStream_t stream);
int launch_matvec_q6k(const GemvArgs &a, const float *x, cudaStream_t stream);
int launch_gemv_f16(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, int ncols, float *out,
                    cudaStream_t stream);
// Several F16 matrices in one launch; QB_E_ARG when the streaming kernel does not take the shape.
int launch_gemv_f16_many(const MatTable &t, int64_t K, const uint16_t *x16, int ncols, cudaStream_t stream);
// F16 from the f32 activation in one launch (rounded to f16 in the prologue); QB_E_ARG when it does not apply.
int launch_matvec_f16(const MatTable &t, int64_t K, const float *x, int ncols, cudaStream_t stream);
int launch_check_weights(int fmt, const void *W, int64_t rows, int64_t K, int *flag, cudaStream_t stream);
// Two-word (16-bit) activation codes (qb_w2.cu); QB_E_ARG when a row's block values do not fit shared memory.
int launch_gemv_w2(int fmt, const void *W, int64_t rows, int64_t K, const int16_t *codes, const qb_scale *scales,
                   int ncols, float *out, cudaStream_t stream);
// FP8 E4M3 weights with 128x128 block scales (qb_fp8.cu).
int launch_gemv_fp8(const uint8_t *W, const float *scales, int64_t rows, int64_t K, const float *x, int ncols,
                    float *out, cudaStream_t stream);
// The int8 cache's score path (qb_kv.cu).
int launch_kv_cache_rows(const float *x, int64_t n, int d, int8_t *codes, uint16_t *scales, cudaStream_t stream);
int launch_kv_quantize_heads(int scaling, const float *q, int nh, int d, int8_t *codes, qb_scale *scales,
                             cudaStream_t stream);
int launch_kv_scores(int scaling, const int8_t *qc, const qb_scale *qs, int nh, int d, const int8_t *kc,
                     const uint16_t *ks, int64_t L, int64_t lcap, int nkv, float scale, float *out,
                     cudaStream_t stream);

constexpr int kMaxDevices = 64;
int num_sms();
// Device address of the library's fault word on the current device (NULL on failure).
int *fault_word();
// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` on the
// current device (once per kernel and device; thread-safe).  QB_OK or QB_E_CUDA.
int ensure_smem_limit(const void *kernel, int bytes);

}  // namespace qb
