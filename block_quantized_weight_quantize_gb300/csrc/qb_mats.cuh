// qb_mats.cuh -- device side of a matrix table (qb_launch.h: MatTable): the
// streaming kernels fill rows and write outputs through it, so several
// matrices that share an activation run as one launch.
#pragma once

#include "qb_common.cuh"
#include "qb_launch.h"

namespace qb {

// The table index of range row v (the last matrix starting at or before v).
__device__ __forceinline__ int mat_of(const MatTable &t, int64_t v) {
    int i = 0;
#pragma unroll
    for (int k = 1; k < kMaxMats; ++k) i = (k < t.n && v >= t.start[k]) ? k : i;
    return i;
}

// The record of range row v.
__device__ __forceinline__ const uint8_t *row_ptr(const MatTable &t, int64_t v, int64_t rec) {
    const int i = mat_of(t, v);
    return t.W[i] + (v - t.start[i]) * rec;
}

// Where column c of range row v goes.
__device__ __forceinline__ float *out_ptr(const MatTable &t, int c, int64_t v) {
    const int i = mat_of(t, v);
    return t.out[i] + (int64_t)c * (t.start[i + 1] - t.start[i]) + (v - t.start[i]);
}

// Bulk copies of range rows [v, v + n) into dst (rows back to back), one per
// matrix the rows fall in, all completing on bar.  Bytes: n * rec in total.
__device__ __forceinline__ void fill_rows(const MatTable &t, uint8_t *dst, int64_t v, int64_t n, int64_t rec,
                                          uint64_t *bar) {
#pragma unroll
    for (int i = 0; i < kMaxMats; ++i) {
        if (i >= t.n) break;
        const int64_t a = v > t.start[i] ? v : t.start[i];
        const int64_t b = (v + n) < t.start[i + 1] ? (v + n) : t.start[i + 1];
        if (a < b)
            bulk_g2s(dst + (a - v) * rec, t.W[i] + (a - t.start[i]) * rec, (uint32_t)((b - a) * rec), bar);
    }
}

}  // namespace qb
