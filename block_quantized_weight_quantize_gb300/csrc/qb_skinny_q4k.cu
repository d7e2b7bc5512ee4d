// qb_skinny_q4k.cu -- the 2..16-column kernels for the Q4_K-like format (a
// translation unit of its own so the formats compile in parallel): the
// tensor-core (tcgen05) kernel from kTcMinCols columns, the warp-per-block
// kernel at 2..4 columns and K = 4096, the dp4a streaming kernel otherwise;
// and the one-column forms (qb_gemv7.cuh, qb_gemv6.cuh, qb_gemv3.cuh) where
// they apply.
#include "qb_gemv.cuh"
#include "qb_gemv3.cuh"
#include "qb_gemv6.cuh"
#include "qb_gemv7.cuh"
#include "qb_tc.cuh"

namespace qb {
template <>
int launch_skinny<kQ4K>(const GemvArgs &a, cudaStream_t stream) {
    if (a.ncols >= kTcMinCols) {
        const int rt = launch_tc<kQ4K>(a, stream);
        if (rt != QB_E_ARG) return rt;
    }
    const int r7 = launch_gemv7_cols<kQ4K>(a, stream, nullptr);  // 2..4 columns at K = 4096
    if (r7 != QB_E_ARG) return r7;
    return launch_gemv3<kQ4K>(a, stream);
}
template <>
int launch_one_col3<kQ4K>(const GemvArgs &a, cudaStream_t stream, const float *x) {
    if (a.ncols > 1) return launch_gemv7_cols<kQ4K>(a, stream, x);  // 2..4 columns from x in one launch
    // K = 4096 (qb_gemv7.cuh): up to 32 rows a CTA with each lane's block held
    // in registers before the dependency wait, up to 64 rows from shared
    // memory; two CTAs a SM.  Longer row ranges stream through rings.
    int r7 = launch_gemv7<kQ4K, 2, 8, true>(a, stream, x);
    if (r7 == QB_E_ARG) r7 = launch_gemv7<kQ4K, 2, 2, false>(a, stream, x);
    if (r7 != QB_E_ARG) return r7;
    const int r6 = launch_gemv6<kQ4K>(a, stream, x);  // K = 4096 (qb_gemv6.cuh: which shapes)
    if (r6 != QB_E_ARG) return r6;
    return launch_gemv3_one<kQ4K>(a, stream, x);
}
}  // namespace qb
