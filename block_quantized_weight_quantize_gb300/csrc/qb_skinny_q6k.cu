// qb_skinny_q6k.cu -- the 2..16-column kernels for the Q6_K-like format (a
// translation unit of its own so the formats compile in parallel): the
// tensor-core (tcgen05) kernel from kTcMinCols columns, the warp-per-block
// kernel at 2..4 columns and K = 4096, the dp4a streaming kernel otherwise.
#include "qb_gemv.cuh"
#include "qb_gemv3.cuh"
#include "qb_gemv6.cuh"
#include "qb_gemv7.cuh"
#include "qb_tc.cuh"

namespace qb {
template <>
int launch_skinny<kQ6K>(const GemvArgs &a, cudaStream_t stream) {
    if (a.ncols >= kTcMinCols) {
        const int rt = launch_tc<kQ6K>(a, stream);
        if (rt != QB_E_ARG) return rt;
    }
    const int r7 = launch_gemv7_cols<kQ6K>(a, stream, nullptr);  // 2..4 columns at K = 4096
    if (r7 != QB_E_ARG) return r7;
    return launch_gemv3<kQ6K>(a, stream);
}
template <>
int launch_one_col3<kQ6K>(const GemvArgs &a, cudaStream_t stream, const float *x) {
    if (a.ncols > 1) return launch_gemv7_cols<kQ6K>(a, stream, x);  // 2..4 columns from x in one launch
    // K = 4096 and up to 64 rows a CTA: a warp per block, a lane per row, two
    // CTAs a SM (qb_gemv7.cuh); longer row ranges stream through rings
    const int r7 = launch_gemv7<kQ6K, 2, 4, false>(a, stream, x);
    if (r7 != QB_E_ARG) return r7;
    const int r6 = launch_gemv6<kQ6K>(a, stream, x);  // K = 4096 (qb_gemv6.cuh: which shapes)
    if (r6 != QB_E_ARG) return r6;
    return launch_gemv3_one<kQ6K>(a, stream, x);
}
}  // namespace qb
