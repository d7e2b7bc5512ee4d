// qb_gemv_q4k.cu -- instantiation of the product kernel for one weight format
// (one translation unit per format so the three compile in parallel).
#include "qb_gemv.cuh"

namespace qb {
int launch_gemv_q4k(const GemvArgs &a, cudaStream_t stream) { return launch_gemv_fmt<kQ4K>(a, stream); }
int launch_matvec_q4k(const GemvArgs &a, const float *x, cudaStream_t stream) {
    const int rc = launch_one_col3<kQ4K>(a, stream, x);
    return rc != QB_E_ARG ? rc : launch_gemv2<kQ4K>(a, stream, x);
}
}  // namespace qb
