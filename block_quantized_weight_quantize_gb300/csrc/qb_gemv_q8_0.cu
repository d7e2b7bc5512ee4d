// qb_gemv_q8_0.cu -- instantiation of the product kernel for one weight format
// (one translation unit per format so the three compile in parallel).
#include "qb_gemv.cuh"

namespace qb {
int launch_gemv_q8_0(const GemvArgs &a, cudaStream_t stream) { return launch_gemv_fmt<kQ8_0>(a, stream); }
int launch_matvec_q8_0(const GemvArgs &a, const float *x, cudaStream_t stream) {
    return launch_gemv2<kQ8_0>(a, stream, x);
}
}  // namespace qb
