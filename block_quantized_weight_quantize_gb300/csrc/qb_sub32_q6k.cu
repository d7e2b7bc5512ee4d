// qb_sub32_q6k.cu -- the ActScaling::Sub32 product for one weight format (a
// translation unit of its own so the formats compile in parallel).
#include "qb_sub32.cuh"

namespace qb {
int launch_gemv_sub32_q6k(const GemvArgs &a, cudaStream_t stream) { return launch_gemv_sub32<kQ6K>(a, stream); }
int launch_matvec_sub32_q6k(const GemvArgs &a, const float *x, cudaStream_t stream) {
    return launch_matvec_sub32<kQ6K>(a, x, stream);
}
}  // namespace qb
