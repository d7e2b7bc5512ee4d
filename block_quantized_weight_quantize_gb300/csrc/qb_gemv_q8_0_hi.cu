// qb_gemv_q8_0_hi.cu -- the product kernel for one weight format at 9..16
// activation columns (compiled apart from 1..8 to halve the build time).
#include "qb_gemv.cuh"

namespace qb {
template <>
int dispatch_hi<kQ8_0>(int nc, const GemvK &k, int threads, int smem, unsigned grid, cudaStream_t s) {
    return dispatch_range<kQ8_0, 9, 16>(nc, k, threads, smem, grid, s);
}
}  // namespace qb
