// qb_gemv_q4k_hi.cu -- the product kernel for one weight format at 9..16
// activation columns (compiled apart from 1..8 to halve the build time).
#include "qb_gemv.cuh"

namespace qb {
template <>
int dispatch_hi<kQ4K>(int nc, const GemvK &k, int threads, int smem, unsigned grid, cudaStream_t s) {
    return dispatch_range<kQ4K, 9, 16>(nc, k, threads, smem, grid, s);
}
}  // namespace qb
