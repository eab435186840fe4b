// Instantiation of the grouped (mixture-of-experts) GEMV for 2-bit codes
// (one translation unit per code width keeps the build parallel).
#include "gemv_moe.cuh"

namespace mnb {
cudaError_t launch_gemv_moe_b2(const MatmulParams& p, const gmma::Geom& geo, const gmoe::MoeArgs& g,
                               unsigned groups, size_t smem_bytes, cudaStream_t s) {
    return gmoe::launch_bits<2>(p, geo, g, groups, smem_bytes, s);
}
}  // namespace mnb
