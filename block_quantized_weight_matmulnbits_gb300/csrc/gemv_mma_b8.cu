// Instantiation of the small-batch tensor-core GEMV for 8-bit codes (one
// translation unit per code width keeps the build parallel).
#include "gemv_pers.cuh"

namespace mnb {
cudaError_t launch_gemv_mma_b8(const MatmulParams& p, const gmma::Geom& geo, cudaStream_t s) {
    return gmma::launch_bits<8>(p, geo, s);
}
cudaError_t launch_gemv_pers_b8(const MatmulParams& p, const gpers::PGeom& geo, int grid, cudaStream_t s) {
    return gpers::launch_bits<8>(p, geo, grid, s);
}
}  // namespace mnb
