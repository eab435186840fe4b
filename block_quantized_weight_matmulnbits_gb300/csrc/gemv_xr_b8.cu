// Instantiation of the register-X decode GEMV for 8-bit codes (one
// translation unit per code width keeps the build parallel).
#include "gemv_xr.cuh"

namespace mnb {
cudaError_t launch_gemv_xr_b8(const MatmulParams& p, const gxr::XGeom& geo, cudaStream_t s) {
    return gxr::launch_bits<8>(p, geo, s);
}
}  // namespace mnb
