// Instantiation of the int8-activation GEMV for 4-bit codes (one translation
// unit per code width keeps the build parallel).
#include "gemv_i8.cuh"

namespace mnb {
cudaError_t launch_gemv_i8_b4(const MatmulParams& p, const gi8::Geom& geo, const int8_t* qa, const float* sa,
                              cudaStream_t s) {
    return gi8::launch_bits<4>(p, geo, qa, sa, s);
}
}  // namespace mnb
