// Instantiation of the streaming decode GEMV for 4-bit codes (one translation
// unit per code width keeps the build parallel).
#include "gemv_stream.cuh"

namespace mnb {
cudaError_t launch_gemv_stream_b4(const MatmulParams& p, const gstr::SGeom& geo, cudaStream_t s) {
    return gstr::launch_bits<4>(p, geo, s);
}
}  // namespace mnb
