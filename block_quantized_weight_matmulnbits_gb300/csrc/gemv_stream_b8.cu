// Instantiation of the streaming decode GEMV for 8-bit codes (one translation
// unit per code width keeps the build parallel).
#include "gemv_stream.cuh"

namespace mnb {
cudaError_t launch_gemv_stream_b8(const MatmulParams& p, const gstr::SGeom& geo, cudaStream_t s) {
    return gstr::launch_bits<8>(p, geo, s);
}
}  // namespace mnb
