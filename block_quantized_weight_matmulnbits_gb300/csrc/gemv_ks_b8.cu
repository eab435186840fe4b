// Instantiation of the k-chunk decode GEMV (gemv_ks.cuh) for 8-bit codes.
#include "gemv_ks.cuh"

namespace mnb {
cudaError_t launch_gemv_ks_b8(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s,
                             const gks::MoeKs* moe, bool a8) {
    return gks::launch_bits<8>(p, geo, s, moe, a8);
}
}  // namespace mnb
