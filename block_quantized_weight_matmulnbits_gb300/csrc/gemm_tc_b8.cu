// Instantiation of the tcgen05 prefill GEMM for 8-bit codes (one translation
// unit per code width keeps the build parallel).
#include "gemm_bs.cuh"
#include "gemm_hl.cuh"

namespace mnb {
cudaError_t launch_gemm_tc_b8(const MatmulParams& p, const gbs::Geom& geo, const gbs::Maps& m, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    return bf ? gbs::launch<8, true>(p, geo, m, s) : gbs::launch<8, false>(p, geo, m, s);
}
cudaError_t launch_gemm_a8_b8(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s) {
    return ghl::launch<8, true>(p, geo, m, s);
}
cudaError_t launch_gemm_hl_b8(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s) {
    return ghl::launch<8>(p, geo, m, s);
}
}  // namespace mnb
