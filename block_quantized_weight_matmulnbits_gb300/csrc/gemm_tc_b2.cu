// Instantiation of the tcgen05 prefill GEMM for 2-bit codes (one
// translation unit per code width keeps the build parallel).
#include "gemm_ta.cuh"

namespace mnb {
cudaError_t launch_gemm_tc_b2(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    return bf ? gtc::launch<2, true>(p, geo, m, s) : gtc::launch<2, false>(p, geo, m, s);
}
cudaError_t launch_gemm_ta_b2(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    return bf ? gtc::launch_ta<2, true>(p, geo, m, s) : gtc::launch_ta<2, false>(p, geo, m, s);
}
}  // namespace mnb
