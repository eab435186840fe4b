// Instantiation of the tcgen05 prefill GEMM for 8-bit codes (one
// translation unit per code width keeps the build parallel).
#include "gemm_ta.cuh"

namespace mnb {
cudaError_t launch_gemm_tc_b8(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    return bf ? gtc::launch<8, true>(p, geo, m, s) : gtc::launch<8, false>(p, geo, m, s);
}
cudaError_t launch_gemm_ta_b8(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    return bf ? gtc::launch_ta<8, true>(p, geo, m, s) : gtc::launch_ta<8, false>(p, geo, m, s);
}
}  // namespace mnb
