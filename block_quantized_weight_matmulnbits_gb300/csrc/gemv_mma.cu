// Host side of the small-batch tensor-core GEMV (kernel in gemv_mma.cuh).
#include "gemv_mma.cuh"

namespace mnb {

cudaError_t launch_gemv_mma_b2(const MatmulParams& p, const gmma::Geom& geo, cudaStream_t s);
cudaError_t launch_gemv_mma_b4(const MatmulParams& p, const gmma::Geom& geo, cudaStream_t s);
cudaError_t launch_gemv_mma_b8(const MatmulParams& p, const gmma::Geom& geo, cudaStream_t s);

static gmma::Geom geom_for(const MatmulParams& p) {
    return gmma::make_geom(p.L, p.M, p.M <= 8 ? 8 : 16);
}

bool gemv_mma_supported(const MatmulParams& p) {
    if (p.M < 1 || p.M > 16 || p.g_idx != nullptr) return false;
    if (p.act_dtype != kBF16 && p.act_dtype != kF16) return false;
    const gmma::Geom g = geom_for(p);
    // K-splits must start on quantisation-block boundaries
    if (g.C > 1 && ((int64_t)g.tiles_cta * p.L.KT) % p.L.bs != 0) return false;
    return g.total_bytes <= device_info().smem_optin && p.L.NT * g.C <= 0x7FFFFFFF;
}

cudaError_t launch_gemv_mma(const MatmulParams& p, cudaStream_t s) {
    const gmma::Geom geo = geom_for(p);
    if (geo.total_bytes > device_info().smem_optin) return cudaErrorNotSupported;
    switch (p.L.bits) {
        case 2: return launch_gemv_mma_b2(p, geo, s);
        case 4: return launch_gemv_mma_b4(p, geo, s);
        case 8: return launch_gemv_mma_b8(p, geo, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
