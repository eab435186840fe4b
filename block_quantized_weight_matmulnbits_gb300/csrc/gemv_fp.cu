// Host side of the FP8 / NVFP4 decode GEMV (gemv_fp.cuh).
#include <cstdlib>
#include <cstring>

#include "gemv_fp.cuh"

namespace mnb {

static bool fp_geom(const FpParams& p, gfp::FGeom* g) {
    if (p.act_dtype != kBF16 && p.act_dtype != kF16) return false;
    const char* e = std::getenv("MNB_FP_KERNEL");
    if (e && std::strcmp(e, "generic") == 0) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    return gfp::make_fgeom(p.L.N, p.L.K, p.fmt, p.M, sms, device_info().smem_optin, g);
}

bool gemv_fp_supported(const FpParams& p) {
    gfp::FGeom g;
    return fp_geom(p, &g);
}

cudaError_t launch_gemv_fp(const FpParams& p, cudaStream_t s) {
    gfp::FGeom g;
    if (!fp_geom(p, &g)) return cudaErrorNotSupported;
    switch (p.fmt) {
        case kWfE4M3: return gfp::launch_fmt<kWfE4M3>(p, g, s);
        case kWfE5M2: return gfp::launch_fmt<kWfE5M2>(p, g, s);
        case kWfNVFP4: return gfp::launch_fmt<kWfNVFP4>(p, g, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
