// Host side of the FP8 / NVFP4 decode GEMVs: gemv_nv.cuh (NVFP4 on the tensor
// cores, the default) and gemv_fp.cuh (decode tables on the CUDA cores: FP8,
// and NVFP4 shapes the first declines or MNB_FP_KERNEL=lut).
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "gemv_fp.cuh"
#include "gemv_nv.cuh"

namespace mnb {

static bool nv_geom(const FpParams& p, gnv::NGeom* g) {
    if (p.fmt != kWfNVFP4 || (p.act_dtype != kBF16 && p.act_dtype != kF16)) return false;
    const char* e = std::getenv("MNB_FP_KERNEL");
    if (e && (std::strcmp(e, "generic") == 0 || std::strcmp(e, "lut") == 0)) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    const bool svec = p.L.N % 16 == 0 && (reinterpret_cast<uintptr_t>(p.scales) & 15u) == 0;
    return gnv::make_ngeom(p.L, p.M, sms, device_info().smem_optin, svec, g);
}

bool gemv_nv_selected(const FpParams& p) {
    gnv::NGeom g;
    return nv_geom(p, &g);
}

static bool fp_geom(const FpParams& p, gfp::FGeom* g) {
    if (p.act_dtype != kBF16 && p.act_dtype != kF16) return false;
    const char* e = std::getenv("MNB_FP_KERNEL");
    if (e && std::strcmp(e, "generic") == 0) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    return gfp::make_fgeom(p.L.N, p.L.K, p.fmt, p.M, sms, device_info().smem_optin, g);
}

bool gemv_fp_supported(const FpParams& p) {
    gfp::FGeom g;
    return gemv_nv_selected(p) || fp_geom(p, &g);
}

cudaError_t launch_gemv_fp(const FpParams& p, cudaStream_t s) {
    gnv::NGeom ng;
    if (nv_geom(p, &ng)) return gnv::launch(p, ng, s);
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
