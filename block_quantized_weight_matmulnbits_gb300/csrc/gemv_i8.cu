// Host side of the int8-activation path (kernels in gemv_i8.cuh).
#include "gemv_i8.cuh"

namespace mnb {
namespace gi8 {

// ---- 1. activation quantisation: one warp per (m, kb) ----
// Codes go to qa (int8, with the block scales to sa [M][KB]) or, for the
// prefill GEMM, to xq as code * s_a rounded to tf32 (f32 containers, the
// activation the GEMM's tf32 MMA multiplies); rows are Kpad long either way.
__global__ void __launch_bounds__(256) quant_act_kernel(const void* x, int dt, int8_t* qa, float* xq, float* sa,
                                                        int64_t M, Layout L) {
    // The previous kernel on the stream may have written x, or may still be
    // reading this workspace; no-op when not launched as a dependent.
    griddep_wait();
    griddep_launch_dependents();  // the next kernel may start streaming its weights
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= M * L.KB) return;
    const int64_t m = w / L.KB, kb = w - m * L.KB;
    const int64_t k0 = kb * L.bs;
    const int64_t k1 = imin64(k0 + L.bs, L.K);
    float amax = 0.f;
    for (int64_t k = k0 + lane; k < k1; k += 32) amax = fmaxf(amax, fabsf(load_f32(x, m * L.K + k, dt)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float s = __fdiv_rn(amax, 127.0f);
    if (sa && lane == 0) sa[m * L.KB + kb] = s;
    for (int64_t k = k0 + lane; k < k0 + L.bs; k += 32) {
        int code = 0;
        if (k < L.K && amax > 0.f) {
            const float r = roundf(__fdiv_rn(load_f32(x, m * L.K + k, dt), s));  // half away from zero
            code = (int)fminf(fmaxf(r, -127.f), 127.f);
        }
        if (xq) {
            uint32_t t;  // code * s_a, rounded to tf32 (nearest, ties away)
            asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(__fmul_rn((float)code, s)));
            xq[m * L.Kpad + k] = __uint_as_float(t);
        } else {
            qa[m * L.Kpad + k] = (int8_t)code;
        }
    }
}

}  // namespace gi8


cudaError_t launch_gemv_i8_b2(const MatmulParams& p, const gi8::Geom& geo, const int8_t* qa, const float* sa,
                              cudaStream_t s);
cudaError_t launch_gemv_i8_b4(const MatmulParams& p, const gi8::Geom& geo, const int8_t* qa, const float* sa,
                              cudaStream_t s);
cudaError_t launch_gemv_i8_b8(const MatmulParams& p, const gi8::Geom& geo, const int8_t* qa, const float* sa,
                              cudaStream_t s);

static gi8::Geom geom_for(const MatmulParams& p) { return gi8::make_geom(p.L, p.M, p.M == 1 ? 1 : 16); }

size_t i8_workspace_bytes(int64_t M, const Layout& L) { return gi8::workspace_bytes(M, L); }

bool gemv_i8_supported(const MatmulParams& p) {
    if (p.M < 1 || p.M > 16 || p.g_idx != nullptr) return false;
    const gi8::Geom g = geom_for(p);
    // K-splits must start on quantisation-block boundaries
    if (g.C > 1 && ((int64_t)g.tiles_cta * p.L.KT) % p.L.bs != 0) return false;
    return g.total_bytes <= device_info().smem_optin && p.L.NT * g.C <= 0x7FFFFFFF;
}

static cudaError_t quant_launch(const void* x, int act_dtype, int8_t* qa, float* xq, float* sa, int64_t M,
                                const Layout& L, bool pdl, cudaStream_t s) {
    const int64_t warps = M * L.KB;
    const int64_t blocks = (warps + 7) / 8;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gi8::quant_act_kernel, x, act_dtype, qa, xq, sa, M, L);
}

cudaError_t launch_quant_act(const void* x, int act_dtype, int8_t* qa, float* sa, int64_t M, const Layout& L,
                             cudaStream_t s) {
    return quant_launch(x, act_dtype, qa, nullptr, sa, M, L, false, s);
}

cudaError_t launch_quant_act_tf32(const void* x, int act_dtype, float* xq, int64_t M, const Layout& L, bool pdl,
                                  cudaStream_t s) {
    return quant_launch(x, act_dtype, nullptr, xq, nullptr, M, L, pdl, s);
}

cudaError_t launch_gemv_i8(const MatmulParams& p, cudaStream_t s) {
    const gi8::Geom geo = geom_for(p);
    if (geo.total_bytes > device_info().smem_optin) return cudaErrorNotSupported;
    int8_t* qa = static_cast<int8_t*>(p.workspace);
    float* sa = reinterpret_cast<float*>(static_cast<uint8_t*>(p.workspace) + gi8::qa_bytes(p.M, p.L));
    cudaError_t e = quant_launch(p.x, p.act_dtype, qa, nullptr, sa, p.M, p.L, (p.flags & kFlagPDL) != 0, s);
    if (e != cudaSuccess) return e;
    switch (p.L.bits) {
        case 2: return launch_gemv_i8_b2(p, geo, qa, sa, s);
        case 4: return launch_gemv_i8_b4(p, geo, qa, sa, s);
        case 8: return launch_gemv_i8_b8(p, geo, qa, sa, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
