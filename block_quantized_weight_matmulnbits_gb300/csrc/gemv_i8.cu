// Host side of the int8-activation path (kernels in gemv_i8.cuh).
#include "gemv_i8.cuh"
#include "gemv_ks.cuh"

namespace mnb {
namespace gi8 {

// ---- 1. activation quantisation: one warp per (m, kb) ----
// Codes to qa (int8, rows Kpad long, zero past K) and the block scales to
// sa [M][KB].
__global__ void __launch_bounds__(256) quant_act_kernel(const void* x, int dt, int8_t* qa, float* sa, int64_t M,
                                                        Layout L) {
    // The previous kernel on the stream may have written x, or may still be
    // reading this workspace; no-op when not launched as a dependent.
    griddep_wait();
    griddep_launch_dependents();  // the GEMV may start streaming its weights
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
    if (lane == 0) sa[m * L.KB + kb] = s;
    for (int64_t k = k0 + lane; k < k0 + L.bs; k += 32) {
        int code = 0;
        if (k < L.K && amax > 0.f) {
            const float r = roundf(__fdiv_rn(load_f32(x, m * L.K + k, dt), s));  // half away from zero
            code = (int)fminf(fmaxf(r, -127.f), 127.f);
        }
        qa[m * L.Kpad + k] = (int8_t)code;
    }
}

// The same quantisation for the decode GEMV on the bf16 K-chunk schedule:
// x' = code * s_a in f32, written as two bf16 rows, hi = RN(x') and
// lo = RN(x' - hi) (|x' - hi - lo| <= 2^-16 |x'|), rows 2m and 2m + 1 of xq
// [2M][Kpad] (zero past K).
__global__ void __launch_bounds__(256) quant_act_hilo_kernel(const void* x, int dt, uint16_t* xq, int64_t M,
                                                             Layout L) {
    griddep_wait();
    griddep_launch_dependents();
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
    for (int64_t k = k0 + lane; k < k0 + L.bs; k += 32) {
        int code = 0;
        if (k < L.K && amax > 0.f) {
            const float r = roundf(__fdiv_rn(load_f32(x, m * L.K + k, dt), s));  // half away from zero
            code = (int)fminf(fmaxf(r, -127.f), 127.f);
        }
        const float v = __fmul_rn((float)code, s);
        const __nv_bfloat16 hi = __float2bfloat16_rn(v);
        const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));  // v - hi is exact in f32
        xq[(2 * m) * L.Kpad + k] = __bfloat16_as_ushort(hi);
        xq[(2 * m + 1) * L.Kpad + k] = __bfloat16_as_ushort(lo);
    }
}

// The same quantisation for the prefill GEMM, 8 consecutive depths per lane
// (one 16-byte load of bf16 / f16 X where the row allows it), a block's
// bs / 8 lanes reducing its |x| max with shuffles: xq[m, k] = code * s_a
// rounded to tf32 (f32 containers, rows Kpad long, zero past K), the
// activation the GEMM's tf32 MMA multiplies.  Codes and scales are those of
// quant_act_kernel (same operations on the same values).
__global__ void __launch_bounds__(256) quant_act_tf32_kernel(const void* x, int dt, float* xq, int64_t M, Layout L) {
    griddep_wait();
    griddep_launch_dependents();
    // grid (lane blocks of a row, rows, row groups of 65535): no division for the lane's row and depth
    const int64_t m = (int64_t)blockIdx.z * 65535 + blockIdx.y;
    const int64_t k0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    const bool live = m < M && k0 < L.Kpad;  // lanes past the row still join the shuffles
    float v[8];
    const int64_t xrow = m * L.K;
    if (live && dt != kF32 && k0 + 8 <= L.K && (L.K & 7) == 0 &&
        (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + xrow + k0));
        const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (dt == kBF16) {
                v[2 * j] = __uint_as_float(wv[j] << 16);
                v[2 * j + 1] = __uint_as_float(wv[j] & 0xFFFF0000u);
            } else {
                v[2 * j] = __half2float(__ushort_as_half((unsigned short)(wv[j] & 0xFFFFu)));
                v[2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(wv[j] >> 16)));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (live && k0 + j < L.K) ? load_f32(x, xrow + k0 + j, dt) : 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
    // the block's lanes are aligned groups of bs / 8 (2 .. 32) lanes
    for (int o = 1; o < L.bs / 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (!live) return;
    const float s = __fdiv_rn(amax, 127.0f);
    float out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        int code = 0;
        if (k0 + j < L.K && amax > 0.f) {
            const float r = roundf(__fdiv_rn(v[j], s));  // half away from zero
            code = (int)fminf(fmaxf(r, -127.f), 127.f);
        }
        uint32_t t;  // code * s_a, rounded to tf32 (nearest, ties away)
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(t) : "f"(__fmul_rn((float)code, s)));
        out[j] = __uint_as_float(t);
    }
    float4* dst = reinterpret_cast<float4*>(xq + m * L.Kpad + k0);  // Kpad % 8 == 0, workspace 256-B aligned
    dst[0] = make_float4(out[0], out[1], out[2], out[3]);
    dst[1] = make_float4(out[4], out[5], out[6], out[7]);
}

}  // namespace gi8


cudaError_t launch_gemv_i8_b2(const MatmulParams& p, const gi8::Geom& geo, const int8_t* qa, const float* sa,
                              cudaStream_t s);
cudaError_t launch_gemv_i8_b4(const MatmulParams& p, const gi8::Geom& geo, const int8_t* qa, const float* sa,
                              cudaStream_t s);
cudaError_t launch_gemv_i8_b8(const MatmulParams& p, const gi8::Geom& geo, const int8_t* qa, const float* sa,
                              cudaStream_t s);
cudaError_t launch_gemv_ks_b2(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s, const gks::MoeKs* moe,
                              bool a8 = false);
cudaError_t launch_gemv_ks_b4(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s, const gks::MoeKs* moe,
                              bool a8 = false);
cudaError_t launch_gemv_ks_b8(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s, const gks::MoeKs* moe,
                              bool a8 = false);

static gi8::Geom geom_for(const MatmulParams& p) { return gi8::make_geom(p.L, p.M, p.M == 1 ? 1 : 16); }

// M <= 4 may run on the bf16 K-chunk schedule over hi / lo activation rows: [2M][Kpad] bf16.
static size_t hilo_bytes(int64_t M, const Layout& L) { return ((size_t)4 * M * (size_t)L.Kpad + 255) & ~size_t(255); }

size_t i8_workspace_bytes(int64_t M, const Layout& L) {
    const size_t a = gi8::workspace_bytes(M, L);
    const size_t b = M <= 4 ? hilo_bytes(M, L) : 0;
    return a > b ? a : b;
}

bool gemv_i8_supported(const MatmulParams& p) {
    if (p.M < 1 || p.M > 16 || p.g_idx != nullptr) return false;
    const gi8::Geom g = geom_for(p);
    // K-splits must start on quantisation-block boundaries
    if (g.C > 1 && ((int64_t)g.tiles_cta * p.L.KT) % p.L.bs != 0) return false;
    return g.total_bytes <= device_info().smem_optin && p.L.NT * g.C <= 0x7FFFFFFF;
}

// xq == nullptr: int8 codes and scales (warp per block); else tf32 activations (thread per block).
static cudaError_t quant_launch(const void* x, int act_dtype, int8_t* qa, float* xq, float* sa, int64_t M,
                                const Layout& L, bool pdl, cudaStream_t s) {
    // tf32: lanes of 8 depths, grid (blocks of 256 lanes along the row, rows): a block never straddles rows
    const int64_t row_blocks = (L.Kpad / 8 + 255) / 256;
    const int64_t blocks = xq ? row_blocks : (M * L.KB + 7) / 8;
    const int64_t ry = M < 65535 ? M : 65535, rz = (M + 65534) / 65535;
    if (blocks > 0x7FFFFFFF || rz > 65535) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = xq ? dim3((unsigned)row_blocks, (unsigned)ry, (unsigned)rz) : dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (xq) return cudaLaunchKernelEx(&cfg, gi8::quant_act_tf32_kernel, x, act_dtype, xq, M, L);
    return cudaLaunchKernelEx(&cfg, gi8::quant_act_kernel, x, act_dtype, qa, sa, M, L);
}

cudaError_t launch_quant_act(const void* x, int act_dtype, int8_t* qa, float* sa, int64_t M, const Layout& L,
                             cudaStream_t s) {
    return quant_launch(x, act_dtype, qa, nullptr, sa, M, L, false, s);
}

cudaError_t launch_quant_act_tf32(const void* x, int act_dtype, float* xq, int64_t M, const Layout& L, bool pdl,
                                  cudaStream_t s) {
    return quant_launch(x, act_dtype, nullptr, xq, nullptr, M, L, pdl, s);
}

// Accuracy level 4 with M <= 4: the quantised activations as hi + lo bf16 rows, then the bf16
// K-chunk decode GEMV over them with each token's two columns summed (exact up to 2^-16 of
// code * s_a per element, and f32 accumulation).  False when that schedule declines the shape.
static bool hilo_ok(const MatmulParams& p, gks::KGeom* kg) {
    const char* ev = std::getenv("MNB_A8_HILO");  // 0: always the int8 kernel (tests, tuning)
    if (p.M > 4 || (ev && ev[0] == '0')) return false;
    if ((reinterpret_cast<uintptr_t>(p.scales) & 15) != 0) return false;
    if (p.zp && (reinterpret_cast<uintptr_t>(p.zp) & 15) != 0) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    if (!gks::make_kgeom(p.L, 2 * p.M, sms, device_info().smem_optin, p.scale_dtype == kF32 ? 4 : 2, kg)) return false;
    kg->pairx = 1;
    return true;
}

cudaError_t launch_gemv_i8(const MatmulParams& p, cudaStream_t s) {
    gks::KGeom kg;
    if (hilo_ok(p, &kg)) {
        // one launch: the decode GEMV quantises X while staging it (block sizes 32 .. 256);
        // MNB_A8_HILO=2 takes the two-launch form below (the same bits, for tests)
        const char* ev = std::getenv("MNB_A8_HILO");
        const bool fused = !(ev && ev[0] == '2');
        MatmulParams f = p;
        f.M = 2 * p.M;  // hi / lo rows; X stays p.x in its own type
        cudaError_t e = cudaErrorNotSupported;
        if (fused) switch (p.L.bits) {
            case 2: e = launch_gemv_ks_b2(f, kg, s, nullptr, true); break;
            case 4: e = launch_gemv_ks_b4(f, kg, s, nullptr, true); break;
            case 8: e = launch_gemv_ks_b8(f, kg, s, nullptr, true); break;
            default: return cudaErrorInvalidValue;
        }
        if (e != cudaErrorNotSupported) return e;
        cudaGetLastError();
        // otherwise the quantised rows through the workspace, then the GEMV over them
        uint16_t* xq = static_cast<uint16_t*>(p.workspace);
        cudaLaunchConfig_t cfg = {};
        const int64_t blocks = (p.M * p.L.KB + 7) / 8;
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = (p.flags & kFlagPDL) ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, gi8::quant_act_hilo_kernel, p.x, p.act_dtype, xq, p.M, p.L);
        if (e != cudaSuccess) return e;
        MatmulParams q = p;
        q.x = xq;
        q.act_dtype = kBF16;
        q.M = 2 * p.M;
        switch (p.L.bits) {
            case 2: e = launch_gemv_ks_b2(q, kg, s, nullptr); break;
            case 4: e = launch_gemv_ks_b4(q, kg, s, nullptr); break;
            case 8: e = launch_gemv_ks_b8(q, kg, s, nullptr); break;
            default: return cudaErrorInvalidValue;
        }
        if (e != cudaErrorNotSupported) return e;
        cudaGetLastError();  // not instantiated for this block size and scale type: the int8 kernel below
    }
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
