// FP8 / NVFP4 weight matmul on CUDA cores, any M:
//   y[m, n] = sum_k x[m, k] * w(k, n)   (+ bias: none on the pages' ops)
//   FP8:   w(k, n) = fp8(code) * s[n]  (s = 1 when no per-column scale is given)
//   NVFP4: w(k, n) = fl32(fl32(e2m1(code) * e4m3(scale8[k / 16][n])) * global_scale)
// which is rlx-cpu 0.2.13, src/thunk/ops/quant.rs, dequant_matmul_fp8 and
// dequant_matmul_nvfp4 (weights [K, N]; re-tiled by mnb_pack_fp_weights into
// the library's packed layout, codes unchanged).  Each weight is decoded
// exactly (fp_formats.cuh) and formed in f32 in the page's order; the
// products are accumulated in f32.  Tiles of 64 weight rows x 16 activation
// rows x 32 depths in shared memory.
#include "fp_formats.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int TN = 64, TM = 16, TK = 32;

__global__ __launch_bounds__(256) void fp_generic_kernel(FpParams p) {
    __shared__ float ws[TN][TK + 1];
    __shared__ float xs[TM][TK + 1];
    const Layout& L = p.L;
    const int tid = threadIdx.x;
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) verify_header(p.packed_hdr, L, p.status, p.fmt);
    const int64_t n0 = (int64_t)blockIdx.x * TN, m0 = (int64_t)blockIdx.y * TM;
    const int nl = tid % TN, mg = tid / TN;
    const int mask = code_mask(L.bits);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t k0 = 0; k0 < L.K; k0 += TK) {
        for (int i = tid; i < TN * TK; i += 256) {
            const int r = i / TK, c = i % TK;
            const int64_t n = n0 + r, k = k0 + c;
            float w = 0.f;
            if (n < L.N && k < L.K) {
                const int64_t bit = L.bit_of(n, k);
                const uint32_t code = (p.packed[bit >> 3] >> (bit & 7)) & mask;
                if (p.fmt == kWfNVFP4) {
                    const uint32_t s8 = __ldg(static_cast<const uint8_t*>(p.scales) + (k >> 4) * L.N + n);
                    const float a = __fmul_rn(fpf::e2m1(code), fpf::e4m3fn(s8));
                    w = __fmul_rn(a, p.global_scale);
                } else {
                    const float v = p.fmt == kWfE5M2 ? fpf::e5m2(code) : fpf::e4m3_page(code);
                    w = p.scales ? __fmul_rn(v, __ldg(static_cast<const float*>(p.scales) + n)) : v;
                }
            }
            ws[r][c] = w;
        }
        for (int i = tid; i < TM * TK; i += 256) {
            const int r = i / TK, c = i % TK;
            const int64_t m = m0 + r, k = k0 + c;
            xs[r][c] = (m < p.M && k < L.K) ? load_f32(p.x, m * L.K + k, p.act_dtype) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < TK; ++c) {
            const float w = ws[nl][c];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(xs[mg * 4 + j][c], w, acc[j]);
        }
        __syncthreads();
    }
    const int64_t n = n0 + nl;
    if (n >= L.N) return;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t m = m0 + mg * 4 + j;
        if (m < p.M) store_f32(p.y, m * L.N + n, acc[j], p.out_dtype);
    }
}

}  // namespace

cudaError_t launch_fp_generic(const FpParams& p, cudaStream_t s) {
    const int64_t gx = (p.L.N + TN - 1) / TN;
    const int64_t gy = (p.M + TM - 1) / TM;
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    fp_generic_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mnb
