// Generic CUDA-core kernel: any M, any activation / scale / output dtype,
// optional g_idx and bias.  It is the correctness baseline of the library and
// the path for shapes the specialised kernels do not take (f32 activations
// with M > 1, g_idx, act-order packs outside the decode GEMV's shapes).  Weights are dequantised into shared memory tile by tile
// as w = (f32(q) - f32(zp)) * f32(scale) (onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs, fn dequantize_nbits_value; with g_idx the
// scale and zero point follow g_idx[k] while the code keeps its block
// position, MatMulNBitsKernel::dequantize_weight), then contracted with fp32
// FMAs.  The bias is added after the product (MatMulNBitsKernel::execute).
//
// g_idx values outside [0, KB) are an error on the page (dequantize_weight
// rejects them).  Here g_idx lives on the device, so the kernel checks each
// value before using it: a bad value is never used as an index, the CTA that
// met it writes none of its outputs, and the device status word becomes
// MNB_ERR_INVALID_ARG.  Every output depends on every depth, so every CTA
// meets the bad value and Y is left entirely unwritten.
#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int TN = 64;   // weight rows per CTA
constexpr int TM = 16;   // activation rows per CTA
constexpr int TK = 32;   // depth per step

__global__ __launch_bounds__(256) void generic_kernel(MatmulParams p) {
    __shared__ float ws[TN][TK + 1];
    __shared__ float xs[TM][TK + 1];
    __shared__ int bad_gidx;
    const Layout& L = p.L;
    const int tid = threadIdx.x;
    const int64_t n0 = (int64_t)blockIdx.x * TN;
    const int64_t m0 = (int64_t)blockIdx.y * TM;
    const int nl = tid % TN;        // this thread's row of W
    const int mg = tid / TN;        // 0..3 -> activation rows mg*4 .. mg*4+3
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int mask = code_mask(L.bits);
    if (tid == 0) bad_gidx = 0;
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) verify_header(p.packed_hdr, L, p.status, kWfInt, p.kperm != nullptr);
    __syncthreads();

    for (int64_t k0 = 0; k0 < L.K; k0 += TK) {
        for (int i = tid; i < TN * TK; i += 256) {
            const int r = i / TK, c = i % TK;
            const int64_t n = n0 + r, k = k0 + c;
            float w = 0.f;
            if (n < L.N && k < L.K) {
                const int64_t bit = L.bit_of(n, k);
                const int q = (p.packed[bit >> 3] >> (bit & 7)) & mask;
                // act-order pack: stored depth k is in group k / bs (its X depth is kperm[k], below)
                const int64_t g = p.g_idx ? (int64_t)p.g_idx[k] : k / L.bs;
                if (g >= 0 && g < L.KB) {
                    const int z = load_zp(p.zp, L, n, g);
                    const float s = load_f32(p.scales, n * L.KB + g, p.scale_dtype);
                    w = __fmul_rn(__fsub_rn((float)q, (float)z), s);
                } else {
                    bad_gidx = 1;  // never used as an index
                }
            }
            ws[r][c] = w;
        }
        for (int i = tid; i < TM * TK; i += 256) {
            const int r = i / TK, c = i % TK;
            const int64_t m = m0 + r, k = k0 + c;
            int64_t kx = k;
            if (p.kperm != nullptr && k < L.K) {
                const int64_t v = p.kperm[k];
                kx = v < 0 ? 0 : (v >= L.K ? L.K - 1 : v);  // a bad pack's permutation never indexes past X
            }
            xs[r][c] = (m < p.M && k < L.K) ? load_f32(p.x, m * L.K + kx, p.act_dtype) : 0.f;
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
    // bad_gidx was written before the loop's last barrier
    if (bad_gidx) {
        if (tid == 0) set_status(p.status, 1 /* MNB_ERR_INVALID_ARG */);
        return;
    }
    const int64_t n = n0 + nl;
    if (n >= L.N) return;
    const float b = p.bias ? load_f32(p.bias, n, p.bias_dtype) : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t m = m0 + mg * 4 + j;
        if (m < p.M) store_f32(p.y, m * L.N + n, acc[j] + b, p.out_dtype);
    }
}

}  // namespace

cudaError_t launch_generic(const MatmulParams& p, cudaStream_t s) {
    const int64_t gx = (p.L.N + TN - 1) / TN;
    const int64_t gy = (p.M + TM - 1) / TM;
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    generic_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace mnb
