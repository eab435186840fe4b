// Decode GEMV for FP8 (E4M3 as the page decodes it, E5M2) and NVFP4 weights,
// 1 <= M <= 4, bf16 / f16 / f32-free X (bf16 or f16):
//   FP8:   Y[m, n] = s[n] * sum_k X[m, k] * fp8(W[k, n])
//   NVFP4: Y[m, n] = global * sum_kb e4m3(S[kb, n]) * sum_{k in kb} X[m, k] * e2m1(W[k, n])
// dequant_matmul_fp8 / dequant_matmul_nvfp4 of rlx-cpu 0.2.13,
// src/thunk/ops/quant.rs, with the scales factored out of the sums (one f32
// rounding per factor; within the library's per-element bound).
//
// Schedule: the K-chunk items of gemv_ks.cuh (one 16-warp CTA per SM, items
// of 4 packed tiles streamed into registers one item ahead, one fixed-order
// reduction per CTA).  Arithmetic on CUDA cores: every code is decoded by an
// exact table in shared memory built from the bit-field decoders of
// fp_formats.cuh, one copy per lane (so the 32 lanes of a lookup hit 32
// distinct banks), and multiplied into f32 accumulators.
//   * FP8: a 256-entry f32 table; 4 instructions per weight (byte select,
//     address, lookup, FMA).  The page's exponent-15 codes decode to infinity
//     or NaN exactly as the exact kernel does.
//   * NVFP4: a byte of the 4-bit tile holds the same depth of rows g and g + 8,
//     so a 256-entry table of f32 pairs decodes two weights per lookup.  The
//     E4M3 block scales of the CTA's rows are staged in shared memory
//     (transposed to [row][block]) and decoded by a 256-entry table.
#pragma once

#include "fp_formats.cuh"
#include "gemv_ks.cuh"

namespace mnb {
namespace gfp {

using gks::Cursor;
using gks::kThreads;
using gks::kTilesPerChunk;
using gks::kW;

struct FGeom {
    int G, KC, max_rt, xrow;
    int KB;                  // NVFP4 scale blocks (K / 16)
    size_t lut_bytes, slut_bytes, sc_bytes, x_bytes, red_bytes, total_bytes;
};

// FP8: 8-bit tiles, chunk of 8 k-steps (128 depths); NVFP4: 4-bit tiles,
// chunk of 16 k-steps (256 depths).  K a multiple of the chunk depth.
inline bool make_fgeom(int64_t N, int64_t K, int fmt, int64_t M, int sms, size_t smem_limit, FGeom* out) {
    if (M < 1 || M > 4) return false;
    const int64_t chunk_k = fmt == kWfNVFP4 ? 256 : 128;
    if (K % chunk_k != 0 || N < 1) return false;
    const int64_t NT = (N + 15) / 16;
    FGeom g{};
    g.KC = (int)(K / chunk_k);
    g.G = (int)(NT < sms ? NT : sms);
    g.max_rt = (int)((NT + g.G - 1) / g.G);
    if (g.max_rt > kThreads / 16) return false;
    g.xrow = (int)(K / 8) + 4;
    g.KB = (int)(K / 16);
    g.lut_bytes = fmt == kWfNVFP4 ? (size_t)256 * 32 * 8 : (size_t)256 * 32 * 4;
    g.slut_bytes = fmt == kWfNVFP4 ? 256 * 4 : 0;
    g.sc_bytes = fmt == kWfNVFP4 ? round16((size_t)g.max_rt * 16 * (g.KB + 16)) : 0;
    g.x_bytes = (size_t)M * g.xrow * 16;
    g.red_bytes = (size_t)g.max_rt * kW * 16 * M * 4;
    g.total_bytes = g.lut_bytes + g.slut_bytes + g.sc_bytes + g.x_bytes + g.red_bytes;
    if (g.total_bytes > smem_limit) return false;
    *out = g;
    return true;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 lds_f32x2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
// byte i of word, zero-extended
__device__ __forceinline__ uint32_t byte_of(uint32_t word, int i) { return prmt(word, 0u, 0x4440u | (uint32_t)i); }

template <bool BF16X>
__device__ __forceinline__ float x_lo(uint32_t v) {
    if constexpr (BF16X) return __uint_as_float(v << 16);
    else return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu)));
}
template <bool BF16X>
__device__ __forceinline__ float x_hi(uint32_t v) {
    if constexpr (BF16X) return __uint_as_float(v & 0xFFFF0000u);
    else return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

template <int FMT, bool BF16X, int MT>
__global__ void __launch_bounds__(kThreads, 1) gemv_fp_kernel(FpParams p, FGeom geo, int pdl) {
    constexpr bool NV = FMT == kWfNVFP4;
    constexpr int SPT = NV ? 4 : 2;            // k-steps per packed tile
    constexpr int CH = kTilesPerChunk * SPT;   // k-steps per chunk
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* lut = smem;                                       // [256][32 lanes] f32 (FP8) or f32x2 (NVFP4)
    float* slut = reinterpret_cast<float*>(smem + geo.lut_bytes);  // [256] block-scale values (NVFP4)
    uint8_t* sc_s = smem + geo.lut_bytes + geo.slut_bytes;    // [rows][KB + 16] block-scale codes (NVFP4)
    uint4* xs = reinterpret_cast<uint4*>(sc_s + geo.sc_bytes);  // [M][xrow] X in B-fragment order
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(xs) + geo.x_bytes);  // [max_rt][kW][16][M]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = MT == 1 ? 1 : (int)p.M;
    const int KC = geo.KC;
    const int64_t rt0 = (int64_t)blockIdx.x * L.NT / geo.G;
    const int nrt = (int)((int64_t)(blockIdx.x + 1) * L.NT / geo.G - rt0);
    const int n_items = nrt * KC;
    const uint8_t* wbase = p.packed + rt0 * L.KTILES * kTileBytes + lane * 16;

    // ---- 1. the first two items' weights (registers), then the tables ----
    uint4 wb[2][kTilesPerChunk];
    auto load = [&](uint4 (&w)[kTilesPerChunk], const Cursor& it) {
        if (it.i < n_items) {
            const uint8_t* src = wbase + (size_t)(uint32_t)it.i * (size_t)(kTilesPerChunk * kTileBytes);
#pragma unroll
            for (int j = 0; j < kTilesPerChunk; ++j) w[j] = ldg_stream(src + j * kTileBytes);
        }
    };
    const int q16 = kW / KC, r16 = kW % KC;
    Cursor cur{warp, warp / KC, warp % KC};
    Cursor nxt = cur;
    nxt.advance(KC, q16, r16);
    load(wb[0], cur);
    load(wb[1], nxt);
    for (int c = tid; c < 256; c += kThreads) {
        if constexpr (NV) {
            const float2 v = make_float2(fpf::e2m1((uint32_t)c & 15u), fpf::e2m1((uint32_t)c >> 4));
            for (int l = 0; l < 32; ++l) reinterpret_cast<float2*>(lut)[c * 32 + l] = v;
            slut[c] = fpf::e4m3fn((uint32_t)c);
        } else {
            const float v = FMT == kWfE5M2 ? fpf::e5m2((uint32_t)c) : fpf::e4m3_page((uint32_t)c);
            for (int l = 0; l < 32; ++l) reinterpret_cast<float*>(lut)[c * 32 + l] = v;
        }
    }
    const int rows_cta = nrt * 16;
    if constexpr (NV) {
        // block-scale codes of the CTA's rows, transposed to [row][block]; rows past N read row N - 1
        const uint8_t* S = static_cast<const uint8_t*>(p.scales);
        const int srow = geo.KB + 16;
        for (int kb = warp; kb < geo.KB; kb += kW) {
            for (int r = lane; r < rows_cta; r += 32) {
                int64_t n = rt0 * 16 + r;
                if (n >= L.N) n = L.N - 1;
                sc_s[r * srow + kb] = __ldg(S + (int64_t)kb * L.N + n);
            }
        }
    }
    for (int o = tid; o < nrt * kW * 16 * M; o += kThreads) red[o] = 0.f;
    if (pdl) {
        griddep_wait();               // X (and Y) may belong to the previous kernel on the stream
        griddep_launch_dependents();  // after the wait: at most two chained kernels overlap
    }
    {
        const uint32_t* x32 = static_cast<const uint32_t*>(p.x);  // K even: rows are 4-byte aligned
        const int64_t kw = L.K / 2;
        const int pairs = (int)(L.K / 32);
        for (int o = tid; o < M * pairs * 4; o += kThreads) {
            const int m = o / (pairs * 4), r = o - m * (pairs * 4);
            const uint32_t* src = x32 + m * kw + (r >> 2) * 16 + (r & 3);
            xs[(size_t)m * geo.xrow + r] = make_uint4(__ldg(src), __ldg(src + 4), __ldg(src + 8), __ldg(src + 12));
        }
    }
    __syncthreads();

    // ---- 2. items ----
    const uint32_t lut_lane = smem_u32(lut) + (uint32_t)lane * (NV ? 8u : 4u);
    const uint32_t slut_a = smem_u32(slut);
    const uint32_t xa_lane = smem_u32(xs + t);
    const uint32_t xrow_bytes = (uint32_t)geo.xrow * 16u;
    const uint32_t srow = (uint32_t)geo.KB + 16u;
    const uint32_t sc_g = smem_u32(sc_s) + (uint32_t)g * srow;
    float acc[2][MT];  // rows g, g + 8 x tokens (this lane's share of the depths)
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

    auto flush = [&](int rt_l) {
        float* dst = red + (size_t)(rt_l * kW + warp) * 16 * M;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float v = acc[r][m];
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);  // the 4 lanes of a row, fixed order
                v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
                if (t == 0 && m < M) dst[(g + 8 * r) * M + m] = v;
                acc[r][m] = 0.f;
            }
        }
    };

    auto compute = [&](const uint4 (&w)[kTilesPerChunk], const Cursor& it) {
        const uint32_t xa = xa_lane + (uint32_t)it.c * (uint32_t)(CH / 2) * 64u;
        uint32_t s0[4], s8[4];  // NVFP4: the chunk's 16 block-scale codes of rows g and g + 8
        if constexpr (NV) {
            const uint32_t sa = sc_g + (uint32_t)it.rt * 16u * srow + (uint32_t)it.c * 16u;
            const uint4 a = lds128(sa), b = lds128(sa + 8u * srow);
            s0[0] = a.x; s0[1] = a.y; s0[2] = a.z; s0[3] = a.w;
            s8[0] = b.x; s8[1] = b.y; s8[2] = b.z; s8[3] = b.w;
        }
        uint4 xv[MT];
#pragma unroll
        for (int s = 0; s < CH; ++s) {
            if ((s & 1) == 0) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < M) xv[m] = lds128(xa + (uint32_t)m * xrow_bytes + (uint32_t)(s >> 1) * 64u);
            }
            const uint4 wt = w[s / SPT];
            const uint32_t words[4] = {wt.x, wt.y, wt.z, wt.w};
            if constexpr (NV) {
                const uint32_t word = words[s % SPT];
                // byte i: (row g, row g + 8) at depth 2t (i = 0), 2t + 8 (1), 2t + 1 (2), 2t + 9 (3)
                const float2 p0 = lds_f32x2(lut_lane + byte_of(word, 0) * 256u);
                const float2 p1 = lds_f32x2(lut_lane + byte_of(word, 1) * 256u);
                const float2 p2 = lds_f32x2(lut_lane + byte_of(word, 2) * 256u);
                const float2 p3 = lds_f32x2(lut_lane + byte_of(word, 3) * 256u);
                const float sg = lds_f32(slut_a + byte_of(s0[s >> 2], s & 3) * 4u);
                const float sg8 = lds_f32(slut_a + byte_of(s8[s >> 2], s & 3) * 4u);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const uint32_t b0 = (s & 1) ? xv[m].z : xv[m].x, b1 = (s & 1) ? xv[m].w : xv[m].y;
                        const float x0 = x_lo<BF16X>(b0), x1 = x_hi<BF16X>(b0);
                        const float x2 = x_lo<BF16X>(b1), x3 = x_hi<BF16X>(b1);
                        float tg = x0 * p0.x;
                        tg = fmaf(x1, p2.x, tg);
                        tg = fmaf(x2, p1.x, tg);
                        tg = fmaf(x3, p3.x, tg);
                        float t8 = x0 * p0.y;
                        t8 = fmaf(x1, p2.y, t8);
                        t8 = fmaf(x2, p1.y, t8);
                        t8 = fmaf(x3, p3.y, t8);
                        acc[0][m] = fmaf(sg, tg, acc[0][m]);
                        acc[1][m] = fmaf(sg8, t8, acc[1][m]);
                    }
                }
            } else {
                // word 2ss: (row g: depths 2t, 2t+1; row g+8: 2t, 2t+1); word 2ss+1: the same at depths + 8
                const uint32_t wa = words[2 * (s % SPT)], wc = words[2 * (s % SPT) + 1];
                float v[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[i] = lds_f32(lut_lane + byte_of(wa, i) * 128u);
                    v[4 + i] = lds_f32(lut_lane + byte_of(wc, i) * 128u);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const uint32_t b0 = (s & 1) ? xv[m].z : xv[m].x, b1 = (s & 1) ? xv[m].w : xv[m].y;
                        const float x0 = x_lo<BF16X>(b0), x1 = x_hi<BF16X>(b0);
                        const float x2 = x_lo<BF16X>(b1), x3 = x_hi<BF16X>(b1);
                        float a0 = acc[0][m], a8 = acc[1][m];
                        a0 = fmaf(x0, v[0], a0);
                        a0 = fmaf(x1, v[1], a0);
                        a0 = fmaf(x2, v[4], a0);
                        a0 = fmaf(x3, v[5], a0);
                        a8 = fmaf(x0, v[2], a8);
                        a8 = fmaf(x1, v[3], a8);
                        a8 = fmaf(x2, v[6], a8);
                        a8 = fmaf(x3, v[7], a8);
                        acc[0][m] = a0;
                        acc[1][m] = a8;
                    }
                }
            }
        }
    };

    auto step = [&](uint4 (&w)[kTilesPerChunk]) {
        compute(w, cur);
        Cursor after = nxt;
        after.advance(KC, q16, r16);
        load(w, after);
        if (nxt.i >= n_items || nxt.rt != cur.rt) flush(cur.rt);
        cur = nxt;
        nxt = after;
        return cur.i < n_items;
    };
    if (cur.i < n_items) {
        while (step(wb[0]) && step(wb[1])) {
        }
    }
    __syncthreads();

    // ---- 3. rows: the 16 warps' partials in a fixed order, times the column / global scale ----
    for (int o = tid; o < nrt * 16 * M; o += kThreads) {
        const int rt_l = o / (16 * M), rem = o - rt_l * 16 * M;
        const int row = rem / M, m = rem - row * M;
        const float* src = red + (size_t)rt_l * kW * 16 * M + row * M + m;
        float v = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kW; ++w2) v += src[(size_t)w2 * 16 * M];
        const int64_t n = (rt0 + rt_l) * 16 + row;
        if (n < L.N) {
            if constexpr (NV) v *= p.global_scale;
            else if (p.scales) v *= __ldg(static_cast<const float*>(p.scales) + n);
            store_f32(p.y, (int64_t)m * L.N + n, v, p.out_dtype);
        }
    }
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status, p.fmt);
}

template <int FMT>
cudaError_t launch_fmt(const FpParams& p, const FGeom& geo, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    const int pdl = (p.flags & kFlagPDL) ? 1 : 0;
    auto go = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)geo.G);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = geo.total_bytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, kern, p, geo, pdl);
    };
    if (p.M == 1) return bf ? go(gemv_fp_kernel<FMT, true, 1>) : go(gemv_fp_kernel<FMT, false, 1>);
    return bf ? go(gemv_fp_kernel<FMT, true, 4>) : go(gemv_fp_kernel<FMT, false, 4>);
}

}  // namespace gfp
}  // namespace mnb
