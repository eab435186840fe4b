// Decode GEMV for NVFP4 weights on the tensor cores, 1 <= M <= 4, bf16 or f16 X:
//   Y[m, n] = global * sum_kb e4m3(S[kb, n]) * sum_{k in kb} X[m, k] * e2m1(W[k, n])
// dequant_matmul_nvfp4 of rlx-cpu 0.2.13, src/thunk/ops/quant.rs, with the
// block scale and the global scale factored out of the sums (the page's first
// rounding, f32(e2m1 * e4m3), is exact: a 2-bit by 4-bit significand product).
//
// A scale block is 16 deep, one mma.sync m16n8k16 k-step.  The schedule is the
// K-chunk one of gemv_ks.cuh (one 16-warp CTA per SM over a contiguous range
// of 16-row tiles, items of 4 packed tiles streamed into registers one item
// ahead, partial sums per row tile in registers, one fixed-order reduction).
//
// Codes to the A fragment, exactly and without tables.  The 4-bit packed tile
// is the int4 one: register r of a k-step's fragment holds nibbles r (low
// half) and r + 4 (high half) of the lane's word, each nibble E2M1 bits
// (m, e0, e1, s) from bit 0.  The two magnitude fields are moved to the two
// low exponent bits and the top mantissa bit of the activation type (bits 6-8
// of bf16, 9-11 of f16, in each half) and the result is multiplied by a
// packed +-2^(bias - 1), the sign taken from the code: a field with e >= 1
// reads 2^(e - bias) (1 + m / 2) and one with e = 0 is the subnormal
// m * 2^(1 - bias) / 2, so the product is the E2M1 value, exactly (the
// packed multiply keeps subnormal operands).  Per k-step: 4 magnitude shifts
// and masks, 3 sign shifts and 4 sign merges, 4 packed multiplies.
//
// Block scales: the CTA's E4M3 scale codes are read once, decoded to f32
// (OCP E4M3 by the hardware conversion to f16, exact) and staged in shared
// memory as [row tile][block][g][row g, row g + 8]: one 8-byte load per lane
// per k-step gives the scales of both of its rows.
#pragma once

#include "gemv_ks.cuh"

namespace mnb {
namespace gnv {

using gks::Cursor;
using gks::kItemBytes;
using gks::kThreads;
using gks::kTilesPerChunk;
using gks::kW;
using gmma::mma16816;

constexpr int kCH = kTilesPerChunk * 4;  // k-steps per chunk (4-bit codes: 4 per packed tile)

struct NGeom {
    int G;         // CTAs
    int KC;        // K-chunks per row tile
    int q16, r16;  // a step of kW items: q16 row tiles and r16 chunks
    int max_rt;    // most row tiles of one CTA
    int xrow;      // X row stride in 16-byte units
    int KB;        // scale blocks (K / 16)
    int svec;      // 1: scale rows read 16 codes at a time (N % 16 == 0, 16-byte aligned scales)
    size_t x_bytes, sc_bytes, red_bytes, total_bytes;
};

// The shapes this kernel takes: K a multiple of the chunk depth (256), M <= 4,
// the CTA's X, f32 block scales and partials in shared memory, offsets in 32 bits.
inline bool make_ngeom(const Layout& L, int64_t M, int sms, size_t smem_limit, bool svec, NGeom* out) {
    if (M < 1 || M > 4 || L.bits != 4 || L.bs != 16) return false;
    const int64_t chunk_k = (int64_t)kCH * 16;
    if (L.K % chunk_k != 0 || L.N < 1) return false;
    NGeom g{};
    g.KC = (int)(L.K / chunk_k);
    g.G = (int)(L.NT < sms ? L.NT : sms);
    g.max_rt = (int)((L.NT + g.G - 1) / g.G);
    if ((uint64_t)L.NT * (uint64_t)(g.G + 1) >= (1ull << 31)) return false;
    if ((uint64_t)g.max_rt * (uint64_t)g.KC * (uint64_t)kItemBytes >= (1ull << 31)) return false;
    g.q16 = kW / g.KC;
    g.r16 = kW % g.KC;
    g.xrow = (int)(L.K / 8) + 4;
    g.KB = (int)(L.K / 16);
    g.svec = svec ? 1 : 0;
    g.x_bytes = (size_t)(M + 1) * g.xrow * 16;
    g.sc_bytes = (size_t)g.max_rt * g.KB * 64;
    g.red_bytes = (size_t)g.max_rt * kW * 16 * M * 4;
    g.total_bytes = g.x_bytes + g.sc_bytes + g.red_bytes;
    if (g.total_bytes > smem_limit || g.sc_bytes >= (1ull << 31)) return false;
    *out = g;
    return true;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 lds64f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// Two OCP E4M3 codes (low byte, high byte) to f32, through the exact
// hardware conversion to an f16 pair.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t lo, uint32_t hi) {
    const unsigned short pair = (unsigned short)((lo & 0xFFu) | ((hi & 0xFFu) << 8));
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(pair));
    const __half h0 = __ushort_as_half((unsigned short)(h & 0xFFFFu));
    const __half h1 = __ushort_as_half((unsigned short)(h >> 16));
    return make_float2(__half2float(h0), __half2float(h1));
}

template <bool BF16X>
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (BF16X) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The A fragment of one k-step from the lane's word of 8 codes (see the top).
template <bool BF16X>
__device__ __forceinline__ void kstep_a(uint32_t w, uint32_t (&a)[4]) {
    constexpr int kMant = BF16X ? 6 : 9;                              // bit of the top mantissa bit
    constexpr uint32_t kMagMask = BF16X ? 0x01C001C0u : 0x0E000E00u;  // e1 e0 m in each half
    constexpr uint32_t kPow = BF16X ? 0x7E807E80u : 0x74007400u;      // 2^126 (bf16) / 2^14 (f16) pairs
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int ms = kMant - 4 * r;  // left shift of nibble r's magnitude bits
        const uint32_t mag = (ms >= 0 ? (w << ms) : (w >> -ms)) & kMagMask;
        const uint32_t sgn = lop3_and_or(w << (12 - 4 * r), 0x80008000u, kPow);  // sign bit 4r + 3 to bit 15
        a[r] = hmul2<BF16X>(mag, sgn);
    }
}

template <bool BF16X, bool M1>
__global__ void __launch_bounds__(kThreads, 1) gemv_nv_kernel(FpParams p, NGeom geo, int pdl) {
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint4* xs = reinterpret_cast<uint4*>(smem);                                 // [M + 1][xrow]: row M is zeros
    float* sc = reinterpret_cast<float*>(smem + geo.x_bytes);                  // [max_rt][KB][8 g][2]
    float* red = reinterpret_cast<float*>(smem + geo.x_bytes + geo.sc_bytes);  // [max_rt][kW][M][16 rows]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = M1 ? 1 : (int)p.M;
    const int KC = geo.KC, KB = geo.KB;
    const uint32_t NT32 = (uint32_t)L.NT;
    const int rt0 = (int)(blockIdx.x * NT32 / (uint32_t)geo.G);
    const int nrt = (int)((blockIdx.x + 1) * NT32 / (uint32_t)geo.G - (uint32_t)rt0);
    const int n_items = nrt * KC;
    const uint8_t* wbase = p.packed + (size_t)rt0 * (size_t)L.KTILES * kTileBytes + lane * 16;

    // ---- 1. the first item's weights, the block scales, X, the second item ----
    uint4 wb[2][kTilesPerChunk];
    auto load = [&](uint4 (&w)[kTilesPerChunk], const Cursor& it) {
        if (it.i < n_items) {
            const uint8_t* src = wbase + (uint32_t)it.i * (uint32_t)kItemBytes;
#pragma unroll
            for (int j = 0; j < kTilesPerChunk; ++j) w[j] = ldg_stream(src + j * kTileBytes);
        }
    };
    Cursor cur{warp, warp / KC, warp % KC};
    Cursor nxt = cur;
    nxt.advance(KC, geo.q16, geo.r16);
    load(wb[0], cur);

    const uint8_t* S = static_cast<const uint8_t*>(p.scales);
    if (geo.svec) {
        // unit o = (block kb, local row tile): the 16 codes of the row tile's rows at block kb,
        // one 16-byte load; four units per thread in flight
        const int units = nrt * KB;
        const float inv_nrt = 1.f / (float)nrt;
        for (int base = 0; base < units; base += 4 * kThreads) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int o = base + u * kThreads + tid;
                if (o < units) {
                    const int kb = __float2int_rz(((float)o + 0.5f) * inv_nrt);  // o < 2^22: exact
                    const int rl = o - kb * nrt;
                    v[u] = __ldg(reinterpret_cast<const uint4*>(S + (size_t)kb * (size_t)L.N +
                                                                (size_t)(rt0 + rl) * 16));
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int o = base + u * kThreads + tid;
                if (o < units) {
                    const int kb = __float2int_rz(((float)o + 0.5f) * inv_nrt);
                    const int rl = o - kb * nrt;
                    const uint32_t c[4] = {v[u].x, v[u].y, v[u].z, v[u].w};  // rows 4i .. 4i + 3 in word i
                    float4* dst = reinterpret_cast<float4*>(sc + ((size_t)rl * KB + kb) * 16);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // float4 q: rows 2q, 2q + 8, 2q + 1, 2q + 9
                        const uint32_t ra = c[(2 * q) >> 2] >> (8 * ((2 * q) & 3));
                        const uint32_t rb = c[(2 * q + 8) >> 2] >> (8 * ((2 * q + 8) & 3));
                        const uint32_t rc = c[(2 * q + 1) >> 2] >> (8 * ((2 * q + 1) & 3));
                        const uint32_t rd = c[(2 * q + 9) >> 2] >> (8 * ((2 * q + 9) & 3));
                        const float2 f0 = e4m3x2_to_f32(ra, rb), f1 = e4m3x2_to_f32(rc, rd);
                        dst[q] = make_float4(f0.x, f0.y, f1.x, f1.y);
                    }
                }
            }
        }
    } else {
        // one code per unit (row-fastest within a block); rows past N read row N - 1
        const int R = nrt * 16;
        const int units = R * KB;
        const float inv_r = 1.f / (float)R;
        for (int base = 0; base < units; base += 8 * kThreads) {
            uint32_t v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int o = base + u * kThreads + tid;
                if (o < units) {
                    const int kb = __float2int_rz(((float)o + 0.5f) * inv_r);
                    int64_t n = (int64_t)rt0 * 16 + (o - kb * R);
                    if (n >= L.N) n = L.N - 1;
                    v[u] = __ldg(S + (size_t)kb * (size_t)L.N + (size_t)n);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int o = base + u * kThreads + tid;
                if (o < units) {
                    const int kb = __float2int_rz(((float)o + 0.5f) * inv_r);
                    const int r = o - kb * R, rl = r >> 4, r16 = r & 15;
                    sc[((size_t)rl * KB + kb) * 16 + 2 * (r16 & 7) + (r16 >> 3)] = e4m3x2_to_f32(v[u], 0u).x;
                }
            }
        }
    }
    for (int o = tid; o < nrt * kW * 16 * M; o += kThreads) red[o] = 0.f;
    const int pairs = (int)(L.K / 32);
    for (int o = tid; o < pairs * 4; o += kThreads) xs[(size_t)M * geo.xrow + o] = make_uint4(0, 0, 0, 0);
    if (pdl) {
        griddep_wait();               // X (and Y) may belong to the previous kernel on the stream
        griddep_launch_dependents();  // after the wait: at most two chained kernels overlap
    }
    {
        // X in B-fragment order: entry (m, pair P, lane class tt) holds depths
        // 32P + 2tt + {0, 1}, + 8, + 16, + 24 of row m
        const uint32_t* x32 = static_cast<const uint32_t*>(p.x);  // K even: rows are 4-byte aligned
        const int64_t kw = L.K / 2;
        for (int r0 = 0; r0 < pairs * 4; r0 += kThreads) {
            const int r = r0 + tid;
            const int P = r >> 2, tt = r & 3;
            uint4 v[M1 ? 1 : 4];
#pragma unroll
            for (int m = 0; m < (M1 ? 1 : 4); ++m) {
                if (m < M && r < pairs * 4) {
                    const uint32_t* src = x32 + (int64_t)m * kw + P * 16 + tt;
                    v[m] = make_uint4(__ldg(src), __ldg(src + 4), __ldg(src + 8), __ldg(src + 12));
                }
            }
#pragma unroll
            for (int m = 0; m < (M1 ? 1 : 4); ++m)
                if (m < M && r < pairs * 4) xs[(size_t)m * geo.xrow + r] = v[m];
        }
    }
    load(wb[1], nxt);
    __syncthreads();

    // ---- 2. items, two buffers: compute one while the next is in flight ----
    const uint32_t xa_lane = smem_u32(xs + (size_t)(g < M ? g : M) * geo.xrow + t);
    const uint32_t sc_lane = smem_u32(sc) + (uint32_t)g * 8u;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    auto flush = [&](int rt_l) {
        float* r = red + (size_t)(rt_l * kW + warp) * 16 * M;
        const int m0 = 2 * t, m1 = 2 * t + 1;
        if (m0 < M) {
            r[m0 * 16 + g] = y[0];
            r[m0 * 16 + g + 8] = y[2];
        }
        if (!M1 && m1 < M) {
            r[m1 * 16 + g] = y[1];
            r[m1 * 16 + g + 8] = y[3];
        }
        y[0] = y[1] = y[2] = y[3] = 0.f;
    };
    auto compute = [&](const uint4 (&w)[kTilesPerChunk], const Cursor& it) {
        const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t xa = xa_lane + (uint32_t)it.c * (uint32_t)(kCH / 2) * 64u;
        const uint32_t sa = sc_lane + ((uint32_t)it.rt * (uint32_t)KB + (uint32_t)it.c * (uint32_t)kCH) * 64u;
        uint4 xv = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int s = 0; s < kCH; ++s) {
            if ((s & 1) == 0) xv = lds128(xa + (uint32_t)(s >> 1) * 64u);
            const uint4 wt = w[s >> 2];
            const uint32_t word = (s & 3) == 0 ? wt.x : (s & 3) == 1 ? wt.y : (s & 3) == 2 ? wt.z : wt.w;
            uint32_t a[4];
            kstep_a<BF16X>(word, a);
            float acc[4];
            const uint32_t b0 = (s & 1) ? xv.z : xv.x, b1 = (s & 1) ? xv.w : xv.y;
            mma16816<BF16X>(acc, a, b0, b1, zero4);
            const float2 sv = lds64f(sa + (uint32_t)s * 64u);  // scales of rows g, g + 8 at this block
            y[0] = fmaf(sv.x, acc[0], y[0]);
            y[2] = fmaf(sv.y, acc[2], y[2]);
            if constexpr (!M1) {
                y[1] = fmaf(sv.x, acc[1], y[1]);
                y[3] = fmaf(sv.y, acc[3], y[3]);
            }
        }
    };
    auto step = [&](uint4 (&w)[kTilesPerChunk]) {
        compute(w, cur);
        Cursor after = nxt;
        after.advance(KC, geo.q16, geo.r16);
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

    // ---- 3. rows: the 16 warps' partials in a fixed order, times the global scale ----
    const float inv_m = 1.f / (float)M;
    for (int o = tid; o < nrt * 16 * M; o += kThreads) {
        const int row = o & 15, q = o >> 4;
        const int rt_l = M1 ? q : __float2int_rz(((float)q + 0.5f) * inv_m);
        const int m = M1 ? 0 : q - rt_l * M;
        const float* src = red + (size_t)rt_l * kW * 16 * M + m * 16 + row;
        float t8[kW / 2];
#pragma unroll
        for (int w2 = 0; w2 < kW / 2; ++w2) t8[w2] = src[(size_t)(2 * w2) * 16 * M] + src[(size_t)(2 * w2 + 1) * 16 * M];
#pragma unroll
        for (int h = kW / 4; h >= 1; h >>= 1) {
#pragma unroll
            for (int w2 = 0; w2 < h; ++w2) t8[w2] = t8[2 * w2] + t8[2 * w2 + 1];
        }
        const int64_t n = (int64_t)(rt0 + rt_l) * 16 + row;
        if (n < L.N) store_f32(p.y, (int64_t)m * L.N + n, t8[0] * p.global_scale, p.out_dtype);
    }
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status, p.fmt);
}

inline cudaError_t launch(const FpParams& p, const NGeom& geo, cudaStream_t s) {
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
    if (p.M == 1) return bf ? go(gemv_nv_kernel<true, true>) : go(gemv_nv_kernel<false, true>);
    return bf ? go(gemv_nv_kernel<true, false>) : go(gemv_nv_kernel<false, false>);
}

}  // namespace gnv
}  // namespace mnb
