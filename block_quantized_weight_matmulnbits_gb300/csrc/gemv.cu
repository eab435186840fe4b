// Decode GEMV, M == 1:  y[n] = sum_k x[k] * (q[n,k] - zp[n,kb]) * scale[n,kb]  (+ bias[n]).
//
// What it computes is the MatMulNBits product of onnx-runtime-ep-cpu
// 0.1.0-dev.5, src/kernels/matmul_nbits.rs (fn dequantize_nbits_value for w,
// the m == 1 branch of MatMulNBitsKernel::execute for the GEMV); the pages'
// own decode kernels are CPU SIMD loops (int4_dot_row_*), so nothing of their
// structure is reused here.
//
// GB300 design (HBM-bound: ~0.56 byte per weight at 4 bits):
//  * Persistent: one CTA per SM, row-tiles (16 rows, all of K) dealt round-robin.
//  * Each of the CTA's warps owns a contiguous K-slice of every row-tile and
//    streams its slice of the packed weights with 1-D bulk copies
//    (cp.async.bulk, TMA engine) into its own ring of shared-memory slots,
//    completion tracked by one mbarrier per slot.  The ring keeps
//    SLOTS * CHUNK bytes per warp in flight independent of registers, which
//    is what lets a few warps per SM saturate HBM3e.
//  * Unpack is exact and cheap: a 4-bit code OR'ed into the mantissa of
//    2^23 (0x4B000000) gives the float 2^23 + q * 2^p exactly (p = 0, or 16
//    for the odd depth of a pair); subtracting 2^23 + zp * 2^p (one packed
//    f32x2 add) gives (q - zp) * 2^p exactly; the activation of the odd depth
//    is pre-scaled by 2^-16 (exact), so one packed f32x2 FMA accumulates
//    x * (q - zp) for two depths.  8-bit codes use PRMT to place the byte.
//  * Per (row, K-block) the scale multiplies the block's partial sum
//    (one f32x2 FMA); scales and the subtraction constants of the next
//    row-tile are loaded during the current one and staged in shared memory.
//  * Partial sums of the warps are reduced in a fixed order through shared
//    memory, so results are bit-identical run to run.
#include <cstdio>

#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSlots = 12;      // ring slots per warp
constexpr int kChunkTiles = 2;  // 512-byte tiles per bulk copy
constexpr int kChunkBytes = kChunkTiles * kTileBytes;
constexpr uint32_t kMagic23 = 0x4B000000u;  // 2^23
constexpr int kStageRegs = 8;   // staged (row, block) entries per thread prefetched into registers

struct GemvGeom {
    int64_t kblocks_pad;  // staged blocks per row (covers KTILES * KT depths)
    int64_t ktw;          // k-tiles per warp slice
    int64_t nch;          // chunks per warp slice
    size_t xs_bytes, ring_bytes, stage_bytes, red_bytes, bar_bytes, total_bytes;
};

__host__ GemvGeom gemv_geom(const Layout& L) {
    GemvGeom g;
    g.kblocks_pad = (L.KTILES * L.KT + L.bs - 1) / L.bs;
    g.ktw = (L.KTILES + kWarps - 1) / kWarps;
    g.nch = (g.ktw + kChunkTiles - 1) / kChunkTiles;
    g.xs_bytes = (size_t)L.KTILES * L.KT * 4;
    g.ring_bytes = (size_t)kWarps * kSlots * kChunkBytes;
    g.stage_bytes = (size_t)2 * 16 * (g.kblocks_pad | 1) * 16;
    g.red_bytes = (size_t)2 * kWarps * 16 * 4;
    g.bar_bytes = (size_t)kWarps * kSlots * 8;
    g.total_bytes = g.ring_bytes + g.xs_bytes + g.stage_bytes + g.red_bytes + g.bar_bytes + 128;
    return g;
}

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ uint64_t pack2u(uint32_t a, uint32_t b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Staged per-(row, block) entry: the pair to subtract, (2^23 + zp, 2^23 + zp*2^pb)
// as floats, and the scale twice.
struct __align__(16) StageEntry {
    uint32_t c0, c1;
    float s0, s1;
};

template <int BITS>
struct Unpack;

// 4-bit: word = one k-step; pair r at nibbles r (even depth) and r+4 (odd depth).
template <>
struct Unpack<4> {
    static constexpr int kPb = 16;
    // d[r] = ((q_even - zp) , (q_odd - zp) * 2^16) for fragment register r.
    __device__ __forceinline__ static void kstep(const uint32_t* w, int s, uint64_t cg, uint64_t cg8,
                                                 uint64_t d[4]) {
        const uint32_t word = w[s];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t sh = word >> (4 * r);
            const uint32_t va = lop3_and_or(sh, 0x0000000Fu, kMagic23);
            const uint32_t vb = lop3_and_or(sh, 0x000F0000u, kMagic23);
            d[r] = fsub2(pack2u(va, vb), (r & 1) ? cg8 : cg);
        }
    }
    static constexpr int kStepsPerTile = 4;
};

// 2-bit: word j holds k-steps 2j and 2j+1; pair i = 4*(s&1) + r at fields i and i+8.
template <>
struct Unpack<2> {
    static constexpr int kPb = 16;
    __device__ __forceinline__ static void kstep(const uint32_t* w, int s, uint64_t cg, uint64_t cg8,
                                                 uint64_t d[4]) {
        const uint32_t word = w[s >> 1];
        const int base = (s & 1) * 4;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t sh = word >> (2 * (base + r));
            const uint32_t va = lop3_and_or(sh, 0x00000003u, kMagic23);
            const uint32_t vb = lop3_and_or(sh, 0x00030000u, kMagic23);
            d[r] = fsub2(pack2u(va, vb), (r & 1) ? cg8 : cg);
        }
    }
    static constexpr int kStepsPerTile = 8;
};

// 8-bit: k-step s in words 2s (depths 2t, 2t+1) and 2s+1 (2t+8, 2t+9);
// byte 2*hi + e, hi selecting row g+8.
template <>
struct Unpack<8> {
    static constexpr int kPb = 0;
    __device__ __forceinline__ static void kstep(const uint32_t* w, int s, uint64_t cg, uint64_t cg8,
                                                 uint64_t d[4]) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t word = w[2 * s + (r >> 1)];
            const uint32_t hi = r & 1;
            const uint32_t va = prmt(word, kMagic23, 0x7650u | (2 * hi));
            const uint32_t vb = prmt(word, kMagic23, 0x7650u | (2 * hi + 1));
            d[r] = fsub2(pack2u(va, vb), hi ? cg8 : cg);
        }
    }
    static constexpr int kStepsPerTile = 2;
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(MatmulParams p, GemvGeom geo) {
    using U = Unpack<BITS>;
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;                                                   // [warps][slots][chunk]
    float* xs = reinterpret_cast<float*>(smem + geo.ring_bytes);            // permuted x'
    StageEntry* stage = reinterpret_cast<StageEntry*>(smem + geo.ring_bytes + geo.xs_bytes);
    float* red = reinterpret_cast<float*>(smem + geo.ring_bytes + geo.xs_bytes + geo.stage_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + geo.ring_bytes + geo.xs_bytes + geo.stage_bytes +
                                                 geo.red_bytes);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t NT = L.NT;
    const int64_t my_tiles = (NT - blockIdx.x + gridDim.x - 1) / gridDim.x;  // row-tiles of this CTA
    if (my_tiles <= 0) return;

    // This warp's K-slice of every row-tile.
    const int64_t kt_begin = imin64((int64_t)warp * geo.ktw, L.KTILES);
    const int64_t kt_end = imin64(kt_begin + geo.ktw, L.KTILES);
    const int64_t nch = (kt_end - kt_begin + kChunkTiles - 1) / kChunkTiles;
    const int64_t total_chunks = nch * my_tiles;
    uint64_t* wbars = bars + warp * kSlots;
    uint8_t* wring = ring + (size_t)warp * kSlots * kChunkBytes;

    auto issue = [&](int64_t qi) {  // lane 0 only
        const int64_t i = qi / nch, c = qi - i * nch;
        const int64_t rt = blockIdx.x + i * gridDim.x;
        const int64_t kt = kt_begin + c * kChunkTiles;
        const uint32_t bytes = (uint32_t)(imin64(kChunkTiles, kt_end - kt) * kTileBytes);
        const int slot = (int)(qi % kSlots);
        mbar_arrive_expect_tx(&wbars[slot], bytes);
        bulk_g2s(wring + slot * kChunkBytes, p.packed + (rt * L.KTILES + kt) * kTileBytes, bytes,
                 &wbars[slot]);
    };

    if (lane == 0) {
        for (int s = 0; s < kSlots; ++s) mbar_init(&wbars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // Start streaming at once: the prologue below overlaps the first copies.
    int64_t issued = imin64(kSlots, total_chunks);
    if (lane == 0)
        for (int64_t qi = 0; qi < issued; ++qi) issue(qi);

    // x': per k-step S and lane class t, (x[16S+2t], x[16S+2t+1]*2^-pb, x[16S+2t+8], x[16S+2t+9]*2^-pb).
    {
        const float odd_scale = (U::kPb == 16) ? (1.0f / 65536.0f) : 1.0f;
        const int64_t ksteps = L.KTILES * L.KT / 16;
        for (int64_t i = tid; i < ksteps * 4; i += kThreads) {
            const int64_t S = i >> 2;
            const int tt = (int)(i & 3);
            const int64_t k0 = 16 * S + 2 * tt;
            float v[4];
            const int64_t ks[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = ks[j] < L.K ? load_f32(p.x, ks[j], p.act_dtype) : 0.f;
            reinterpret_cast<float4*>(xs)[i] = make_float4(v[0], v[1] * odd_scale, v[2], v[3] * odd_scale);
        }
    }

    // Staging of (subtract constants, scale) per (row, block) of a row-tile.
    // Entry (r, kb) lives at r * kbs + kb; kbs is odd so the 8 row groups of a
    // warp hit different banks.
    const int64_t kbp = geo.kblocks_pad;
    const int64_t kbs = kbp | 1;
    const int64_t stage_entries = 16 * kbp;
    const int64_t stage_stride = 16 * kbs;
    auto make_entry = [&](uint32_t z, float sc) {
        StageEntry se;
        se.c0 = kMagic23 | z;
        se.c1 = kMagic23 | (z << U::kPb);
        se.s0 = se.s1 = sc;
        return se;
    };
    auto raw_value = [&](int64_t rt, int64_t e, uint32_t* z, float* sc) {
        const int64_t r = e / kbp, kb = e - r * kbp;
        const int64_t n = rt * 16 + r;
        if (n < L.N && kb < L.KB) {
            *z = (uint32_t)load_zp(p.zp, L, n, kb);
            *sc = load_f32(p.scales, n * L.KB + kb, p.scale_dtype);
        } else {
            *z = 0;
            *sc = 0.f;
        }
    };
    const bool stage_in_regs = stage_entries <= (int64_t)kStageRegs * kThreads;
    float pre_s[kStageRegs];
    uint32_t pre_z[kStageRegs / 4];
    auto stage_prefetch = [&](int64_t rt) {
#pragma unroll
        for (int j = 0; j < kStageRegs; ++j) {
            const int64_t e = tid + (int64_t)j * kThreads;
            uint32_t z = 0;
            float sc = 0.f;
            if (e < stage_entries) raw_value(rt, e, &z, &sc);
            pre_s[j] = sc;
            if ((j & 3) == 0) pre_z[j >> 2] = 0;
            pre_z[j >> 2] |= z << (8 * (j & 3));
        }
    };
    auto stage_commit = [&](int buf) {
        StageEntry* dst = stage + buf * stage_stride;
#pragma unroll
        for (int j = 0; j < kStageRegs; ++j) {
            const int64_t e = tid + (int64_t)j * kThreads;
            if (e < stage_entries) {
                const int64_t r = e / kbp, kb = e - r * kbp;
                dst[r * kbs + kb] = make_entry((pre_z[j >> 2] >> (8 * (j & 3))) & 0xFF, pre_s[j]);
            }
        }
    };
    auto stage_direct = [&](int64_t rt, int buf) {
        StageEntry* dst = stage + buf * stage_stride;
        for (int64_t e = tid; e < stage_entries; e += kThreads) {
            uint32_t z;
            float sc;
            raw_value(rt, e, &z, &sc);
            const int64_t r = e / kbp, kb = e - r * kbp;
            dst[r * kbs + kb] = make_entry(z, sc);
        }
    };

    if (stage_in_regs) {
        stage_prefetch(blockIdx.x);
        stage_commit(0);
    } else {
        stage_direct(blockIdx.x, 0);
    }
    __syncthreads();

    // Blocks are powers of two >= 16 depths, i.e. 2^spb_log k-steps.
    const int spb_log = __ffs(L.bs / 16) - 1;
    const int spb_mask = (1 << spb_log) - 1;
    bool bad = false;
    int64_t q = 0;  // chunks consumed by this warp
    for (int64_t i = 0; i < my_tiles; ++i) {
        const int64_t rt = blockIdx.x + i * gridDim.x;
        const int buf = (int)(i & 1);
        const bool has_next = (i + 1) < my_tiles;
        if (has_next && stage_in_regs) stage_prefetch(rt + gridDim.x);
        const StageEntry* st_g = stage + buf * stage_stride + g * kbs;
        const StageEntry* st_g8 = st_g + 8 * kbs;

        uint64_t acc_g = 0, acc_g8 = 0;  // (even, odd) partial sums of the current block
        uint64_t y_g = 0, y_g8 = 0;
        int S = (int)(kt_begin * U::kStepsPerTile);  // k-step index inside the row
        uint64_t cg = 0, cg8 = 0, sg = 0, sg8 = 0;
        bool first = true;

        for (int64_t c = 0; c < nch; ++c, ++q) {
            const int slot = (int)(q % kSlots);
            if (!bad) bad = !mbar_wait(&wbars[slot], (uint32_t)((q / kSlots) & 1), p.status);
            if (bad) continue;
            const int64_t kt = kt_begin + c * kChunkTiles;
            const int ntile = (int)imin64(kChunkTiles, kt_end - kt);
            uint4 wv[kChunkTiles];
            const uint8_t* sbase = wring + slot * kChunkBytes;
#pragma unroll
            for (int tl = 0; tl < kChunkTiles; ++tl)
                if (tl < ntile) wv[tl] = reinterpret_cast<const uint4*>(sbase + tl * kTileBytes)[lane];
#pragma unroll
            for (int tl = 0; tl < kChunkTiles; ++tl) {
                if (tl >= ntile) break;
                const uint32_t* w = reinterpret_cast<const uint32_t*>(&wv[tl]);
#pragma unroll
                for (int s = 0; s < U::kStepsPerTile; ++s, ++S) {
                    if (first || (S & spb_mask) == 0) {
                        first = false;
                        const int kb = S >> spb_log;
                        const uint4 eg = *reinterpret_cast<const uint4*>(st_g + kb);
                        const uint4 eg8 = *reinterpret_cast<const uint4*>(st_g8 + kb);
                        cg = pack2u(eg.x, eg.y);
                        sg = pack2u(eg.z, eg.w);
                        cg8 = pack2u(eg8.x, eg8.y);
                        sg8 = pack2u(eg8.z, eg8.w);
                    }
                    const float4 xv = reinterpret_cast<const float4*>(xs)[S * 4 + t];
                    const uint64_t p1 = pack2(xv.x, xv.y), p2 = pack2(xv.z, xv.w);
                    uint64_t d[4];
                    U::kstep(w, s, cg, cg8, d);
                    acc_g = ffma2(p1, d[0], acc_g);
                    acc_g8 = ffma2(p1, d[1], acc_g8);
                    acc_g = ffma2(p2, d[2], acc_g);
                    acc_g8 = ffma2(p2, d[3], acc_g8);
                    if (((S + 1) & spb_mask) == 0) {
                        y_g = ffma2(sg, acc_g, y_g);
                        y_g8 = ffma2(sg8, acc_g8, y_g8);
                        acc_g = 0;
                        acc_g8 = 0;
                    }
                }
            }
            __syncwarp();
            // Refill this slot with the chunk kSlots ahead (its data has been consumed).
            if (issued < total_chunks) {
                if (lane == 0) {
                    fence_proxy_async_smem();
                    issue(issued);
                }
                ++issued;
            }
        }
        // Flush a block cut by the end of this warp's slice.
        y_g = ffma2(sg, acc_g, y_g);
        y_g8 = ffma2(sg8, acc_g8, y_g8);
        const float2 yg = unpack2(y_g), yg8 = unpack2(y_g8);
        float vg = yg.x + yg.y, vg8 = yg8.x + yg8.y;
        vg += __shfl_xor_sync(0xffffffffu, vg, 1);
        vg8 += __shfl_xor_sync(0xffffffffu, vg8, 1);
        vg += __shfl_xor_sync(0xffffffffu, vg, 2);
        vg8 += __shfl_xor_sync(0xffffffffu, vg8, 2);
        float* rb = red + buf * kWarps * 16;
        if (t == 0) {
            rb[warp * 16 + g] = vg;
            rb[warp * 16 + g + 8] = vg8;
        }
        if (has_next) {
            if (stage_in_regs) stage_commit(buf ^ 1);
            else stage_direct(rt + gridDim.x, buf ^ 1);
        }
        __syncthreads();
        if (warp == (int)(i % kWarps) && lane < 16) {
            float v = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kWarps; ++w2) v += rb[w2 * 16 + lane];
            const int64_t n = rt * 16 + lane;
            if (n < L.N) {
                if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
                store_f32(p.y, n, v, p.out_dtype);
            }
        }
    }
    // After a timed-out wait, give copies still in flight a bounded chance to land before exit.
    if (bad && lane == 0) {
        for (int64_t qq = q; qq < issued; ++qq) {
            const int slot = (int)(qq % kSlots);
            for (int it = 0; it < (1 << 16); ++it)
                if (mbar_try_wait(&wbars[slot], (uint32_t)((qq / kSlots) & 1))) break;
        }
    }
}

}  // namespace

bool gemv_supported(const MatmulParams& p) {
    if (p.M != 1 || p.g_idx != nullptr) return false;
    const GemvGeom g = gemv_geom(p.L);
    return g.total_bytes <= device_info().smem_optin;
}

cudaError_t launch_gemv(const MatmulParams& p, cudaStream_t s) {
    const GemvGeom geo = gemv_geom(p.L);
    const DeviceInfo& di = device_info();
    const int64_t grid = imin64(p.L.NT, di.sm_count);
    cudaError_t e = cudaSuccess;
    switch (p.L.bits) {
        case 2:
            e = cudaFuncSetAttribute(gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)geo.total_bytes);
            if (e == cudaSuccess) gemv_kernel<2><<<(unsigned)grid, kThreads, geo.total_bytes, s>>>(p, geo);
            break;
        case 4:
            e = cudaFuncSetAttribute(gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)geo.total_bytes);
            if (e == cudaSuccess) gemv_kernel<4><<<(unsigned)grid, kThreads, geo.total_bytes, s>>>(p, geo);
            break;
        case 8:
            e = cudaFuncSetAttribute(gemv_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)geo.total_bytes);
            if (e == cudaSuccess) gemv_kernel<8><<<(unsigned)grid, kThreads, geo.total_bytes, s>>>(p, geo);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mnb
