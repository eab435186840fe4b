// Persistent small-batch GEMV on warp-level tensor-core MMA (1 <= M <= 16,
// bf16 or f16 X) for the common decode shape: many 16-row tiles whose whole
// K fits one pass of 16 warps (K <= 64 packed tiles).  Same arithmetic as the
// per-tile kernel in gemv_mma.cuh (MatMulNBits of onnx-runtime-ep-cpu
// 0.1.0-dev.5, src/kernels/matmul_nbits.rs, fn dequantize_nbits_value); the
// difference is the schedule.
//
// Why: HBM3e reaches its bandwidth only with many independent requests in
// flight per SM (on GB300 about 256 warp-wide 16-byte loads per SM); loads
// into registers cap that at what the register file holds, and a grid of one
// CTA per row tile runs in one and a half waves whose CTAs each wait out a
// full memory latency.  Here one CTA of 16 warps per SM takes a contiguous,
// balanced range of row tiles and streams them through a ring of kDepth
// shared-memory slots with cp.async (16 bytes per request, no registers held):
// every thread keeps 4 requests per row tile, kDepth - 1 row tiles ahead.  A
// row tile's 16 rows of scales and zero points are contiguous in the ORT
// layout and travel in the same copy groups, one row tile earlier, so that
// each row tile's (zero-point constant, scale) table is decoded while the
// previous tile is computed.  X is staged once per CTA; the 16 warps' partial
// sums of a row tile are reduced (fixed order) one iteration later, so each
// row tile costs one barrier.
#pragma once

#include "gemv_mma.cuh"

namespace mnb {
namespace gpers {

using gmma::Entry;
using gmma::Unpack;

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kDepth = 4;   // shared-memory slots of the row-tile ring
constexpr int kMaxTPW = 4;  // k-tiles per warp per row tile
constexpr int kRun = 4;     // blocks per thread in the scale loads

struct PGeom {
    int tpw;     // k-tiles per warp per row tile
    int kbn;     // blocks reachable by the packed depths (ceil(KTILES * KT / bs))
    int kbs;     // row stride of the (zero-point constant, scale) table (kbn | 1)
    int ks;      // k-steps of X staged (KTILES * KT / 16)
    int runs;    // scale runs of kRun blocks per row
    size_t w_slot;                      // packed codes of one row tile (KTILES * 512 bytes)
    size_t raw_row, raw_zoff, raw_slot;  // raw copy: bytes per row of scales, offset of zero points, slot size
    size_t xb_bytes, stage_bytes, red_bytes, total_bytes;
};

inline PGeom make_pgeom(const Layout& L, int64_t M, int MT) {
    PGeom g{};
    g.tpw = (int)((L.KTILES + kWarps - 1) / kWarps);
    g.kbn = (int)((L.KTILES * L.KT + L.bs - 1) / L.bs);
    g.kbs = g.kbn | 1;
    g.ks = (int)(L.KTILES * L.KT / 16);
    g.runs = (g.kbn + kRun - 1) / kRun;
    g.xb_bytes = (size_t)M * g.ks * 32;
    g.stage_bytes = (size_t)2 * 16 * g.kbs * sizeof(Entry);
    g.red_bytes = (size_t)2 * kWarps * 16 * MT * 4;
    g.w_slot = (size_t)L.KTILES * kTileBytes;
    g.raw_row = 0;  // set by the caller (needs the scale dtype)
    g.total_bytes = kDepth * g.w_slot + g.xb_bytes + g.stage_bytes + g.red_bytes;  // + raw slots (caller)
    return g;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int BITS, bool BF16X, int MT, int SPB_LOG, int TPW>
__global__ void __launch_bounds__(kThreads, 1) gemv_pers_kernel(MatmulParams p, PGeom geo, int pdl) {
    using U = Unpack<BITS, BF16X>;
    constexpr int NTILE = MT / 8;
    constexpr int SPT = U::kStepsPerTile;
    constexpr int kMask = (1 << SPB_LOG) - 1;
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* wring = smem;                                                   // [kDepth][w_slot]
    uint8_t* raw = wring + kDepth * geo.w_slot;                              // [kDepth][raw_slot]
    uint8_t* xb = raw + kDepth * geo.raw_slot;                               // [M][ks][32 B]
    Entry* stage = reinterpret_cast<Entry*>(xb + geo.xb_bytes);              // [2][16][kbs]
    float* red = reinterpret_cast<float*>(xb + geo.xb_bytes + geo.stage_bytes);  // [2][kWarps][16][MT]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = (int)p.M;
    const int kbs = geo.kbs;
    const int KS = geo.ks;
    const int64_t rbeg = (int64_t)blockIdx.x * L.NT / gridDim.x;
    const int n_my = (int)((int64_t)(blockIdx.x + 1) * L.NT / gridDim.x - rbeg);
    const int wt0 = warp * TPW;  // first k-tile of this warp in every row tile
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;

    // ---- asynchronous copies (all threads): packed codes and raw scales of a row tile ----
    auto copy_w = [&](int64_t rt, int slot) {
        const uint8_t* src = p.packed + rt * L.KTILES * kTileBytes;
        uint8_t* dst = wring + slot * geo.w_slot;
        const int chunks = (int)(geo.w_slot / 16);
        for (int c = tid; c < chunks; c += kThreads) cp_async16(dst + c * 16, src + c * 16);
    };
    auto copy_raw = [&](int64_t rt, int slot) {
        const int64_t rows = imin64(16, L.N - rt * 16);
        const int sch = (int)(rows * geo.raw_row / 16);
        const int zch = p.zp ? (int)(rows * L.zp_row / 16) : 0;
        const uint8_t* ssrc = static_cast<const uint8_t*>(p.scales) + rt * 16 * geo.raw_row;
        const uint8_t* zsrc = p.zp ? p.zp + rt * 16 * L.zp_row : nullptr;
        uint8_t* dst = raw + slot * geo.raw_slot;
        for (int c = tid; c < sch + zch; c += kThreads) {
            if (c < sch) cp_async16(dst + c * 16, ssrc + c * 16);
            else cp_async16(dst + geo.raw_zoff + (c - sch) * 16, zsrc + (c - sch) * 16);
        }
    };
    // group q holds the codes of local row tile q and the scales of row tile q + 1
    // (group 0 also those of row tile 0)
    if (n_my > 0) copy_raw(rbeg, 0);
    for (int q = 0; q < kDepth - 1; ++q) {
        if (q < n_my) copy_w(rbeg + q, q);
        if (q + 1 < n_my) copy_raw(rbeg + q + 1, (q + 1) % kDepth);
        cp_async_commit();
    }

    // ---- decode a landed raw slot into the table: thread -> (row, run of kRun blocks) ----
    const int items = 16 * geo.runs;
    auto decode_raw = [&](int slot, int i, Entry* dst) {
        const uint8_t* src = raw + slot * geo.raw_slot;
        const int64_t rt = rbeg + i;
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {
            const int it = tid + ps * kThreads;
            if (it < items) {
                const int r = it / geo.runs, run = it - r * geo.runs;
                const bool row_ok = rt * 16 + r < L.N;
#pragma unroll
                for (int j = 0; j < kRun; ++j) {
                    const int kb = run * kRun + j;
                    if (kb < geo.kbn) {
                        const bool ok = row_ok && kb < L.KB;
                        float sc = 0.f;
                        uint32_t z = 1u << (BITS - 1);
                        if (ok) {
                            const uint8_t* sp = src + r * geo.raw_row + kb * sbytes;
                            if (sbytes == 4) {
                                sc = *reinterpret_cast<const float*>(sp);
                            } else {
                                const unsigned short u = *reinterpret_cast<const unsigned short*>(sp);
                                sc = p.scale_dtype == kF16 ? __half2float(__ushort_as_half(u))
                                                           : __uint_as_float((uint32_t)u << 16);
                            }
                            if (p.zp) {
                                const int bit = kb * BITS;
                                z = ((uint32_t)src[geo.raw_zoff + r * L.zp_row + (bit >> 3)] >> (bit & 7)) &
                                    code_mask(BITS);
                            }
                        } else if (p.zp) {
                            z = 0;
                        }
                        dst[r * kbs + kb] = Entry{U::zconst(z), sc};
                    }
                }
            }
        }
    };

    if (pdl) {
        griddep_wait();  // X (and Y) may belong to the previous kernel on the stream
        griddep_launch_dependents();  // after the wait: at most two chained kernels overlap
    }

    // ---- activations (B fragments) of all K, staged once: item (m, k-step S) = 32 bytes ----
    {
        const int xitems = M * KS;
        const bool vec = (L.K % 8) == 0;
        const uint16_t* x16 = static_cast<const uint16_t*>(p.x);
        for (int it = tid; it < xitems; it += kThreads) {
            const int m = it / KS, S = it - m * KS;
            const int64_t k0 = 16 * (int64_t)S;
            uint4 v0, v1;
            if (vec && k0 + 16 <= L.K) {
                const uint4* src = reinterpret_cast<const uint4*>(x16 + m * L.K + k0);
                v0 = __ldg(src);
                v1 = __ldg(src + 1);
            } else {
                uint32_t h[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int64_t ka = k0 + 2 * j, kb2 = ka + 1;
                    const uint32_t lo = ka < L.K ? x16[m * L.K + ka] : 0u;
                    const uint32_t hi = kb2 < L.K ? x16[m * L.K + kb2] : 0u;
                    h[j] = lo | (hi << 16);
                }
                v0 = make_uint4(h[0], h[1], h[2], h[3]);
                v1 = make_uint4(h[4], h[5], h[6], h[7]);
            }
            uint4* dst = reinterpret_cast<uint4*>(xb) + (int64_t)it * 2;
            dst[0] = make_uint4(v0.x, v1.x, v0.y, v1.y);
            dst[1] = make_uint4(v0.z, v1.z, v0.w, v1.w);
        }
    }
    // the scales of row tile 0 (group 0) -> table 0
    cp_async_wait<kDepth - 2>();
    __syncthreads();
    if (n_my > 0) decode_raw(0, 0, stage);

    auto lds2 = [](uint32_t addr) {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
        return v;
    };
    const uint32_t xa0 = smem_u32(reinterpret_cast<const uint2*>(xb) + (int64_t)(g % M) * KS * 4 + t) +
                         (uint32_t)(wt0 * SPT) * 32u;
    const uint32_t xa1 = smem_u32(reinterpret_cast<const uint2*>(xb) + (int64_t)((g + 8) % M) * KS * 4 + t) +
                         (uint32_t)(wt0 * SPT) * 32u;
    const int kb_w = (wt0 * SPT) >> SPB_LOG;  // first block of this warp's slice
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

    // reduce the 16 warps' partial sums of local row tile i (buffer i & 1) and store Y
    auto reduce_store = [&](int i) {
        if (tid < 16 * M) {
            const int row = tid & 15, m = tid >> 4;
            const float* rb = red + (size_t)(i & 1) * kWarps * 16 * MT + row * MT + m;
            float v = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kWarps; ++w2) v += rb[w2 * 16 * MT];
            const int64_t n = (rbeg + i) * 16 + row;
            if (n < L.N) {
                if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
                store_f32(p.y, (int64_t)m * L.N + n, v, p.out_dtype);
            }
        }
    };

    for (int i = 0; i < n_my; ++i) {
        cp_async_wait<kDepth - 2>();  // groups <= i complete: codes of row tile i, scales of i + 1
        __syncthreads();
        if (i >= 1) reduce_store(i - 1);
        {
            const int q = i + kDepth - 1;  // next group
            if (q < n_my) copy_w(rbeg + q, q % kDepth);
            if (q + 1 < n_my) copy_raw(rbeg + q + 1, (q + 1) % kDepth);
            cp_async_commit();
        }
        const Entry* st = stage + (size_t)(i & 1) * 16 * kbs;
        const uint8_t* wsl = wring + (i % kDepth) * geo.w_slot + lane * 16;
        const uint32_t st_g = smem_u32(st + g * kbs + kb_w);
        const uint32_t st_off8 = (uint32_t)(8 * kbs * sizeof(Entry));
        float y[NTILE][4], acc[NTILE][4];
#pragma unroll
        for (int q = 0; q < NTILE; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c) y[q][c] = acc[q][c] = 0.f;
        uint32_t zg = 0, zg8 = 0;
        float sg = 0.f, sg8 = 0.f;
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
            if (wt0 + j < L.KTILES) {
                const uint4 wj = *reinterpret_cast<const uint4*>(wsl + (wt0 + j) * kTileBytes);
#pragma unroll
                for (int s = 0; s < SPT; ++s) {
                    const int ks = j * SPT + s;  // k-step inside the warp's slice
                    if ((ks & kMask) == 0) {
                        const uint32_t ea = st_g + (uint32_t)(ks >> SPB_LOG) * (uint32_t)sizeof(Entry);
                        const uint2 eg = lds2(ea), eg8 = lds2(ea + st_off8);
                        zg = eg.x;
                        sg = __uint_as_float(eg.y);
                        zg8 = eg8.x;
                        sg8 = __uint_as_float(eg8.y);
                    }
                    uint32_t a[4];
                    U::kstep(wj, s, zg, zg8, a);
                    const bool fresh = (ks & kMask) == 0;
                    const uint2 b0 = lds2(xa0 + (uint32_t)ks * 32u);
                    if (fresh) gmma::mma16816<BF16X>(acc[0], a, b0.x, b0.y, zero4);
                    else gmma::mma16816<BF16X>(acc[0], a, b0.x, b0.y, acc[0]);
                    if constexpr (NTILE == 2) {
                        const uint2 b1 = lds2(xa1 + (uint32_t)ks * 32u);
                        if (fresh) gmma::mma16816<BF16X>(acc[1], a, b1.x, b1.y, zero4);
                        else gmma::mma16816<BF16X>(acc[1], a, b1.x, b1.y, acc[1]);
                    }
                    if (((ks + 1) & kMask) == 0) {
#pragma unroll
                        for (int q = 0; q < NTILE; ++q) {
                            y[q][0] = fmaf(sg, acc[q][0], y[q][0]);
                            y[q][1] = fmaf(sg, acc[q][1], y[q][1]);
                            y[q][2] = fmaf(sg8, acc[q][2], y[q][2]);
                            y[q][3] = fmaf(sg8, acc[q][3], y[q][3]);
                        }
                    }
                }
            }
        }
        // the next row tile's table (its scales landed with this tile's codes)
        if (i + 1 < n_my) decode_raw((i + 1) % kDepth, i + 1, stage + (size_t)((i + 1) & 1) * 16 * kbs);

        float* mine = red + ((size_t)(i & 1) * kWarps + warp) * 16 * MT;
#pragma unroll
        for (int q = 0; q < NTILE; ++q) {
            const int col = q * 8 + 2 * t;
            mine[g * MT + col] = y[q][0];
            mine[g * MT + col + 1] = y[q][1];
            mine[(g + 8) * MT + col] = y[q][2];
            mine[(g + 8) * MT + col + 1] = y[q][3];
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    if (n_my > 0) reduce_store(n_my - 1);
    if (blockIdx.x == 0 && threadIdx.x == 0) verify_header(p.packed_hdr, p.L, p.status);
}

template <int BITS, bool BF16X, int MT, int SPB_LOG, int TPW>
cudaError_t launch_p(const MatmulParams& p, const PGeom& geo, int grid, cudaStream_t s) {
    const int pdl = (p.flags & kFlagPDL) ? 1 : 0;
    auto kern = gemv_pers_kernel<BITS, BF16X, MT, SPB_LOG, TPW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = geo.total_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p, geo, pdl);
}

template <int BITS, bool BF16X, int MT, int SPB_LOG>
cudaError_t launch_tpw(const MatmulParams& p, const PGeom& geo, int grid, cudaStream_t s) {
    switch (geo.tpw) {
        case 1: return launch_p<BITS, BF16X, MT, SPB_LOG, 1>(p, geo, grid, s);
        case 2: return launch_p<BITS, BF16X, MT, SPB_LOG, 2>(p, geo, grid, s);
        case 3: return launch_p<BITS, BF16X, MT, SPB_LOG, 3>(p, geo, grid, s);
        case 4: return launch_p<BITS, BF16X, MT, SPB_LOG, 4>(p, geo, grid, s);
        default: return cudaErrorNotSupported;
    }
}

template <int BITS, bool BF16X, int MT>
cudaError_t launch_spb(const MatmulParams& p, const PGeom& geo, int grid, cudaStream_t s) {
    switch (p.L.bs / 16) {
        case 1: return launch_tpw<BITS, BF16X, MT, 0>(p, geo, grid, s);
        case 2: return launch_tpw<BITS, BF16X, MT, 1>(p, geo, grid, s);
        case 4: return launch_tpw<BITS, BF16X, MT, 2>(p, geo, grid, s);
        case 8: return launch_tpw<BITS, BF16X, MT, 3>(p, geo, grid, s);
        default: return cudaErrorNotSupported;
    }
}

template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const PGeom& geo, int grid, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    if (p.M <= 8)
        return bf ? launch_spb<BITS, true, 8>(p, geo, grid, s) : launch_spb<BITS, false, 8>(p, geo, grid, s);
    return bf ? launch_spb<BITS, true, 16>(p, geo, grid, s) : launch_spb<BITS, false, 16>(p, geo, grid, s);
}

}  // namespace gpers
}  // namespace mnb
