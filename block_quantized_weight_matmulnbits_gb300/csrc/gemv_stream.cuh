// Streaming decode GEMV on warp-level tensor-core MMA, 1 <= M <= 16, bf16 or
// f16 X:  Y[m, n] = sum_kb scale[n, kb] * sum_{k in kb} X[m, k] * (q[n, k] - zp[n, kb])  (+ bias[n]),
// MatMulNBits as restated by onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs (fn dequantize_nbits_value; MatMulNBitsKernel::
// execute).  The arithmetic is that of gemv_mma.cuh: a code pair masked into
// the mantissa of 128.0 (bf16) or 1024.0 (f16) and one packed subtract give
// (q - zp) exactly, one mma.sync m16n8k16 multiplies 256 of them by the
// activations in f32, and the block's f32 scale multiplies the fragment once
// per block.
//
// Schedule (a GB300 design; measured on GB300: a 26 MB read streams at about
// 7.5 TB/s only when every SM keeps ~16 KB or more in flight without pause,
// and kernels chained with programmatic dependent launch overlap their tails):
//   * persistent CTAs of 8 warps, a whole number per SM, with registers and
//     shared memory left for one CTA of the next chained kernel; CTA c owns a
//     contiguous range of 16-row tiles;
//   * warp w owns a fixed K-slice (whole quantisation blocks) of every row
//     tile and walks it in chunks of up to 4 packed tiles held in registers
//     (16 bytes per lane per tile); as soon as a tile has been used its
//     register takes the load of the same tile of the next chunk, across
//     row-tile boundaries, so a chunk of loads is always in flight and the
//     weight stream never waits for the compute;
//   * the (zero-point constant, scale) entries of a chunk's blocks are loaded
//     into registers together with the chunk's codes and written to the
//     warp's own double-buffered shared-memory slot just before the chunk is
//     computed;
//   * X is staged once per CTA, after the dependency wait;
//   * the warps' partial sums of a row tile are summed through shared memory
//     in a fixed order by one warp (a different one per row tile); mbarriers
//     let the other warps run on without waiting for that reduction.
// Reduction orders are fixed, so results are bit-identical run to run.
#pragma once

#include "gemv_mma.cuh"

namespace mnb {
namespace gstr {

using gmma::Entry;
using gmma::mma16816;
using gmma::Unpack;

constexpr int kW = 8;                 // warps per CTA
constexpr int kThreads = kW * 32;

// Packed tiles per chunk: 256 depths for 2- and 4-bit codes, 128 for 8-bit
// (16 bytes per lane per tile: 64 or 32 bytes of codes in flight per lane).
template <int BITS>
struct Chunk {
    static constexpr int kTiles = BITS == 2 ? 2 : 4;
    static constexpr int kDepth = kTiles * 256 / BITS;
};

// Entry slots per row per chunk (blocks in a chunk) and entries per lane.
template <int BITS, int SPB_LOG>
struct Slots {
    static constexpr int kEB = SPB_LOG < 0 ? 1 : ((Chunk<BITS>::kDepth / 16) >> SPB_LOG) > 0
                                                   ? ((Chunk<BITS>::kDepth / 16) >> SPB_LOG) : 1;
    static constexpr int kEPL = kEB >= 2 ? kEB / 2 : 1;  // 16 rows x kEB slots over 32 lanes
};

struct SGeom {
    int G;            // CTAs
    int utiles;       // packed tiles per K-unit (max(1, bs / KT)): slices are whole units
    int nunits;       // K-units per row tile
    int eb;           // entry slots per row per chunk (blocks per chunk, >= 1)
    int ks_total;     // k-steps staged for X (KTILES * KT / 16)
    size_t x_bytes, ent_bytes, red_bytes, bar_off, total_bytes;
};

// SPB_LOG: log2 of k-steps per quantisation block when a block fits in a
// chunk (every chunk then starts and ends on block boundaries); -1 when a
// block spans chunks (one block per chunk, its ends found at run time).
template <int BITS, bool BF16X, int MT, int SPB_LOG>
__global__ void __launch_bounds__(kThreads, 3) gemv_stream_kernel(MatmulParams p, SGeom geo, int pdl) {
    using U = Unpack<BITS, BF16X>;
    constexpr int NTILE = MT / 8;
    constexpr int SPT = U::kStepsPerTile;  // k-steps per packed tile
    constexpr int kCH = Chunk<BITS>::kTiles;
    constexpr int EB = Slots<BITS, SPB_LOG>::kEB;
    constexpr int kEPL = Slots<BITS, SPB_LOG>::kEPL;
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* xb = smem;                                                         // [M][ks_total][32 B]
    Entry* ent = reinterpret_cast<Entry*>(smem + geo.x_bytes);                  // [kW][2][16][eb]
    float* red = reinterpret_cast<float*>(smem + geo.x_bytes + geo.ent_bytes);  // [2][kW][16][MT]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + geo.bar_off);
    uint64_t* red_full = bars;      // [2]: one arrival per warp
    uint64_t* red_free = bars + 2;  // [2]: the reducing warp

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = (int)p.M;

    // ---- this CTA's row tiles and this warp's K-slice ----
    const int64_t rt0 = (int64_t)blockIdx.x * L.NT / geo.G;
    const int nrt = (int)((int64_t)(blockIdx.x + 1) * L.NT / geo.G - rt0);
    const int u0 = warp * geo.nunits / kW, u1 = (warp + 1) * geo.nunits / kW;
    const int64_t tw0 = (int64_t)u0 * geo.utiles;
    const int ntw = (int)(imin64((int64_t)u1 * geo.utiles, L.KTILES) - tw0);  // >= 1 (nunits >= kW)
    const int nch = (ntw + kCH - 1) / kCH;                                   // chunks per row tile
    const int64_t k_w0 = tw0 * L.KT;                                         // first depth of the slice

    if (tid == 0) {
        mbar_init(&red_full[0], kW);
        mbar_init(&red_full[1], kW);
        mbar_init(&red_free[0], 1);
        mbar_init(&red_free[1], 1);
        fence_barrier_init();
    }

    // ---- weights: chunk i = (row tile i / nch, chunk i % nch) ----
    const int total_ch = nrt * nch;
    const uint8_t* wbase = p.packed + (size_t)lane * 16;
    // address of tile 0 of chunk i and its tile count (0 past the last chunk)
    auto chunk_src = [&](int i, int* nt) -> const uint8_t* {
        if (i >= total_ch) {
            *nt = 0;
            return wbase;
        }
        const int r = i / nch, c = i - r * nch;
        *nt = min(kCH, ntw - c * kCH);
        return wbase + ((rt0 + r) * L.KTILES + tw0 + (int64_t)c * kCH) * kTileBytes;
    };

    // ---- entries of chunk i: lane l holds row l & 15, block slots (l >> 4) + 2q ----
    const int erow = lane & 15, ej0 = lane >> 4;
    uint32_t es[kEPL], ez[kEPL];
    auto fetch_entries = [&](int i) {
        const int r = i / nch, c = i - r * nch;
        const int64_t n = (rt0 + r) * 16 + erow;
        const bool row_ok = i < total_ch && n < L.N;
        const int64_t kb0 = (k_w0 + (int64_t)c * Chunk<BITS>::kDepth) / L.bs;
#pragma unroll
        for (int q = 0; q < kEPL; ++q) {
            const int j = ej0 + 2 * q;
            const int64_t kb = kb0 + j;
            es[q] = 0;
            ez[q] = 0;
            if (row_ok && j < EB && kb < L.KB) {
                const int64_t si = n * L.KB + kb;
                es[q] = p.scale_dtype == kF32 ? __ldg(reinterpret_cast<const uint32_t*>(p.scales) + si)
                                              : (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p.scales) + si);
                if (p.zp) ez[q] = __ldg(p.zp + n * L.zp_row + ((kb * BITS) >> 3)) >> ((kb * BITS) & 7);
            }
        }
    };
    // slots past the chunk's blocks get a zero scale and a zero-point constant
    // that cancels zero codes (padding codes are zero, their activations too)
    auto store_entries = [&](int b) {
        Entry* dst = ent + ((size_t)warp * 2 + b) * 16 * EB + (size_t)erow * EB;
#pragma unroll
        for (int q = 0; q < kEPL; ++q) {
            const int j = ej0 + 2 * q;
            if (j < EB) {
                float sc;
                if (p.scale_dtype == kF32) sc = __uint_as_float(es[q]);
                else if (p.scale_dtype == kF16) sc = __half2float(__ushort_as_half((unsigned short)es[q]));
                else sc = __uint_as_float(es[q] << 16);
                const uint32_t z = p.zp ? (ez[q] & (uint32_t)code_mask(BITS)) : (1u << (BITS - 1));
                dst[j] = Entry{U::zconst(z), sc};
            }
        }
    };

    uint4 wv[kCH];
    {
        int nt0;
        const uint8_t* src0 = chunk_src(0, &nt0);
#pragma unroll
        for (int j = 0; j < kCH; ++j)
            if (j < nt0) wv[j] = ldg_stream(src0 + j * kTileBytes);
    }
    fetch_entries(0);
    __syncthreads();          // barrier init visible
    if (pdl) {
        griddep_wait();       // X (and Y) may belong to the previous kernel on the stream
        // only now may the next kernel launch: at most two chained kernels overlap
        griddep_launch_dependents();
    }

    // ---- X once per CTA: item (m, k-step S) = 32 bytes; lane class t reads 8 bytes at t * 8 ----
    {
        const int KS = geo.ks_total;
        const int items = M * KS;
        const bool vec = (L.K % 8) == 0;
        const uint16_t* x16 = static_cast<const uint16_t*>(p.x);
        for (int it = tid; it < items; it += kThreads) {
            const int m = it / KS, S = it - m * KS;
            const int64_t k0 = 16 * (int64_t)S;
            uint4 v0, v1;
            if (vec && k0 + 16 <= L.K) {
                const uint4* src = reinterpret_cast<const uint4*>(x16 + (int64_t)m * L.K + k0);
                v0 = __ldg(src);
                v1 = __ldg(src + 1);
            } else {
                uint32_t h[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int64_t ka = k0 + 2 * j, kb2 = ka + 1;
                    const uint32_t lo = ka < L.K ? x16[(int64_t)m * L.K + ka] : 0u;
                    const uint32_t hi = kb2 < L.K ? x16[(int64_t)m * L.K + kb2] : 0u;
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
    __syncthreads();

    const int S_w0 = (int)(k_w0 / 16);  // first k-step of the slice
    const uint32_t xa0 =
        smem_u32(reinterpret_cast<const uint2*>(xb) + (int64_t)(g % M) * geo.ks_total * 4 + t) + (uint32_t)S_w0 * 32u;
    const uint32_t xa1 =
        smem_u32(reinterpret_cast<const uint2*>(xb) + (int64_t)((g + 8) % M) * geo.ks_total * 4 + t) +
        (uint32_t)S_w0 * 32u;
    const int spb_log = SPB_LOG >= 0 ? SPB_LOG : __ffs(L.bs / 16) - 1;
    const int spb_mask = (1 << spb_log) - 1;
    constexpr int kSMask = SPB_LOG >= 0 ? (1 << (SPB_LOG >= 0 ? SPB_LOG : 0)) - 1 : 0;
    constexpr int kSLog = SPB_LOG >= 0 ? SPB_LOG : 0;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    auto lds2 = [](uint32_t addr) {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
        return v;
    };

    float y[NTILE][4], acc[NTILE][4];
    uint32_t zg = 0, zg8 = 0;
    float sg = 0.f, sg8 = 0.f;
    int cur_r = 0, cur_c = 0, ci = 0;
    bool ok = true;
    const uint32_t e8 = 8u * (uint32_t)EB * (uint32_t)sizeof(Entry);  // entry of row g + 8

    // one chunk: global chunk ci = row tile cur_r, chunk cur_c, codes in wv;
    // the chunk's entries are already in registers (es, ez)
    auto step = [&]() {
        if (cur_c == 0) {
#pragma unroll
            for (int q = 0; q < NTILE; ++q)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) y[q][c4] = 0.f;
        }
        // this chunk's entries into slot ci & 1 (its last reader was chunk ci - 2), then the next chunk's loads
        store_entries(ci & 1);
        fetch_entries(ci + 1);
        __syncwarp();
        const uint32_t ebase = smem_u32(ent + ((size_t)warp * 2 + (ci & 1)) * 16 * EB + (size_t)g * EB);
        int nt_next;
        const uint8_t* src_next = chunk_src(ci + 1, &nt_next);
        ++ci;
        const int nt = min(kCH, ntw - cur_c * kCH);
        const int Sc = cur_c * kCH * SPT;  // first k-step of the chunk inside the slice
#pragma unroll
        for (int j = 0; j < kCH; ++j) {
            if (j < nt) {
#pragma unroll
                for (int s = 0; s < SPT; ++s) {
                    const int ks = j * SPT + s;  // k-step inside the chunk (static)
                    const int Sk = Sc + ks;      // k-step inside the slice
                    const bool bstart = SPB_LOG >= 0 ? ((ks & kSMask) == 0) : ((Sk & spb_mask) == 0);
                    if (SPB_LOG >= 0 ? bstart : (ks == 0)) {  // a chunk inside a block reads its one slot
                        const uint32_t ea = ebase + (uint32_t)(SPB_LOG >= 0 ? (ks >> kSLog) : 0) * (uint32_t)sizeof(Entry);
                        const uint2 eg = lds2(ea), eg8 = lds2(ea + e8);
                        zg = eg.x;
                        sg = __uint_as_float(eg.y);
                        zg8 = eg8.x;
                        sg8 = __uint_as_float(eg8.y);
                    }
                    uint32_t a[4];
                    U::kstep(wv[j], s, zg, zg8, a);
                    const uint2 b0 = lds2(xa0 + (uint32_t)Sk * 32u);
                    if (bstart) mma16816<BF16X>(acc[0], a, b0.x, b0.y, zero4);
                    else mma16816<BF16X>(acc[0], a, b0.x, b0.y, acc[0]);
                    if constexpr (NTILE == 2) {
                        const uint2 b1 = lds2(xa1 + (uint32_t)Sk * 32u);
                        if (bstart) mma16816<BF16X>(acc[1], a, b1.x, b1.y, zero4);
                        else mma16816<BF16X>(acc[1], a, b1.x, b1.y, acc[1]);
                    }
                    const bool bend = SPB_LOG >= 0 ? (((ks + 1) & kSMask) == 0) : (((Sk + 1) & spb_mask) == 0);
                    if (bend) {
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
            // tile j is used: its register takes tile j of the next chunk
            if (j < nt_next) wv[j] = ldg_stream(src_next + j * kTileBytes);
        }
        if (++cur_c < nch) return;
        // ---- end of row tile cur_r ----
        const int r = cur_r;
        cur_c = 0;
        ++cur_r;
        const int rb = r & 1;
        if (r >= 2 && !mbar_wait(&red_free[rb], (uint32_t)(((r >> 1) - 1) & 1), p.status)) {
            ok = false;
            return;
        }
        float* mine = red + ((size_t)rb * kW + warp) * 16 * MT;
#pragma unroll
        for (int q = 0; q < NTILE; ++q) {
            const int col = q * 8 + 2 * t;
            *reinterpret_cast<float2*>(&mine[g * MT + col]) = make_float2(y[q][0], y[q][1]);
            *reinterpret_cast<float2*>(&mine[(g + 8) * MT + col]) = make_float2(y[q][2], y[q][3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_full[rb]);
        if (warp == r % kW) {
            if (!mbar_wait(&red_full[rb], (uint32_t)((r >> 1) & 1), p.status)) {
                ok = false;
                return;
            }
            const float* base = red + (size_t)rb * kW * 16 * MT;
            for (int o = lane; o < 16 * M; o += 32) {
                const int row = o & 15, m = o >> 4;
                float v = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kW; ++w2) v += base[(w2 * 16 + row) * MT + m];
                const int64_t n = (rt0 + r) * 16 + row;
                if (n < L.N) {
                    if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
                    store_f32(p.y, (int64_t)m * L.N + n, v, p.out_dtype);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&red_free[rb]);
        }
    };

    // ---- main loop over the chunks of this CTA's row tiles ----
    for (int i = 0; i < total_ch && ok; ++i) step();
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status);
}

// Geometry; false when the shape is not for this schedule.
inline bool make_sgeom(const Layout& L, int64_t M, int MT, int sms, size_t smem_limit, SGeom* out) {
    SGeom g{};
    const int cdepth = L.bits == 8 ? 128 : 256;  // Chunk<BITS>::kDepth
    g.utiles = (int)(L.bs > L.KT ? L.bs / L.KT : 1);
    g.nunits = (int)((L.KTILES + g.utiles - 1) / g.utiles);
    if (g.nunits < kW) return false;  // every warp needs a slice
    g.eb = L.bs >= cdepth ? 1 : cdepth / L.bs;  // Slots<BITS, SPB_LOG>::kEB
    g.ks_total = (int)(L.KTILES * L.KT / 16);
    g.x_bytes = round16((size_t)M * g.ks_total * 32);
    g.ent_bytes = round16((size_t)kW * 2 * 16 * g.eb * sizeof(Entry));
    g.red_bytes = (size_t)2 * kW * 16 * MT * 4;
    g.bar_off = g.x_bytes + g.ent_bytes + g.red_bytes;
    g.total_bytes = g.bar_off + 4 * 8;
    if (g.total_bytes > smem_limit) return false;
    // CTAs: two per SM when shared memory leaves room for a third (one CTA of
    // the next chained kernel), else one
    const int per_sm = 3 * (g.total_bytes + 1024) <= (size_t)228 * 1024 ? 2 : 1;
    int64_t G = (int64_t)sms * per_sm;
    if (G > L.NT) G = L.NT;
    g.G = (int)G;
    *out = g;
    return true;
}

template <int BITS, bool BF16X, int MT, int SPB_LOG>
cudaError_t launch_s(const MatmulParams& p, const SGeom& geo, cudaStream_t s) {
    const int pdl = (p.flags & kFlagPDL) ? 1 : 0;
    auto kern = gemv_stream_kernel<BITS, BF16X, MT, SPB_LOG>;
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
}

template <int BITS, bool BF16X, int MT>
cudaError_t launch_spb(const MatmulParams& p, const SGeom& geo, cudaStream_t s) {
    if (p.L.bs > Chunk<BITS>::kDepth) return launch_s<BITS, BF16X, MT, -1>(p, geo, s);
    switch (p.L.bs / 16) {
        case 1: return launch_s<BITS, BF16X, MT, 0>(p, geo, s);
        case 2: return launch_s<BITS, BF16X, MT, 1>(p, geo, s);
        case 4: return launch_s<BITS, BF16X, MT, 2>(p, geo, s);
        case 8: return launch_s<BITS, BF16X, MT, 3>(p, geo, s);
        default: return launch_s<BITS, BF16X, MT, BITS == 8 ? -1 : 4>(p, geo, s);
    }
}

template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const SGeom& geo, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    if (p.M <= 8) return bf ? launch_spb<BITS, true, 8>(p, geo, s) : launch_spb<BITS, false, 8>(p, geo, s);
    return bf ? launch_spb<BITS, true, 16>(p, geo, s) : launch_spb<BITS, false, 16>(p, geo, s);
}

}  // namespace gstr
}  // namespace mnb
