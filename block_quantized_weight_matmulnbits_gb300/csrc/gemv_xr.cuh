// Decode GEMV for 1 <= M <= 8, bf16 or f16 X, shaped for the least work per
// weight byte:  Y[m, n] = sum_kb scale[n, kb] * sum_{k in kb} X[m, k] * (q[n, k] - zp[n, kb])  (+ bias[n]),
// MatMulNBits as restated by onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs (fn dequantize_nbits_value; MatMulNBitsKernel::
// execute), with the arithmetic of gemv_mma.cuh: (q - zp) exact in the
// activation type (mantissa magic and one packed subtract), one mma.sync
// m16n8k16 per 256 weights, the block's f32 scale applied to the fragment.
//
// Schedule (measured on GB300: a 26 MB weight streams at ~7.5 TB/s when every
// SM keeps ~16 KB+ of reads in flight; the per-tile kernels spent about three
// times the necessary instructions per k-step on staging and addressing):
//   * one CTA of 16 warps per SM, owning a contiguous range of 16-row tiles;
//   * warp w owns the same K-slice (at most 16 k-steps, whole quantisation
//     blocks) of every row tile, so its X fragments are loaded once into
//     registers;
//   * each warp streams its slice of successive row tiles through its own
//     ring of 4 shared-memory slots with 1-D bulk copies (cp.async.bulk; one
//     instruction per slice, up to 16 KB per SM in flight per ring step);
//     the first copies are issued before anything else, ahead of the
//     dependency wait, since the weights are constant;
//   * the scales and zero points of the CTA's rows (contiguous in the ORT
//     layout) arrive by two bulk copies and are decoded once into a table of
//     (zero-point constant, scale) entries, also before the dependency wait;
//   * the 16 partial sums of a row tile are reduced in a fixed order through
//     shared memory by one warp (a different one per row tile), with
//     mbarriers, so the other warps never wait for the reduction.
// Reduction orders are fixed, so results are bit-identical run to run.
#pragma once

#include "gemv_mma.cuh"

namespace mnb {
namespace gxr {

using gmma::Entry;
using gmma::mma16816;
using gmma::Unpack;

constexpr int kW = 16;
constexpr int kThreads = kW * 32;
constexpr int kMaxD = 4;     // ring slots per warp (at most)
constexpr int kMaxKS = 16;   // k-steps per warp slice (X fragments in registers)
constexpr int kEntPad = 16;  // zero entries after the last row: blocks past KB of a padded last tile

struct XGeom {
    int G;               // CTAs
    int ntw;             // packed tiles per warp slice (the last warps may take fewer)
    int tpw_max;         // ntw rounded: tiles per warp except possibly the last ones
    int max_rt;          // most row tiles of one CTA
    int D;               // ring slots per warp (2 .. kMaxD)
    int raw_copy;        // scales / zero points by bulk copy (16-byte aligned bases, 16-byte row groups)
    size_t slot_bytes;   // ntw * 512
    size_t raw_s_bytes, raw_z_bytes;  // raw staging of one CTA (max_rt * 16 rows)
    size_t ent_bytes, ring_bytes, raw_bytes, red_bytes, bar_off, total_bytes;
};

// Slices: warp w takes tiles [w * tpw, min((w + 1) * tpw, KTILES)) of every row
// tile; tpw is a multiple of the tiles per quantisation block.
inline bool make_xgeom(const Layout& L, int64_t M, int sms, size_t smem_limit, XGeom* out, int sbytes,
                       bool raw_aligned) {
    XGeom g{};
    if (M < 1 || M > 8) return false;
    const int64_t utiles = L.bs > L.KT ? L.bs / L.KT : 1;
    const int64_t units = (L.KTILES + utiles - 1) / utiles;
    const int64_t upw = (units + kW - 1) / kW;
    g.tpw_max = (int)(upw * utiles);
    if ((int64_t)(kW - 1) * g.tpw_max >= L.KTILES) return false;  // every warp gets a slice
    const int spt = 16 / L.bits;
    if (g.tpw_max * spt != kMaxKS && g.tpw_max * spt != kMaxKS / 2) return false;  // instantiated depths
    if (L.bs / 16 > kMaxKS) return false;
    g.ntw = g.tpw_max;
    g.G = (int)(L.NT < sms ? L.NT : sms);
    g.max_rt = (int)((L.NT + g.G - 1) / g.G);
    g.slot_bytes = (size_t)g.tpw_max * kTileBytes;
    g.ent_bytes = round16(((size_t)g.max_rt * 16 * L.KB + kEntPad) * sizeof(Entry));
    g.red_bytes = (size_t)2 * kW * 16 * 8 * 4;
    // raw copies: every row group of 16 rows must be a multiple of 16 bytes (always true) and the
    // valid rows of a partial last row tile too; the bases must be 16-byte aligned
    g.raw_s_bytes = round16((size_t)g.max_rt * 16 * L.KB * sbytes);
    g.raw_z_bytes = round16((size_t)g.max_rt * 16 * L.zp_row);
    const int64_t tail_rows = L.N % 16;
    g.raw_copy = raw_aligned && (tail_rows == 0 || ((tail_rows * L.KB * sbytes) % 16 == 0 &&
                                                    (tail_rows * L.zp_row) % 16 == 0));
    g.raw_bytes = g.raw_copy ? g.raw_s_bytes + g.raw_z_bytes : 0;
    const size_t fixed = g.ent_bytes + g.raw_bytes + g.red_bytes + (size_t)(kW * kMaxD + 6) * 8 + 128;
    if (g.ent_bytes > (size_t)96 * 1024 || fixed >= smem_limit) return false;
    g.D = (int)((smem_limit - fixed) / ((size_t)kW * g.slot_bytes));
    if (g.D > kMaxD) g.D = kMaxD;
    if (g.D < 2) return false;
    g.ring_bytes = (size_t)kW * g.D * g.slot_bytes;
    g.bar_off = g.ring_bytes + g.ent_bytes + g.raw_bytes + g.red_bytes;
    g.total_bytes = g.bar_off + (size_t)(kW * kMaxD + 6) * 8 + 128;
    *out = g;
    return true;
}

// TPW: packed tiles per warp slice (static); SPB_LOG: log2 k-steps per block.
template <int BITS, bool BF16X, int TPW, int SPB_LOG>
__global__ void __launch_bounds__(kThreads, 1) gemv_xr_kernel(MatmulParams p, XGeom geo, int pdl) {
    using U = Unpack<BITS, BF16X>;
    constexpr int SPT = U::kStepsPerTile;
    constexpr int KSW = TPW * SPT;           // k-steps of a full slice (<= 16)
    constexpr int SPB = 1 << SPB_LOG;        // k-steps per block
    static_assert(KSW <= kMaxKS, "slice too deep");
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;                                                   // [kW][D][slot]
    Entry* ent = reinterpret_cast<Entry*>(smem + geo.ring_bytes);           // [max_rt * 16][KB]
    uint8_t* raw = smem + geo.ring_bytes + geo.ent_bytes;                   // raw scales, then zero points
    float* red = reinterpret_cast<float*>(raw + geo.raw_bytes);             // [2][kW][16][8]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + geo.bar_off);
    uint64_t* ring_full = bars;                 // [kW][kMaxD]
    uint64_t* red_full = bars + kW * kMaxD;     // [2]
    uint64_t* red_free = red_full + 2;          // [2]
    uint64_t* raw_full = red_free + 2;          // [1]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = (int)p.M;

    const int64_t rt0 = (int64_t)blockIdx.x * L.NT / geo.G;
    const int nrt = (int)((int64_t)(blockIdx.x + 1) * L.NT / geo.G - rt0);
    const int64_t tw0 = (int64_t)warp * TPW;
    const int ntw = (int)imin64(TPW, L.KTILES - tw0);      // tiles of this warp's slice (>= 1)
    const uint32_t slice_bytes = (uint32_t)ntw * kTileBytes;
    const int D = geo.D;
    uint8_t* wring = ring + (size_t)warp * D * geo.slot_bytes;
    uint64_t* wbar = ring_full + warp * kMaxD;
    int issued = 0;  // row tiles whose slices lane 0 has requested

    const int sb = p.scale_dtype == kF32 ? 4 : 2;
    const int64_t nrows = imin64((int64_t)nrt * 16, L.N - rt0 * 16);  // valid rows of the CTA
    const uint32_t raw_s = (uint32_t)(nrows * L.KB * sb), raw_z = p.zp ? (uint32_t)(nrows * L.zp_row) : 0u;
    // ---- 1. barriers, the raw scales / zero points of the CTA's rows, then the first D slices
    //         of this warp (constant data: all before the dependency wait) ----
    if (lane == 0) {
        for (int d = 0; d < D; ++d) mbar_init(&wbar[d], 1);
        if (warp == 0) {
            mbar_init(&red_full[0], kW);
            mbar_init(&red_full[1], kW);
            mbar_init(&red_free[0], 1);
            mbar_init(&red_free[1], 1);
            mbar_init(raw_full, 1);
        }
        fence_barrier_init();
        if (warp == 0 && geo.raw_copy && nrows > 0) {
            mbar_arrive_expect_tx(raw_full, raw_s + raw_z);
            bulk_g2s(raw, static_cast<const uint8_t*>(p.scales) + rt0 * 16 * L.KB * sb, raw_s, raw_full);
            if (raw_z) bulk_g2s(raw + geo.raw_s_bytes, p.zp + rt0 * 16 * L.zp_row, raw_z, raw_full);
        }
        for (int d = 0; d < D && d < nrt; ++d) {
            mbar_arrive_expect_tx(&wbar[d], slice_bytes);
            bulk_g2s(wring + d * geo.slot_bytes, p.packed + ((rt0 + d) * L.KTILES + tw0) * kTileBytes, slice_bytes,
                     &wbar[d]);
            ++issued;
        }
    }

    // ---- 2. entries of every (row, block) of this CTA's row tiles ----
    __syncthreads();  // barrier init visible
    {
        const int rows = nrt * 16;
        bool have_raw = geo.raw_copy != 0;
        if (have_raw && nrows > 0 && !mbar_wait_lim(raw_full, 0, p.status, p.wait_limit, p.wait_hint_ns)) have_raw = false;
        for (int rr = warp; rr < rows; rr += kW) {  // local row rr: lanes walk its blocks
            const int64_t n = rt0 * 16 + rr;
            Entry* dst = ent + (size_t)rr * L.KB;
            for (int64_t kb = lane; kb < L.KB; kb += 32) {
                uint32_t zc = U::zconst(0u);
                float sc = 0.f;
                if (n < L.N) {
                    uint32_t z = 1u << (BITS - 1);
                    if (have_raw) {
                        const int64_t i = (int64_t)rr * L.KB + kb;
                        if (sb == 4) sc = reinterpret_cast<const float*>(raw)[i];
                        else if (p.scale_dtype == kF16)
                            sc = __half2float(__ushort_as_half(reinterpret_cast<const unsigned short*>(raw)[i]));
                        else sc = __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(raw)[i] << 16);
                        if (p.zp) {
                            const int64_t bit = kb * BITS;
                            z = (raw[geo.raw_s_bytes + (size_t)rr * L.zp_row + (bit >> 3)] >> (bit & 7)) &
                                (uint32_t)code_mask(BITS);
                        }
                    } else {
                        sc = load_f32(p.scales, n * L.KB + kb, p.scale_dtype);
                        if (p.zp) z = (uint32_t)load_zp(p.zp, L, n, kb);
                    }
                    zc = U::zconst(z);
                }
                dst[kb] = Entry{zc, sc};
            }
        }
        if (tid < kEntPad) ent[(size_t)rows * L.KB + tid] = Entry{U::zconst(0u), 0.f};
    }
    __syncthreads();  // entries visible
    if (pdl) {
        griddep_wait();              // X (and Y) may belong to the previous kernel on the stream
        griddep_launch_dependents();  // after the wait: at most two chained kernels overlap
    }

    // ---- 3. this lane's X fragments of the slice (token g; zeros for g >= M or past K) ----
    uint32_t xb[KSW][2];
    {
        const uint16_t* x16 = static_cast<const uint16_t*>(p.x);
        const int64_t xr = (int64_t)(g < M ? g : 0) * L.K;
#pragma unroll
        for (int s = 0; s < KSW; ++s) {
            const int64_t k0 = (tw0 * SPT + s) * 16 + 2 * t;
            uint32_t v[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t ka = k0 + 8 * h;
                uint32_t lo = 0, hi = 0;
                if (g < M) {
                    if (ka + 1 < L.K && (((xr + ka) & 1) == 0)) {
                        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(x16 + xr + ka));
                        lo = w & 0xFFFFu;
                        hi = w >> 16;
                    } else {
                        lo = ka < L.K ? x16[xr + ka] : 0u;
                        hi = ka + 1 < L.K ? x16[xr + ka + 1] : 0u;
                    }
                }
                v[h] = lo | (hi << 16);
            }
            xb[s][0] = v[0];
            xb[s][1] = v[1];
        }
    }

    // ---- 4. row tiles ----
    const int64_t kb_w0 = tw0 * L.KT / L.bs;  // first block of the slice
    const uint32_t ent_g = smem_u32(ent + (size_t)g * L.KB + kb_w0);
    const uint32_t row_stride = (uint32_t)(16 * L.KB * sizeof(Entry));
    const uint32_t e8 = (uint32_t)(8 * L.KB * sizeof(Entry));
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    auto lds2 = [](uint32_t addr) {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
        return v;
    };
    bool ok = true;
    for (int r = 0; r < nrt && ok; ++r) {
        const int d = r % D;
        if (!mbar_wait_lim(&wbar[d], (uint32_t)((r / D) & 1), p.status, p.wait_limit, p.wait_hint_ns)) {
            ok = false;
            break;
        }
        const uint8_t* slot = wring + d * geo.slot_bytes + lane * 16;
        const uint32_t er = ent_g + (uint32_t)r * row_stride;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        float acc[4];
        uint32_t zg = 0, zg8 = 0;
        float sg = 0.f, sg8 = 0.f;
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
            if (j < ntw) {
                const uint4 wv = *reinterpret_cast<const uint4*>(slot + j * kTileBytes);
#pragma unroll
                for (int s = 0; s < SPT; ++s) {
                    const int S = j * SPT + s;
                    const bool bstart = (S % SPB) == 0;
                    const bool bend = ((S + 1) % SPB) == 0 || S == KSW - 1;
                    if (bstart) {
                        const uint32_t ea = er + (uint32_t)(S / SPB) * (uint32_t)sizeof(Entry);
                        const uint2 eg = lds2(ea), eg8 = lds2(ea + e8);
                        zg = eg.x;
                        sg = __uint_as_float(eg.y);
                        zg8 = eg8.x;
                        sg8 = __uint_as_float(eg8.y);
                    }
                    uint32_t a[4];
                    U::kstep(wv, s, zg, zg8, a);
                    if (bstart) mma16816<BF16X>(acc, a, xb[S][0], xb[S][1], zero4);
                    else mma16816<BF16X>(acc, a, xb[S][0], xb[S][1], acc);
                    if (bend || (S + 1 == ntw * SPT)) {
                        y[0] = fmaf(sg, acc[0], y[0]);
                        y[1] = fmaf(sg, acc[1], y[1]);
                        y[2] = fmaf(sg8, acc[2], y[2]);
                        y[3] = fmaf(sg8, acc[3], y[3]);
                    }
                }
            }
        }
        __syncwarp();
        // the slot is consumed: refill it with row tile r + D
        if (lane == 0 && r + D < nrt) {
            mbar_arrive_expect_tx(&wbar[d], slice_bytes);
            bulk_g2s(wring + d * geo.slot_bytes, p.packed + ((rt0 + r + D) * L.KTILES + tw0) * kTileBytes,
                     slice_bytes, &wbar[d]);
            ++issued;
        }
        // ---- partial sums of row tile r: write, then one warp reduces ----
        const int rb = r & 1;
        if (r >= 2 && !mbar_wait_lim(&red_free[rb], (uint32_t)(((r >> 1) - 1) & 1), p.status, p.wait_limit,
                                    p.wait_hint_ns)) {
            ok = false;
            break;
        }
        float* mine = red + ((size_t)rb * kW + warp) * 16 * 8;
        *reinterpret_cast<float2*>(&mine[g * 8 + 2 * t]) = make_float2(y[0], y[1]);
        *reinterpret_cast<float2*>(&mine[(g + 8) * 8 + 2 * t]) = make_float2(y[2], y[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_full[rb]);
        if (warp == r % kW) {
            if (!mbar_wait_lim(&red_full[rb], (uint32_t)((r >> 1) & 1), p.status, p.wait_limit, p.wait_hint_ns)) {
                ok = false;
                break;
            }
            const float* base = red + (size_t)rb * kW * 16 * 8;
            for (int o = lane; o < 16 * M; o += 32) {
                const int row = o & 15, m = o >> 4;
                float v = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kW; ++w2) v += base[(w2 * 16 + row) * 8 + m];
                const int64_t n = (rt0 + r) * 16 + row;
                if (n < L.N) {
                    if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
                    store_f32(p.y, (int64_t)m * L.N + n, v, p.out_dtype);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&red_free[rb]);
        }
    }
    if (!ok && lane == 0) {
        // copies still in flight must land before the CTA exits (fixed bound):
        // the last request of each slot is row tile issued - 1 - i (i < D)
        for (int i = 0; i < D && i < issued; ++i) {
            const int last = issued - 1 - i;
            for (int it = 0; it < (1 << 16); ++it)
                if (mbar_try_wait_sleep(&wbar[last % D], (uint32_t)((last / D) & 1), 2000)) break;
        }
    }
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status);
}

template <int BITS, bool BF16X, int TPW, int SPB_LOG>
cudaError_t launch_x(const MatmulParams& p, const XGeom& geo, cudaStream_t s) {
    const int pdl = (p.flags & kFlagPDL) ? 1 : 0;
    auto kern = gemv_xr_kernel<BITS, BF16X, TPW, SPB_LOG>;
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

// Instantiated slice depths: 16 k-steps per slice (4 tiles of 4-bit, 2 of
// 2-bit, 8 of 8-bit) and 8 k-steps; block sizes of 1, 2, 4, 8 and 16 k-steps.
template <int BITS, bool BF16X, int TPW>
cudaError_t launch_spb(const MatmulParams& p, const XGeom& geo, cudaStream_t s) {
    switch (p.L.bs / 16) {
        case 1: return launch_x<BITS, BF16X, TPW, 0>(p, geo, s);
        case 2: return launch_x<BITS, BF16X, TPW, 1>(p, geo, s);
        case 4: return launch_x<BITS, BF16X, TPW, 2>(p, geo, s);
        case 8: return launch_x<BITS, BF16X, TPW, 3>(p, geo, s);
        case 16: return launch_x<BITS, BF16X, TPW, 4>(p, geo, s);
        default: return cudaErrorNotSupported;
    }
}

template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const XGeom& geo, cudaStream_t s) {
    constexpr int kFull = 16 / (16 / BITS);  // tiles of a 16-k-step slice: 4 (4-bit), 2 (2-bit), 8 (8-bit)
    const bool bf = p.act_dtype == kBF16;
    if (geo.tpw_max == kFull)
        return bf ? launch_spb<BITS, true, kFull>(p, geo, s) : launch_spb<BITS, false, kFull>(p, geo, s);
    if (geo.tpw_max * 2 == kFull)
        return bf ? launch_spb<BITS, true, kFull / 2>(p, geo, s) : launch_spb<BITS, false, kFull / 2>(p, geo, s);
    return cudaErrorNotSupported;
}

}  // namespace gxr
}  // namespace mnb
