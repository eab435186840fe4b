// Prefill GEMM on 5th-generation tensor cores with exact block-scaled
// accumulation, M >= 1, bf16 or f16 X:
//
//   Y[m, n] = sum_kb scale[n, kb] * ( sum_{k in kb} X[m, k] * (q[n, k] - zp[n, kb]) )   (+ bias[n])
//
// which is MatMulNBits, w = (q - zp) * scale (onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs, fn dequantize_nbits_value), with the block
// scale taken out of the inner sum in the way the page's own int4 / int8 dot
// kernels factor it (int4_dot_row_*, int8_row: one integer-weighted dot per
// block, rescaled once).
//
// Why this form: the tensor core multiplies bf16 (or f16) operands.  (q - zp)
// is a small integer and exact in either type, and a bf16 / f16 activation
// times it is exact in the f32 accumulator, so each block's partial sum is
// exact up to f32 accumulation.  The block scale is then applied in f32.  A
// weight rounded to bf16 before the MMA would carry a relative error of up to
// 2^-8 per weight, more than the per-element bound the library promises;
// this kernel never forms that product.
//
// Tile: 128 W rows (TMEM lanes, the MMA's M) x BT tokens (the MMA's N), K in
// 128-deep stages.  The transposed tile D[n, m] is accumulated per
// quantisation block into one of NP partial accumulators in tensor memory.
//   warp 0       producer: per stage one TMA copy of the X tile (two 64-deep
//                boxes, 128-byte swizzle, zero fill past M and K) and one of
//                the 128 rows' packed codes (a 5-D tensor map that stores each
//                512-byte tile as [chunk t][row group g][16 B], so a warp's
//                rows read distinct shared-memory banks).
//   warp 1       allocates tensor memory and issues the MMAs: per k-step one
//                tcgen05.mma (M = 128, N = BT, K = 16, A from tensor memory, B
//                the X tile in shared memory) into the partial of its block;
//                one commit per block (partial complete) and one per stage
//                (ring slot free).
//   warps 4-11   write A = (q - zp) in the MMA's type into tensor memory: one
//                W row per thread (its TMEM lane), 64 depths of every stage.
//   warps 12-27  rescale: per block, read the partial (one W row per thread,
//                BT / 4 tokens per warp), release it, and add scale * partial
//                into f32 registers with packed FMAs.  Then the epilogue: bias,
//                round to the output type, stores coalesced along N.
// Every mbarrier wait is bounded: on a timeout the kernel records
// MNB_ERR_TIMEOUT, lets its copies and MMAs in flight finish (fixed bound),
// frees tensor memory and returns.  The reduction order over K is fixed, so
// results are deterministic.
#pragma once

#include "tc_ptx.cuh"

namespace mnb {
namespace gbs {

constexpr int kRows = 128;        // W rows per tile = TMEM lanes = MMA M
constexpr int kBK = 128;          // depths per stage
constexpr int kACols = 64;        // TMEM columns of one A stage (128 depths as 16-bit pairs)
constexpr int kCtlWarps = 4;      // producer, MMA issuer, two idle
constexpr int kDqWarps = 8;       // write A
constexpr int kRsWarps = 16;      // rescale + epilogue
constexpr int kThreads = (kCtlWarps + kDqWarps + kRsWarps) * 32;
constexpr int kMaxR = 4;
constexpr int kMaxNP = 4;
// mbarriers, the tensor-memory address and the abort flag
constexpr size_t kBarBytes = (3 * kMaxR + 2 * kMaxNP + 1) * 8 + 16;

struct Geom {
    int BT;             // tokens per tile (MMA N): 32, 64 or 128
    int NP;             // partial accumulators in tensor memory
    int R;              // ring depth: shared-memory X / code slots and TMEM A slots
    int n_tiles, m_tiles;
    int k_stages;       // ceil(KB * bs / 128)
    int tmem_cols;      // allocated columns (power of two)
    int a_col0;         // first column of the A ring (= NP * BT)
    size_t x_stage, wp_stage, total_bytes;
};

struct Maps {
    CUtensorMap x, w;
};

template <int BITS, bool BF16X, int BT>
__global__ void __launch_bounds__(kThreads, 1) gemm_bs_kernel(MatmulParams p, Geom geo,
                                                               const __grid_constant__ CUtensorMap xmap,
                                                               const __grid_constant__ CUtensorMap wmap) {
    constexpr int KT = 256 / BITS;        // depths per packed tile
    constexpr int TILES = kBK / KT;       // packed tiles per 16-row tile per stage: 2-bit 1, 4-bit 2, 8-bit 4
    constexpr int CW = BT / 4;            // token columns per rescale warp
    constexpr uint32_t kMag = BF16X ? 0x43004300u : 0x64006400u;  // 128.0 / 1024.0 in both halves
    const Layout& L = p.L;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int R = geo.R, NP = geo.NP;
    uint8_t* xs = smem;                                    // [R][2][BT x 128 B] (SW128, TMA)
    uint8_t* wp = xs + R * geo.x_stage;                    // [R][8 row tiles][TILES][512 B] (transposed, TMA)
    uint64_t* bars = reinterpret_cast<uint64_t*>(wp + R * geo.wp_stage);
    uint64_t* tma_full = bars;                             // X tile and codes of the slot landed
    uint64_t* a_full = bars + kMaxR;                       // A slot written (kDqWarps arrivals)
    uint64_t* mma_done = bars + 2 * kMaxR;                 // MMAs of the slot's stage finished: slot free
    uint64_t* part_full = bars + 3 * kMaxR;                // partial of a block complete
    uint64_t* part_free = part_full + kMaxNP;              // partial read out (kRsWarps arrivals)
    uint64_t* done = part_free + kMaxNP;                   // every MMA finished
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int n_tile = blockIdx.x % geo.n_tiles;
    const int m_tile = blockIdx.x / geo.n_tiles;
    const int64_t n0 = (int64_t)n_tile * kRows;
    const int64_t m0 = (int64_t)m_tile * BT;
    const int KS = geo.k_stages;
    const int spb = L.bs / 16;                       // k-steps per quantisation block
    const int64_t n_ksteps = L.KB * (int64_t)spb;    // k-steps that carry data
    const uint32_t wl = p.wait_limit, wh = p.wait_hint_ns;

    if (tid == 0) {
        for (int s = 0; s < kMaxR; ++s) {
            mbar_init(&tma_full[s], 1);
            mbar_init(&a_full[s], kDqWarps);
            mbar_init(&mma_done[s], 1);
        }
        for (int b = 0; b < kMaxNP; ++b) {
            mbar_init(&part_full[b], 1);
            mbar_init(&part_free[b], kRsWarps);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tc::alloc(tmem_slot, (uint32_t)geo.tmem_cols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t a_base = tmem + (uint32_t)geo.a_col0;
    volatile int* abort_v = abort_flag;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(geo.x_stage + geo.wp_stage);
            const int nrt = (int)(n0 / 16);
            int issued = 0;
            for (int ks = 0; ks < KS; ++ks) {
                const int s = ks % R;
                const uint32_t ph = (uint32_t)((ks / R) & 1);
                if (ks >= R && !tc::wait_bounded(&mma_done[s], ph ^ 1u, p.status, wl, wh)) {
                    *abort_v = 1;
                    break;
                }
                if (*abort_v) break;
                mbar_arrive_expect_tx(&tma_full[s], bytes);
                uint8_t* xd = xs + s * geo.x_stage;
                tc::tma_load_2d(xd, &xmap, ks * kBK, (int)m0, &tma_full[s]);
                tc::tma_load_2d(xd + BT * 128, &xmap, ks * kBK + 64, (int)m0, &tma_full[s]);
                tc::tma_load_5d(wp + s * geo.wp_stage, &wmap, 0, 0, 0, ks * TILES, nrt, &tma_full[s]);
                issued = ks + 1;
            }
            if (*abort_v) {  // let the copies in flight land before the CTA can exit
                for (int ks = issued - R < 0 ? 0 : issued - R; ks < issued; ++ks)
                    tc::drain_wait(&tma_full[ks % R], (uint32_t)((ks / R) & 1));
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = tc::idesc_f16(BF16X, kRows, BT);
        const uint64_t dx0 = tc::sdesc_sw128(smem_u32(xs));
        const uint64_t x_step = geo.x_stage >> 4;
        const uint64_t x_half = (uint64_t)(BT * 128) >> 4;
        bool ok = true;
        int64_t gk = 0;  // global k-step
        for (int ks = 0; ks < KS && ok; ++ks) {
            const int s = ks % R;
            const uint32_t ph = (uint32_t)((ks / R) & 1);
            if (!tc::wait_bounded(&a_full[s], ph, p.status, wl, wh)) {
                ok = false;
                break;
            }
            tc::fence_after();
            if (lane == 0) {
                const uint64_t dxs = dx0 + (uint64_t)s * x_step;
                const uint32_t as = a_base + (uint32_t)(s * kACols);
                for (int kk = 0; kk < 8; ++kk, ++gk) {
                    if (gk >= n_ksteps) continue;
                    const int64_t b = gk / spb;
                    const int within = (int)(gk - b * spb);
                    const int pb = (int)(b % NP);
                    if (within == 0 && b >= NP) {
                        if (!tc::wait_bounded(&part_free[pb], (uint32_t)(((b / NP) - 1) & 1), p.status, wl, wh)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after();
                    }
                    const uint64_t bd = dxs + (uint64_t)(kk & 3) * 2 + (uint64_t)(kk >> 2) * x_half;
                    tc::mma_ta(tmem + (uint32_t)(pb * BT), as + (uint32_t)kk * 8u, bd, idesc, within ? 1u : 0u);
                    if (within == spb - 1) tc::commit(&part_full[pb]);
                }
                tc::commit(&mma_done[s]);
            } else {
                gk += 8;
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        if (!ok) *abort_v = 1;
        // every MMA this thread issued must finish before tensor memory is freed
        if (lane == 0) {
            tc::commit(done);
            tc::drain_wait(done, 0);
        }
        __syncwarp();
    } else if (warp >= kCtlWarps && warp < kCtlWarps + kDqWarps) {
        // ---------------- A = (q - zp), one W row per thread ----------------
        const int dw = warp - kCtlWarps;
        const int q4 = warp & 3;        // TMEM lane quadrant of this warp
        const int jh = dw >> 2;         // k-steps 4 jh .. 4 jh + 3 of every stage
        const int r = q4 * 32 + lane;   // W row inside the tile = TMEM lane
        const int rt = r >> 4, g = r & 7, hi = (r >> 3) & 1;
        const int64_t n = n0 + r;
        const bool row_ok = n < L.N;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        const int zmask = code_mask(BITS);
        const int nb = L.bs >= 64 ? 1 : 64 / L.bs;  // blocks in a thread's 64 depths of a stage
        // raw zero-point bytes of the blocks of stage ks (at most 4), fetched a stage ahead
        auto zp_fetch = [&](int ks, uint32_t (&zb)[4]) {
            const int64_t fb = ((int64_t)ks * kBK + 64 * jh) / L.bs;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t kb = fb + i;
                zb[i] = 0;
                if (p.zp && row_ok && i < nb && kb < L.KB)
                    zb[i] = __ldg(p.zp + n * L.zp_row + ((kb * BITS) >> 3));
            }
        };
        uint32_t zb_next[4];
        zp_fetch(0, zb_next);
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks) {
            const int s = ks % R;
            const uint32_t ph = (uint32_t)((ks / R) & 1);
            uint32_t zb[4] = {zb_next[0], zb_next[1], zb_next[2], zb_next[3]};
            if (ks + 1 < KS) zp_fetch(ks + 1, zb_next);
            if (ks >= R && !tc::wait_bounded(&mma_done[s], ph ^ 1u, p.status, wl, wh)) {
                ok = false;
                break;
            }
            if (!tc::wait_bounded(&tma_full[s], ph, p.status, wl, wh)) {
                ok = false;
                break;
            }
            if (*abort_v) break;
            // subtraction constant (magic + zp) of each of the thread's four k-steps
            uint32_t zc[4];
            {
                const int64_t fb = ((int64_t)ks * kBK + 64 * jh) / L.bs;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int64_t kb = ((int64_t)ks * kBK + 64 * jh + 16 * kk) / L.bs;
                    const int i = (int)(kb - fb);
                    uint32_t z = 1u << (BITS - 1);
                    if (p.zp) z = (zb[i & 3] >> ((kb * BITS) & 7)) & (uint32_t)zmask;
                    if constexpr (BITS == 8 && BF16X) zc[kk] = 0x4B000000u | z;  // f32 2^23 + z
                    else zc[kk] = ((kMag & 0xFFFFu) + z) * 0x10001u;
                }
            }
            // codes: chunk t of packed tile tl at tl * 512 + t * 128 + g * 16 of the row tile
            const uint8_t* cb = wp + s * geo.wp_stage + rt * TILES * kTileBytes + g * 16;
            uint32_t v[32];  // column 8 kk + c of the thread's half stage: depths 2c, 2c + 1 of k-step kk
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if constexpr (BITS == 4) {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(cb + jh * kTileBytes + t * 128);
                    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t ws = w[kk] >> (4 * hi);
                        v[8 * kk + t] = tc::hsub2(lop3_and_or(ws, 0x000F000Fu, kMag), zc[kk], BF16X);
                        v[8 * kk + t + 4] = tc::hsub2(lop3_and_or(ws >> 8, 0x000F000Fu, kMag), zc[kk], BF16X);
                    }
                } else if constexpr (BITS == 2) {
                    const uint2 w2 = *reinterpret_cast<const uint2*>(cb + t * 128 + 8 * jh);
                    const uint32_t w[2] = {w2.x, w2.y};
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const int f = 4 * (kk & 1) + hi + 2 * hf;
                            v[8 * kk + t + 4 * hf] =
                                tc::hsub2(lop3_and_or(w[kk >> 1] >> (2 * f), 0x00030003u, kMag), zc[kk], BF16X);
                        }
                    }
                } else {
#pragma unroll
                    for (int tp = 0; tp < 2; ++tp) {  // two packed tiles (2 k-steps each) per half stage
                        const uint4 w4 = *reinterpret_cast<const uint4*>(cb + (2 * jh + tp) * kTileBytes + t * 128);
                        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int ss = 0; ss < 2; ++ss) {
                            const int kk = 2 * tp + ss;
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const uint32_t word = w[2 * ss + hf];
                                const uint32_t b0 = 2 * hi, b1 = b0 + 1;
                                uint32_t qv;
                                if constexpr (BF16X) {
                                    const uint32_t va = prmt(word, 0x4B000000u, 0x7650u | b0);
                                    const uint32_t vb = prmt(word, 0x4B000000u, 0x7650u | b1);
                                    const float2 d = unpack2(fsub2(pack2u(va, vb), pack2u(zc[kk], zc[kk])));
                                    qv = tc::cvt_bf16x2(d.x, d.y);  // |q - zp| <= 255: exact in bf16
                                } else {
                                    qv = tc::hsub2(prmt(word, 0x64646464u, b0 | (4u << 4) | (b1 << 8) | (4u << 12)),
                                                   zc[kk], false);
                                }
                                v[8 * kk + t + 4 * hf] = qv;
                            }
                        }
                    }
                }
            }
            tc::st_32x32b_x32(a_base + (uint32_t)(s * kACols + 32 * jh) + lane_addr, v);
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[s]);
        }
        if (!ok) *abort_v = 1;
    } else if (warp >= kCtlWarps + kDqWarps) {
        // ---------------- rescale: y += scale * partial, then the epilogue ----------------
        const int rw = warp - kCtlWarps - kDqWarps;
        const int q4 = warp & 3;
        const int cs = rw >> 2;           // token columns cs * CW .. cs * CW + CW - 1
        const int r = q4 * 32 + lane;
        const int64_t n = n0 + r;
        const bool row_ok = n < L.N;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        const int sdt = p.scale_dtype;
        auto scale_at = [&](int64_t b) -> float {
            return (row_ok && b < L.KB) ? load_f32(p.scales, n * L.KB + b, sdt) : 0.f;
        };
        uint64_t y2[CW / 2];
#pragma unroll
        for (int i = 0; i < CW / 2; ++i) y2[i] = 0;
        float s0 = scale_at(0), s1 = scale_at(1), s2 = scale_at(2);
        bool ok = true;
        for (int64_t b = 0; b < L.KB; ++b) {
            const int pb = (int)(b % NP);
            if (!tc::wait_bounded(&part_full[pb], (uint32_t)((b / NP) & 1), p.status, wl, wh)) {
                ok = false;
                break;
            }
            if (*abort_v) break;
            tc::fence_after();
            const float sc = s0;
            s0 = s1;
            s1 = s2;
            s2 = scale_at(b + 3);
            const uint64_t sc2 = pack2(sc, sc);
            // the partial in chunks of up to 16 columns (register pressure)
            constexpr int CH = CW < 16 ? CW : 16;
#pragma unroll
            for (int c0 = 0; c0 < CW; c0 += CH) {
                uint32_t P[CH];
                tc::ld_32x32b<CH>(tmem + (uint32_t)(pb * BT + cs * CW + c0) + lane_addr, P);
                tc::wait_ld();
                if (c0 + CH == CW) {  // the whole partial is in registers: release it
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&part_free[pb]);
                }
#pragma unroll
                for (int i = 0; i < CH / 2; ++i) {
                    y2[c0 / 2 + i] = ffma2(pack2u(P[2 * i], P[2 * i + 1]), sc2, y2[c0 / 2 + i]);
                }
            }
        }
        if (!ok) *abort_v = 1;
        if (ok && !*abort_v && row_ok) {
            const float bias = p.bias ? load_f32(p.bias, n, p.bias_dtype) : 0.f;
#pragma unroll
            for (int i = 0; i < CW / 2; ++i) {
                const float2 v = unpack2(y2[i]);
                const int64_t m = m0 + cs * CW + 2 * i;
                if (m < p.M) store_f32(p.y, m * L.N + n, v.x + bias, p.out_dtype);
                if (m + 1 < p.M) store_f32(p.y, (m + 1) * L.N + n, v.y + bias, p.out_dtype);
            }
        }
    }

    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, (uint32_t)geo.tmem_cols);
    }
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status, kWfInt, p.kperm != nullptr ? 1 : 0);
}

template <int BITS, bool BF16X>
cudaError_t launch(const MatmulParams& p, const Geom& geo, const Maps& m, cudaStream_t s) {
    auto go = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)(geo.n_tiles * geo.m_tiles), kThreads, geo.total_bytes, s>>>(p, geo, m.x, m.w);
        return cudaGetLastError();
    };
    switch (geo.BT) {
        case 32: return go(gemm_bs_kernel<BITS, BF16X, 32>);
        case 64: return go(gemm_bs_kernel<BITS, BF16X, 64>);
        default: return go(gemm_bs_kernel<BITS, BF16X, 128>);
    }
}

}  // namespace gbs
}  // namespace mnb
