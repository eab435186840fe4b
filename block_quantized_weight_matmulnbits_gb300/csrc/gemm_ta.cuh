// Prefill GEMM with the dequantised weights in tensor memory (tcgen05, A
// operand from TMEM):  Y^T tile [128 W rows x BT tokens] = W_tile . X_tile^T,
// w = (q - zp) * scale as in onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs, fn dequantize_nbits_value.
//
// Why: with W as the B operand in shared memory (gemm_tc.cuh) every stage
// writes the dequantised tile into shared memory and the MMA reads it back,
// and together with the X tile and the packed codes that is ~67 KB of
// shared-memory traffic per 64-deep stage at BN = 112 - the kernel's floor.
// Here W is the MMA's A operand (M = 128 W rows) and lives in tensor memory:
// each dequantising thread owns one W row (one TMEM lane) and writes its 32
// bf16 pairs per stage with one tcgen05.st; X (BT tokens) is the B operand
// read from shared memory as staged by TMA.  Shared memory then carries only
// the X tile (TMA write + MMA read) and the packed codes (TMA write + one
// read).
//
//   warp 0      : producer (TMA X tile, TMA packed codes of the 128 rows, raw
//                 scales / zero points SB blocks at a time).  The packed codes
//                 are loaded through a 5-D tensor map that stores each 512-byte
//                 tile as [chunk t][row group g][16 bytes] instead of the
//                 global [g][t]: a warp's rows then read distinct banks.
//   warp 1      : TMEM owner and MMA issuer: per 128-deep stage 8 MMAs
//                 (M = 128, N = BT, K = 16) from the A slot of the stage,
//                 one commit per stage.  It waits only for the A slot: every
//                 dequantising warp saw the stage's TMA barrier complete before
//                 it arrived, so the X tile has landed too.  Its loop has a
//                 fixed cost per stage, hence the deep stages.
//   warps 2-3   : idle.
//   warps 4-19  : dequantise; warp (quadrant q = warp % 4, j = (warp - 4) / 4)
//                 writes TMEM lanes 32q..32q+31 (W rows), k-steps 2j, 2j+1
//                 of every stage.  Then the epilogue: tcgen05.ld of the
//                 accumulator (lane = W row, column = token), bias, RNE,
//                 coalesced stores along N.
// Every mbarrier wait is bounded (MNB_ERR_TIMEOUT, bounded drain of copies in
// flight, TMEM freed); the K order is fixed, so results are deterministic.
#pragma once

#include "gemm_tc.cuh"

namespace mnb {
namespace gtc {

constexpr int kTaRows = 128;  // W rows per tile (the MMA's M)

__device__ __forceinline__ void tc_mma_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// Packed codes of one stage through the 5-D map {16 B, g, t, k tile, row tile}.
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, int kt, int rt, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(0), "r"(0), "r"(0), "r"(kt), "r"(rt), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// SPB_LOG: log2 of 16-deep k-steps per quantisation block, 3 meaning "at least
// 8" (one block per 128 depths or more).
template <int BITS, bool BF16X, int SPB_LOG>
__global__ void __launch_bounds__(kThreads, 1) gemm_ta_kernel(MatmulParams p, TcGeom geo,
                                                               const __grid_constant__ CUtensorMap xmap,
                                                               const __grid_constant__ CUtensorMap wmap,
                                                               const __grid_constant__ CUtensorMap smap,
                                                               const __grid_constant__ CUtensorMap zmap) {
    constexpr int KT = 256 / BITS;
    constexpr int BKC = 128;                         // depths per stage
    constexpr int TILES = BKC / KT;                  // packed tiles per 16-row tile per stage
    constexpr int SSTAGE = BKC / 16;                 // 16-deep k-steps per stage
    constexpr uint32_t kMag = BF16X ? 0x43004300u : 0x64006400u;
    constexpr int NB = (SSTAGE >> SPB_LOG) > 0 ? (SSTAGE >> SPB_LOG) : 1;  // blocks per stage
    constexpr int A_COLS = SSTAGE * 8;               // TMEM columns of one A stage
    const Layout& L = p.L;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int R = geo.R;
    const int BT = geo.BN;  // tokens per tile (the MMA's N)
    uint8_t* xs = smem;                                   // [R][BK/64][BT x 64] bf16, SW128 (TMA)
    uint8_t* wp = xs + R * geo.x_stage;                   // [R][8][TILES][512 B] packed codes (TMA)
    uint8_t* sraw = wp + R * geo.wp_stage;                // [2][128][sb] raw scales
    uint8_t* zraw = sraw + 2 * geo.sraw_bytes;            // [2][128][sb * bits / 8] raw zero points
    uint64_t* bars = reinterpret_cast<uint64_t*>(zraw + 2 * geo.zraw_bytes);
    uint64_t* tma_full = bars;                            // X tile + packed codes landed
    uint64_t* a_full = bars + kMaxR;                      // A slot written (4 quadrant warps)
    uint64_t* mma_done = bars + 2 * kMaxR;                // MMAs of the stage finished: slots free
    uint64_t* raw_full = bars + 3 * kMaxR;                // raw scale buffer b landed
    uint64_t* done = raw_full + 2;                        // accumulator complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int BK = geo.BK;
    const int n_tile = blockIdx.x % geo.n_tiles;
    const int m_tile = blockIdx.x / geo.n_tiles;
    const int64_t n0 = (int64_t)n_tile * kTaRows;
    const int64_t m0 = (int64_t)m_tile * BT;
    const int KS = geo.k_stages;

    if (tid == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&tma_full[s], 1);
            mbar_init(&a_full[s], kDqWarps);
            mbar_init(&mma_done[s], 1);
        }
        mbar_init(&raw_full[0], 1);
        mbar_init(&raw_full[1], 1);
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(geo.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;  // accumulator at columns [0, BT); A ring after it
    const uint32_t a_base = tmem + (uint32_t)geo.a_col0;  // first column of the A ring
    volatile int* abort_v = abort_flag;
    const int SB = geo.sb, G = geo.sb_stages;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(geo.x_stage + geo.wp_stage);
            const int nrt = (int)(n0 / 16);
            int s = 0, issued = 0;
            uint32_t ph = 0;
            const int nq = (int)((L.KB + SB - 1) / SB);
            const uint32_t rbytes = (uint32_t)(geo.sraw_bytes + (p.zp ? geo.zraw_bytes : 0));
            int q_next = 0;
            auto issue_raw = [&](int q) {
                const int b = q & 1;
                mbar_arrive_expect_tx(&raw_full[b], rbytes);
                tma_load_2d(sraw + b * geo.sraw_bytes, &smap, q * SB, (int)n0, &raw_full[b]);
                if (p.zp) tma_load_2d(zraw + b * geo.zraw_bytes, &zmap, q * SB * BITS / 8, (int)n0, &raw_full[b]);
            };
            for (; q_next < nq && q_next < 2; ++q_next) issue_raw(q_next);
            for (int ks = 0; ks < KS; ++ks) {
                if (ks >= R && !mbar_wait(&mma_done[s], ph ^ 1u, p.status)) {
                    *abort_v = 1;
                    break;
                }
                if (*abort_v) break;
                const int stages_done = ks >= R ? ks - R + 1 : 0;
                for (; q_next < nq && (q_next - 1) * G <= stages_done; ++q_next) issue_raw(q_next);
                mbar_arrive_expect_tx(&tma_full[s], bytes);
                uint8_t* xd = xs + s * geo.x_stage;
                tma_load_2d(xd, &xmap, ks * BK, (int)m0, &tma_full[s]);
                tma_load_2d(xd + BT * 128, &xmap, ks * BK + 64, (int)m0, &tma_full[s]);
                tma_load_5d(wp + s * geo.wp_stage, &wmap, ks * TILES, nrt, &tma_full[s]);
                issued = ks + 1;
                if (++s == R) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_v) {
                for (int ks = issued - R < 0 ? 0 : issued - R; ks < issued; ++ks)
                    for (int it = 0; it < (1 << 16); ++it)
                        if (mbar_try_wait(&tma_full[ks % R], (uint32_t)((ks / R) & 1))) break;
                for (int q = q_next - 2 < 0 ? 0 : q_next - 2; q < q_next; ++q)
                    for (int it = 0; it < (1 << 16); ++it)
                        if (mbar_try_wait(&raw_full[q & 1], (uint32_t)((q >> 1) & 1))) break;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = idesc_f16(BF16X, BT);
        const uint64_t dx0 = sdesc_sw128(smem_u32(xs));
        const uint64_t x_step = geo.x_stage >> 4;
        const uint64_t x_half = (uint64_t)(BT * 128) >> 4;
        uint64_t dxs = dx0;
        uint32_t as = a_base;
        int s = 0;
        uint32_t ph = 0;
        for (int ks = 0; ks < KS; ++ks) {
            if (!mbar_wait(&a_full[s], ph, p.status)) {
                *abort_v = 1;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < SSTAGE; ++kk) {
                    const uint64_t bd = dxs + (uint64_t)(kk & 3) * 2 + (kk >> 2) * x_half;
                    tc_mma_ta(tmem, as + (uint32_t)kk * 8u, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&mma_done[s]);
            }
            __syncwarp();
            if (++s == R) {
                s = 0;
                ph ^= 1u;
                dxs = dx0;
                as = a_base;
            } else {
                dxs += x_step;
                as += A_COLS;
            }
        }
        if (lane == 0) tc_commit(done);
        __syncwarp();
    } else if (warp >= kCtlWarps) {
        // ---------------- dequantiser (one W row per thread), then epilogue ----------------
        const int dw = warp - kCtlWarps;
        const int q4 = warp & 3;       // TMEM lane quadrant of this warp
        const int jw = dw >> 2;        // k-steps 2 jw, 2 jw + 1 of every stage
        const int r = q4 * 32 + lane;  // W row inside the tile = TMEM lane
        const int rt = r >> 4, g = r & 7, hi = (r >> 3) & 1;
        const int bs_log = __ffs(L.bs) - 1;
        const int g_log = __ffs(G) - 1;
        const int sdt = p.scale_dtype;
        const int zmask = code_mask(BITS);
        const int zrow = SB * BITS / 8;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        constexpr int NBW = (2 >> SPB_LOG) > 0 ? (2 >> SPB_LOG) : 1;  // blocks in the warp's two k-steps
        bool ok = true;
        int q_cur = -1;
        int s = 0;
        uint32_t ph = 0;
        for (int ks = 0; ks < KS; ++ks) {
            if (ks >= R && !mbar_wait(&mma_done[s], ph ^ 1u, p.status)) {
                ok = false;
                break;
            }
            if (!mbar_wait(&tma_full[s], ph, p.status)) {
                ok = false;
                break;
            }
            const int q = ks >> g_log;
            if (q != q_cur) {
                if (!mbar_wait(&raw_full[q & 1], (uint32_t)((q >> 1) & 1), p.status)) {
                    ok = false;
                    break;
                }
                q_cur = q;
            }
            // this row's constants for the blocks of k-steps 2 jw, 2 jw + 1
            uint32_t zc[NBW], sp[NBW];
            {
                const int kl0 = (int)((((int64_t)ks * BKC + 32 * jw) >> bs_log) - ((int64_t)q * SB));
                const uint8_t* sbuf = sraw + (q & 1) * geo.sraw_bytes;
                const uint8_t* zbuf = zraw + (q & 1) * geo.zraw_bytes;
#pragma unroll
                for (int j = 0; j < NBW; ++j) {
                    const int idx = r * SB + kl0 + j;
                    float sc;
                    if (sdt == kF32) {
                        sc = reinterpret_cast<const float*>(sbuf)[idx];
                    } else {
                        const unsigned short v = reinterpret_cast<const unsigned short*>(sbuf)[idx];
                        sc = sdt == kF16 ? __half2float(__ushort_as_half(v)) : __uint_as_float((uint32_t)v << 16);
                    }
                    uint32_t z = 1u << (BITS - 1);
                    if (p.zp) {
                        const uint32_t bit = (uint32_t)(kl0 + j) * BITS;
                        z = ((uint32_t)zbuf[r * zrow + (bit >> 3)] >> (bit & 7)) & zmask;
                    }
                    sp[j] = to_pair(sc, BF16X);
                    if constexpr (BITS == 8 && BF16X) zc[j] = 0x4B000000u | z;
                    else zc[j] = ((kMag & 0xFFFFu) + z) * 0x10001u;
                }
            }
            // the row's codes (rows g and g + 8 share them): chunk t of packed tile tl
            // at tl * 512 + t * 128 + g * 16 (the transposed tile layout of the load)
            const uint8_t* cb = wp + s * geo.wp_stage + rt * TILES * kTileBytes + g * 16;
            uint32_t v[16];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                // this thread's code words of k-steps 2 jw, 2 jw + 1 in chunk t, in one load:
                //   4-bit: packed tile jw / 2, words 2 (jw % 2) + ss
                //   2-bit: packed tile 0, word jw (both k-steps)
                //   8-bit: packed tile jw, words 2 ss + half
                uint32_t wd[4];
                if constexpr (BITS == 4) {
                    const uint2 w2 = *reinterpret_cast<const uint2*>(cb + (jw >> 1) * kTileBytes + t * 128 + 8 * (jw & 1));
                    wd[0] = w2.x;
                    wd[1] = w2.y;
                } else if constexpr (BITS == 2) {
                    wd[0] = *reinterpret_cast<const uint32_t*>(cb + t * 128 + 4 * jw);
                } else {
                    const uint4 w4 = *reinterpret_cast<const uint4*>(cb + jw * kTileBytes + t * 128);
                    wd[0] = w4.x;
                    wd[1] = w4.y;
                    wd[2] = w4.z;
                    wd[3] = w4.w;
                }
#pragma unroll
                for (int ss = 0; ss < 2; ++ss) {
                    const int j = (ss >> SPB_LOG) < NBW ? (ss >> SPB_LOG) : 0;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t pr;
                        if constexpr (BITS == 4) {
                            const uint32_t x = lop3_and_or(wd[ss] >> (4 * (hi + 2 * half)), 0x000F000Fu, kMag);
                            pr = hmul2(hsub2(x, zc[j], BF16X), sp[j], BF16X);
                        } else if constexpr (BITS == 2) {
                            const int f = 4 * ss + hi + 2 * half;
                            const uint32_t x = lop3_and_or(wd[0] >> (2 * f), 0x00030003u, kMag);
                            pr = hmul2(hsub2(x, zc[j], BF16X), sp[j], BF16X);
                        } else {
                            const uint32_t word = wd[2 * ss + half];
                            const uint32_t b0 = 2 * hi, b1 = b0 + 1;
                            uint32_t qv;
                            if constexpr (BF16X) {
                                const uint32_t va = prmt(word, 0x4B000000u, 0x7650u | b0);
                                const uint32_t vb = prmt(word, 0x4B000000u, 0x7650u | b1);
                                const float2 d = unpack2(fsub2(pack2u(va, vb), pack2u(zc[j], zc[j])));
                                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(qv) : "f"(d.y), "f"(d.x));
                            } else {
                                qv = hsub2(prmt(word, 0x64646464u, b0 | (4u << 4) | (b1 << 8) | (4u << 12)), zc[j],
                                           BF16X);
                            }
                            pr = hmul2(qv, sp[j], BF16X);
                        }
                        v[ss * 8 + 4 * half + t] = pr;  // depths 16 st + 2t + 8 half (+1), st = 2 jw + ss
                    }
                }
            }
            tc_st16(a_base + (uint32_t)(s * A_COLS + 16 * jw) + lane_addr, v);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[s]);
            if (++s == R) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) *abort_v = 1;

        // ---------------- epilogue: TMEM (lane = W row, column = token) -> Y ----------------
        if (ok && !*abort_v && mbar_wait(done, 0, p.status)) {
            tc_fence_after();
            const int64_t n = n0 + r;
            float bias = 0.f;
            if (p.bias && n < L.N) bias = load_f32(p.bias, n, p.bias_dtype);
            for (int c0 = jw * 16; c0 < BT; c0 += 64) {
                uint32_t rr[16];
                tc_ld16(tmem + lane_addr + (uint32_t)c0, rr);
                if (n < L.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int64_t m = m0 + c0 + j;
                        if (m < p.M) store_f32(p.y, m * L.N + n, __uint_as_float(rr[j]) + bias, p.out_dtype);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(geo.tmem_cols)
                     : "memory");
    }
}

template <int BITS, bool BF16X>
cudaError_t launch_ta(const MatmulParams& p, const TcGeom& geo, const Maps& m, cudaStream_t s) {
    const int spb = p.L.bs / 16;
    const int spb_log = spb >= 8 ? 3 : (spb == 4 ? 2 : (spb == 2 ? 1 : 0));
    auto pick = [&](auto kern) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)(geo.n_tiles * geo.m_tiles), kThreads, geo.total_bytes, s>>>(p, geo, m.x, m.w, m.s, m.z);
        return cudaGetLastError();
    };
    switch (spb_log) {
        case 0: return pick(gemm_ta_kernel<BITS, BF16X, 0>);
        case 1: return pick(gemm_ta_kernel<BITS, BF16X, 1>);
        case 2: return pick(gemm_ta_kernel<BITS, BF16X, 2>);
        default: return pick(gemm_ta_kernel<BITS, BF16X, 3>);
    }
}

}  // namespace gtc
}  // namespace mnb
