// Prefill GEMM for bf16 activations on 5th-generation tensor cores, with the
// weight carried exactly enough as a sum of two bf16 values:
//
//   w = (q - zp) * scale                      (onnx-runtime-ep-cpu 0.1.0-dev.5,
//                                              src/kernels/matmul_nbits.rs, fn dequantize_nbits_value)
//   w ~ hi + lo,   |w - (hi + lo)| <= 2^-15 |w|
//   Y^T tile = A_hi . X^T + A_lo . X^T        (two bf16 MMAs per k-step, one f32 accumulator)
//
// Why: a weight rounded once to bf16 carries a relative error of up to 2^-8,
// above the per-element bound of the library (2e-3 of sum |x w|); hi + lo is
// within 2^-15.  The split costs three packed bf16 operations per pair of
// weights and is exact where it must be:
//   qz  = q - zp                              (exact: a small integer)
//   s   = s_hi + s_lo (+ at most 2^-16 |s|)   (s_hi = bf16(s), s_lo = bf16(s - s_hi), per block)
//   hi  = RN(qz * s_hi)                       (mul.rn.bf16x2)
//   r   = RN(qz * s_hi - hi)                  (fma.rn.bf16x2; the rounding error of a product of
//                                              two 8-bit significands fits 8 bits: exact)
//   lo  = RN(qz * s_lo + r)                   (fma.rn.bf16x2; |lo| <~ 2^-7 |w|, error <= 2^-8 |lo|)
// and the tensor core multiplies bf16 by bf16 exactly and accumulates in f32.
//
// Tile: 128 W rows (TMEM lanes, the MMA's M) x BT = 256 tokens (the MMA's N,
// the width at which tcgen05.mma runs at full rate on GB300), K in 64-deep
// stages.  When one tile per CTA leaves SMs idle, the K range is split
// between the two CTAs of a cluster, which add their accumulators through
// distributed shared memory in a fixed order.
//   warp 0       producer: per stage one TMA copy of the X tile (64-deep box,
//                128-byte swizzle, zero fill past M and K) and one of the 128
//                rows' packed codes (5-D tensor map: each 512-byte tile as
//                [chunk t][row group g][16 B]).
//   warp 1       allocates tensor memory; issues, per stage, 4 k-steps x
//                (hi, lo) MMAs (M = 128, N = BT, K = 16) from the stage's A
//                slot and one commit that frees the slot.
//   warps 4-11   write A_hi, A_lo for one W row per thread (its TMEM lane),
//                32 depths of every stage each; then the epilogue.
//
// TF32 variant (accuracy level 4 above 16 rows): X holds the activations as
// the per-block int8 codes times their block scales (onnx-runtime-ep-cpu
// matmul_nbits.rs, fn quantize_activation_signed: x ~ code * s_a), rounded to
// tf32 by the quantising kernel, and A holds w = (q - zp) * scale rounded to
// tf32: one kind::tf32 MMA (K = 8) per 8 depths, BT = 256 tokens, a 64 KB X
// stage (f32) and a ring of three stages, A slots of 64 columns (one per
// depth).  Each
// operand carries at most 2^-11 relative error, so a product is within
// 2^-10 of x * w, inside the library's bound, and no per-block rescale of a
// partial is needed (the block scales are in the operands).
// Every mbarrier wait is bounded (MNB_ERR_TIMEOUT, copies and MMAs in flight
// drained with a fixed bound, tensor memory freed).  Reduction orders are
// fixed, so results are deterministic.
#pragma once

#include "tc_ptx.cuh"

namespace mnb {
namespace ghl {

constexpr int kRows = 128;       // W rows per tile = TMEM lanes = MMA M
constexpr int kBT = 256;         // tokens per tile = MMA N
constexpr int kBK = 64;          // depths per stage (4 k-steps)
constexpr int kACols = 64;       // TMEM columns of one A slot: A_hi (32) then A_lo (32)
constexpr int kCtlWarps = 4;
constexpr int kDqWarps = 16;
constexpr int kKK = 16 / kDqWarps;  // k-steps a dequant warp writes per stage
constexpr int kThreads = (kCtlWarps + kDqWarps) * 32;
constexpr int kR = 4;            // ring depth (shared-memory stages and TMEM A slots)
constexpr int kXStage = kBT * kBK * 2;  // 32 KB
// mbarriers, tensor-memory address and abort flag
__host__ __device__ constexpr size_t hl_bar_bytes(int r) { return (3 * r + 1) * 8 + 16; }

struct Geom {
    int ystore;         // 1: Y written by TMA from a shared-memory stage (Maps::y valid)
    int pdl;            // launched as a programmatic dependent: X is read only after the dependency wait
    int n_tiles, m_tiles;
    int splitk;         // 1, or 2: the two CTAs of a cluster take halves of K
    int k_stages;       // stages of the whole K (ceil(Kpad / 64))
    size_t wp_stage, total_bytes;
};

struct Maps {
    CUtensorMap x, w, y;
};

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// s -> (s_hi, s_lo) bf16 pairs (both halves equal): s_hi = RN(s), s_lo = RN(s - s_hi).
__device__ __forceinline__ void split_scale(float s, uint32_t* hi2, uint32_t* lo2) {
    const uint32_t h = tc::cvt_bf16x2(s, s);
    const float hf = __uint_as_float(h << 16);
    const float rest = s - hf;  // exact in f32
    *hi2 = h;
    *lo2 = tc::cvt_bf16x2(rest, rest);
}

template <int BITS, bool TF32>
__global__ void __launch_bounds__(kThreads, 1) gemm_hl_kernel(MatmulParams p, Geom geo,
                                                               const __grid_constant__ CUtensorMap xmap,
                                                               const __grid_constant__ CUtensorMap wmap,
                                                               const __grid_constant__ CUtensorMap ymap) {
    constexpr int KT = 256 / BITS;                  // depths per packed tile
    constexpr int TILES = kBK >= KT ? kBK / KT : 1;  // packed tiles per 16-row tile per stage
    constexpr uint32_t kMag = 0x43004300u;           // bf16 128.0 in both halves
    constexpr int BT = kBT;                           // tokens per tile (MMA N)
    constexpr int R = TF32 ? 3 : kR;                  // ring depth
    constexpr int XST = TF32 ? 2 * kXStage : kXStage; // X bytes per stage (f32 in the tf32 variant)
    const Layout& L = p.L;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* xs = smem;                                      // [R][BT x 128 B] (SW128, TMA)
    uint8_t* wp = xs + R * XST;                         // [R][8 row tiles][TILES][512 B]
    uint64_t* bars = reinterpret_cast<uint64_t*>(wp + R * geo.wp_stage);
    uint64_t* tma_full = bars;                               // [R]
    uint64_t* a_full = bars + R;                            // [R] kDqWarps arrivals
    uint64_t* mma_done = bars + 2 * R;                      // [R]
    uint64_t* done = bars + 3 * R;                          // the accumulator is complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int tile = geo.splitk == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int rank = geo.splitk == 2 ? (int)cluster_ctarank() : 0;
    const int n_tile = tile % geo.n_tiles, m_tile = tile / geo.n_tiles;
    const int64_t n0 = (int64_t)n_tile * kRows;
    const int64_t m0 = (int64_t)m_tile * BT;
    // stages of this CTA: all of K, or its half
    const int ks_lo = geo.splitk == 2 ? (rank == 0 ? 0 : geo.k_stages / 2) : 0;
    const int ks_hi = geo.splitk == 2 ? (rank == 0 ? geo.k_stages / 2 : geo.k_stages) : geo.k_stages;
    const int KS = ks_hi - ks_lo;
    const int64_t n_ksteps = L.Kpad / 16;  // k-steps that carry data
    const uint32_t wl = p.wait_limit, wh = p.wait_hint_ns;

    if (tid == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&tma_full[s], 1);
            mbar_init(&a_full[s], kDqWarps);
            mbar_init(&mma_done[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tc::alloc(tmem_slot, 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;           // accumulator: columns [0, BT)
    const uint32_t a_base = tmem + (uint32_t)BT;  // A ring: columns [BT, BT + 256)
    volatile int* abort_v = abort_flag;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(XST + geo.wp_stage);
            const int nrt = (int)(n0 / 16);
            int issued = 0;
            auto load_x = [&](int i) {
                const int s = i % R, ks = ks_lo + i;
                if constexpr (TF32) {  // 64 depths of f32: two 128-byte boxes
                    tc::tma_load_2d(xs + s * XST, &xmap, ks * kBK, (int)m0, &tma_full[s]);
                    tc::tma_load_2d(xs + s * XST + BT * 128, &xmap, ks * kBK + 32, (int)m0, &tma_full[s]);
                } else {
                    tc::tma_load_2d(xs + s * XST, &xmap, ks * kBK, (int)m0, &tma_full[s]);
                }
            };
            auto load_w = [&](int i) {
                const int s = i % R, ks = ks_lo + i;
                // packed tiles of this stage: KT >= 64 tiles span whole stages (one load per tile)
                if constexpr (KT > kBK) {
                    tc::tma_load_5d(wp + s * geo.wp_stage, &wmap, 0, 0, 0, (ks * kBK) / KT, nrt, &tma_full[s]);
                } else {
                    tc::tma_load_5d(wp + s * geo.wp_stage, &wmap, 0, 0, 0, ks * TILES, nrt, &tma_full[s]);
                }
            };
            // the first ring fill's weights do not depend on the previous kernel: they are
            // requested before the dependency wait, X after it
            const int pre = KS < R ? KS : R;
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&tma_full[i], bytes);
                load_w(i);
            }
            if (geo.pdl) {
                griddep_wait();               // X (and Y) may belong to the previous kernel on the stream
                griddep_launch_dependents();  // after the wait: at most two chained kernels overlap
            }
            for (int i = 0; i < pre; ++i) load_x(i);
            issued = pre;
            for (int i = pre; i < KS; ++i) {
                const int s = i % R;
                const uint32_t ph = (uint32_t)((i / R) & 1);
                if (!tc::wait_bounded(&mma_done[s], ph ^ 1u, p.status, wl, wh)) {
                    *abort_v = 1;
                    break;
                }
                if (*abort_v) break;
                mbar_arrive_expect_tx(&tma_full[s], bytes);
                load_x(i);
                load_w(i);
                issued = i + 1;
            }
            if (*abort_v) {
                for (int i = issued - R < 0 ? 0 : issued - R; i < issued; ++i)
                    tc::drain_wait(&tma_full[i % R], (uint32_t)((i / R) & 1));
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = TF32 ? tc::idesc_tf32(kRows, BT) : tc::idesc_f16(true, kRows, kBT);
        const uint64_t dx0 = tc::sdesc_sw128(smem_u32(xs));
        constexpr uint64_t x_step = (uint64_t)XST >> 4;
        bool ok = true;
        for (int i = 0; i < KS; ++i) {
            const int s = i % R;
            const uint32_t ph = (uint32_t)((i / R) & 1);
            if (!tc::wait_bounded(&a_full[s], ph, p.status, wl, wh)) {
                ok = false;
                break;
            }
            tc::fence_after();
            if (lane == 0) {
                const uint64_t dxs = dx0 + (uint64_t)s * x_step;
                const uint32_t as = a_base + (uint32_t)(s * kACols);
                const int64_t gk0 = (int64_t)(ks_lo + i) * 4;
                if constexpr (TF32) {
                    // 8 MMAs of 8 depths: 32 bytes along K each, the second box from the 5th on
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        if (gk0 + (kk >> 1) < n_ksteps) {
                            const uint64_t bd = dxs + (uint64_t)(kk >> 2) * ((uint64_t)(BT * 128) >> 4) + (uint64_t)(kk & 3) * 2;
                            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                            tc::mma_ta_tf32(tmem, as + (uint32_t)(kk * 8), bd, idesc, acc);
                        }
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if (gk0 + kk < n_ksteps) {
                            const uint64_t bd = dxs + (uint64_t)kk * 2;  // 32 bytes along K per k-step
                            const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                            tc::mma_ta(tmem, as + (uint32_t)(kk * 8), bd, idesc, acc);
                            tc::mma_ta(tmem, as + 32u + (uint32_t)(kk * 8), bd, idesc, 1u);
                        }
                    }
                }
                tc::commit(&mma_done[s]);
            }
            __syncwarp();
        }
        if (!ok) *abort_v = 1;
        if (lane == 0) {
            tc::commit(done);
            if (!ok) tc::drain_wait(done, 0);
        }
        __syncwarp();
    } else if (warp >= kCtlWarps) {
        // ---------------- A_hi, A_lo: one W row per thread ----------------
        const int dw = warp - kCtlWarps;
        const int q4 = warp & 3;          // TMEM lane quadrant
        const int jh = dw >> 2;           // k-steps kKK jh .. kKK jh + kKK - 1 of every stage
        const int r = q4 * 32 + lane;     // W row inside the tile
        const int rt = r >> 4, g = r & 7, hi = (r >> 3) & 1;
        const int64_t n = n0 + r;
        const bool row_ok = n < L.N;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        const int zmask = code_mask(BITS);
        const int sdt = p.scale_dtype;
        // block of the thread's 32 depths (bs >= 32) or of each of its two k-steps (bs = 16)
        const int bs_log = __ffs(L.bs) - 1;  // block sizes are powers of two
        auto blocks_of = [&](int ks, int64_t* kb0, int64_t* kb1) {
            const int64_t d0 = (int64_t)ks * kBK + 16 * kKK * jh;
            *kb0 = d0 >> bs_log;
            *kb1 = (d0 + 16) >> bs_log;
        };
        // raw loads only (a decode here would wait for the load): scale bits and the
        // zero-point byte of the thread's block(s) of a stage; decoded when used
        const bool two_blocks = kKK == 2 && L.bs < 32;
        auto raw_scale = [&](int64_t kb) -> uint32_t {
            if (!row_ok || kb >= L.KB) return 0u;
            const int64_t i = n * L.KB + kb;
            return sdt == kF32 ? __ldg(static_cast<const uint32_t*>(p.scales) + i)
                               : (uint32_t)__ldg(static_cast<const unsigned short*>(p.scales) + i);
        };
        auto raw_zp = [&](int64_t kb) -> uint32_t {
            if (!p.zp || !row_ok || kb >= L.KB) return 0u;
            return __ldg(p.zp + n * L.zp_row + ((kb * BITS) >> 3));
        };
        auto fetch = [&](int ks, uint32_t* s0, uint32_t* s1, uint32_t* z0, uint32_t* z1) {
            int64_t kb0, kb1;
            blocks_of(ks, &kb0, &kb1);
            *s0 = raw_scale(kb0);
            *z0 = raw_zp(kb0);
            if (two_blocks) {
                *s1 = raw_scale(kb1);
                *z1 = raw_zp(kb1);
            }
        };
        auto dec_scale = [&](uint32_t r) -> float {
            if (sdt == kF32) return __uint_as_float(r);
            if (sdt == kF16) return __half2float(__ushort_as_half((unsigned short)r));
            return __uint_as_float(r << 16);
        };
        auto dec_zp = [&](uint32_t r, int ks, int half) -> uint32_t {
            if (!p.zp) return 1u << (BITS - 1);
            int64_t kb0, kb1;
            blocks_of(ks, &kb0, &kb1);
            const int64_t kb = half ? kb1 : kb0;
            return (r >> ((kb * BITS) & 7)) & (uint32_t)zmask;
        };
        // scales and zero points are scattered loads (one row per thread): each is
        // fetched kPF stages ahead into one of kPF named register slots, and the
        // stage loop is unrolled kPF times so a slot is read in place (copying a
        // register whose load is still in flight would wait for it)
        constexpr int kPF = 3;
        uint32_t ps0[kPF], ps1[kPF] = {}, pz0[kPF], pz1[kPF] = {};
#pragma unroll
        for (int q = 0; q < kPF; ++q)
            if (q < KS) fetch(ks_lo + q, &ps0[q], &ps1[q], &pz0[q], &pz1[q]);
        auto stage = [&](int i, uint32_t& slot_s0, uint32_t& slot_s1, uint32_t& slot_z0, uint32_t& slot_z1) -> bool {
            const int s = i % R;
            const uint32_t ph = (uint32_t)((i / R) & 1);
            const int ks = ks_lo + i;
            if (i >= R && !tc::wait_bounded(&mma_done[s], ph ^ 1u, p.status, wl, wh)) {
                return false;
            }
            if (!tc::wait_bounded(&tma_full[s], ph, p.status, wl, wh)) {
                return false;
            }
            if (*abort_v) return false;
            const float sc0 = dec_scale(slot_s0);
            const float sc1 = two_blocks ? dec_scale(slot_s1) : sc0;
            const uint32_t z0 = dec_zp(slot_z0, ks, 0);
            const uint32_t z1 = two_blocks ? dec_zp(slot_z1, ks, 1) : z0;
            if (i + kPF < KS) fetch(ks + kPF, &slot_s0, &slot_s1, &slot_z0, &slot_z1);
            uint32_t shi[2], slo[2], zc[2];
            split_scale(sc0, &shi[0], &slo[0]);
            split_scale(sc1, &shi[1], &slo[1]);
            zc[0] = ((kMag & 0xFFFFu) + z0) * 0x10001u;
            zc[1] = ((kMag & 0xFFFFu) + z1) * 0x10001u;
            // (q - zp) pairs of the thread's two k-steps: column c of k-step kk = depths 2c, 2c + 1
            uint32_t qz[8 * kKK];
            const uint8_t* cb = wp + s * geo.wp_stage + rt * TILES * kTileBytes + g * 16;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
#pragma unroll
                for (int kk = 0; kk < kKK; ++kk) {
                    const int st = kKK * jh + kk;  // k-step inside the stage
                    uint32_t v0, v1;             // depths 2t/2t+1 and 2t+8/2t+9 of the row
                    if constexpr (BITS == 4) {
                        // stage = one packed tile (4 k-steps): word st of chunk t
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(cb + t * 128 + 4 * st) >> (4 * hi);
                        v0 = tc::hsub2(lop3_and_or(w, 0x000F000Fu, kMag), zc[kk], true);
                        v1 = tc::hsub2(lop3_and_or(w >> 8, 0x000F000Fu, kMag), zc[kk], true);
                    } else if constexpr (BITS == 2) {
                        // a packed tile spans 8 k-steps (two stages): k-step gs of the tile
                        const int gs = (ks & 1) * 4 + st;
                        const uint32_t w = *reinterpret_cast<const uint32_t*>(cb + t * 128 + 4 * (gs >> 1));
                        const int f0 = 4 * (gs & 1) + hi;
                        v0 = tc::hsub2(lop3_and_or(w >> (2 * f0), 0x00030003u, kMag), zc[kk], true);
                        v1 = tc::hsub2(lop3_and_or(w >> (2 * (f0 + 2)), 0x00030003u, kMag), zc[kk], true);
                    } else {
                        // 8-bit: tile st >> 1 of the stage, k-step st & 1 of the tile: words 2 (st & 1) + half
                        const uint2 w2 =
                            *reinterpret_cast<const uint2*>(cb + (st >> 1) * kTileBytes + t * 128 + 8 * (st & 1));
                        const uint32_t b0 = 2 * hi, b1 = b0 + 1;
                        const uint32_t zf = 0x4B000000u | (kk ? z1 : z0);
                        float2 d;
                        d = unpack2(fsub2(pack2u(prmt(w2.x, 0x4B000000u, 0x7650u | b0), prmt(w2.x, 0x4B000000u, 0x7650u | b1)),
                                          pack2u(zf, zf)));
                        v0 = tc::cvt_bf16x2(d.x, d.y);  // |q - zp| <= 255: exact in bf16
                        d = unpack2(fsub2(pack2u(prmt(w2.y, 0x4B000000u, 0x7650u | b0), prmt(w2.y, 0x4B000000u, 0x7650u | b1)),
                                          pack2u(zf, zf)));
                        v1 = tc::cvt_bf16x2(d.x, d.y);
                    }
                    qz[8 * kk + t] = v0;
                    qz[8 * kk + t + 4] = v1;
                }
            }
            if constexpr (TF32) {
                // w = (q - zp) * scale in f32, rounded to tf32: one column per depth
                static_assert(kKK == 1, "the tf32 variant writes one k-step per warp");
                uint32_t av[16];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t v0 = qz[t], v1 = qz[t + 4];  // depths 2t, 2t+1 and 2t+8, 2t+9
                    av[2 * t] = tc::cvt_tf32(__fmul_rn(__uint_as_float(v0 << 16), sc0));
                    av[2 * t + 1] = tc::cvt_tf32(__fmul_rn(__uint_as_float(v0 & 0xFFFF0000u), sc0));
                    av[2 * t + 8] = tc::cvt_tf32(__fmul_rn(__uint_as_float(v1 << 16), sc0));
                    av[2 * t + 9] = tc::cvt_tf32(__fmul_rn(__uint_as_float(v1 & 0xFFFF0000u), sc0));
                }
                tc::st_32x32b_x16(a_base + (uint32_t)(s * kACols + 16 * jh) + lane_addr, av);
                tc::wait_st();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[s]);
                return true;
            }
            uint32_t ah[8 * kKK], al[8 * kKK];
#pragma unroll
            for (int c = 0; c < 8 * kKK; ++c) {
                const int kk = c >> 3;
                const uint32_t h = bmul2(qz[c], shi[kk]);
                const uint32_t rr = bfma2(qz[c], shi[kk], h ^ 0x80008000u);  // qz * s_hi - h, exact
                ah[c] = h;
                al[c] = bfma2(qz[c], slo[kk], rr);
            }
            const uint32_t col = a_base + (uint32_t)(s * kACols + 8 * kKK * jh) + lane_addr;
            if constexpr (kKK == 2) {
                tc::st_32x32b_x16(col, *reinterpret_cast<const uint32_t(*)[16]>(ah));
                tc::st_32x32b_x16(col + 32u, *reinterpret_cast<const uint32_t(*)[16]>(al));
            } else {
                tc::st_32x32b_x8(col, *reinterpret_cast<const uint32_t(*)[8]>(ah));
                tc::st_32x32b_x8(col + 32u, *reinterpret_cast<const uint32_t(*)[8]>(al));
            }
            tc::wait_st();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[s]);
            return true;
        };
        bool ok = true;
        for (int i = 0; i < KS && ok; i += kPF) {
            ok = stage(i, ps0[0], ps1[0], pz0[0], pz1[0]);
            if (ok && i + 1 < KS) ok = stage(i + 1, ps0[1], ps1[1], pz0[1], pz1[1]);
            if (ok && i + 2 < KS) ok = stage(i + 2, ps0[2], ps1[2], pz0[2], pz1[2]);
        }
        if (!ok) *abort_v = 1;

        // ---------------- epilogue ----------------
        bool fine = ok && !*abort_v && tc::wait_bounded(done, 0, p.status, wl, wh);
        tc::fence_after();
        const float bias = (p.bias && row_ok) ? load_f32(p.bias, n, p.bias_dtype) : 0.f;
        // Y: this CTA's tokens [tok0, tok0 + T) of its 128 rows, staged in the idle X ring as
        // [128-byte row chunk][token][row] and written by TMA (out-of-range rows and tokens are
        // clipped), or stored element by element
        const int T = geo.splitk == 2 ? kBT / 2 : BT;
        const int64_t tok0 = m0 + (geo.splitk == 2 ? (int64_t)(kBT / 2) * rank : 0);
        const int es = p.out_dtype == kF32 ? 4 : 2;
        const int rowc = 128 / es;
        uint8_t* ystage = smem + (geo.splitk == 2 ? 65536 : 0);  // past the split-K exchange buffer
        auto put = [&](int t, float v) {
            if (geo.ystore) {
                uint8_t* d = ystage + (size_t)(r / rowc) * (size_t)(T * 128) + (size_t)t * 128 + (size_t)(r % rowc) * es;
                if (es == 4) {
                    *reinterpret_cast<float*>(d) = v;
                } else if (p.out_dtype == kF16) {
                    *reinterpret_cast<__half*>(d) = __float2half_rn(v);
                } else {
                    *reinterpret_cast<__nv_bfloat16*>(d) = __float2bfloat16_rn(v);
                }
            } else {
                const int64_t m = tok0 + t;
                if (row_ok && m < p.M) store_f32(p.y, m * L.N + n, v, p.out_dtype);
            }
        };
        if (geo.splitk == 1) {
            // columns kEpi jh .. kEpi jh + kEpi - 1 of this thread's row
            constexpr int kEpi = BT / (kDqWarps / 4);
            for (int c0 = kEpi * jh; c0 < kEpi * jh + kEpi && fine; c0 += 32) {
                uint32_t v[32];
                tc::ld_32x32b<32>(tmem + (uint32_t)c0 + lane_addr, v);
                tc::wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) put(c0 + j, __uint_as_float(v[j]) + bias);
            }
        } else {
            // rank r outputs tokens 128 r .. 128 r + 127; it hands the partner its half
            // of the other 128 columns through shared memory ([col / 4][row][4] floats)
            float4* xbuf = reinterpret_cast<float4*>(smem);  // 64 KB, the X ring is idle now
            const int other = 128 * (rank ^ 1), mine = 128 * rank;
            constexpr int kHalf = (kBT / 2) / (kDqWarps / 4);  // columns of a half a thread moves
            if (fine) {
                for (int c0 = other + kHalf * jh; c0 < other + kHalf * jh + kHalf; c0 += 32) {
                    uint32_t v[32];
                    tc::ld_32x32b<32>(tmem + (uint32_t)c0 + lane_addr, v);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        xbuf[((c0 - other + j) >> 2) * kRows + r] =
                            make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                        __uint_as_float(v[j + 3]));
                }
            }
            // both CTAs' buffers written (every thread of both CTAs joins both cluster barriers)
            asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
            if (fine) {
                const uint32_t peer = rank ^ 1;
                for (int c0 = mine + kHalf * jh; c0 < mine + kHalf * jh + kHalf; c0 += 32) {
                    uint32_t v[32];
                    tc::ld_32x32b<32>(tmem + (uint32_t)c0 + lane_addr, v);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4* src = &xbuf[((c0 - mine + j) >> 2) * kRows + r];
                        uint32_t remote;
                        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(src)), "r"(peer));
                        float4 o;
                        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(o.x), "=f"(o.y), "=f"(o.z), "=f"(o.w) : "r"(remote) : "memory");
                        const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // D_rank0 + D_rank1 in either CTA (f32 addition of two terms commutes)
                            put(c0 - mine + j + e, __uint_as_float(v[j + e]) + ov[e] + bias);
                        }
                    }
                }
            }
        }
        if (geo.ystore) {
            fence_proxy_async_smem();  // the stage's generic writes, before the TMA reads them
            asm volatile("bar.sync 1, %0;" ::"n"(kDqWarps * 32) : "memory");
            if (warp == kCtlWarps && lane == 0 && fine) {
                for (int c = 0; c < 128 / rowc; ++c)
                    tc::tma_store_2d(&ymap, ystage + (size_t)c * (size_t)(T * 128), (int)(n0 + c * rowc), (int)tok0);
                tc::bulk_commit();
                tc::bulk_wait_read0();
            }
        }
    }
    if (geo.splitk == 2 && warp < kCtlWarps) {
        // the control warps join the epilogue's cluster barrier
        asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    }

    tc::fence_before();
    __syncthreads();
    if (geo.splitk == 2) cluster_sync();  // the partner has read this CTA's buffer
    if (warp == 1) {
        tc::fence_after();
        tc::dealloc(tmem, 512);
    }
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status, kWfInt, p.kperm != nullptr ? 1 : 0);
}

template <int BITS, bool TF32 = false>
cudaError_t launch(const MatmulParams& p, const Geom& geo, const Maps& m, cudaStream_t s) {
    auto kern = gemm_hl_kernel<BITS, TF32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(geo.n_tiles * geo.m_tiles * geo.splitk));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = geo.total_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)geo.splitk;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = geo.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p, geo, m.x, m.w, m.y);
}

}  // namespace ghl
}  // namespace mnb
