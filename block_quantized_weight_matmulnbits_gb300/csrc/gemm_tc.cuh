// Prefill GEMM on 5th-generation tensor cores (tcgen05 + TMEM + TMA), M >= 1,
// bf16 or f16 X:  Y[m, n] = sum_k X[m, k] * w[n, k]  (+ bias[n]),
// w = (q - zp) * scale as in onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs, fn dequantize_nbits_value.  The pages' prefill
// paths (AMX tile GEMM, dequantise-then-sgemm) are CPU designs; this is a
// GB300 design.
//
// One CTA computes one 128 x BN tile of Y (128 rows of X, BN rows of W) over
// K in stages of BK depths (64; 128 for 2-bit codes).  Every shared-memory
// ring (X tile, packed codes, dequantised W) has the same depth R, stage ks
// lives in slot ks % R, and one tcgen05.commit per stage frees the slot.
//   warp 0      : producer.  Per stage, one 2-D TMA copy of the X tile
//                 (128B swizzle, zero fill past M and K) and one 3-D TMA
//                 copy of the BN rows' packed 512-byte tiles.
//   warp 1      : owns the TMEM accumulator (128 lanes x BN f32 columns); one
//                 lane issues tcgen05.mma kind::f16 (M = 128, N = BN, K = 16)
//                 and one tcgen05.commit per stage.  Its loop is kept to a
//                 few instructions per stage (slot and phase counters,
//                 descriptors advanced by addition): it shares an SM
//                 sub-partition with dequantising warps, and its per-stage
//                 latency paces the whole pipeline.
//   warps 2-3   : per stage, convert the BN rows' block scales and zero
//                 points into 32-bit entries (zero-point constant | scale in
//                 the MMA's input type) in a small shared-memory ring; the two
//                 warps take alternate stages and keep the next stage's
//                 global loads in flight while they store the current one.
//   warps 4-19  : dequantise.  The stage's (16-row tile, packed tile) units
//                 are dealt round-robin over the 16 warps (unit U of the
//                 kernel to warp U % 16); every warp still visits every stage
//                 only at most R - 1 stages apart, so each barrier is only
//                 ever waited on for its current or next phase.  A code pair is masked into the mantissa of 128.0 / 1024.0,
//                 (q - zp) is one exact packed subtract and one packed
//                 multiply by the block scale rounds w once to the MMA's input
//                 type, written straight into the canonical K-major
//                 128B-swizzled layout.  After the K loop the same warps read
//                 the accumulator out of TMEM (tcgen05.ld), add the bias,
//                 round to the output dtype and store Y with 16-byte stores.
// Every mbarrier wait is bounded: on timeout the kernel records
// MNB_ERR_TIMEOUT, lets its copies in flight land (bounded), frees TMEM and
// returns.  The reduction order over K is fixed, so results are deterministic.
#pragma once

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cuda.h>

#include "mnb_internal.h"

namespace mnb {
namespace gtc {

constexpr int kBM = 128;
constexpr int kCtlWarps = 4;
constexpr int kDqWarps = 16;
constexpr int kThreads = (kCtlWarps + kDqWarps) * 32;
constexpr int kMaxR = 8;

struct TcGeom {
    int BN;          // W rows per tile (multiple of 16, <= 256)
    int BK;          // depths per stage (64, or 128 for 2-bit codes)
    int tmem_cols;   // power of two >= BN
    int n_tiles;     // ceil(N / BN)
    int m_tiles;     // ceil(M / 128)
    int k_stages;    // ceil(KTILES * KT / BK)
    int units;       // (16-row tile, packed tile) units per stage
    int nbs;         // quantisation blocks per stage (max(1, BK / bs)); BN * nbs <= 256
    int R;           // ring depth
    int scale_tma;   // raw scales / zero points arrive by TMA, SB blocks at a time
    int sb;          // blocks per raw scale buffer (TMA path)
    int sb_stages;   // stages per raw scale buffer (sb * bs / BK, >= R)
    int ta;          // W in tensor memory (gemm_ta.cuh): BN = tokens per tile, 128 W rows per tile
    int a_col0;      // (ta) first TMEM column of the A ring
    size_t x_stage, wp_stage, wd_stage, ent_stage, sraw_bytes, zraw_bytes, total_bytes;
};

// ---- PTX wrappers specific to tcgen05 / TMA tensor copies ----

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: 8-row x 128-byte
// atoms stacked along M/N every 1024 bytes (SBO); LBO unused for this layout.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused), 16 B
    d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
    d |= (uint64_t)1 << 46;                          // descriptor version for sm_100 family
    d |= (uint64_t)2 << 61;                          // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16: f32 accumulator, A/B bf16 or f16,
// both K-major, M = 128, N = n.
__host__ __device__ inline uint32_t idesc_f16(bool bf16, int n) {
    uint32_t d = 0;
    d |= 1u << 4;                     // D format f32
    d |= (bf16 ? 1u : 0u) << 7;       // A format
    d |= (bf16 ? 1u : 0u) << 10;      // B format
    d |= (uint32_t)(n >> 3) << 17;    // N / 8
    d |= (uint32_t)(kBM >> 4) << 24;  // M / 16
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b, bool bf16) {
    uint32_t d;
    if (bf16) asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b, bool bf16) {
    uint32_t d;
    if (bf16) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Round an f32 to the MMA input type, replicated in both halves.
__device__ __forceinline__ uint32_t to_pair(float v, bool bf16) {
    uint32_t d;
    if (bf16) asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(v));
    else asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(v));
    return d;
}


template <int BITS, bool BF16X, int NBU, bool RAW>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(MatmulParams p, TcGeom geo,
                                                               const __grid_constant__ CUtensorMap xmap,
                                                               const __grid_constant__ CUtensorMap wmap,
                                                               const __grid_constant__ CUtensorMap smap,
                                                               const __grid_constant__ CUtensorMap zmap) {
    constexpr int KT = 256 / BITS;              // depths per packed tile
    constexpr int kSteps = 16 / BITS;           // 16-deep k-steps per packed tile
    constexpr int SPB = kSteps / NBU;           // k-steps per quantisation block inside a unit
    constexpr int TILES = BITS == 8 ? 2 : 1;    // packed tiles per 16-row tile per stage
    constexpr uint32_t kMag = BF16X ? 0x43004300u : 0x64006400u;
    const Layout& L = p.L;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic so the compiler keeps
    // the shared address space (plain loads / stores compile to LDS / STS)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int R = geo.R;
    uint8_t* xs = smem;                                   // [R][BK/64][128 x 64] bf16, SW128 (TMA)
    uint8_t* wd = xs + R * geo.x_stage;                   // [R][BK/64][BN x 64] bf16, SW128
    uint8_t* wp = wd + R * geo.wd_stage;                  // [R][BN/16][TILES][512 B] packed codes (TMA)
    uint8_t* ent = wp + R * geo.wp_stage;                 // [R][BN][nbs] u32 (zero-point constant | scale << 16)
    uint8_t* sraw = ent + R * geo.ent_stage;              // [2][BN][sb] raw scales (TMA path)
    uint8_t* zraw = sraw + 2 * geo.sraw_bytes;            // [2][BN][sb * bits / 8] raw zero points (TMA path)
    uint64_t* bars = reinterpret_cast<uint64_t*>(zraw + 2 * geo.zraw_bytes);
    uint64_t* tma_full = bars;                            // X tile + packed codes landed
    uint64_t* wd_full = bars + kMaxR;                     // all units of the stage dequantised
    uint64_t* mma_done = bars + 2 * kMaxR;                // MMAs of the stage finished: slot free
    uint64_t* ent_full = bars + 3 * kMaxR;                // scale / zero-point entries of the stage written
    uint64_t* raw_full = bars + 4 * kMaxR;                // raw scale buffer b landed (TMA path)
    uint64_t* done = raw_full + 2;                        // accumulator complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int BN = geo.BN, BK = geo.BK;
    const int n_tile = blockIdx.x % geo.n_tiles;
    const int m_tile = blockIdx.x / geo.n_tiles;
    const int64_t n0 = (int64_t)n_tile * BN;
    const int64_t m0 = (int64_t)m_tile * kBM;
    const int KS = geo.k_stages;

    if (tid == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&tma_full[s], 1);
            mbar_init(&wd_full[s], geo.units);
            mbar_init(&mma_done[s], 1);
            mbar_init(&ent_full[s], 1);
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
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_v = abort_flag;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)(geo.x_stage + geo.wp_stage);
            const int nrt = (int)(n0 / 16);
            int s = 0, issued = 0;
            uint32_t ph = 0;
            // raw scales (RAW): super-slot q (SB blocks = G stages) in buffer q & 1;
            // super-slot q is loaded once super-slot q - 2 is fully consumed
            const int SB = geo.sb, G = geo.sb_stages;
            const int nq = (int)((L.KB + SB - 1) / SB);
            const uint32_t rbytes = (uint32_t)(geo.sraw_bytes + (p.zp ? geo.zraw_bytes : 0));
            int q_next = 0;
            auto issue_raw = [&](int q) {
                const int b = q & 1;
                mbar_arrive_expect_tx(&raw_full[b], rbytes);
                tma_load_2d(sraw + b * geo.sraw_bytes, &smap, q * SB, (int)n0, &raw_full[b]);
                if (p.zp) tma_load_2d(zraw + b * geo.zraw_bytes, &zmap, q * SB * BITS / 8, (int)n0, &raw_full[b]);
            };
            if constexpr (RAW) {
                for (; q_next < nq && q_next < 2; ++q_next) issue_raw(q_next);
            }
            for (int ks = 0; ks < KS; ++ks) {
                if (ks >= R && !mbar_wait(&mma_done[s], ph ^ 1u, p.status)) {
                    *abort_v = 1;
                    break;
                }
                if (*abort_v) break;
                if constexpr (RAW) {
                    const int stages_done = ks >= R ? ks - R + 1 : 0;
                    for (; q_next < nq && (q_next - 1) * G <= stages_done; ++q_next) issue_raw(q_next);
                }
                mbar_arrive_expect_tx(&tma_full[s], bytes);
                uint8_t* xd = xs + s * geo.x_stage;
                tma_load_2d(xd, &xmap, ks * BK, (int)m0, &tma_full[s]);
                if (BITS == 2) tma_load_2d(xd + kBM * 128, &xmap, ks * BK + 64, (int)m0, &tma_full[s]);
                tma_load_3d(wp + s * geo.wp_stage, &wmap, 0, ks * TILES, nrt, &tma_full[s]);
                issued = ks + 1;
                if (++s == R) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (*abort_v) {
                // let copies still in flight land (bounded) before the CTA exits
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
        const uint32_t idesc = idesc_f16(BF16X, BN);
        const uint64_t dx0 = sdesc_sw128(smem_u32(xs)), dw0 = sdesc_sw128(smem_u32(wd));
        const uint64_t x_step = geo.x_stage >> 4, w_step = geo.wd_stage >> 4;
        const uint64_t w_half = (uint64_t)(BN * 128) >> 4;
        uint64_t dxs = dx0, dws = dw0;
        int s = 0;
        uint32_t ph = 0;
        for (int ks = 0; ks < KS; ++ks) {
            if (!mbar_wait(&tma_full[s], ph, p.status) || !mbar_wait(&wd_full[s], ph, p.status)) {
                *abort_v = 1;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < (BITS == 2 ? 8 : 4); ++kk) {
                    const uint64_t off = (uint64_t)(kk & 3) * 2;  // 32 bytes along K inside the swizzle atom
                    const uint64_t ad = dxs + off + (kk >> 2) * (uint64_t)((kBM * 128) >> 4);
                    const uint64_t bd = dws + off + (kk >> 2) * w_half;
                    tc_mma(tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&mma_done[s]);
            }
            __syncwarp();
            if (++s == R) {
                s = 0;
                ph ^= 1u;
                dxs = dx0;
                dws = dw0;
            } else {
                dxs += x_step;
                dws += w_step;
            }
        }
        if (lane == 0) tc_commit(done);
        __syncwarp();
    } else if (warp < kCtlWarps) {
        // ---------------- scale / zero-point entries ----------------
        const int nsw = R >= 3 ? 2 : 1;  // consecutive stages of a warp stay within R - 1
        const int sw = warp - 2;
        if (!RAW && sw < nsw) {
            const int nbs = geo.nbs;
            const int nbs_log = __ffs(nbs) - 1;
            const int per_stage = BN * nbs;  // <= 256: at most 8 entries per lane
            const int bs_log = __ffs(L.bs) - 1;
            const int sdt = p.scale_dtype;
            const int zmask = code_mask(BITS);
            float sa[8], sb[8];
            uint32_t za[8], zb[8];
            auto load = [&](int ks, float (&sc)[8], uint32_t (&zz)[8]) {
                const int64_t kbs = ((int64_t)ks * BK) >> bs_log;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = lane + 32 * i;
                    const int64_t n = n0 + (e >> nbs_log), kb = kbs + (e & (nbs - 1));
                    const bool ok = e < per_stage && n < L.N && kb < L.KB;
                    sc[i] = ok ? load_f32(p.scales, n * L.KB + kb, sdt) : 0.f;
                    uint32_t z = 1u << (BITS - 1);
                    if (p.zp != nullptr) {
                        const int64_t bit = kb * BITS;
                        z = ok ? ((uint32_t)__ldg(p.zp + n * L.zp_row + (bit >> 3)) >> (bit & 7)) & zmask : 0u;
                    }
                    zz[i] = z;
                }
            };
            if (sw < KS) load(sw, sa, za);
            for (int ks = sw; ks < KS; ks += nsw) {
                if (ks + nsw < KS) load(ks + nsw, sb, zb);
                const int s = ks % R;
                const uint32_t ph = (uint32_t)((ks / R) & 1);
                if (ks >= R && !mbar_wait(&mma_done[s], ph ^ 1u, p.status)) {
                    *abort_v = 1;
                    break;
                }
                uint32_t* dst = reinterpret_cast<uint32_t*>(ent + s * geo.ent_stage);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = lane + 32 * i;
                    if (e < per_stage) {
                        uint32_t lo;
                        if constexpr (BITS == 8 && BF16X) lo = za[i];
                        else lo = (kMag & 0xFFFFu) + za[i];
                        dst[e] = lo | (to_pair(sa[i], BF16X) << 16);
                    }
                    sa[i] = sb[i];
                    za[i] = zb[i];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&ent_full[s]);
            }
        }
    } else {
        // ---------------- dequantiser, then epilogue ----------------
        const int dw = warp - kCtlWarps;
        const int units = geo.units;
        const int total_units = KS * units;
        const int g = lane >> 2, t = lane & 3;
        const int bs_log = __ffs(L.bs) - 1;
        const int nbs = geo.nbs;
        const int g_log = __ffs(geo.sb_stages) - 1;  // RAW: stages per raw super-slot (power of two)
        const int sdt = p.scale_dtype;
        const int zmask = code_mask(BITS);
        const int zrow = geo.sb * BITS / 8;
        int q_cur = -1;
        // Active warps: at most units * (R - 1), so consecutive stages a warp works
        // on are at most R - 1 apart and every barrier it waits on is at its
        // current or next phase.
        const int A = units * (R - 1) < kDqWarps ? units * (R - 1) : kDqWarps;
        bool ok = true;
        if (dw < A) {
            int ks = dw / units, u = dw - ks * units;
            int s = ks % R;
            uint32_t ph = (uint32_t)((ks / R) & 1);
            const int dks = A / units, du = A - dks * units;  // advance per unit of this warp
            for (int U = dw; U < total_units; U += A) {
                if (ks >= R && !mbar_wait(&mma_done[s], ph ^ 1u, p.status)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&tma_full[s], ph, p.status) ||
                    (!RAW && !mbar_wait(&ent_full[s], ph, p.status))) {
                    ok = false;
                    break;
                }
                const int rt = u / TILES, tl = u - rt * TILES;
                // this unit's constants for rows g, g + 8 and its NBU blocks
                uint32_t zc[2][NBU], sp[2][NBU];
                if constexpr (RAW) {
                    const int q = ks >> g_log;
                    if (q != q_cur) {
                        if (!mbar_wait(&raw_full[q & 1], (uint32_t)((q >> 1) & 1), p.status)) {
                            ok = false;
                            break;
                        }
                        q_cur = q;
                    }
                    const int kl = (int)((((int64_t)ks * BK + tl * KT) >> bs_log) - ((int64_t)q * geo.sb));
                    const uint8_t* sbuf = sraw + (q & 1) * geo.sraw_bytes;
                    const uint8_t* zbuf = zraw + (q & 1) * geo.zraw_bytes;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int row = rt * 16 + g + 8 * h;
#pragma unroll
                        for (int j = 0; j < NBU; ++j) {
                            const int idx = row * geo.sb + kl + j;
                            float sc;
                            if (sdt == kF32) {
                                sc = reinterpret_cast<const float*>(sbuf)[idx];
                            } else {
                                const unsigned short v = reinterpret_cast<const unsigned short*>(sbuf)[idx];
                                sc = sdt == kF16 ? __half2float(__ushort_as_half(v)) : __uint_as_float((uint32_t)v << 16);
                            }
                            uint32_t z = 1u << (BITS - 1);
                            if (p.zp) {
                                const uint32_t bit = (uint32_t)(kl + j) * BITS;
                                z = ((uint32_t)zbuf[row * zrow + (bit >> 3)] >> (bit & 7)) & zmask;
                            }
                            sp[h][j] = to_pair(sc, BF16X);
                            if constexpr (BITS == 8 && BF16X) zc[h][j] = 0x4B000000u | z;
                            else zc[h][j] = ((kMag & 0xFFFFu) + z) * 0x10001u;
                        }
                    }
                } else {
                    const int j0 = (L.bs <= KT) ? ((tl * KT) >> bs_log) : 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t* ea = reinterpret_cast<const uint32_t*>(ent + s * geo.ent_stage) +
                                             (rt * 16 + g + 8 * h) * nbs + j0;
                        uint32_t e[NBU];
                        if constexpr (NBU == 1) {
                            e[0] = ea[0];
                        } else if constexpr (NBU == 2) {
                            const uint2 v = *reinterpret_cast<const uint2*>(ea);
                            e[0] = v.x;
                            e[1] = v.y;
                        } else {
#pragma unroll
                            for (int q = 0; q < NBU; q += 4) {
                                const uint4 v = *reinterpret_cast<const uint4*>(ea + q);
                                e[q] = v.x;
                                e[q + 1] = v.y;
                                e[q + 2] = v.z;
                                e[q + 3] = v.w;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < NBU; ++j) {
                            sp[h][j] = prmt(e[j], e[j], 0x3232u);  // scale in both halves
                            if constexpr (BITS == 8 && BF16X) zc[h][j] = 0x4B000000u | (e[j] & 0xFFu);
                            else zc[h][j] = prmt(e[j], e[j], 0x1010u);  // zero-point constant in both halves
                        }
                    }
                }

                const uint4 wv = *reinterpret_cast<const uint4*>(wp + s * geo.wp_stage + u * kTileBytes + lane * 16);
                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                // swizzled row bases: row r at (r/8)*1024 + (r%8)*128, 16-byte chunk index xor (r%8)
                uint8_t* base0 = wd + s * geo.wd_stage + (rt * 2048 + g * 128 + 4 * t);
                uint8_t* base1 = base0 + 1024;  // row r0 + 8
#pragma unroll
                for (int st = 0; st < kSteps; ++st) {
                    const int j = st / SPB;
                    const uint32_t zc0 = zc[0][j], zc1 = zc[1][j];
                    const uint32_t sp0 = sp[0][j], sp1 = sp[1][j];
                    uint32_t a[4];
                    if constexpr (BITS == 4) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t v = lop3_and_or(w[st] >> (4 * r), 0x000F000Fu, kMag);
                            a[r] = hmul2(hsub2(v, (r & 1) ? zc1 : zc0, BF16X), (r & 1) ? sp1 : sp0, BF16X);
                        }
                    } else if constexpr (BITS == 2) {
                        const uint32_t word = w[st >> 1];
                        const int base = (st & 1) * 4;
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t v = lop3_and_or(word >> (2 * (base + r)), 0x00030003u, kMag);
                            a[r] = hmul2(hsub2(v, (r & 1) ? zc1 : zc0, BF16X), (r & 1) ? sp1 : sp0, BF16X);
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t word = w[2 * st + (r >> 1)];
                            const uint32_t b0 = 2 * (r & 1), b1 = b0 + 1;
                            uint32_t q;
                            if constexpr (BF16X) {
                                const uint32_t va = prmt(word, 0x4B000000u, 0x7650u | b0);
                                const uint32_t vb = prmt(word, 0x4B000000u, 0x7650u | b1);
                                const uint32_t z = (r & 1) ? zc1 : zc0;
                                const float2 d = unpack2(fsub2(pack2u(va, vb), pack2u(z, z)));
                                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(q) : "f"(d.y), "f"(d.x));
                            } else {
                                q = hsub2(prmt(word, 0x64646464u, b0 | (4u << 4) | (b1 << 8) | (4u << 12)),
                                          (r & 1) ? zc1 : zc0, BF16X);
                            }
                            a[r] = hmul2(q, (r & 1) ? sp1 : sp0, BF16X);
                        }
                    }
                    // register r: row r0 (r even) / r0 + 8 (r odd), depths 2t(+1) (+8 for r >= 2)
                    const int kl = tl * KT + 16 * st;  // depth inside the stage
                    const uint32_t tile = (uint32_t)(kl >> 6) * (uint32_t)(BN * 128);
                    const uint32_t c0 = tile + (uint32_t)((((kl & 63) >> 3) ^ g) << 4);        // depths 2t, 2t+1
                    const uint32_t c1 = tile + (uint32_t)(((((kl & 63) >> 3) + 1) ^ g) << 4);  // depths 2t+8, 2t+9
                    *reinterpret_cast<uint32_t*>(base0 + c0) = a[0];
                    *reinterpret_cast<uint32_t*>(base1 + c0) = a[1];
                    *reinterpret_cast<uint32_t*>(base0 + c1) = a[2];
                    *reinterpret_cast<uint32_t*>(base1 + c1) = a[3];
                }
                fence_proxy_async_smem();  // generic-proxy writes -> tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(&wd_full[s]);
                // advance (stage, unit) by A units
                u += du;
                int adv = dks;
                if (u >= units) {
                    u -= units;
                    ++adv;
                }
                ks += adv;
                s += adv;
                while (s >= R) {
                    s -= R;
                    ph ^= 1u;
                }
            }
        }
        if (!ok) *abort_v = 1;

        // ---------------- epilogue: TMEM -> registers -> Y ----------------
        if (ok && !*abort_v && mbar_wait(done, 0, p.status)) {
            tc_fence_after();
            const int quad = warp & 3;  // TMEM lane quadrant this warp may access
            const int part = dw >> 2;   // which 16-column groups
            const int64_t m = m0 + quad * 32 + lane;
            const int osz = p.out_dtype == kF32 ? 4 : 2;
            const bool vec = (L.N * osz) % 16 == 0;
            for (int c0 = part * 16; c0 < BN; c0 += 64) {
                uint32_t r[16];
                tc_ld16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, r);
                if (m >= p.M) continue;
                const int64_t nb = n0 + c0;
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    v[j] = __uint_as_float(r[j]);
                    if (p.bias && nb + j < L.N) v[j] += load_f32(p.bias, nb + j, p.bias_dtype);
                }
                if (vec && nb + 16 <= L.N) {
                    uint8_t* yp = static_cast<uint8_t*>(p.y) + (size_t)(m * L.N + nb) * osz;
                    if (p.out_dtype == kF32) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            reinterpret_cast<float4*>(yp)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                                                           v[4 * j + 3]);
                    } else {
                        uint32_t h[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (p.out_dtype == kBF16)
                                asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(v[2 * j + 1]), "f"(v[2 * j]));
                            else
                                asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h[j]) : "f"(v[2 * j + 1]), "f"(v[2 * j]));
                        }
                        reinterpret_cast<uint4*>(yp)[0] = make_uint4(h[0], h[1], h[2], h[3]);
                        reinterpret_cast<uint4*>(yp)[1] = make_uint4(h[4], h[5], h[6], h[7]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (nb + j < L.N) store_f32(p.y, m * L.N + nb + j, v[j], p.out_dtype);
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

struct Maps {
    CUtensorMap x, w, s, z;
};

template <int BITS, bool BF16X, int NBU>
cudaError_t launch_nbu(const MatmulParams& p, const TcGeom& geo, const Maps& m, cudaStream_t s) {
    auto kern = geo.scale_tma ? gemm_tc_kernel<BITS, BF16X, NBU, true> : gemm_tc_kernel<BITS, BF16X, NBU, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(geo.n_tiles * geo.m_tiles), kThreads, geo.total_bytes, s>>>(p, geo, m.x, m.w, m.s, m.z);
    return cudaGetLastError();
}

// NBU = quantisation blocks per packed tile (1 when a block covers the tile).
template <int BITS, bool BF16X>
cudaError_t launch(const MatmulParams& p, const TcGeom& geo, const Maps& m, cudaStream_t s) {
    constexpr int KT = 256 / BITS;
    const int nbu = p.L.bs >= KT ? 1 : (int)(KT / p.L.bs);
    switch (nbu) {
        case 1: return launch_nbu<BITS, BF16X, 1>(p, geo, m, s);
        case 2: return launch_nbu<BITS, BF16X, 2>(p, geo, m, s);
        case 4:
            if constexpr (BITS != 8) return launch_nbu<BITS, BF16X, 4>(p, geo, m, s);
            break;
        case 8:
            if constexpr (BITS == 2) return launch_nbu<BITS, BF16X, 8>(p, geo, m, s);
            break;
        default: break;
    }
    return cudaErrorNotSupported;
}

}  // namespace gtc
}  // namespace mnb
