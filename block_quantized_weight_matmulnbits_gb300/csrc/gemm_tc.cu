// Prefill GEMM on 5th-generation tensor cores (tcgen05 + TMEM + TMA), M >= 1,
// bf16 or f16 X:  Y[m, n] = sum_k X[m, k] * w[n, k]  (+ bias[n]),
// w = (q - zp) * scale as in onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs, fn dequantize_nbits_value.  The pages' prefill
// paths (AMX tile GEMM, dequantise-then-sgemm) are CPU designs; this is a
// GB300 design.
//
// One CTA computes one 128 x BN tile of Y (128 rows of X, BN rows of W):
//   warp 0      : producer.  Per 64-deep K stage (128 for 2-bit codes) it
//                 loads the X tile with a 2-D TMA copy (128B swizzle, zero
//                 fill past M and K) and the packed codes of the BN W rows
//                 with 1-D bulk copies (a 16-row tile is contiguous along K).
//   warp 1      : owns the TMEM accumulator (128 lanes x BN f32 columns) and,
//                 from one elected lane, issues tcgen05.mma kind::f16
//                 (M = 128, N = BN, K = 16) on the staged tiles; a
//                 tcgen05.commit per stage releases the stage.
//   warps 2-9   : dequantise the stage's codes to bf16/f16 straight into
//                 the canonical K-major 128B-swizzled layout the MMA reads:
//                 a code pair is masked into the mantissa of 128.0 / 1024.0,
//                 (q - zp) is one exact packed subtract, then one packed
//                 multiply by the block scale rounds w once to the MMA's
//                 input type.  After the K loop the same warps read the
//                 accumulator out of TMEM (tcgen05.ld), add the bias, round
//                 to the output dtype and store Y.
// Shared-memory stages are tracked by mbarriers (TMA bytes, dequant done,
// MMA done); every wait is bounded and reports MNB_ERR_TIMEOUT instead of
// hanging.  The reduction order over K is fixed, so results are
// deterministic.
#include <cstdio>
#include <cstdlib>
#include <cuda.h>

#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int kMaxRaw = 8;   // ring of X tiles + packed W (TMA destination)
constexpr int kWd = 4;       // ring of dequantised W tiles
constexpr int kBM = 128;
constexpr int kDequantWarps = 16;
constexpr int kThreads = (2 + kDequantWarps) * 32;

struct TcGeom {
    int BN;          // W rows per tile (multiple of 16, <= 256)
    int BK;          // depths per stage (64, or 128 for 2-bit codes)
    int tmem_cols;   // power of two >= BN
    int n_tiles;     // ceil(N / BN)
    int m_tiles;     // ceil(M / 128)
    int k_stages;    // ceil(Kpad / BK)
    int tiles_per_stage_row;  // packed 512-byte tiles per 16-row tile per stage
    int raw_stages;  // depth of the X + packed-W ring (<= kMaxRaw)
    int tab_stride;  // entries per row of the converted (zero point, scale) table (odd)
    size_t x_stage, wp_stage, wd_stage, scale_bytes, zp_bytes, tab_bytes, total_bytes;
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

// Byte offset of element (r, k) in a (rows x 64) K-major SW128 tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) + ((k & 7) << 1));
}

template <int BITS, bool BF16X>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(MatmulParams p, TcGeom geo,
                                                               const __grid_constant__ CUtensorMap xmap,
                                                               const __grid_constant__ CUtensorMap wmap) {
    const Layout& L = p.L;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int RS = geo.raw_stages;
    uint8_t* xs = smem;                                          // [RS][128 x BK] bf16, SW128 (TMA)
    uint8_t* wd = xs + RS * geo.x_stage;                         // [kWd][BN x BK] bf16, SW128
    uint8_t* wp = wd + kWd * geo.wd_stage;                       // [RS][BN/16][tiles][512 B] packed
    uint8_t* sraw = wp + RS * geo.wp_stage;                      // [BN][KB] raw scales of this tile's rows
    uint8_t* zraw = sraw + geo.scale_bytes;                      // [BN][zp_row] raw zero points
    uint32_t* tab = reinterpret_cast<uint32_t*>(zraw + geo.zp_bytes);  // [BN][tab_stride] converted
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(tab) + geo.tab_bytes);
    uint64_t* raw_full = bars;                   // X tile + packed W landed
    uint64_t* raw_empty = bars + kMaxRaw;        // MMA finished with the X tile (and so the codes)
    uint64_t* wd_full = bars + 2 * kMaxRaw;      // dequantised W written
    uint64_t* wd_empty = wd_full + kWd;          // MMA finished reading the dequantised W
    uint64_t* done = wd_empty + kWd;             // accumulator complete
    uint64_t* sbar = done + 1;                   // scales / zero points landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbar + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int BN = geo.BN, BK = geo.BK;
    const int n_tile = blockIdx.x % geo.n_tiles;
    const int m_tile = blockIdx.x / geo.n_tiles;
    const int64_t n0 = (int64_t)n_tile * BN;
    const int64_t m0 = (int64_t)m_tile * kBM;
    const int rows = (int)imin64(BN, L.N - n0);  // valid W rows of this tile
    const int KS = geo.k_stages;
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;

    if (tid == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 1);
        }
        for (int s = 0; s < kWd; ++s) {
            mbar_init(&wd_full[s], kDequantWarps / kWd);  // the dequant warps that own the slot
            mbar_init(&wd_empty[s], 1);
        }
        mbar_init(done, 1);
        mbar_init(sbar, 1);
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

    // Scales and zero points of this tile's rows: contiguous in the ORT layout.
    const size_t sc_bytes = (size_t)rows * L.KB * sbytes;
    const size_t z_bytes = p.zp ? (size_t)rows * L.zp_row : 0;
    const uint8_t* sc_src = static_cast<const uint8_t*>(p.scales) + (size_t)n0 * L.KB * sbytes;
    const uint8_t* z_src = p.zp ? p.zp + (size_t)n0 * L.zp_row : nullptr;
    const bool sc_bulk = (sc_bytes % 16 == 0) && ((reinterpret_cast<uintptr_t>(sc_src) & 15) == 0) &&
                         (z_bytes % 16 == 0) && (!z_src || (reinterpret_cast<uintptr_t>(z_src) & 15) == 0);

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            if (sc_bulk) {
                mbar_arrive_expect_tx(sbar, (uint32_t)(sc_bytes + z_bytes));
                bulk_g2s(sraw, sc_src, (uint32_t)sc_bytes, sbar);
                if (z_bytes) bulk_g2s(zraw, z_src, (uint32_t)z_bytes, sbar);
            }
            int issued = 0;
            for (int ks = 0; ks < KS; ++ks) {
                const int s = ks % RS;
                if (ks >= RS) {
                    if (!mbar_wait(&raw_empty[s], (uint32_t)(((ks / RS) - 1) & 1), p.status)) {
                        *abort_flag = 1;
                        break;
                    }
                }
                if (*reinterpret_cast<volatile int*>(abort_flag)) break;
                // one tensor copy of the stage's packed tiles for all BN / 16 row tiles
                // ([row tile][k tile][512 B], zero fill past N and past the last k tile)
                const int kt0 = ks * geo.tiles_per_stage_row;
                const uint32_t bytes = (uint32_t)(geo.x_stage + geo.wp_stage);
                mbar_arrive_expect_tx(&raw_full[s], bytes);
                for (int half = 0; half < BK / 64; ++half)
                    tma_load_2d(xs + s * geo.x_stage + half * (kBM * 128), &xmap, ks * BK + half * 64, (int)m0,
                                &raw_full[s]);
                tma_load_3d(wp + s * geo.wp_stage, &wmap, 0, kt0, (int)(n0 / 16), &raw_full[s]);
                issued = ks + 1;
            }
            if (*reinterpret_cast<volatile int*>(abort_flag)) {
                // give copies still in flight a bounded chance to land before the CTA exits
                for (int ks = issued - RS < 0 ? 0 : issued - RS; ks < issued; ++ks)
                    for (int it = 0; it < (1 << 16); ++it)
                        if (mbar_try_wait(&raw_full[ks % RS], (uint32_t)((ks / RS) & 1))) break;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        const uint32_t idesc = idesc_f16(BF16X, BN);
        for (int ks = 0; ks < KS; ++ks) {
            const int s = ks % RS, w = ks % kWd;
            bool ok = mbar_wait(&raw_full[s], (uint32_t)((ks / RS) & 1), p.status) &&
                      mbar_wait(&wd_full[w], (uint32_t)((ks / kWd) & 1), p.status);
            if (!ok) *abort_flag = 1;
            if (*reinterpret_cast<volatile int*>(abort_flag)) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t xa = smem_u32(xs + s * geo.x_stage);
                const uint32_t wa = smem_u32(wd + w * geo.wd_stage);
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const int half = kk >> 2, sub = kk & 3;
                    const uint64_t ad = sdesc_sw128(xa + half * (kBM * 128) + sub * 32);
                    const uint64_t bd = sdesc_sw128(wa + half * (BN * 128) + sub * 32);
                    tc_mma(tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&raw_empty[s]);
                tc_commit(&wd_empty[w]);
                if (ks == KS - 1) tc_commit(done);
            }
            __syncwarp();
        }
    } else {
        // ---------------- dequantiser, then epilogue ----------------
        const int dw = warp - 2;  // 0..7
        const bool bf = BF16X;
        constexpr uint32_t kMag = BF16X ? 0x43004300u : 0x64006400u;
        const int zmask = code_mask(BITS);
        if (!sc_bulk) {
            // cooperative plain copy of the scales / zero points (rare: ragged last tile)
            for (size_t i = (size_t)(tid - 64); i < sc_bytes; i += kDequantWarps * 32) sraw[i] = sc_src[i];
            for (size_t i = (size_t)(tid - 64); i < z_bytes; i += kDequantWarps * 32) zraw[i] = z_src[i];
            asm volatile("bar.sync 1, %0;" ::"n"(kDequantWarps * 32) : "memory");
        } else if (!mbar_wait(sbar, 0, p.status)) {
            *abort_flag = 1;
        }
        constexpr int KT = 256 / BITS;          // depths per packed tile
        constexpr int kSteps = 16 / BITS;       // k-steps per packed tile
        const int bs_log = __ffs(L.bs) - 1;     // block size is a power of two
        const int KBi = (int)L.KB;
        const int zrow = (int)L.zp_row;
        const int tstr = geo.tab_stride;
        // Table of (row, block): low 16 bits the zero-point constant (magic + zp
        // for the 16-bit paths, zp for 8-bit bf16), high 16 bits the scale
        // rounded once to the MMA input type; rows past N and blocks past KB
        // hold scale 0.  Built once per CTA; the odd row stride keeps the 8 row
        // groups of a warp on different banks.
        for (int r = dw; r < BN; r += kDequantWarps) {
            for (int kb = lane; kb < tstr; kb += 32) {
                float sc = 0.f;
                uint32_t z = 0;
                if (r < rows && kb < KBi) {
                    const int i = r * KBi + kb;
                    if (sbytes == 4) {
                        sc = reinterpret_cast<const float*>(sraw)[i];
                    } else {
                        const uint16_t u = reinterpret_cast<const uint16_t*>(sraw)[i];
                        sc = p.scale_dtype == kF16 ? __half2float(__ushort_as_half(u))
                                                   : __uint_as_float((uint32_t)u << 16);
                    }
                    if (p.zp) {
                        const int bit = kb * BITS;
                        z = (zraw[r * zrow + (bit >> 3)] >> (bit & 7)) & zmask;
                    } else {
                        z = 1u << (BITS - 1);
                    }
                }
                const uint32_t zc = (BITS == 8 && BF16X) ? z : ((kMag & 0xFFFFu) + z);
                tab[r * tstr + kb] = zc | (to_pair(sc, bf) << 16);
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kDequantWarps * 32) : "memory");
        auto consts = [&](int r, int kb, uint32_t& zc, uint32_t& sp) {
            const uint32_t e = tab[r * tstr + kb];
            sp = prmt(e, e, 0x3232u);  // scale in both halves
            if constexpr (BITS == 8 && BF16X) zc = 0x4B000000u | (e & 0xFFu);
            else zc = prmt(e, e, 0x1010u);  // zero-point constant in both halves
        };
        const int rts = BN / 16;
        const int tiles = geo.tiles_per_stage_row;
        const int g = lane >> 2, t = lane & 3;
        // Stage ks belongs to the kDequantWarps / kWd warps with dw % kWd == ks % kWd;
        // warp dw / kWd of them takes every (kDequantWarps / kWd)-th unit.  Each warp
        // so works on every kWd-th stage, and kWd stages are dequantised at once.
        constexpr int kOwners = kDequantWarps / kWd;
        const int my_slot = dw % kWd, my_part = dw / kWd;
        constexpr int kMaxUnits = 4;               // units of one warp per stage (BN <= 256)
        const int units = rts * tiles;
        for (int ks = my_slot; ks < KS; ks += kWd) {
            const int s = ks % RS, w = my_slot;
            if (ks >= kWd && !mbar_wait(&wd_empty[w], (uint32_t)(((ks / kWd) - 1) & 1), p.status)) *abort_flag = 1;
            if (!mbar_wait(&raw_full[s], (uint32_t)((ks / RS) & 1), p.status)) *abort_flag = 1;
            if (*reinterpret_cast<volatile int*>(abort_flag)) break;
            const uint8_t* src = wp + s * geo.wp_stage;
            uint8_t* dst = wd + w * geo.wd_stage;
            // unit = (16-row tile, packed tile of the stage); one lane's 16 bytes each
#pragma unroll
            for (int ui = 0; ui < kMaxUnits; ++ui) {
                const int u = kOwners * ui + my_part;
                if (u >= units) continue;
                const int rt = u / tiles, tl = u - rt * tiles;
                const int r0 = rt * 16 + g, r1 = r0 + 8;
                const int kbase = ks * BK + tl * KT;
                uint32_t zcs[2][kSteps], sps[2][kSteps];
#pragma unroll
                for (int st = 0; st < kSteps; ++st) {
                    const int kb = (kbase + 16 * st) >> bs_log;
                    const int kb_prev = st ? (kbase + 16 * (st - 1)) >> bs_log : -1;
                    if (kb != kb_prev) {
                        consts(r0, kb, zcs[0][st], sps[0][st]);
                        consts(r1, kb, zcs[1][st], sps[1][st]);
                    } else {
                        zcs[0][st] = zcs[0][st - 1];
                        sps[0][st] = sps[0][st - 1];
                        zcs[1][st] = zcs[1][st - 1];
                        sps[1][st] = sps[1][st - 1];
                    }
                }
                const uint4 wv = reinterpret_cast<const uint4*>(src + (size_t)u * kTileBytes)[lane];
                const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
                // swizzled row bases: row r at (r/8)*1024 + (r%8)*128, chunk index xor (r%8)
                const uint32_t base0 = (uint32_t)((r0 >> 3) * 1024 + (r0 & 7) * 128 + 4 * t);
                const uint32_t base1 = (uint32_t)((r1 >> 3) * 1024 + (r1 & 7) * 128 + 4 * t);
                const uint32_t xr = (uint32_t)(r0 & 7);  // r1 & 7 == r0 & 7
#pragma unroll
                for (int st = 0; st < kSteps; ++st) {
                    const uint32_t zc0 = zcs[0][st], zc1 = zcs[1][st];
                    const uint32_t sp0 = sps[0][st], sp1 = sps[1][st];
                    uint32_t a[4];
                    if constexpr (BITS == 4) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t v = lop3_and_or(w[st] >> (4 * r), 0x000F000Fu, kMag);
                            a[r] = hmul2(hsub2(v, (r & 1) ? zc1 : zc0, bf), (r & 1) ? sp1 : sp0, bf);
                        }
                    } else if constexpr (BITS == 2) {
                        const uint32_t word = w[st >> 1];
                        const int base = (st & 1) * 4;
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const uint32_t v = lop3_and_or(word >> (2 * (base + r)), 0x00030003u, kMag);
                            a[r] = hmul2(hsub2(v, (r & 1) ? zc1 : zc0, bf), (r & 1) ? sp1 : sp0, bf);
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
                                          (r & 1) ? zc1 : zc0, bf);
                            }
                            a[r] = hmul2(q, (r & 1) ? sp1 : sp0, bf);
                        }
                    }
                    // register r: row r0 (r even) / r1 (r odd), depths 2t(+1) (+8 for r >= 2)
                    const int kl = tl * KT + 16 * st;   // depth inside the stage
                    uint8_t* tile = dst + (size_t)(kl >> 6) * (BN * 128);
                    const uint32_t c0 = (uint32_t)((((kl & 63) >> 3) ^ xr) << 4);      // depths 2t, 2t+1
                    const uint32_t c1 = (uint32_t)(((((kl & 63) >> 3) + 1) ^ xr) << 4); // depths 2t+8, 2t+9
                    *reinterpret_cast<uint32_t*>(tile + base0 + c0) = a[0];
                    *reinterpret_cast<uint32_t*>(tile + base1 + c0) = a[1];
                    *reinterpret_cast<uint32_t*>(tile + base0 + c1) = a[2];
                    *reinterpret_cast<uint32_t*>(tile + base1 + c1) = a[3];
                }
            }
            fence_proxy_async_smem();  // make the generic-proxy writes visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&wd_full[w]);
        }

        // ---------------- epilogue: TMEM -> registers -> Y ----------------
        if (dw < 4) {
            const int quad = warp & 3;  // TMEM lane quadrant this warp may access
            bool ok = !*reinterpret_cast<volatile int*>(abort_flag) && mbar_wait(done, 0, p.status);
            if (ok) {
                tc_fence_after();
                const int64_t m = m0 + quad * 32 + lane;
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t r[16];
                    tc_ld16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)c0, r);
                    if (m < p.M) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int64_t n = n0 + c0 + j;
                            if (n < L.N) {
                                float v = __uint_as_float(r[j]);
                                if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
                                store_f32(p.y, m * L.N + n, v, p.out_dtype);
                            }
                        }
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

// ---- host side ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &ptr, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

TcGeom make_geom(const MatmulParams& p) {
    TcGeom g{};
    const Layout& L = p.L;
    g.BK = L.bits == 2 ? 128 : 64;
    g.tiles_per_stage_row = (int)(g.BK / L.KT);  // 4-bit: 1, 8-bit: 2, 2-bit: 1
    g.m_tiles = (int)((p.M + kBM - 1) / kBM);
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    // BN (multiple of 16, <= 256): fewest waves, then least padded work
    const char* env = std::getenv("MNB_TC_BN");
    const int forced = env ? std::atoi(env) : 0;
    double best = 1e30;
    // the four warps that own a stage handle at most 4 (16-row tile, packed tile) units each
    const int max_bn = 16 * 4 * (kDequantWarps / kWd) / g.tiles_per_stage_row;
    for (int bn = 32; bn <= 256 && bn <= max_bn; bn += 16) {
        if (forced && bn != forced) continue;
        const int64_t nt = (L.N + bn - 1) / bn;
        const int64_t tiles = nt * g.m_tiles;
        const int64_t waves = (tiles + sms - 1) / sms;
        const double cost = (double)waves * bn + 1e-3 * (double)(nt * bn - L.N);
        if (cost < best) {
            best = cost;
            g.BN = bn;
        }
    }
    g.n_tiles = (int)((L.N + g.BN - 1) / g.BN);
    g.tmem_cols = 32;
    while (g.tmem_cols < g.BN) g.tmem_cols <<= 1;
    g.k_stages = (int)((L.KTILES * L.KT + g.BK - 1) / g.BK);
    g.x_stage = (size_t)kBM * g.BK * 2;
    g.wd_stage = (size_t)g.BN * g.BK * 2;
    g.wp_stage = (size_t)(g.BN / 16) * g.tiles_per_stage_row * kTileBytes;
    g.scale_bytes = round16((size_t)g.BN * L.KB * (p.scale_dtype == kF32 ? 4 : 2));
    g.zp_bytes = round16(p.zp ? (size_t)g.BN * L.zp_row : 0);
    // blocks reachable by the staged depths (the packed rows run to KTILES * KT)
    g.tab_stride = (int)(((L.KTILES * L.KT + L.bs - 1) / L.bs) | 1);
    g.tab_bytes = round16((size_t)g.BN * g.tab_stride * 4);
    const size_t fixed = 1024 + kWd * g.wd_stage + g.scale_bytes + g.zp_bytes + g.tab_bytes +
                         (2 * kMaxRaw + 2 * kWd + 4) * 8 + 16;
    const size_t limit = device_info().smem_optin ? device_info().smem_optin : 232448;
    g.raw_stages = kMaxRaw;
    while (g.raw_stages > 2 && fixed + g.raw_stages * (g.x_stage + g.wp_stage) > limit) --g.raw_stages;
    g.total_bytes = fixed + g.raw_stages * (g.x_stage + g.wp_stage);
    return g;
}

template <int BITS, bool BF16X>
cudaError_t launch(const MatmulParams& p, const TcGeom& geo, const CUtensorMap& map, const CUtensorMap& wmap,
                   cudaStream_t s) {
    auto kern = gemm_tc_kernel<BITS, BF16X>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(geo.n_tiles * geo.m_tiles), kThreads, geo.total_bytes, s>>>(p, geo, map, wmap);
    return cudaGetLastError();
}

}  // namespace

bool gemm_tc_supported(const MatmulParams& p) {
    if (p.g_idx != nullptr || p.M < 1) return false;
    if (p.act_dtype != kBF16 && p.act_dtype != kF16) return false;
    const DeviceInfo& di = device_info();
    if (di.major != 10) return false;                   // tcgen05 needs the sm_100 family
    if ((p.L.K * 2) % 16 != 0) return false;            // TMA row stride of X
    if ((reinterpret_cast<uintptr_t>(p.x) & 15) != 0) return false;
    if (p.L.K > (int64_t)1 << 31 || p.M > (int64_t)1 << 31) return false;
    if (!encode_fn()) return false;
    const TcGeom g = make_geom(p);
    return g.total_bytes <= di.smem_optin && (int64_t)g.n_tiles * g.m_tiles < (int64_t)1 << 31;
}

cudaError_t launch_gemm_tc(const MatmulParams& p, cudaStream_t s) {
    const TcGeom geo = make_geom(p);
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)p.L.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.L.K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBM};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        p.act_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(&map, dt, 2, const_cast<void*>(p.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // Packed codes as a 3-D tensor of 16-bit elements: [row tile][k tile][256 x u16].
    CUtensorMap wmap;
    const cuuint64_t wdims[3] = {256, (cuuint64_t)p.L.KTILES, (cuuint64_t)p.L.NT};
    const cuuint64_t wstrides[2] = {(cuuint64_t)kTileBytes, (cuuint64_t)p.L.KTILES * kTileBytes};
    const cuuint32_t wbox[3] = {256, (cuuint32_t)geo.tiles_per_stage_row, (cuuint32_t)(geo.BN / 16)};
    const cuuint32_t westr[3] = {1, 1, 1};
    r = enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint8_t*>(p.packed), wdims, wstrides, wbox, westr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const bool bf = p.act_dtype == kBF16;
    switch (p.L.bits) {
        case 2: return bf ? launch<2, true>(p, geo, map, wmap, s) : launch<2, false>(p, geo, map, wmap, s);
        case 4: return bf ? launch<4, true>(p, geo, map, wmap, s) : launch<4, false>(p, geo, map, wmap, s);
        case 8: return bf ? launch<8, true>(p, geo, map, wmap, s) : launch<8, false>(p, geo, map, wmap, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
