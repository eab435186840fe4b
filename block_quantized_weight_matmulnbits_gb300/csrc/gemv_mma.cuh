// Small-batch GEMV on warp-level tensor-core MMA, 1 <= M <= 16, bf16 or f16 X:
//   Y[m, n] = sum_k X[m, k] * (q[n, k] - zp[n, kb]) * scale[n, kb]   (+ bias[n]).
//
// The operation is MatMulNBits as restated by onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs (fn dequantize_nbits_value; MatMulNBitsKernel::
// execute).  The pages' decode kernels are CPU SIMD loops; this kernel is a
// GB300 design.
//
// Why tensor cores for an HBM-bound GEMV: exact unpacking costs at least two
// issue slots per weight (mask into a float's mantissa, subtract), and a
// CUDA-core FMA per weight on top of that exceeds the issue budget GB300
// leaves per weight when HBM3e streams ~7 TB/s.  With W rows as the MMA's M
// dimension (16 rows) and activation rows as its N dimension (8 or 16), one
// mma.sync m16n8k16 consumes 256 weights per warp, so the contraction costs
// almost no issue slots and the unpack dominates:
//   * the packed layout gives each lane its A fragment directly: a 16-bit
//     code pair is masked into the mantissa of 128.0 (bf16) or 1024.0 (f16),
//     and one packed 16-bit subtract of (magic + zp) yields (q - zp) exactly;
//   * the MMA accumulates one quantisation block in f32 (products of small
//     integers and bf16/f16 activations are exact), then the fragment is
//     scaled by the block's f32 scale into the running sum.
//
// Work decomposition (measured on GB300: many resident CTAs with loads in
// registers stream a ~26 MB weight faster per launch than persistent
// bulk-copy rings): one CTA of 8 warps per (16-row tile, K-split); each warp
// issues all its 16-byte weight loads (up to 8 tiles) before anything else,
// then stages the CTA's activations and per-block scales / zero points in
// shared memory, then computes.  When K needs more than one CTA the K-splits
// of a row tile form a thread-block cluster and are summed through
// distributed shared memory in a fixed order; no global scratch is used.
// Every reduction order is fixed, so results are bit-identical run to run.
#pragma once

#include <cstdlib>

#include "mnb_internal.h"

namespace mnb {
namespace gmma {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxTPW = 8;       // tiles per warp per round (all loads in flight together)
constexpr int kMaxCluster = 8;   // portable cluster size
constexpr uint32_t kMagic23 = 0x4B000000u;

struct Geom {
    int C;            // K-splits = cluster size
    int tiles_cta;    // k-tiles per CTA (a multiple of kWarps * tpw, except the last split)
    int tpw;          // k-tiles per warp per round
    int rounds;       // rounds per warp
    int kb_cta;       // staged blocks per CTA (covers tiles_cta * KT depths)
    int ks_cta;       // k-steps per CTA
    size_t xb_bytes, stage_bytes, red_bytes, part_bytes, total_bytes;
};

struct __align__(8) Entry {
    uint32_t zc;  // subtraction constant for the row-block (see Unpack::zconst)
    float s;      // scale
};

__device__ __forceinline__ uint32_t hsub2_bf16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_f16(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
template <bool BF16X>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
    if constexpr (BF16X) {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%11,%12,%13};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
              "f"(c[3]));
    } else {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%11,%12,%13};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
              "f"(c[3]));
    }
}

// A fragment (4 registers of bf16/f16 pairs, exact q - zp) of k-step s of a
// lane's 16 packed bytes; zg / zg8 are the subtraction constants of rows g / g+8.
template <int BITS, bool BF16X>
struct Unpack {
    static constexpr int kStepsPerTile = 16 / BITS;  // 4-bit: 4, 2-bit: 8, 8-bit: 2
    static constexpr uint32_t kMagic16x2 = BF16X ? 0x43004300u : 0x64006400u;  // 128.0 / 1024.0 pairs

    __device__ __forceinline__ static uint32_t zconst(uint32_t z) {
        if constexpr (BITS == 8 && BF16X) {
            return kMagic23 | z;  // f32 2^23 + z (8-bit codes do not fit a bf16 mantissa)
        } else {
            const uint32_t h = (kMagic16x2 & 0xFFFFu) + z;  // magic + z in one 16-bit lane
            return h | (h << 16);
        }
    }

    __device__ __forceinline__ static void kstep(const uint4& wv, int s, uint32_t zg, uint32_t zg8,
                                                 uint32_t (&a)[4]) {
        const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
        if constexpr (BITS == 4) {
            const uint32_t word = w[s];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t v = lop3_and_or(word >> (4 * r), 0x000F000Fu, kMagic16x2);
                a[r] = BF16X ? hsub2_bf16(v, (r & 1) ? zg8 : zg) : hsub2_f16(v, (r & 1) ? zg8 : zg);
            }
        } else if constexpr (BITS == 2) {
            const uint32_t word = w[s >> 1];
            const int base = (s & 1) * 4;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t v = lop3_and_or(word >> (2 * (base + r)), 0x00030003u, kMagic16x2);
                a[r] = BF16X ? hsub2_bf16(v, (r & 1) ? zg8 : zg) : hsub2_f16(v, (r & 1) ? zg8 : zg);
            }
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t word = w[2 * s + (r >> 1)];
                const uint32_t b0 = 2 * (r & 1), b1 = b0 + 1;
                if constexpr (BF16X) {
                    const uint32_t va = prmt(word, kMagic23, 0x7650u | b0);
                    const uint32_t vb = prmt(word, kMagic23, 0x7650u | b1);
                    const uint32_t zc = (r & 1) ? zg8 : zg;
                    const float2 d = unpack2(fsub2(pack2u(va, vb), pack2u(zc, zc)));
                    a[r] = cvt_bf16x2(d.x, d.y);
                } else {
                    const uint32_t v = prmt(word, 0x64646464u, b0 | (4u << 4) | (b1 << 8) | (4u << 12));
                    a[r] = hsub2_f16(v, (r & 1) ? zg8 : zg);
                }
            }
        }
    }
};

inline int env_or(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

// Host-side geometry.  Each warp takes up to kMaxTPW k-tiles per round; a CTA
// takes kWarps warps' worth of tiles; the K-splits of a row tile form a
// cluster of at most kMaxCluster CTAs (more rounds per warp beyond that).
// MNB_MMA_TPW overrides the tiles per warp (1..8).
inline Geom make_geom(const Layout& L, int64_t M, int MT) {
    Geom g{};
    const int64_t KT = L.KTILES;
    int tpw = env_or("MNB_MMA_TPW", 0);
    if (tpw < 1 || tpw > kMaxTPW) {
        // enough tiles per warp that all warps work, at most kMaxTPW
        tpw = (int)((KT + kWarps - 1) / kWarps);
        if (tpw > kMaxTPW) tpw = kMaxTPW;
        if (tpw < 1) tpw = 1;
    }
    const int64_t per_round = (int64_t)kWarps * tpw;
    int64_t rounds_total = (KT + per_round - 1) / per_round;  // CTA-rounds along K
    int C = (int)(rounds_total < kMaxCluster ? rounds_total : kMaxCluster);
    if (C < 1) C = 1;
    const int rounds = (int)((rounds_total + C - 1) / C);
    g.C = C;
    g.tpw = tpw;
    g.rounds = rounds;
    g.tiles_cta = (int)(per_round * rounds);
    g.kb_cta = (int)((g.tiles_cta * L.KT + L.bs - 1) / L.bs);
    g.ks_cta = (int)(g.tiles_cta * L.KT / 16);
    g.xb_bytes = (size_t)M * g.ks_cta * 32;
    g.stage_bytes = (size_t)16 * (g.kb_cta | 1) * sizeof(Entry);
    g.red_bytes = (size_t)kWarps * 16 * MT * 4;
    g.part_bytes = (size_t)16 * MT * 4;
    g.total_bytes = g.xb_bytes + g.stage_bytes + g.red_bytes + g.part_bytes + 64;
    return g;
}

// Activation and output rows of one CTA: local row m (0 <= m < M <= MT)
// reads X row x_row(m) and writes Y row y_row(m).  prepare() runs once the
// weight loads are in flight and before X is staged (every thread calls it;
// it may synchronise the CTA) and fixes M.  The plain product uses rows
// 0 .. M-1 of both; the grouped product gathers and scatters.
struct DenseRows {
    int M;
    __device__ __forceinline__ void prepare() {}
    __device__ __forceinline__ int64_t x_row(int m) const { return m; }
    __device__ __forceinline__ int64_t y_row(int m) const { return m; }
};

// One CTA's share of the product: row tile rt, K-split `split` of its
// cluster, rows given by `rows`.  SPB_LOG >= 0: blocks of 2^SPB_LOG k-steps
// start at every warp slice (static block structure); -1: any block size,
// run-time checks.
template <int BITS, bool BF16X, int MT, int SPB_LOG, class Rows>
__device__ __forceinline__ void gemv_tile(const MatmulParams& p, const Geom& geo, int pdl, int64_t rt, int split,
                                          Rows& rows, uint8_t* smem) {
    using U = Unpack<BITS, BF16X>;
    constexpr int NTILE = MT / 8;  // MMA n8 tiles (activation rows 0-7, 8-15)
    constexpr int SPT = U::kStepsPerTile;
    const Layout& L = p.L;
    uint8_t* xb = smem;
    Entry* stage = reinterpret_cast<Entry*>(smem + geo.xb_bytes);
    float* red = reinterpret_cast<float*>(smem + geo.xb_bytes + geo.stage_bytes);
    float* part = red + kWarps * 16 * MT;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int C = geo.C;
    const int64_t cta_t0 = (int64_t)split * geo.tiles_cta;  // first k-tile of this CTA
    const int64_t cta_t1 = imin64(cta_t0 + geo.tiles_cta, L.KTILES);
    const int tpw = geo.tpw;

    const int64_t k_cta0 = cta_t0 * L.KT;
    const int kb_cta = geo.kb_cta;
    const int kbs = kb_cta | 1;
    const int64_t kb0 = k_cta0 / L.bs;

    // ---- 1. loads, in the order their data is needed: this thread's run of 8
    //         (row, block) scales and zero points, then the warp's weight tiles.
    //         Decoding the small first loads overlaps the weight stream. ----
    const int runs = (kb_cta + 7) / 8;
    const bool stage_fast = 16 * runs <= kThreads;  // one run per thread (the common case)
    const int srow = tid / (runs > 0 ? runs : 1), srun = tid - srow * (runs > 0 ? runs : 1);
    const int64_t s_n = rt * 16 + srow;
    const int64_t s_kb = kb0 + (int64_t)srun * 8;
    const bool s_active = stage_fast && tid < 16 * runs;
    const bool s_row_ok = s_active && s_n < L.N;
    const bool s_full = s_row_ok && s_kb + 8 <= L.KB;
    const int64_t s_si = s_n * L.KB + s_kb;
    const bool s_vec16 = s_full && p.scale_dtype != kF32 && (s_si & 7) == 0 &&
                         (reinterpret_cast<uintptr_t>(p.scales) & 15) == 0;
    const bool s_vec32 = s_full && p.scale_dtype == kF32 && (s_si & 3) == 0 &&
                         (reinterpret_cast<uintptr_t>(p.scales) & 15) == 0;
    const uint8_t* s_zsrc = p.zp ? p.zp + s_n * L.zp_row + s_kb * BITS / 8 : nullptr;
    const bool z_vec = s_full && p.zp && (reinterpret_cast<uintptr_t>(s_zsrc) & (BITS - 1)) == 0;
    uint4 sv0 = make_uint4(0, 0, 0, 0), sv1 = make_uint4(0, 0, 0, 0);
    uint64_t zraw = 0;
    if (s_vec16) {
        sv0 = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.scales) + s_si));
    } else if (s_vec32) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(p.scales) + s_si);
        sv0 = __ldg(src);
        sv1 = __ldg(src + 1);
    }
    if (z_vec) {
        if (BITS == 2) zraw = __ldg(reinterpret_cast<const uint16_t*>(s_zsrc));
        else if (BITS == 4) zraw = __ldg(reinterpret_cast<const uint32_t*>(s_zsrc));
        else zraw = __ldg(reinterpret_cast<const unsigned long long*>(s_zsrc));
    }

    const uint8_t* wrow = p.packed + (rt * L.KTILES) * kTileBytes + lane * 16;
    auto warp_tile0 = [&](int round) { return cta_t0 + ((int64_t)round * kWarps + warp) * tpw; };
    uint4 wv[kMaxTPW];
    auto load_round = [&](int round) {
        const int64_t t0 = warp_tile0(round);
#pragma unroll
        for (int j = 0; j < kMaxTPW; ++j)
            if (j < tpw && t0 + j < cta_t1) wv[j] = ldg_stream(wrow + (t0 + j) * kTileBytes);
    };
    load_round(0);

    // ---- 2. per (row, block) subtraction constant and scale; entry (r, j) at r * kbs + j ----
    auto decode_run = [&](int r, int run, int64_t n, int64_t kbr, bool vec16, bool vec32, bool zv,
                          const uint4& a0, const uint4& a1, uint64_t zr) {
        const bool row_ok = n < L.N;
        const int64_t si = n * L.KB + kbr;
        float sc[8];
        uint32_t z[8];
        if (vec16) {
            const uint32_t h[4] = {a0.x, a0.y, a0.z, a0.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t lo = h[j] & 0xFFFFu, hi = h[j] >> 16;
                if (p.scale_dtype == kF16) {
                    sc[2 * j] = __half2float(__ushort_as_half((uint16_t)lo));
                    sc[2 * j + 1] = __half2float(__ushort_as_half((uint16_t)hi));
                } else {
                    sc[2 * j] = __uint_as_float(lo << 16);
                    sc[2 * j + 1] = __uint_as_float(hi << 16);
                }
            }
        } else if (vec32) {
            sc[0] = __uint_as_float(a0.x); sc[1] = __uint_as_float(a0.y);
            sc[2] = __uint_as_float(a0.z); sc[3] = __uint_as_float(a0.w);
            sc[4] = __uint_as_float(a1.x); sc[5] = __uint_as_float(a1.y);
            sc[6] = __uint_as_float(a1.z); sc[7] = __uint_as_float(a1.w);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                sc[j] = (row_ok && kbr + j < L.KB) ? load_f32(p.scales, si + j, p.scale_dtype) : 0.f;
        }
        uint64_t packed = zr;
        if (p.zp != nullptr && !zv) {
            packed = 0;
            const uint8_t* zsrc = p.zp + n * L.zp_row + kbr * BITS / 8;
#pragma unroll
            for (int j = 0; j < BITS; ++j) {
                // byte j holds blocks kbr + 8j/BITS ...; read it only if its first block exists
                if (row_ok && kbr + (8 * j) / BITS < L.KB) packed |= (uint64_t)__ldg(zsrc + j) << (8 * j);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            z[j] = p.zp ? ((uint32_t)(packed >> (j * BITS)) & code_mask(BITS)) : (1u << (BITS - 1));
        // two entries per 16-byte store
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const int jl = run * 8 + j;
            const bool v0 = row_ok && kbr + j < L.KB, v1 = row_ok && kbr + j + 1 < L.KB;
            const Entry e0{U::zconst(v0 ? z[j] : 0u), v0 ? sc[j] : 0.f};
            const Entry e1{U::zconst(v1 ? z[j + 1] : 0u), v1 ? sc[j + 1] : 0.f};
            Entry* dst = stage + r * kbs + jl;
            if (jl + 1 < kb_cta) {
                dst[0] = e0;
                dst[1] = e1;
            } else if (jl < kb_cta) {
                dst[0] = e0;
            }
        }
    };
    if (stage_fast) {
        if (s_active) decode_run(srow, srun, s_n, s_kb, s_vec16, s_vec32, z_vec, sv0, sv1, zraw);
    } else {
        for (int it = tid; it < 16 * runs; it += kThreads) {
            const int r = it / runs, run = it - r * runs;
            decode_run(r, run, rt * 16 + r, kb0 + (int64_t)run * 8, false, false, false, sv0, sv1, 0);
        }
    }
    if (pdl) {
        griddep_wait();  // X (and Y) may belong to the previous kernel on the stream
        // Only now may the next kernel launch: at most two kernels of a
        // programmatic chain overlap (this one, once its predecessor is
        // complete, and its successor's pre-wait part).
        griddep_launch_dependents();
    }
    rows.prepare();
    const int M = rows.M;

    // ---- 3. activations (B fragments) of this CTA's k-steps:
    //         row m, local k-step S, lane class t -> (X[m][k+2t..], X[m][k+2t+8..]);
    //         item (m, S) is 32 bytes written as two 16-byte stores ----
    {
        const int KS = geo.ks_cta;
        const int items = M * KS;
        const bool vec = (L.K % 8) == 0;  // rows of X are 16-byte aligned
        const uint16_t* x16 = static_cast<const uint16_t*>(p.x);
        for (int it = tid; it < items; it += kThreads) {
            const int m = it / KS, S = it - m * KS;
            const int64_t k0 = k_cta0 + 16 * (int64_t)S;
            const int64_t xr = rows.x_row(m);
            uint4 v0, v1;
            if (vec && k0 + 16 <= L.K) {
                const uint4* src = reinterpret_cast<const uint4*>(x16 + xr * L.K + k0);
                v0 = __ldg(src);
                v1 = __ldg(src + 1);
            } else {
                uint32_t h[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int64_t ka = k0 + 2 * j, kb2 = ka + 1;
                    const uint32_t lo = ka < L.K ? x16[xr * L.K + ka] : 0u;
                    const uint32_t hi = kb2 < L.K ? x16[xr * L.K + kb2] : 0u;
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

    // ---- 4. contraction ----
    // Shared-memory addresses as 32-bit values so every per-k-step access is a
    // base register plus a compile-time offset.
    const uint32_t st_base = smem_u32(stage + g * kbs);     // row g; row g + 8 is 8 * kbs entries on
    const uint32_t st_off8 = (uint32_t)(8 * kbs * sizeof(Entry));
    const uint32_t xa0 = smem_u32(reinterpret_cast<const uint2*>(xb) + (int64_t)(g % M) * geo.ks_cta * 4 + t);
    const uint32_t xa1 = smem_u32(reinterpret_cast<const uint2*>(xb) + (int64_t)((g + 8) % M) * geo.ks_cta * 4 + t);
    const int spb_log = SPB_LOG >= 0 ? SPB_LOG : __ffs(L.bs / 16) - 1;
    const int spb_mask = (1 << spb_log) - 1;
    constexpr int kStaticMask = SPB_LOG >= 0 ? (1 << (SPB_LOG >= 0 ? SPB_LOG : 0)) - 1 : 0;
    constexpr int kStaticLog = SPB_LOG >= 0 ? SPB_LOG : 0;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float y[NTILE][4];
    float acc[NTILE][4];
#pragma unroll
    for (int j = 0; j < NTILE; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) y[j][c] = acc[j][c] = 0.f;
    uint32_t zg = 0, zg8 = 0;
    float sg = 0.f, sg8 = 0.f;
    bool fresh = true, first = true;

    auto lds2 = [](uint32_t addr) {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
        return v;
    };

    for (int round = 0; round < geo.rounds; ++round) {
        const int64_t t0 = warp_tile0(round);
        if (round > 0) load_round(round);
        const int ntile = (int)imin64(tpw, cta_t1 - t0);  // may be <= 0
        const int S0 = (int)((t0 - cta_t0) * SPT);        // local k-step of this warp's first tile
        const uint32_t xr0 = xa0 + (uint32_t)S0 * 32u, xr1 = xa1 + (uint32_t)S0 * 32u;
        const uint32_t er = st_base + (uint32_t)(SPB_LOG >= 0 ? (S0 >> kStaticLog) : 0) * (uint32_t)sizeof(Entry);
#pragma unroll
        for (int j = 0; j < kMaxTPW; ++j) {
            if (j < ntile) {
#pragma unroll
                for (int s = 0; s < SPT; ++s) {
                    const int ks = j * SPT + s;  // k-step inside this warp's slice (static)
                    const int Sk = S0 + ks;      // k-step inside the CTA
                    const bool block_start =
                        SPB_LOG >= 0 ? ((ks & kStaticMask) == 0) : (first || (Sk & spb_mask) == 0);
                    if (block_start) {
                        first = false;
                        const uint32_t ea = SPB_LOG >= 0
                                                ? er + (uint32_t)(ks >> kStaticLog) * (uint32_t)sizeof(Entry)
                                                : st_base + (uint32_t)(Sk >> spb_log) * (uint32_t)sizeof(Entry);
                        const uint2 eg = lds2(ea), eg8 = lds2(ea + st_off8);
                        zg = eg.x;
                        sg = __uint_as_float(eg.y);
                        zg8 = eg8.x;
                        sg8 = __uint_as_float(eg8.y);
                    }
                    uint32_t a[4];
                    U::kstep(wv[j], s, zg, zg8, a);
                    const bool from_zero = SPB_LOG >= 0 ? ((ks & kStaticMask) == 0) : fresh;
                    const uint2 b0 = lds2(xr0 + (uint32_t)ks * 32u);
                    if (from_zero) mma16816<BF16X>(acc[0], a, b0.x, b0.y, zero4);
                    else mma16816<BF16X>(acc[0], a, b0.x, b0.y, acc[0]);
                    if constexpr (NTILE == 2) {
                        const uint2 b1 = lds2(xr1 + (uint32_t)ks * 32u);
                        if (from_zero) mma16816<BF16X>(acc[1], a, b1.x, b1.y, zero4);
                        else mma16816<BF16X>(acc[1], a, b1.x, b1.y, acc[1]);
                    }
                    fresh = false;
                    const bool block_end =
                        SPB_LOG >= 0 ? (((ks + 1) & kStaticMask) == 0) : (((Sk + 1) & spb_mask) == 0);
                    if (block_end) {
#pragma unroll
                        for (int q = 0; q < NTILE; ++q) {
                            y[q][0] = fmaf(sg, acc[q][0], y[q][0]);
                            y[q][1] = fmaf(sg, acc[q][1], y[q][1]);
                            y[q][2] = fmaf(sg8, acc[q][2], y[q][2]);
                            y[q][3] = fmaf(sg8, acc[q][3], y[q][3]);
                        }
                        fresh = true;
                    }
                }
            }
        }
        if (!fresh) {  // a block cut by the end of this warp's tiles
#pragma unroll
            for (int q = 0; q < NTILE; ++q) {
                y[q][0] = fmaf(sg, acc[q][0], y[q][0]);
                y[q][1] = fmaf(sg, acc[q][1], y[q][1]);
                y[q][2] = fmaf(sg8, acc[q][2], y[q][2]);
                y[q][3] = fmaf(sg8, acc[q][3], y[q][3]);
            }
            fresh = true;
        }
        first = true;
    }

    // ---- 5. reduce the warps' K-slices (fixed order), then the cluster's K-splits ----
    float* mine = red + warp * 16 * MT;
#pragma unroll
    for (int q = 0; q < NTILE; ++q) {
        const int col = q * 8 + 2 * t;
        mine[g * MT + col] = y[q][0];
        mine[g * MT + col + 1] = y[q][1];
        mine[(g + 8) * MT + col] = y[q][2];
        mine[(g + 8) * MT + col + 1] = y[q][3];
    }
    __syncthreads();
    const bool owner = tid < 16 * M;
    const int row = tid & 15, m = tid >> 4;
    float v = 0.f;
    if (owner) {
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) v += red[w2 * 16 * MT + row * MT + m];
    }
    if (C > 1) {
        if (owner) part[row * MT + m] = v;
        cluster_sync();
        if (split == 0 && owner) {
            v = part[row * MT + m];
            for (int c2 = 1; c2 < C; ++c2) v += ld_dsmem_f32(&part[row * MT + m], (uint32_t)c2);
        }
        cluster_sync();  // peers keep their shared memory until the leader has read it
    }
    if (split == 0 && owner) {
        const int64_t n = rt * 16 + row;
        if (n < L.N) {
            if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
            store_f32(p.y, rows.y_row(m) * L.N + n, v, p.out_dtype);
        }
    }
}

// The plain product: one CTA per (row tile, K-split), rows 0 .. M-1.
// Occupancy by code width (measured on GB300): 8-bit codes are the longest K
// (K-split clusters) and gain from 4 CTAs per SM; 2- and 4-bit codes are
// faster with 3 CTAs per SM and spill-free registers.
template <int BITS, bool BF16X, int MT, int SPB_LOG>
__global__ void __launch_bounds__(kThreads, BITS == 8 ? 4 : 3) gemv_mma_kernel(MatmulParams p, Geom geo, int pdl) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int64_t rt = blockIdx.x / geo.C;
    DenseRows rows{(int)p.M};
    gemv_tile<BITS, BF16X, MT, SPB_LOG>(p, geo, pdl, rt, (int)(blockIdx.x - rt * geo.C), rows, smem);
    if (blockIdx.x == 0 && threadIdx.x == 0) verify_header(p.packed_hdr, p.L, p.status);
}

template <int BITS, bool BF16X, int MT, int SPB_LOG>
cudaError_t launch_variant(const MatmulParams& p, const Geom& geo, cudaStream_t s) {
    const int pdl = (p.flags & kFlagPDL) ? 1 : 0;
    auto kern = gemv_mma_kernel<BITS, BF16X, MT, SPB_LOG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.L.NT * geo.C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = geo.total_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)geo.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p, geo, pdl);
}

// Static block structure when every warp slice starts on a block boundary and
// blocks are at most 8 k-steps.
template <int BITS, bool BF16X, int MT>
cudaError_t launch_spb(const MatmulParams& p, const Geom& geo, cudaStream_t s) {
    const int spb = p.L.bs / 16;
    const int steps_per_warp = geo.tpw * (16 / BITS);
    if (steps_per_warp % spb == 0) {
        switch (spb) {
            case 1: return launch_variant<BITS, BF16X, MT, 0>(p, geo, s);
            case 2: return launch_variant<BITS, BF16X, MT, 1>(p, geo, s);
            case 4: return launch_variant<BITS, BF16X, MT, 2>(p, geo, s);
            case 8: return launch_variant<BITS, BF16X, MT, 3>(p, geo, s);
            default: break;
        }
    }
    return launch_variant<BITS, BF16X, MT, -1>(p, geo, s);
}

template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const Geom& geo, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    if (p.M <= 8) return bf ? launch_spb<BITS, true, 8>(p, geo, s) : launch_spb<BITS, false, 8>(p, geo, s);
    return bf ? launch_spb<BITS, true, 16>(p, geo, s) : launch_spb<BITS, false, 16>(p, geo, s);
}

}  // namespace gmma
}  // namespace mnb
