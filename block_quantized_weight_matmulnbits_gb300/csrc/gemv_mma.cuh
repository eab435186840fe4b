// Small-batch GEMV on warp-level tensor-core MMA, 1 <= M <= 16, bf16 or f16 X:
//   Y[m, n] = sum_k X[m, k] * (q[n, k] - zp[n, kb]) * scale[n, kb]   (+ bias[n]).
//
// The operation is MatMulNBits as restated by onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs (fn dequantize_nbits_value; MatMulNBitsKernel::
// execute).  The pages' decode kernels are CPU SIMD loops; this kernel is a
// GB300 design.
//
// Why tensor cores for an HBM-bound GEMV: exact unpacking costs at least two
// issue slots per weight (mask into a float's mantissa, subtract), and a CUDA-
// core FMA per weight on top of that exceeds the issue budget GB300 leaves per
// weight when HBM3e streams ~7 TB/s.  With W rows as the MMA's M dimension
// (16 rows) and activation rows as its N dimension (8 or 16), one mma.sync
// m16n8k16 consumes 256 weights per warp, so the contraction costs almost no
// issue slots and the unpack dominates:
//   * the packed layout gives each lane its A fragment directly: a 16-bit
//     code pair is masked into the mantissa of 128.0 (bf16) or 1024.0 (f16),
//     and one packed 16-bit subtract of (magic + zp) yields (q - zp) exactly;
//   * the MMA accumulates one quantisation block in f32 (products of bf16 or
//     f16 integers and activations are exact), then the fragment is scaled by
//     the block's f32 scale into the running sum;
//   * weights stream through a per-warp ring of shared-memory slots filled by
//     1-D bulk copies (cp.async.bulk, TMA engine), scales and zero points of
//     whole row-tiles are bulk-copied ahead and converted once per CTA.
// Partial sums of the warps (K-slices) are reduced in a fixed order, so
// results are bit-identical run to run.
#pragma once

#include <cstdlib>

#include "mnb_internal.h"

namespace mnb {
namespace gmma {

constexpr int kMaxSlots = 12;
constexpr int kMinSlots = 3;
constexpr int kRawSlots = 4;
constexpr uint32_t kMagic23 = 0x4B000000u;

struct Geom {
    int warps;            // consumer warps per CTA (8 or 16)
    int chunk_tiles;      // 512-byte tiles per bulk copy (1, 2 or 4)
    int slots;            // ring slots per warp
    int stage_bufs;       // 1 or 2
    int64_t ktw;          // k-tiles per warp slice (multiple of chunk_tiles)
    int64_t kblocks_pad;  // staged blocks per row
    int64_t ks_total;     // k-steps per row (KTILES * KT / 16)
    int raw_scale_bytes, raw_zp_bytes;
    size_t ring_bytes, xb_bytes, raw_bytes, stage_bytes, red_bytes, bar_bytes, total_bytes;
};

struct __align__(8) Entry {
    uint32_t zc;  // subtraction constant for the row-block (see unpack)
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
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%10,%11,%12,%13};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
              "f"(c[3]));
    } else {
        asm volatile(
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

    // Subtraction constant of a row-block with zero point z.
    __device__ __forceinline__ static uint32_t zconst(uint32_t z) {
        if constexpr (BITS == 8 && BF16X) {
            return kMagic23 | z;  // f32 2^23 + z
        } else {
            const uint32_t h = (kMagic16x2 & 0xFFFFu) + z;  // magic + z, one 16-bit lane
            return h | (h << 16);
        }
    }

    __device__ __forceinline__ static void kstep(const uint32_t* w, int s, uint32_t zg, uint32_t zg8,
                                                 uint32_t (&a)[4]) {
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

// Host-side geometry: the widest CTA and deepest ring that fit shared memory.
// Overrides for tuning: MNB_MMA_WARPS (8/16), MNB_MMA_CHUNK (1/2/4 tiles),
// MNB_MMA_SLOTS (max ring slots per warp), MNB_MMA_STAGE_BUFS (1/2).
inline Geom make_geom(const Layout& L, int64_t M, int scale_dtype, bool has_zp, size_t smem_limit, int MT) {
    Geom best{};
    best.total_bytes = (size_t)-1;
    const int fw = env_or("MNB_MMA_WARPS", 0), fc = env_or("MNB_MMA_CHUNK", 0);
    const int fs = env_or("MNB_MMA_SLOTS", kMaxSlots), fb = env_or("MNB_MMA_STAGE_BUFS", 0);
    const int warps_opts[2] = {16, 8};
    for (int wi = 0; wi < 2; ++wi) {
        const int W = warps_opts[wi];
        if (fw && fw != W) continue;
        for (int ct = 4; ct >= 1; ct >>= 1) {
            if (fc && fc != ct) continue;
            Geom g{};
            g.warps = W;
            g.chunk_tiles = ct;
            const int64_t per = (L.KTILES + W - 1) / W;
            g.ktw = (per + ct - 1) / ct * ct;
            // skip chunk sizes that would leave a quarter or more of the warps idle
            if ((L.KTILES + g.ktw - 1) / g.ktw < (W * 3 + 3) / 4 && ct > 1) continue;
            g.kblocks_pad = (L.KTILES * L.KT + L.bs - 1) / L.bs;
            g.ks_total = L.KTILES * L.KT / 16;
            g.raw_scale_bytes = (int)(16 * L.KB * (scale_dtype == kF32 ? 4 : 2));
            g.raw_zp_bytes = has_zp ? (int)(16 * L.zp_row) : 0;
            g.xb_bytes = (size_t)M * g.ks_total * 32;
            g.raw_bytes = (size_t)kRawSlots * (round16(g.raw_scale_bytes) + round16(g.raw_zp_bytes));
            g.red_bytes = (size_t)2 * W * 16 * MT * 4;
            g.bar_bytes = (size_t)(W * kMaxSlots + kRawSlots) * 8;
            for (int bufs = 2; bufs >= 1; --bufs) {
                if (fb && fb != bufs) continue;
                g.stage_bufs = bufs;
                g.stage_bytes = (size_t)bufs * 16 * (g.kblocks_pad | 1) * sizeof(Entry);
                const size_t fixed = g.xb_bytes + g.raw_bytes + g.stage_bytes + g.red_bytes + g.bar_bytes + 128;
                const size_t chunk = (size_t)ct * kTileBytes;
                int slots = fs > kMaxSlots ? kMaxSlots : fs;
                while (slots > kMinSlots && fixed + (size_t)W * slots * chunk > smem_limit) --slots;
                g.slots = slots;
                g.ring_bytes = (size_t)W * slots * chunk;
                g.total_bytes = g.ring_bytes + fixed;
                if (g.total_bytes <= smem_limit && g.ring_bytes >= (96u << 10)) return g;
                if (g.total_bytes <= smem_limit && (best.total_bytes == (size_t)-1 || g.ring_bytes > best.ring_bytes))
                    best = g;
            }
        }
    }
    return best;
}

// SPB_LOG >= 0: blocks of 2^SPB_LOG k-steps tile every chunk (static block
// structure); -1: any block size, run-time checks.
template <int BITS, bool BF16X, int MT, int SPB_LOG>
__global__ void __launch_bounds__(512, 1) gemv_mma_kernel(MatmulParams p, Geom geo) {
    using U = Unpack<BITS, BF16X>;
    constexpr int NTILE = MT / 8;  // MMA n8 tiles (activation rows 0-7, 8-15)
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    const int W = geo.warps;
    const int T = W * 32;
    const int chunk_bytes = geo.chunk_tiles * kTileBytes;
    uint8_t* ring = smem;
    uint8_t* xb = smem + geo.ring_bytes;
    uint8_t* raw = xb + geo.xb_bytes;
    Entry* stage = reinterpret_cast<Entry*>(raw + geo.raw_bytes);
    float* red = reinterpret_cast<float*>(raw + geo.raw_bytes + geo.stage_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(raw + geo.raw_bytes + geo.stage_bytes + geo.red_bytes);
    uint64_t* rbars = bars + W * kMaxSlots;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = (int)p.M;
    const int my_tiles = (int)((L.NT - blockIdx.x + gridDim.x - 1) / gridDim.x);
    if (my_tiles <= 0) return;
    const int S_SLOTS = geo.slots;
    const int CT = geo.chunk_tiles;

    // ---- weight stream of this warp's K-slice ----
    const int64_t kt_begin = imin64((int64_t)warp * geo.ktw, L.KTILES);
    const int64_t kt_end = imin64(kt_begin + geo.ktw, L.KTILES);
    const int nch = (int)((kt_end - kt_begin + CT - 1) / CT);
    const int total_chunks = nch * my_tiles;
    uint64_t* wbars = bars + warp * kMaxSlots;
    uint8_t* wring = ring + (size_t)warp * S_SLOTS * chunk_bytes;
    int iss_i = 0, iss_c = 0, iss_slot = 0, issued = 0;
    auto issue_next = [&]() {  // lane 0 only
        const int64_t rt = blockIdx.x + (int64_t)iss_i * gridDim.x;
        const int64_t kt = kt_begin + (int64_t)iss_c * CT;
        const uint32_t bytes = (uint32_t)(imin64(CT, kt_end - kt) * kTileBytes);
        mbar_arrive_expect_tx(&wbars[iss_slot], bytes);
        bulk_g2s(wring + iss_slot * chunk_bytes, p.packed + (rt * L.KTILES + kt) * kTileBytes, bytes,
                 &wbars[iss_slot]);
    };
    auto advance_issue = [&]() {
        ++issued;
        if (++iss_c == nch) { iss_c = 0; ++iss_i; }
        if (++iss_slot == S_SLOTS) iss_slot = 0;
    };

    // ---- raw scales / zero points of whole row-tiles ----
    const bool raw_ok = ((reinterpret_cast<uintptr_t>(p.scales) & 15) == 0) &&
                        (p.zp == nullptr || (reinterpret_cast<uintptr_t>(p.zp) & 15) == 0);
    const int raw_slot_bytes = (int)(round16(geo.raw_scale_bytes) + round16(geo.raw_zp_bytes));
    auto tile_by_copy = [&](int i) {
        const int64_t rt = blockIdx.x + (int64_t)i * gridDim.x;
        return raw_ok && (rt * 16 + 16 <= L.N);
    };
    auto issue_raw = [&](int i) {  // thread 0 only
        if (i >= my_tiles || !tile_by_copy(i)) return;
        const int64_t rt = blockIdx.x + (int64_t)i * gridDim.x;
        const int slot = i % kRawSlots;
        uint8_t* dst = raw + slot * raw_slot_bytes;
        mbar_arrive_expect_tx(&rbars[slot], (uint32_t)(geo.raw_scale_bytes + geo.raw_zp_bytes));
        bulk_g2s(dst, static_cast<const uint8_t*>(p.scales) + rt * geo.raw_scale_bytes,
                 (uint32_t)geo.raw_scale_bytes, &rbars[slot]);
        if (geo.raw_zp_bytes)
            bulk_g2s(dst + round16(geo.raw_scale_bytes), p.zp + rt * geo.raw_zp_bytes, (uint32_t)geo.raw_zp_bytes,
                     &rbars[slot]);
    };

    if (lane == 0)
        for (int s = 0; s < S_SLOTS; ++s) mbar_init(&wbars[s], 1);
    if (tid == 0)
        for (int s = 0; s < kRawSlots; ++s) mbar_init(&rbars[s], 1);
    fence_barrier_init();
    __syncthreads();
    {
        const int n0 = total_chunks < S_SLOTS ? total_chunks : S_SLOTS;
        for (int q0 = 0; q0 < n0; ++q0) {
            if (lane == 0) issue_next();
            advance_issue();
        }
    }
    if (tid == 0)
        for (int i = 0; i < kRawSlots; ++i) issue_raw(i);

    // ---- B operand: activation row m, k-step S, lane class t -> 8 bytes
    //      (X[m][16S+2t], X[m][16S+2t+1]) | (X[m][16S+2t+8], X[m][16S+2t+9]) ----
    {
        const int64_t KS = geo.ks_total;
        const int64_t items = (int64_t)M * KS;
        const bool vec = (L.K % 8) == 0;  // rows of X are 16-byte aligned
        const uint16_t* x16 = static_cast<const uint16_t*>(p.x);
        constexpr int kRound = 4;
        for (int64_t i0 = tid; i0 < items; i0 += (int64_t)T * kRound) {
            uint4 v[kRound][2];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const int64_t it = i0 + (int64_t)u * T;
                if (it >= items) continue;
                const int64_t m = it / KS, S = it - m * KS;
                const int64_t k0 = 16 * S;
                if (vec && k0 + 16 <= L.K) {
                    const uint4* src = reinterpret_cast<const uint4*>(x16 + m * L.K + k0);
                    v[u][0] = __ldg(src);
                    v[u][1] = __ldg(src + 1);
                } else {
                    uint32_t h[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int64_t ka = k0 + 2 * j, kb2 = ka + 1;
                        const uint32_t lo = ka < L.K ? x16[m * L.K + ka] : 0u;
                        const uint32_t hi = kb2 < L.K ? x16[m * L.K + kb2] : 0u;
                        h[j] = lo | (hi << 16);
                    }
                    v[u][0] = make_uint4(h[0], h[1], h[2], h[3]);
                    v[u][1] = make_uint4(h[4], h[5], h[6], h[7]);
                }
            }
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const int64_t it = i0 + (int64_t)u * T;
                if (it >= items) continue;
                uint2* dst = reinterpret_cast<uint2*>(xb) + it * 4;
                dst[0] = make_uint2(v[u][0].x, v[u][1].x);
                dst[1] = make_uint2(v[u][0].y, v[u][1].y);
                dst[2] = make_uint2(v[u][0].z, v[u][1].z);
                dst[3] = make_uint2(v[u][0].w, v[u][1].w);
            }
        }
    }

    // ---- staged (constant, scale) per row-block; entry (r, kb) at r * kbs + kb ----
    const int kbp = (int)geo.kblocks_pad;
    const int kbs = kbp | 1;
    const int stage_stride = 16 * kbs;
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;
    const int zmask = code_mask(BITS);
    const int tpr = T / 16;  // converting threads per row
    const int conv_r = tid / tpr, conv_j = tid % tpr;
    auto convert = [&](int i, int buf) {
        Entry* dst = stage + buf * stage_stride + conv_r * kbs;
        const int64_t rt = blockIdx.x + (int64_t)i * gridDim.x;
        const int64_t n = rt * 16 + conv_r;
        const int kbv = (int)L.KB;
        if (tile_by_copy(i)) {
            const int slot = i % kRawSlots;
            mbar_wait(&rbars[slot], (uint32_t)((i / kRawSlots) & 1), p.status);
            const uint8_t* rs = raw + slot * raw_slot_bytes;
            const uint8_t* rz = rs + round16(geo.raw_scale_bytes) + conv_r * L.zp_row;
            const float* rs32 = reinterpret_cast<const float*>(rs) + conv_r * kbv;
            const uint16_t* rs16 = reinterpret_cast<const uint16_t*>(rs) + conv_r * kbv;
            const bool has_zp = geo.raw_zp_bytes != 0;
            for (int kb = conv_j; kb < kbp; kb += tpr) {
                uint32_t z = 0;
                float sc = 0.f;
                if (kb < kbv) {
                    if (sbytes == 4) {
                        sc = rs32[kb];
                    } else {
                        const uint16_t u = rs16[kb];
                        sc = p.scale_dtype == kF16 ? __half2float(__ushort_as_half(u))
                                                   : __uint_as_float((uint32_t)u << 16);
                    }
                    const int bit = kb * BITS;
                    z = has_zp ? ((rz[bit >> 3] >> (bit & 7)) & zmask) : (1u << (BITS - 1));
                }
                dst[kb] = Entry{U::zconst(z), sc};
            }
        } else {
            for (int kb = conv_j; kb < kbp; kb += tpr) {
                uint32_t z = 0;
                float sc = 0.f;
                if (n < L.N && kb < kbv) {
                    z = (uint32_t)load_zp(p.zp, L, n, kb);
                    sc = load_f32(p.scales, n * L.KB + kb, p.scale_dtype);
                }
                dst[kb] = Entry{U::zconst(z), sc};
            }
        }
    };

    convert(0, 0);
    __syncthreads();
    if (tid == 0) issue_raw(kRawSlots);

    // Lane's B-operand rows: activation rows g and g + 8, folded into [0, M)
    // (columns past M compute duplicates that are never stored).
    const uint2* xrow0 = reinterpret_cast<const uint2*>(xb) + (int64_t)(g % M) * geo.ks_total * 4 + t;
    const uint2* xrow1 = reinterpret_cast<const uint2*>(xb) + (int64_t)((g + 8) % M) * geo.ks_total * 4 + t;

    const int spb_log = SPB_LOG >= 0 ? SPB_LOG : __ffs(L.bs / 16) - 1;
    const int spb_mask = (1 << spb_log) - 1;
    constexpr int kStaticMask = SPB_LOG >= 0 ? (1 << (SPB_LOG >= 0 ? SPB_LOG : 0)) - 1 : 0;
    bool bad = false;
    int q = 0, slot = 0;
    uint32_t parity = 0;
    for (int i = 0; i < my_tiles; ++i) {
        const int64_t rt = blockIdx.x + (int64_t)i * gridDim.x;
        const int buf = geo.stage_bufs == 2 ? (i & 1) : 0;
        const Entry* st_g = stage + buf * stage_stride + g * kbs;
        const Entry* st_g8 = st_g + 8 * kbs;

        float y[NTILE][4];
        float acc[NTILE][4];
#pragma unroll
        for (int j = 0; j < NTILE; ++j)
#pragma unroll
            for (int c = 0; c < 4; ++c) y[j][c] = acc[j][c] = 0.f;
        const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
        int S = (int)(kt_begin * U::kStepsPerTile);
        uint32_t zg = 0, zg8 = 0;
        float sg = 0.f, sg8 = 0.f;
        bool first = true, fresh = true;

        for (int c = 0; c < nch; ++c, ++q) {
            if (!bad) bad = !mbar_wait(&wbars[slot], parity, p.status);
            if (!bad) {
                const int64_t kt = kt_begin + (int64_t)c * CT;
                const int ntile = (int)imin64(CT, kt_end - kt);
                const uint8_t* sbase = wring + slot * chunk_bytes;
#pragma unroll
                for (int tl = 0; tl < 4; ++tl) {
                    if (tl >= ntile) break;
                    const uint4 wv = reinterpret_cast<const uint4*>(sbase + tl * kTileBytes)[lane];
                    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int s = 0; s < U::kStepsPerTile; ++s) {
                        const int ks = tl * U::kStepsPerTile + s;
                        const int Sk = S + ks;
                        const bool block_start =
                            SPB_LOG >= 0 ? ((ks & kStaticMask) == 0) : (first || (Sk & spb_mask) == 0);
                        if (block_start) {
                            first = false;
                            const int kb = Sk >> spb_log;
                            const Entry eg = st_g[kb], eg8 = st_g8[kb];
                            zg = eg.zc;
                            sg = eg.s;
                            zg8 = eg8.zc;
                            sg8 = eg8.s;
                        }
                        uint32_t a[4];
                        U::kstep(w, s, zg, zg8, a);
                        // a block's first MMA starts from zero (static when blocks tile chunks)
                        const bool from_zero = SPB_LOG >= 0 ? ((ks & kStaticMask) == 0) : fresh;
                        const uint2 b0 = xrow0[(int64_t)Sk * 4];
                        if (from_zero) mma16816<BF16X>(acc[0], a, b0.x, b0.y, zero4);
                        else mma16816<BF16X>(acc[0], a, b0.x, b0.y, acc[0]);
                        if constexpr (NTILE == 2) {
                            const uint2 b1 = xrow1[(int64_t)Sk * 4];
                            if (from_zero) mma16816<BF16X>(acc[1], a, b1.x, b1.y, zero4);
                            else mma16816<BF16X>(acc[1], a, b1.x, b1.y, acc[1]);
                        }
                        fresh = false;
                        const bool block_end =
                            SPB_LOG >= 0 ? (((ks + 1) & kStaticMask) == 0) : (((Sk + 1) & spb_mask) == 0);
                        if (block_end) {
#pragma unroll
                            for (int j = 0; j < NTILE; ++j) {
                                y[j][0] = fmaf(sg, acc[j][0], y[j][0]);
                                y[j][1] = fmaf(sg, acc[j][1], y[j][1]);
                                y[j][2] = fmaf(sg8, acc[j][2], y[j][2]);
                                y[j][3] = fmaf(sg8, acc[j][3], y[j][3]);
                            }
                            fresh = true;
                        }
                    }
                }
                S += CT * U::kStepsPerTile;
                __syncwarp();
                if (issued < total_chunks) {
                    if (lane == 0) issue_next();
                    advance_issue();
                }
            }
            if (++slot == S_SLOTS) {
                slot = 0;
                parity ^= 1u;
            }
        }
        if (!fresh) {  // a block cut by the end of this warp's slice
#pragma unroll
            for (int j = 0; j < NTILE; ++j) {
                y[j][0] = fmaf(sg, acc[j][0], y[j][0]);
                y[j][1] = fmaf(sg, acc[j][1], y[j][1]);
                y[j][2] = fmaf(sg8, acc[j][2], y[j][2]);
                y[j][3] = fmaf(sg8, acc[j][3], y[j][3]);
            }
        }
        // red[buf2][warp][row][col]
        float* rb = red + (size_t)(i & 1) * W * 16 * MT;
        float* mine = rb + (size_t)warp * 16 * MT;
#pragma unroll
        for (int j = 0; j < NTILE; ++j) {
            const int col = j * 8 + 2 * t;
            mine[g * MT + col] = y[j][0];
            mine[g * MT + col + 1] = y[j][1];
            mine[(g + 8) * MT + col] = y[j][2];
            mine[(g + 8) * MT + col + 1] = y[j][3];
        }
        if (i + 1 < my_tiles) {
            if (geo.stage_bufs == 1) __syncthreads();
            convert(i + 1, geo.stage_bufs == 2 ? (buf ^ 1) : 0);
        }
        __syncthreads();
        if (tid == 0) issue_raw(i + 1 + kRawSlots);
        if (tid < 16 * M) {
            const int row = tid & 15, m = tid >> 4;
            float v = 0.f;
            for (int w2 = 0; w2 < W; ++w2) v += rb[(size_t)w2 * 16 * MT + row * MT + m];
            const int64_t n = rt * 16 + row;
            if (n < L.N) {
                if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
                store_f32(p.y, (int64_t)m * L.N + n, v, p.out_dtype);
            }
        }
    }
    if (bad && lane == 0) {
        for (int qq = q; qq < issued; ++qq) {
            const int sl = qq % S_SLOTS;
            const uint32_t ph = (uint32_t)((qq / S_SLOTS) & 1);
            for (int it = 0; it < (1 << 16); ++it)
                if (mbar_try_wait(&wbars[sl], ph)) break;
        }
    }
}

template <int BITS, bool BF16X, int MT, int SPB_LOG>
cudaError_t launch_variant(const MatmulParams& p, const Geom& geo, int64_t grid, cudaStream_t s) {
    auto kern = gemv_mma_kernel<BITS, BF16X, MT, SPB_LOG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)geo.total_bytes);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, geo.warps * 32, geo.total_bytes, s>>>(p, geo);
    return cudaGetLastError();
}

template <int BITS, bool BF16X, int MT>
cudaError_t launch_spb(const MatmulParams& p, const Geom& geo, int64_t grid, cudaStream_t s) {
    const int steps_per_chunk = geo.chunk_tiles * (16 / BITS);
    const int spb = p.L.bs / 16;
    if (steps_per_chunk % spb == 0) {
        switch (spb) {
            case 1: return launch_variant<BITS, BF16X, MT, 0>(p, geo, grid, s);
            case 2: return launch_variant<BITS, BF16X, MT, 1>(p, geo, grid, s);
            case 4: return launch_variant<BITS, BF16X, MT, 2>(p, geo, grid, s);
            case 8: return launch_variant<BITS, BF16X, MT, 3>(p, geo, grid, s);
            default: break;
        }
    }
    return launch_variant<BITS, BF16X, MT, -1>(p, geo, grid, s);
}

template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const Geom& geo, int64_t grid, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    if (p.M <= 8) return bf ? launch_spb<BITS, true, 8>(p, geo, grid, s) : launch_spb<BITS, false, 8>(p, geo, grid, s);
    return bf ? launch_spb<BITS, true, 16>(p, geo, grid, s) : launch_spb<BITS, false, 16>(p, geo, grid, s);
}

}  // namespace gmma
}  // namespace mnb
