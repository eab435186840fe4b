// Decode GEMV for 1 <= M <= 8, bf16 or f16 X, f32 / f16 / bf16 scales:
//   Y[m, n] = sum_kb scale[n, kb] * sum_{k in kb} X[m, k] * (q[n, k] - zp[n, kb])   (+ bias[n]),
// MatMulNBits as restated by onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs (fn dequantize_nbits_value; MatMulNBitsKernel::
// execute), with the arithmetic of gemv_mma.cuh: (q - zp) exact in the
// activation type (mantissa magic and one packed subtract), one mma.sync
// m16n8k16 per 256 weights, the block's f32 scale applied to the fragment.
//
// Schedule, shaped for the fewest issue slots per weight byte (a 26 MB int4
// weight must stream in ~4 us, so a k-step of 128 bytes has a budget of about
// 16 warp instructions on 152 SMs):
//   * one CTA of 16 warps per SM owns a contiguous range of 16-row tiles;
//   * work items are (row tile, K-chunk) pairs, a K-chunk being 4 packed
//     tiles: 64 bytes per lane, 16 k-steps of 4-bit codes (32 of 2-bit, 8 of
//     8-bit); warp w takes items w, w + 16, ... of its CTA, so every warp
//     gets the same number of items to within one;
//   * each item's weights, raw scales and raw zero points go straight from
//     global memory into registers one item ahead (double-buffered; no
//     shared-memory staging, no tables); scales and zero points are decoded
//     when their block starts (measured on GB300: asynchronous copies into a
//     deeper shared-memory ring, with or without staged scales, were slower);
//   * X is staged once in shared memory in B-fragment order, one 16-byte
//     load per lane per two k-steps;
//   * each warp keeps its partial sums of a row tile in registers and writes
//     them once per row tile; one pass at the end adds the 16 warps' partials
//     of every row in a fixed order, so results are bit-identical run to run.
// There are no waits on other threads besides two CTA barriers.
#pragma once

#include "gemv_mma.cuh"

namespace mnb {
namespace gks {

using gmma::mma16816;
using gmma::Unpack;

constexpr int kW = 16;
constexpr int kThreads = kW * 32;
constexpr int kTilesPerChunk = 4;  // 64 bytes per lane
constexpr int kItemBytes = kTilesPerChunk * kTileBytes;

struct KGeom {
    int G;        // CTAs
    int KC;       // K-chunks per row tile
    int q16, r16; // a step of kW items: q16 row tiles and r16 chunks
    int max_rt;   // most row tiles of one CTA
    int xrow;     // X row stride in 16-byte units (K / 8 + 4: padded against bank conflicts)
    int pairx;    // 1: X rows 2m, 2m + 1 are the hi and lo bf16 parts of one activation row m
                  // (accuracy level 4); Y row m is the sum of their two columns
    size_t x_bytes, red_bytes, total_bytes;
};

// Act-order pack: X as given (M rows of K 16-bit values) in shared memory after the partials.
inline size_t kperm_x_bytes(const Layout& L, int64_t M) { return (size_t)M * (size_t)L.K * 2; }

// k-steps per chunk for a code width: 4 packed tiles.
__host__ __device__ constexpr int chunk_steps(int bits) { return kTilesPerChunk * (16 / bits); }

// The shapes this schedule takes: the chunk depth divides K, a quantisation
// block lies inside one chunk, a row's scales of one chunk are at most 32
// bytes, and X (M + 1 rows) plus the partial sums fit in shared memory.
inline bool make_kgeom(const Layout& L, int64_t M, int sms, size_t smem_limit, int sbytes, KGeom* out) {
    if (M < 1 || M > 8) return false;
    const int ch = chunk_steps(L.bits);
    const int64_t chunk_k = (int64_t)ch * 16;
    if (L.K % chunk_k != 0) return false;
    const int spb = (int)(L.bs / 16);
    if (L.bs % 16 != 0 || spb < 1 || spb > ch || (spb & (spb - 1)) != 0) return false;
    if ((ch / spb) * sbytes > 32) return false;
    // scale, zero-point and a CTA's weight offsets are formed in 32 bits
    if ((uint64_t)L.N * (uint64_t)L.KB * 4u >= (1ull << 32) || (uint64_t)L.N * (uint64_t)L.zp_row >= (1ull << 32))
        return false;
    KGeom g{};
    g.KC = (int)(L.K / chunk_k);
    g.G = (int)(L.NT < sms ? L.NT : sms);
    g.max_rt = (int)((L.NT + g.G - 1) / g.G);
    if ((uint64_t)g.max_rt * (uint64_t)g.KC * (uint64_t)kItemBytes >= (1ull << 32)) return false;
    // CTA ranges are formed in 32 bits
    if ((uint64_t)L.NT * (uint64_t)(g.G + 1) >= (1ull << 31)) return false;
    g.q16 = kW / g.KC;
    g.r16 = kW % g.KC;
    g.xrow = (int)(L.K / 8) + 4;
    g.x_bytes = (size_t)(M + 1) * g.xrow * 16;
    g.red_bytes = (size_t)g.max_rt * kW * 16 * M * 4;
    g.total_bytes = g.x_bytes + g.red_bytes;
    if (g.total_bytes > smem_limit) return false;
    *out = g;
    return true;
}

template <int BYTES>
__device__ __forceinline__ void ld_raw(const void* src, uint32_t (&w)[BYTES >= 4 ? BYTES / 4 : 1]) {
    if constexpr (BYTES == 32) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else if constexpr (BYTES == 16) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    } else if constexpr (BYTES == 8) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(src));
        w[0] = a.x; w[1] = a.y;
    } else if constexpr (BYTES == 4) {
        w[0] = __ldg(reinterpret_cast<const uint32_t*>(src));
    } else if constexpr (BYTES == 2) {
        w[0] = __ldg(reinterpret_cast<const uint16_t*>(src));
    } else {
        w[0] = __ldg(reinterpret_cast<const uint8_t*>(src));
    }
}

template <int BITS, bool BF16X, int SPB_LOG, int SDT>
struct Item {
    static constexpr int SPT = 16 / BITS;              // k-steps per packed tile
    static constexpr int CH = kTilesPerChunk * SPT;     // k-steps per chunk
    static constexpr int SPB = 1 << SPB_LOG;            // k-steps per block
    static constexpr int BPC = CH / SPB;                // blocks per chunk
    static constexpr int SBYTES = BPC * (SDT == kF32 ? 4 : 2);  // raw scales of a row
    static constexpr int SW = SBYTES >= 4 ? SBYTES / 4 : 1;
    static constexpr int ZBITS = BPC * BITS;            // raw zero-point bits of a row
    static constexpr int ZBYTES = ZBITS >= 8 ? ZBITS / 8 : 1;
    static constexpr int ZW = ZBYTES >= 4 ? ZBYTES / 4 : 1;
    // zero points spread one per byte: block b in byte (b / NZS) % 4 of word
    // (b % NZS) + NZS * (b / (4 * NZS)), NZS = 8 / BITS words per raw word
    static constexpr int NZS = 8 / BITS;
    static constexpr int ZSW = BITS == 8 ? ZW : ZW * NZS;
    // every code field holding 2^(bits - 1): the zero point when none is given
    static constexpr uint32_t kZDefault = BITS == 2 ? 0xAAAAAAAAu : BITS == 4 ? 0x88888888u : 0x80808080u;
    // high byte of the subtraction constant (magic + z) in each 16-bit lane,
    // or the f32 magic 2^23 for 8-bit codes under bf16 activations
    static constexpr bool kF32Magic = BITS == 8 && BF16X;
    static constexpr uint32_t kZHigh = kF32Magic ? 0x4B000000u : ((Unpack<BITS, BF16X>::kMagic16x2 >> 8) & 0xFFu);
    static_assert(SPB <= CH && SBYTES <= 32, "block outside the chunk");

    uint4 w[kTilesPerChunk];
    uint32_t s0[SW], s8[SW];
    uint32_t z0[ZW], z8[ZW];  // raw code fields (spread when the item is computed)
    uint32_t zshift;          // bit offset of the chunk's first field (fields under 8 bits a chunk)

    // Loads of item (local row tile, chunk c): wp is the lane's 16 bytes of the
    // item's first packed tile; sb / zb the scale / zero-point bytes of the
    // CTA's first row; r0, r8 the lane's two rows (local, clamped to the last
    // row: rows past N read row N - 1, whose results are never stored, so the
    // loads need no predicates).  Offsets fit 32 bits.
    __device__ __forceinline__ void load(const uint8_t* wp, const uint8_t* sb, const uint8_t* zb, uint32_t srow,
                                         uint32_t zrow, uint32_t r0, uint32_t r8, uint32_t c) {
#pragma unroll
        for (int j = 0; j < kTilesPerChunk; ++j) w[j] = ldg_stream(wp + j * kTileBytes);
        const uint32_t cs = c * (uint32_t)SBYTES;
        ld_raw<SBYTES>(sb + (r0 * srow + cs), s0);
        ld_raw<SBYTES>(sb + (r8 * srow + cs), s8);
        if (zb != nullptr) {
            const uint32_t zbit = c * (uint32_t)ZBITS;
            const uint32_t zo = zbit >> 3;
            ld_raw<ZBYTES>(zb + (r0 * zrow + zo), z0);
            ld_raw<ZBYTES>(zb + (r8 * zrow + zo), z8);
            zshift = ZBITS < 8 ? (zbit & 7u) : 0u;
        } else {
#pragma unroll
            for (int i = 0; i < ZW; ++i) z0[i] = z8[i] = kZDefault;
            zshift = 0;
        }
    }

    // Raw code fields to one field per byte (done once per item, so that a
    // block's subtraction constant is a single byte permute).
    __device__ __forceinline__ static void spread(const uint32_t (&raw)[ZW], uint32_t shift, uint32_t (&z)[ZSW]) {
        uint32_t r[ZW];
#pragma unroll
        for (int i = 0; i < ZW; ++i) r[i] = raw[i];
        if constexpr (ZBITS < 8) r[0] >>= shift;
#pragma unroll
        for (int i = 0; i < ZW; ++i) {
            if constexpr (BITS == 8) {
                z[i] = r[i];
            } else if constexpr (BITS == 4) {
                z[2 * i] = r[i] & 0x0F0F0F0Fu;
                z[2 * i + 1] = (r[i] >> 4) & 0x0F0F0F0Fu;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) z[4 * i + j] = (r[i] >> (2 * j)) & 0x03030303u;
            }
        }
    }

    __device__ __forceinline__ static float scale(const uint32_t (&s)[SW], int b) {
        if constexpr (SDT == kF32) return __uint_as_float(s[b]);
        const uint32_t word = s[b >> 1];
        if constexpr (SDT == kBF16) {
            return __uint_as_float((b & 1) ? (word & 0xFFFF0000u) : (word << 16));
        } else {
            return __half2float(__ushort_as_half((unsigned short)((b & 1) ? (word >> 16) : (word & 0xFFFFu))));
        }
    }
    // Subtraction constant of block b (Unpack::zconst of its zero point):
    // (magic + z) in both 16-bit lanes, or the f32 2^23 + z.
    __device__ __forceinline__ static uint32_t zconst(const uint32_t (&z)[ZSW], int b) {
        const int word = (b % NZS) + NZS * (b / (4 * NZS));
        const uint32_t byte = (uint32_t)((b / NZS) % 4);
        const uint32_t sel = kF32Magic ? (0x7440u | byte) : (0x4040u | (byte << 8) | byte);
        return prmt(z[word], kZHigh, sel);
    }

    // Adds this item's products to y (rows g, g+8 x tokens 2t, 2t+1); xa is the
    // shared-memory address of the lane's B fragments of the chunk's first
    // k-step pair.  M1: one activation row, so only token 0's sums are kept.
    template <bool M1>
    __device__ __forceinline__ void compute(uint32_t xa, float (&y)[4]) const {
        using U = Unpack<BITS, BF16X>;
        const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
        float acc[4];
        uint32_t zg = 0, zg8 = 0;
        float sg = 0.f, sg8 = 0.f;
        uint4 xv = make_uint4(0, 0, 0, 0);
        uint32_t zs0[ZSW], zs8[ZSW];
        spread(z0, zshift, zs0);
        spread(z8, zshift, zs8);
#pragma unroll
        for (int s = 0; s < CH; ++s) {
            if (s % SPB == 0) {
                const int b = s / SPB;
                sg = scale(s0, b);
                sg8 = scale(s8, b);
                zg = zconst(zs0, b);
                zg8 = zconst(zs8, b);
            }
            if ((s & 1) == 0) {
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                             : "r"(xa + (uint32_t)(s >> 1) * 64u));
            }
            uint32_t a[4];
            U::kstep(w[s / SPT], s % SPT, zg, zg8, a);
            const uint32_t b0 = (s & 1) ? xv.z : xv.x, b1 = (s & 1) ? xv.w : xv.y;
            if (s % SPB == 0) mma16816<BF16X>(acc, a, b0, b1, zero4);
            else mma16816<BF16X>(acc, a, b0, b1, acc);
            if (s % SPB == SPB - 1) {
                y[0] = fmaf(sg, acc[0], y[0]);
                y[2] = fmaf(sg8, acc[2], y[2]);
                if constexpr (!M1) {
                    y[1] = fmaf(sg, acc[1], y[1]);
                    y[3] = fmaf(sg8, acc[3], y[3]);
                }
            }
        }
    }
};

// Position of a warp in its CTA's item list.
// Grouped (mixture-of-experts) calls with at most 8 (token, slot) pairs: the
// experts present in ids, in ascending order, are laid end to end as one
// matrix of n_active x NT row tiles, and the CTAs split that range as they
// split a plain matrix.  Row tile R belongs to active expert R / NT; its MMA
// columns are that expert's pairs (ascending token-then-slot order), the
// other columns read a zero X row.  This is ggml's MUL_MAT_ID grouping as the
// SpacemiT backend computes it (toy 0.8.0, data/vendor/ggml/src/ggml-cpu/
// spacemit/ime.cpp, forward_mul_mat_id).
constexpr int kMoeMaxPairs = 8;
struct MoeKs {
    const int32_t* ids;        // [T, S] expert of each (token, slot); nullptr: a plain call
    int pairs, S, E, x_per_slot;
    size_t expert_bytes;       // packed bytes per expert (header included)
    size_t expert_scale_bytes, expert_zp_bytes;
};

// Position of a warp in its CTA's item list: item i = (local row tile rt,
// chunk c); a step of kW items moves q16 row tiles and r16 chunks.
struct Cursor {
    int i, rt, c;
    __device__ __forceinline__ void advance(int KC, int q16, int r16) {
        i += kW;
        c += r16;
        rt += q16;
        if (c >= KC) {
            c -= KC;
            ++rt;
        }
    }
};

// A8: accuracy level 4 (bf16 MMAs, M = 2 x the activation rows, pairx): X is read
// raw (p.act_dtype bf16, f16 or f32) and quantised while it is staged, per (row,
// block) as quantize_activation_signed of onnx-runtime-ep-cpu 0.1.0-dev.5,
// src/kernels/matmul_nbits.rs does it (s_a = amax / 127, code = round(x / s_a)
// half away from zero, clamped to +-127), each x' = code * s_a in f32 staged as
// its hi = RN_bf16(x') and lo = RN_bf16(x' - hi) in rows 2a and 2a + 1: the same
// operations on the same values as quant_act_hilo_kernel, so the same bits.
// Needs 32 <= bs <= 256 (a block's bs / 8 staging lanes reduce its max).
// KP: act-order pack (p.kperm set): X gathered through the stored permutation while it is staged.
template <int BITS, bool BF16X, int SPB_LOG, int SDT, bool M1, bool MOE, bool A8 = false, bool KP = false>
__global__ void __launch_bounds__(kThreads, 1) gemv_ks_kernel(MatmulParams p, KGeom geo, int pdl, MoeKs moe) {
    static_assert(!A8 || (BF16X && !M1 && !MOE), "accuracy level 4 staging: bf16 hi / lo rows");
    static_assert(!KP || (!MOE && !A8), "act-order pack: plain calls");
    using It = Item<BITS, BF16X, SPB_LOG, SDT>;
    constexpr int CH = It::CH;
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint4* xs = reinterpret_cast<uint4*>(smem);                  // [M + 1][xrow]: row M is zeros
    float* red = reinterpret_cast<float*>(smem + geo.x_bytes);   // [max_rt][kW][M][16 rows]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = M1 ? 1 : (int)p.M;  // grouped: the pairs (every X row staged, one per pair)
    const int KC = geo.KC;
    uint32_t NT32 = (uint32_t)L.NT;
    // grouped call: the active experts (ascending), each one's X row and Y row per MMA column
    __shared__ int moe_ak[MOE ? kMoeMaxPairs : 1];                      // expert id of active index k
    __shared__ int moe_col[MOE ? kMoeMaxPairs * 8 : 1];                 // [k][column g]: X row (M: zero row)
    __shared__ int moe_yrow[MOE ? kMoeMaxPairs * kMoeMaxPairs : 1];     // [k][column m]: Y row, -1: none
    int n_active = 1;
    float inv_nt = 0.f;
    if constexpr (MOE) {
        int id[kMoeMaxPairs];
#pragma unroll
        for (int q = 0; q < kMoeMaxPairs; ++q) id[q] = q < moe.pairs ? __ldg(moe.ids + q) : -1;
        bool first[kMoeMaxPairs];
        int rank[kMoeMaxPairs];
        bool bad = false;
        n_active = 0;
#pragma unroll
        for (int q = 0; q < kMoeMaxPairs; ++q) {
            const bool valid = q < moe.pairs && id[q] >= 0 && id[q] < moe.E;
            bad = bad || (q < moe.pairs && !valid);
            first[q] = valid;
#pragma unroll
            for (int q2 = 0; q2 < q; ++q2)
                if (id[q2] == id[q]) first[q] = false;
            n_active += first[q] ? 1 : 0;
        }
#pragma unroll
        for (int q = 0; q < kMoeMaxPairs; ++q) {
            rank[q] = 0;  // distinct valid ids below id[q]
#pragma unroll
            for (int q2 = 0; q2 < kMoeMaxPairs; ++q2)
                if (first[q2] && id[q2] < id[q]) ++rank[q];
        }
        if (bad && blockIdx.x == 0 && tid == 0) set_status(p.status, 1 /* MNB_ERR_INVALID_ARG */);
        if (tid < kMoeMaxPairs * 8) {  // entry (k, c) of the tables, c a column
            const int k = tid >> 3, c = tid & 7;
            int e = -1;
#pragma unroll
            for (int q = 0; q < kMoeMaxPairs; ++q)
                if (first[q] && rank[q] == k) e = id[q];
            int pos = 0, xr = M, yr = -1;  // the c-th pair of expert e
#pragma unroll
            for (int q = 0; q < kMoeMaxPairs; ++q) {
                if (e >= 0 && q < moe.pairs && id[q] == e) {
                    if (pos == c) xr = yr = q;
                    ++pos;
                }
            }
            if (c == 0) moe_ak[k] = e;
            moe_col[k * 8 + c] = xr;
            moe_yrow[k * kMoeMaxPairs + c] = yr;
        }
        inv_nt = 1.f / (float)NT32;
        NT32 *= (uint32_t)n_active;  // the experts' row tiles end to end
        __syncthreads();             // the tables, before the first item's loads read them
    }
    const int64_t rt0 = (int64_t)(blockIdx.x * NT32 / (uint32_t)geo.G);
    const int nrt = (int)((blockIdx.x + 1) * NT32 / (uint32_t)geo.G - (uint32_t)rt0);
    const int n_items = nrt * KC;
    // the packed tiles of (row tile, chunk) follow each other in item order
    const uint8_t* wbase = p.packed + rt0 * L.KTILES * kTileBytes + lane * 16;
    const uint32_t srow = (uint32_t)L.KB * (SDT == kF32 ? 4u : 2u), zrow = (uint32_t)L.zp_row;
    const uint8_t* sb = static_cast<const uint8_t*>(p.scales) + (size_t)rt0 * 16 * srow;
    const uint8_t* zb = p.zp != nullptr ? p.zp + (size_t)rt0 * 16 * zrow : nullptr;
    const uint32_t nlast = (uint32_t)(L.N - 1 - rt0 * 16);  // last row, local
    const int q16 = geo.q16, r16 = geo.r16;
    // grouped: active expert k of a CTA-local row tile, and its row tile within the expert
    auto expert_of = [&](int rt_l, int* rt_e) -> int {
        const int R = (int)rt0 + rt_l;
        const int k = __float2int_rz(((float)R + 0.5f) * inv_nt);  // R < 2^24: exact
        *rt_e = R - k * (int)L.NT;
        return k;
    };
    // grouped: warp w takes whole row tiles w, w + kW, ... below qW (every chunk in order), so a
    // row's sum stays in one warp's registers and is stored when the row tile ends; the last
    // nrt - qW (< kW) row tiles are split by chunks over all warps (item j = (row tile - qW) * KC +
    // chunk, warp w takes j = w, w + kW, ...), their partials summed at the end, so every warp gets
    // the same number of items to within one (geo.red_bytes == 0: whole row tiles only)
    const int qW = MOE && geo.red_bytes > 0 ? (nrt / kW) * kW : nrt;
    const int pb_rt = qW + warp / KC, pb_c = warp % KC;  // this warp's first split item
    auto valid = [&](const Cursor& it) { return MOE ? it.rt < nrt : it.i < n_items; };
    auto advance = [&](Cursor& it) {
        if constexpr (MOE) {
            if (it.rt < qW) {
                if (++it.c == KC) {
                    it.c = 0;
                    it.rt += kW;
                }
                if (it.rt >= qW) it = Cursor{warp, pb_rt, pb_c};
            } else {
                it.advance(KC, q16, r16);
            }
        } else {
            it.advance(KC, q16, r16);
        }
    };
    // grouped: a warp's items are the chunks of one row tile in a row, so the row tile's expert,
    // bases and rows are worked out once per row tile (for the loads and for the X fragments)
    int lc_rt = -1, cc_rt = -1;
    const uint8_t *lc_w = nullptr, *lc_s = nullptr, *lc_z = nullptr;
    uint32_t lc_r0 = 0, lc_r8 = 0, cc_xa = 0;
    auto load = [&](It& b, const Cursor& it) {
        if (valid(it)) {
            if constexpr (MOE) {
                if (it.rt != lc_rt) {
                    lc_rt = it.rt;
                    int rt_e;
                    const int e = moe_ak[expert_of(it.rt, &rt_e)];
                    const uint32_t nl = (uint32_t)rt_e * 16u + (uint32_t)g, nmax = (uint32_t)L.N - 1u;
                    lc_r0 = min(nl, nmax);
                    lc_r8 = min(nl + 8u, nmax);
                    lc_w = p.packed + (size_t)e * moe.expert_bytes + (size_t)rt_e * (size_t)KC * kItemBytes + lane * 16;
                    lc_s = static_cast<const uint8_t*>(p.scales) + (size_t)e * moe.expert_scale_bytes;
                    lc_z = p.zp != nullptr ? p.zp + (size_t)e * moe.expert_zp_bytes : nullptr;
                }
                b.load(lc_w + (uint32_t)it.c * (uint32_t)kItemBytes, lc_s, lc_z, srow, zrow, lc_r0, lc_r8,
                       (uint32_t)it.c);
            } else {
                const uint32_t nl = (uint32_t)it.rt * 16u + (uint32_t)g;
                const uint32_t r0 = min(nl, nlast), r8 = min(nl + 8u, nlast);
                b.load(wbase + (uint32_t)it.i * (uint32_t)kItemBytes, sb, zb, srow, zrow, r0, r8, (uint32_t)it.c);
            }
        }
    };

    // ---- 1. this warp's first item (constant data: before the dependency
    //         wait), X staged in B-fragment order, then the second item: X
    //         queues behind one item of weights, not two ----
    // items in flight per warp: 3 for 8-bit codes in blocks of 32 or more (plain calls: registers
    // allow a third buffer, and the loop is bound by the bytes in flight, not by issue), else 2
    constexpr int DEPTH = (BITS == 8 && SPB_LOG >= 1 && !MOE && !A8) ? 3 : 2;
    It buf[DEPTH];
    Cursor cur = !MOE ? Cursor{warp, 0, warp} : warp < qW ? Cursor{0, warp, 0} : Cursor{warp, pb_rt, pb_c};
    while (cur.c >= KC) {  // at most kW - 1 times
        cur.c -= KC;
        ++cur.rt;
    }
    Cursor nxt = cur;
    advance(nxt);
    Cursor nxt2 = nxt;  // DEPTH 3: the item after nxt
    if constexpr (DEPTH == 3) advance(nxt2);
    load(buf[0], cur);
    const int pairs = (int)(L.K / 32);
    // one K-chunk per warp (KC == kW) and one staging pass (K / 8 == kThreads): warp w stages
    // exactly the X entries of its own chunk (entry r = thread r) and flushes every (row tile,
    // warp) slot of the partials, so it needs neither a CTA barrier before its items nor zeroed
    // partials
    const bool wlocal = !MOE && KC == kW && pairs * 4 == kThreads;
    if constexpr (!MOE) {
        if (!wlocal)
            for (int o = tid; o < nrt * kW * 16 * M; o += kThreads) red[o] = 0.f;
    } else {
        for (int o = tid; o < (nrt - qW) * kW * 16 * M; o += kThreads) red[o] = 0.f;
    }
    for (int o = tid; o < pairs * 4; o += kThreads) xs[(size_t)M * geo.xrow + o] = make_uint4(0, 0, 0, 0);
    // act-order pack: the stored depths of this thread's first staging entry come from these original
    // depths (constant data, read before the dependency wait)
    int kk0[KP ? 8 : 1] = {0};
    if (KP && tid < pairs * 4) {
        const int j0 = 32 * (tid >> 2) + 2 * (tid & 3);
#pragma unroll
        for (int e = 0; e < (KP ? 8 : 1); ++e) kk0[e] = __ldg(p.kperm + j0 + 8 * (e >> 1) + (e & 1));
    }
    if (pdl) {
        griddep_wait();               // X (and Y) may belong to the previous kernel on the stream
        griddep_launch_dependents();  // after the wait: at most two chained kernels overlap
    }
    if constexpr (A8) {
        // entry (row, pair P, lane class tt) holds depths 32P + 2tt + {0, 1}, + 8, + 16, + 24 (pairs);
        // a block's entries are bs / 8 consecutive lanes, whose max |x| is reduced with shuffles
        const int MA = M >> 1;  // activation rows
        const int G = (int)(L.bs >> 3);
        for (int r0 = 0; r0 < pairs * 4; r0 += kThreads) {
            const int r = r0 + tid;
            const bool live = r < pairs * 4;
            const int P = r >> 2, tt = r & 3;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (a < MA) {
                    float v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = 0.f;
                    const int64_t k0 = (int64_t)a * L.K + 32 * P + 2 * tt;
                    if (live) {
                        if (p.act_dtype == kF32) {
                            const float* xf = static_cast<const float*>(p.x) + k0;  // 8-byte aligned pairs
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float2 f = __ldg(reinterpret_cast<const float2*>(xf + 8 * j));
                                v[2 * j] = f.x;
                                v[2 * j + 1] = f.y;
                            }
                        } else {
                            const uint32_t* xw = static_cast<const uint32_t*>(p.x) + (k0 >> 1);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t wv = __ldg(xw + 4 * j);
                                if (p.act_dtype == kBF16) {
                                    v[2 * j] = __uint_as_float(wv << 16);
                                    v[2 * j + 1] = __uint_as_float(wv & 0xFFFF0000u);
                                } else {
                                    v[2 * j] = __half2float(__ushort_as_half((unsigned short)(wv & 0xFFFFu)));
                                    v[2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(wv >> 16)));
                                }
                            }
                        }
                    }
                    float amax = 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
                    for (int o = G >> 1; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                    const float sa = __fdiv_rn(amax, 127.0f);
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t h2[2], l2[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            int code = 0;
                            if (amax > 0.f) {
                                const float q = roundf(__fdiv_rn(v[2 * j + e], sa));  // half away from zero
                                code = (int)fminf(fmaxf(q, -127.f), 127.f);
                            }
                            const float xq = __fmul_rn((float)code, sa);
                            const __nv_bfloat16 hi = __float2bfloat16_rn(xq);
                            const __nv_bfloat16 lo = __float2bfloat16_rn(xq - __bfloat162float(hi));  // exact difference
                            h2[e] = __bfloat16_as_ushort(hi);
                            l2[e] = __bfloat16_as_ushort(lo);
                        }
                        hw[j] = h2[0] | (h2[1] << 16);
                        lw[j] = l2[0] | (l2[1] << 16);
                    }
                    if (live) {
                        xs[(size_t)(2 * a) * geo.xrow + r] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        xs[(size_t)(2 * a + 1) * geo.xrow + r] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                }
            }
        }
    } else {
        // item (m, pair P, lane class tt), k0 = 32 P:
        // (x[k0 + 2tt..], x[k0 + 8 + 2tt..], x[k0 + 16 + 2tt..], x[k0 + 24 + 2tt..])
        const uint32_t* x32 = static_cast<const uint32_t*>(p.x);  // K even: rows are 4-byte aligned
        const int64_t kw = L.K / 2;
        // act-order pack: X is copied as it is (coalesced, 16 bytes a thread) into shared memory after the
        // partials, and gathered from there through the permutation
        const uint16_t* xraw = reinterpret_cast<const uint16_t*>(smem + geo.x_bytes + geo.red_bytes);
        if constexpr (KP) {
            const uint4* xg = static_cast<const uint4*>(p.x);  // 16-byte aligned rows (K % 8 == 0)
            uint4* xw = reinterpret_cast<uint4*>(smem + geo.x_bytes + geo.red_bytes);
            for (int o = tid; o < M * (int)(L.K / 8); o += kThreads) xw[o] = __ldg(xg + o);
            __syncthreads();
        }
        // every row's words of a thread are requested before any is stored, so
        // the M rows cost one round trip, not M
        for (int r0 = 0; r0 < pairs * 4; r0 += kThreads) {
            const int r = r0 + tid;
            const int P = r >> 2, tt = r & 3;
            if constexpr (KP) {
                // act-order pack: stored depth 32P + 2tt + {0, 1, 8, 9, 16, 17, 24, 25} is X's depth kk[e]
                if (r < pairs * 4) {
                    int kk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int v = r0 == 0 ? kk0[KP ? e : 0] : __ldg(p.kperm + 32 * P + 2 * tt + 8 * (e >> 1) + (e & 1));
                        kk[e] = min(max(v, 0), (int)L.K - 1);  // a bad pack's permutation never indexes past X
                    }
                    for (int m0 = 0; m0 < M; m0 += 2) {
                        uint32_t hv[2][8];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                hv[h][e] = m0 + h < M ? (uint32_t)xraw[(int64_t)(m0 + h) * L.K + kk[e]] : 0u;
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (m0 + h < M)
                                xs[(size_t)(m0 + h) * geo.xrow + r] =
                                    make_uint4(hv[h][0] | (hv[h][1] << 16), hv[h][2] | (hv[h][3] << 16),
                                               hv[h][4] | (hv[h][5] << 16), hv[h][6] | (hv[h][7] << 16));
                    }
                }
            } else {
                uint4 v[M1 ? 1 : 8];
#pragma unroll
                for (int m = 0; m < (M1 ? 1 : 8); ++m) {
                    if (m < M && r < pairs * 4) {
                        // grouped call: row m is pair m = t * S + s: row t of X (or row t * S + s)
                        const int xr = MOE ? (moe.x_per_slot ? m : m / moe.S) : m;
                        const uint32_t* src = x32 + (int64_t)xr * kw + P * 16 + tt;
                        v[m] = make_uint4(__ldg(src), __ldg(src + 4), __ldg(src + 8), __ldg(src + 12));
                    }
                }
#pragma unroll
                for (int m = 0; m < (M1 ? 1 : 8); ++m)
                    if (m < M && r < pairs * 4) xs[(size_t)m * geo.xrow + r] = v[m];
            }
        }
    }
    load(buf[1], nxt);
    if constexpr (DEPTH == 3) load(buf[2], nxt2);
    if (wlocal) __syncwarp();
    else __syncthreads();

    // ---- 2. items, two buffers: compute one while the next is in flight ----
    const uint32_t xa_lane = smem_u32(xs + (size_t)(g < M ? g : M) * geo.xrow + t);
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    const float bias_none = 0.f;
    auto flush = [&](int rt_l) {
        if (MOE && rt_l >= qW) {  // a split row tile: this warp's partial, summed at the end
            float* r = red + (size_t)((rt_l - qW) * kW + warp) * 16 * M;
            const int m0 = 2 * t, m1 = 2 * t + 1;
            if (m0 < M) {
                r[m0 * 16 + g] = y[0];
                r[m0 * 16 + g + 8] = y[2];
            }
            if (m1 < M) {
                r[m1 * 16 + g] = y[1];
                r[m1 * 16 + g + 8] = y[3];
            }
            y[0] = y[1] = y[2] = y[3] = 0.f;
            return;
        }
        if constexpr (MOE) {  // the row tile's sums are complete: store them (bias added here)
            int rt_e;
            const int k = expert_of(rt_l, &rt_e);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int m = 2 * t + (j & 1);
                const int64_t n = (int64_t)rt_e * 16 + g + ((j >> 1) << 3);
                const int yr = m < M ? moe_yrow[k * kMoeMaxPairs + m] : -1;
                if (yr >= 0 && n < L.N) {
                    const float b = p.bias ? load_f32(p.bias, n, p.bias_dtype) : bias_none;
                    store_f32(p.y, (int64_t)yr * L.N + n, y[j] + b, p.out_dtype);
                }
            }
            y[0] = y[1] = y[2] = y[3] = 0.f;
            return;
        }
        if (!M1 && geo.pairx) {  // columns 2t, 2t + 1 are the hi and lo parts of token t
            float* r = red + (size_t)(rt_l * kW + warp) * 16 * (M >> 1);
            if (2 * t < M) {
                r[t * 16 + g] = y[0] + y[1];
                r[t * 16 + g + 8] = y[2] + y[3];
            }
            y[0] = y[1] = y[2] = y[3] = 0.f;
            return;
        }
        float* r = red + (size_t)(rt_l * kW + warp) * 16 * M;
        const int m0 = 2 * t, m1 = 2 * t + 1;
        if (m0 < M) {
            r[m0 * 16 + g] = y[0];
            r[m0 * 16 + g + 8] = y[2];
        }
        if (!M1 && m1 < M) {
            r[m1 * 16 + g] = y[1];
            r[m1 * 16 + g + 8] = y[3];
        }
        y[0] = y[1] = y[2] = y[3] = 0.f;
    };
    // step: compute `cur` from b, refill b with the item DEPTH after it, move on
    auto step = [&](It& b) {
        uint32_t xa = xa_lane;
        if constexpr (MOE) {  // this item's expert: its columns' X rows
            if (cur.rt != cc_rt) {
                cc_rt = cur.rt;
                int rt_e;
                const int k = expert_of(cur.rt, &rt_e);
                cc_xa = smem_u32(xs + (size_t)moe_col[k * 8 + g] * geo.xrow + t);
            }
            xa = cc_xa;
        }
        b.template compute<M1>(xa + (uint32_t)cur.c * (uint32_t)(CH / 2) * 64u, y);
        Cursor after = DEPTH == 3 ? nxt2 : nxt;
        advance(after);
        load(b, after);
        if (!valid(nxt) || nxt.rt != cur.rt) flush(cur.rt);
        cur = nxt;
        if constexpr (DEPTH == 3) {
            nxt = nxt2;
            nxt2 = after;
        } else {
            nxt = after;
        }
        return valid(cur);
    };
    if (valid(cur)) {
        if constexpr (DEPTH == 3) {
            while (step(buf[0]) && step(buf[1]) && step(buf[2])) {
            }
        } else {
            while (step(buf[0]) && step(buf[1])) {
            }
        }
    }
    if constexpr (MOE) {  // whole row tiles already stored; the split ones: their 16 warps' partials
        if (nrt > qW) {
            __syncthreads();
            const float inv_mp = 1.f / (float)M;
            for (int o = tid; o < (nrt - qW) * 16 * M; o += kThreads) {
                const int row = o & 15, q = o >> 4;
                const int rr = __float2int_rz(((float)q + 0.5f) * inv_mp);  // q < 2^16: exact
                const int m = q - rr * M;
                const float* src = red + (size_t)rr * kW * 16 * M + m * 16 + row;
                float t8[kW / 2];
#pragma unroll
                for (int w2 = 0; w2 < kW / 2; ++w2)
                    t8[w2] = src[(size_t)(2 * w2) * 16 * M] + src[(size_t)(2 * w2 + 1) * 16 * M];
#pragma unroll
                for (int h = kW / 4; h >= 1; h >>= 1) {
#pragma unroll
                    for (int w2 = 0; w2 < h; ++w2) t8[w2] = t8[2 * w2] + t8[2 * w2 + 1];
                }
                int rt_e;
                const int k = expert_of(qW + rr, &rt_e);
                const int yr = moe_yrow[k * kMoeMaxPairs + m];
                const int64_t n = (int64_t)rt_e * 16 + row;
                if (yr >= 0 && n < L.N) {
                    const float b = p.bias ? load_f32(p.bias, n, p.bias_dtype) : 0.f;
                    store_f32(p.y, (int64_t)yr * L.N + n, t8[0] + b, p.out_dtype);
                }
            }
        }
        if (blockIdx.x == 0 && tid == 0)
            for (int k = 0; k < n_active; ++k)
                verify_header(static_cast<const uint8_t*>(p.packed_hdr) + (size_t)moe_ak[k] * moe.expert_bytes, L, p.status);
        return;
    }
    __syncthreads();

    // ---- 4. rows: the 16 warps' partials in a fixed order ----
    // consecutive threads take consecutive rows of one token (coalesced stores,
    // conflict-free reads); q = rt_l * M + m is split with a float reciprocal
    // (q < 2^16: exact after truncation of (q + 0.5) / M)
    const int MO = (!M1 && geo.pairx) ? M >> 1 : M;  // output columns
    const float inv_m = M1 ? 1.f : 1.f / (float)MO;
    for (int o = tid; o < nrt * 16 * MO; o += kThreads) {
        const int row = o & 15, q = o >> 4;
        const int rt_l = M1 ? q : __float2int_rz(((float)q + 0.5f) * inv_m);
        const int m = M1 ? 0 : q - rt_l * MO;
        const float* src = red + (size_t)rt_l * kW * 16 * MO + m * 16 + row;
        // the 16 warps' partials as a fixed pairwise tree (independent loads, depth 4)
        float t8[kW / 2];
#pragma unroll
        for (int w2 = 0; w2 < kW / 2; ++w2) t8[w2] = src[(size_t)(2 * w2) * 16 * MO] + src[(size_t)(2 * w2 + 1) * 16 * MO];
#pragma unroll
        for (int h = kW / 4; h >= 1; h >>= 1) {
#pragma unroll
            for (int w2 = 0; w2 < h; ++w2) t8[w2] = t8[2 * w2] + t8[2 * w2 + 1];
        }
        float v = t8[0];
        const int64_t n = (rt0 + rt_l) * 16 + row;
        if (n < L.N) {
            if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
            store_f32(p.y, (int64_t)m * L.N + n, v, p.out_dtype);
        }
    }
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status, kWfInt, KP ? 1 : 0);
}

template <int BITS, bool BF16X, int SPB_LOG, int SDT>
cudaError_t launch_k(const MatmulParams& p, const KGeom& geo, cudaStream_t s, const MoeKs* moe, bool a8) {
    const int pdl = (p.flags & kFlagPDL) ? 1 : 0;
    auto kern = moe ? gemv_ks_kernel<BITS, BF16X, SPB_LOG, SDT, false, true>
                : p.M == 1 ? gemv_ks_kernel<BITS, BF16X, SPB_LOG, SDT, true, false>
                           : gemv_ks_kernel<BITS, BF16X, SPB_LOG, SDT, false, false>;
    if constexpr (BF16X && SPB_LOG >= 1) {
        if (a8) kern = gemv_ks_kernel<BITS, true, SPB_LOG, SDT, false, false, true>;
    } else {
        if (a8) return cudaErrorNotSupported;
    }
    KGeom gk = geo;
    if (p.kperm != nullptr) {
        if (moe || a8) return cudaErrorNotSupported;
        kern = p.M == 1 ? gemv_ks_kernel<BITS, BF16X, SPB_LOG, SDT, true, false, false, true>
                        : gemv_ks_kernel<BITS, BF16X, SPB_LOG, SDT, false, false, false, true>;
        gk.total_bytes = geo.x_bytes + geo.red_bytes + kperm_x_bytes(p.L, p.M);  // X as given, for the gather
    }
    const MoeKs none{};
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gk.total_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)gk.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = gk.total_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p, gk, pdl, moe ? *moe : none);
}

template <int BITS, bool BF16X, int SPB_LOG>
cudaError_t launch_sdt(const MatmulParams& p, const KGeom& geo, cudaStream_t s, const MoeKs* moe, bool a8) {
    constexpr int BPC = chunk_steps(BITS) >> SPB_LOG;
    switch (p.scale_dtype) {
        case kF32:
            if constexpr (BPC * 4 <= 32) return launch_k<BITS, BF16X, SPB_LOG, kF32>(p, geo, s, moe, a8);
            break;
        case kF16: return launch_k<BITS, BF16X, SPB_LOG, kF16>(p, geo, s, moe, a8);
        case kBF16: return launch_k<BITS, BF16X, SPB_LOG, kBF16>(p, geo, s, moe, a8);
        default: break;
    }
    return cudaErrorNotSupported;
}

template <int BITS, bool BF16X>
cudaError_t launch_bs(const MatmulParams& p, const KGeom& geo, cudaStream_t s, const MoeKs* moe, bool a8) {
    constexpr int CH = chunk_steps(BITS);
    switch (p.L.bs) {
        case 16:
            if constexpr (CH <= 16) return launch_sdt<BITS, BF16X, 0>(p, geo, s, moe, a8);
            break;
        case 32: return launch_sdt<BITS, BF16X, 1>(p, geo, s, moe, a8);
        case 64: return launch_sdt<BITS, BF16X, 2>(p, geo, s, moe, a8);
        case 128: return launch_sdt<BITS, BF16X, 3>(p, geo, s, moe, a8);
        case 256:
            if constexpr (CH >= 16) return launch_sdt<BITS, BF16X, 4>(p, geo, s, moe, a8);
            break;
        default: break;
    }
    return cudaErrorNotSupported;
}

// a8: accuracy level 4 with X quantised in the staging (bf16 MMAs whatever X's type; p.M counts the
// hi / lo rows, twice the activation rows); cudaErrorNotSupported where that mode is not built.
template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const KGeom& geo, cudaStream_t s, const MoeKs* moe = nullptr,
                        bool a8 = false) {
    if (a8) return launch_bs<BITS, true>(p, geo, s, nullptr, true);
    return p.act_dtype == kBF16 ? launch_bs<BITS, true>(p, geo, s, moe, false)
                                : launch_bs<BITS, false>(p, geo, s, moe, false);
}

}  // namespace gks
}  // namespace mnb
