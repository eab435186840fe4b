// Decode GEMV, M == 1:  y[n] = sum_k x[k] * (q[n,k] - zp[n,kb]) * scale[n,kb]  (+ bias[n]).
//
// What it computes is the MatMulNBits product of onnx-runtime-ep-cpu
// 0.1.0-dev.5, src/kernels/matmul_nbits.rs (fn dequantize_nbits_value for w,
// the m == 1 branch of MatMulNBitsKernel::execute for the GEMV); the pages'
// own decode kernels are CPU SIMD loops (int4_dot_row_*), so nothing of their
// structure is reused here.
//
// GB300 design (HBM-bound: ~0.56 byte per weight at 4 bits):
//  * Persistent: one CTA per SM, row-tiles (16 rows, all of K) dealt round-robin.
//  * Each of the CTA's warps owns a contiguous K-slice of every row-tile and
//    streams its slice of the packed weights with 1-D bulk copies
//    (cp.async.bulk, TMA engine) into its own ring of shared-memory slots,
//    completion tracked by one mbarrier per slot.  The ring keeps
//    SLOTS * CHUNK bytes per warp in flight independent of registers, which
//    is what lets a few warps per SM saturate HBM3e.
//  * Unpack is exact and cheap: a 4-bit code OR'ed into the mantissa of
//    2^23 (0x4B000000) gives the float 2^23 + q * 2^p exactly (p = 0, or 16
//    for the odd depth of a pair); subtracting 2^23 + zp * 2^p (one packed
//    f32x2 add) gives (q - zp) * 2^p exactly; the activation of the odd depth
//    is pre-scaled by 2^-16 (exact), so one packed f32x2 FMA accumulates
//    x * (q - zp) for two depths.  8-bit codes use PRMT to place the byte.
//  * Per (row, K-block) the scale multiplies the block's partial sum
//    (one f32x2 FMA); scales and the subtraction constants of the next
//    row-tile are loaded during the current one and staged in shared memory.
//  * Partial sums of the warps are reduced in a fixed order through shared
//    memory, so results are bit-identical run to run.
#include <cstdio>
#include <cstdlib>

#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSlots = 12;   // ring slots per warp (as many as shared memory allows, >= kMinSlots)
constexpr int kMinSlots = 4;
constexpr int kChunkTiles = 4;  // 512-byte tiles per bulk copy
constexpr int kChunkBytes = kChunkTiles * kTileBytes;
constexpr int kRawSlots = 4;    // row-tiles of raw scales / zero points in flight
constexpr uint32_t kMagic23 = 0x4B000000u;  // 2^23


struct GemvGeom {
    int64_t kblocks_pad;  // staged blocks per row (covers KTILES * KT depths)
    int64_t ktw;          // k-tiles per warp slice
    int slots;            // ring slots per warp
    int stage_bufs;       // 2: convert the next row-tile while others finish; 1: extra barrier
    int raw_scale_bytes;  // scales of one row-tile (16 rows)
    int raw_zp_bytes;     // zero points of one row-tile (0 when absent)
    size_t ring_bytes, xs_bytes, raw_bytes, stage_bytes, red_bytes, bar_bytes, total_bytes;
};

// Tuning overrides (environment, read per call): MNB_GEMV_STAGE_BUFS = 1 or 2,
// MNB_GEMV_MAX_SLOTS = 4..12.  Defaults pick the deepest ring that fits.
static int env_or(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

__host__ GemvGeom gemv_geom(const Layout& L, int scale_dtype, bool has_zp, size_t smem_limit) {
    const int force_bufs = env_or("MNB_GEMV_STAGE_BUFS", 0);
    int max_slots = env_or("MNB_GEMV_MAX_SLOTS", kMaxSlots);
    max_slots = max_slots < kMinSlots ? kMinSlots : (max_slots > kMaxSlots ? kMaxSlots : max_slots);
    GemvGeom g;
    g.kblocks_pad = (L.KTILES * L.KT + L.bs - 1) / L.bs;
    // whole chunks per warp slice, so quantisation blocks never straddle a chunk
    g.ktw = ((L.KTILES + kWarps - 1) / kWarps + kChunkTiles - 1) / kChunkTiles * kChunkTiles;
    g.raw_scale_bytes = (int)(16 * L.KB * (scale_dtype == kF32 ? 4 : 2));
    g.raw_zp_bytes = has_zp ? (int)(16 * L.zp_row) : 0;
    g.xs_bytes = (size_t)L.KTILES * L.KT * 4;
    g.raw_bytes = (size_t)kRawSlots * (round16(g.raw_scale_bytes) + round16(g.raw_zp_bytes));
    g.red_bytes = (size_t)2 * kWarps * 16 * 4;
    g.bar_bytes = (size_t)(kWarps * kMaxSlots + kRawSlots) * 8;
    // Prefer a double-buffered stage and the deepest ring that fits.
    for (int bufs = 2; bufs >= 1; --bufs) {
        if (force_bufs && bufs != force_bufs) continue;
        g.stage_bufs = bufs;
        g.stage_bytes = (size_t)bufs * 16 * (g.kblocks_pad | 1) * 16;
        const size_t fixed = g.xs_bytes + g.raw_bytes + g.stage_bytes + g.red_bytes + g.bar_bytes + 128;
        int slots = max_slots;
        while (slots > kMinSlots && fixed + (size_t)kWarps * slots * kChunkBytes > smem_limit) --slots;
        g.slots = slots;
        g.ring_bytes = (size_t)kWarps * slots * kChunkBytes;
        g.total_bytes = g.ring_bytes + fixed;
        if (g.total_bytes <= smem_limit && (bufs == 1 || slots >= 6)) break;
    }
    return g;
}

// Staged per-(row, block) entry: the pair to subtract, (2^23 + zp, 2^23 + zp*2^pb)
// as floats, and the scale twice.
struct __align__(16) StageEntry {
    uint32_t c0, c1;
    float s0, s1;
};

template <int BITS>
struct Unpack;

// 4-bit: word = one k-step; pair r at nibbles r (even depth) and r+4 (odd depth).
template <>
struct Unpack<4> {
    static constexpr int kPb = 16;
    // d[r] = ((q_even - zp) , (q_odd - zp) * 2^16) for fragment register r.
    __device__ __forceinline__ static void kstep(const uint32_t* w, int s, uint64_t cg, uint64_t cg8,
                                                 uint64_t d[4]) {
        const uint32_t word = w[s];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t sh = word >> (4 * r);
            const uint32_t va = lop3_and_or(sh, 0x0000000Fu, kMagic23);
            const uint32_t vb = lop3_and_or(sh, 0x000F0000u, kMagic23);
            d[r] = fsub2(pack2u(va, vb), (r & 1) ? cg8 : cg);
        }
    }
    static constexpr int kStepsPerTile = 4;
};

// 2-bit: word j holds k-steps 2j and 2j+1; pair i = 4*(s&1) + r at fields i and i+8.
template <>
struct Unpack<2> {
    static constexpr int kPb = 16;
    __device__ __forceinline__ static void kstep(const uint32_t* w, int s, uint64_t cg, uint64_t cg8,
                                                 uint64_t d[4]) {
        const uint32_t word = w[s >> 1];
        const int base = (s & 1) * 4;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t sh = word >> (2 * (base + r));
            const uint32_t va = lop3_and_or(sh, 0x00000003u, kMagic23);
            const uint32_t vb = lop3_and_or(sh, 0x00030000u, kMagic23);
            d[r] = fsub2(pack2u(va, vb), (r & 1) ? cg8 : cg);
        }
    }
    static constexpr int kStepsPerTile = 8;
};

// 8-bit: k-step s in words 2s (depths 2t, 2t+1) and 2s+1 (2t+8, 2t+9);
// byte 2*hi + e, hi selecting row g+8.
template <>
struct Unpack<8> {
    static constexpr int kPb = 0;
    __device__ __forceinline__ static void kstep(const uint32_t* w, int s, uint64_t cg, uint64_t cg8,
                                                 uint64_t d[4]) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t word = w[2 * s + (r >> 1)];
            const uint32_t hi = r & 1;
            const uint32_t va = prmt(word, kMagic23, 0x7650u | (2 * hi));
            const uint32_t vb = prmt(word, kMagic23, 0x7650u | (2 * hi + 1));
            d[r] = fsub2(pack2u(va, vb), hi ? cg8 : cg);
        }
    }
    static constexpr int kStepsPerTile = 2;
};

// SPB_LOG: log2 of the k-steps per quantisation block when the block
// structure inside a chunk is static (blocks of 1, 2, 4 or 8 k-steps that tile
// the chunk); -1 handles any block size with run-time checks.
template <int BITS, int SPB_LOG>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(MatmulParams p, GemvGeom geo) {
    using U = Unpack<BITS>;
    const Layout& L = p.L;
    if (blockIdx.x == 0 && threadIdx.x == 0) verify_header(p.packed_hdr, L, p.status);
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;                                               // [warps][slots][chunk]
    float* xs = reinterpret_cast<float*>(smem + geo.ring_bytes);        // permuted x'
    uint8_t* raw = smem + geo.ring_bytes + geo.xs_bytes;                // [kRawSlots][scales | zp]
    StageEntry* stage = reinterpret_cast<StageEntry*>(raw + geo.raw_bytes);
    float* red = reinterpret_cast<float*>(raw + geo.raw_bytes + geo.stage_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(raw + geo.raw_bytes + geo.stage_bytes + geo.red_bytes);
    uint64_t* rbars = bars + kWarps * kMaxSlots;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int my_tiles = (int)((L.NT - blockIdx.x + gridDim.x - 1) / gridDim.x);  // row-tiles of this CTA
    if (my_tiles <= 0) return;
    const int S_SLOTS = geo.slots;

    // ---- weight stream: this warp's K-slice of every row-tile of the CTA ----
    const int64_t kt_begin = imin64((int64_t)warp * geo.ktw, L.KTILES);
    const int64_t kt_end = imin64(kt_begin + geo.ktw, L.KTILES);
    const int nch = (int)((kt_end - kt_begin + kChunkTiles - 1) / kChunkTiles);
    const int total_chunks = nch * my_tiles;
    uint64_t* wbars = bars + warp * kMaxSlots;
    uint8_t* wring = ring + (size_t)warp * S_SLOTS * kChunkBytes;
    int iss_i = 0, iss_c = 0, iss_slot = 0, issued = 0;  // next chunk to issue (row-tile, chunk, slot)
    auto issue_next = [&]() {  // lane 0 only; caller checks issued < total_chunks
        const int64_t rt = blockIdx.x + (int64_t)iss_i * gridDim.x;
        const int64_t kt = kt_begin + (int64_t)iss_c * kChunkTiles;
        const uint32_t bytes = (uint32_t)(imin64(kChunkTiles, kt_end - kt) * kTileBytes);
        mbar_arrive_expect_tx(&wbars[iss_slot], bytes);
        bulk_g2s(wring + iss_slot * kChunkBytes, p.packed + (rt * L.KTILES + kt) * kTileBytes, bytes,
                 &wbars[iss_slot]);
    };
    auto advance_issue = [&]() {
        ++issued;
        if (++iss_c == nch) { iss_c = 0; ++iss_i; }
        if (++iss_slot == S_SLOTS) iss_slot = 0;
    };

    // ---- raw scales / zero points of whole row-tiles, bulk-copied ahead ----
    const bool raw_ok = ((reinterpret_cast<uintptr_t>(p.scales) & 15) == 0) &&
                        (p.zp == nullptr || (reinterpret_cast<uintptr_t>(p.zp) & 15) == 0);
    const int raw_slot_bytes = (int)(round16(geo.raw_scale_bytes) + round16(geo.raw_zp_bytes));
    auto tile_by_copy = [&](int i) {  // full row-tile with 16-byte aligned sources
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

    if (lane == 0) {
        for (int s = 0; s < S_SLOTS; ++s) mbar_init(&wbars[s], 1);
    }
    if (tid == 0) {
        for (int s = 0; s < kRawSlots; ++s) mbar_init(&rbars[s], 1);
    }
    fence_barrier_init();
    __syncthreads();
    // Start both streams at once: the prologue below overlaps the first copies.
    if (lane == 0) {
        while (issued < total_chunks && issued < S_SLOTS) {
            issue_next();
            advance_issue();
        }
    } else {
        const int n0 = total_chunks < S_SLOTS ? total_chunks : S_SLOTS;
        for (int q0 = 0; q0 < n0; ++q0) advance_issue();
    }
    if (tid == 0)
        for (int i = 0; i < kRawSlots; ++i) issue_raw(i);

    // x': per k-step S and lane class t, (x[16S+2t], x[16S+2t+1]*2^-pb, x[16S+2t+8], x[16S+2t+9]*2^-pb).
    // Each thread stages whole k-steps (16 activations, two or four 16-byte
    // loads), four k-steps per round with every load issued before use.
    {
        const float odd_scale = (U::kPb == 16) ? (1.0f / 65536.0f) : 1.0f;
        const int ksteps = (int)(L.KTILES * L.KT / 16);
        const int full_steps = (int)(L.K / 16);  // k-steps lying wholly inside K
        constexpr int kRound = 4;
        for (int S0 = tid; S0 < ksteps; S0 += kThreads * kRound) {
            float v[kRound][16];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const int S = S0 + u * kThreads;
                if (S < full_steps) {
                    if (p.act_dtype == kF32) {
                        const float4* src = reinterpret_cast<const float4*>(p.x) + (int64_t)S * 4;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 f = __ldg(src + j);
                            v[u][4 * j] = f.x;
                            v[u][4 * j + 1] = f.y;
                            v[u][4 * j + 2] = f.z;
                            v[u][4 * j + 3] = f.w;
                        }
                    } else {
                        const uint4* src = reinterpret_cast<const uint4*>(p.x) + (int64_t)S * 2;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint4 h = __ldg(src + j);
                            const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const uint32_t lo = hw[e] & 0xFFFFu, hi = hw[e] >> 16;
                                if (p.act_dtype == kBF16) {
                                    v[u][8 * j + 2 * e] = __uint_as_float(lo << 16);
                                    v[u][8 * j + 2 * e + 1] = __uint_as_float(hi << 16);
                                } else {
                                    v[u][8 * j + 2 * e] = __half2float(__ushort_as_half((uint16_t)lo));
                                    v[u][8 * j + 2 * e + 1] = __half2float(__ushort_as_half((uint16_t)hi));
                                }
                            }
                        }
                    }
                } else if (S < ksteps) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int64_t k = 16 * (int64_t)S + j;
                        v[u][j] = k < L.K ? load_f32(p.x, k, p.act_dtype) : 0.f;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const int S = S0 + u * kThreads;
                if (S < ksteps) {
#pragma unroll
                    for (int tt = 0; tt < 4; ++tt)
                        reinterpret_cast<float4*>(xs)[S * 4 + tt] =
                            make_float4(v[u][2 * tt], v[u][2 * tt + 1] * odd_scale, v[u][2 * tt + 8],
                                        v[u][2 * tt + 9] * odd_scale);
                }
            }
        }
    }

    // Staged entry (r, kb) of a row-tile lives at r * kbs + kb; kbs is odd so the
    // 8 row groups of a warp read different banks.
    const int kbp = (int)geo.kblocks_pad;
    const int kbs = kbp | 1;
    const int stage_entries = 16 * kbp;
    const int stage_stride = 16 * kbs;
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;
    const int zmask = code_mask(L.bits);
    auto make_entry = [&](uint32_t z, float sc) {
        StageEntry se;
        se.c0 = kMagic23 | z;
        se.c1 = kMagic23 | (z << U::kPb);
        se.s0 = se.s1 = sc;
        return se;
    };
    // Convert row-tile i's scales and zero points into staged entries of buffer
    // buf.  Thread (r = tid / 16, j = tid % 16) handles blocks j, j+16, ... of
    // row r, so the 16 threads of a row read consecutive scales.
    const int conv_r = tid >> 4, conv_j = tid & 15;
    auto convert = [&](int i, int buf) {
        StageEntry* dst = stage + buf * stage_stride + conv_r * kbs;
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
            for (int kb = conv_j; kb < kbp; kb += 16) {
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
                dst[kb] = make_entry(z, sc);
            }
        } else {
            for (int kb = conv_j; kb < kbp; kb += 16) {
                uint32_t z = 0;
                float sc = 0.f;
                if (n < L.N && kb < kbv) {
                    z = (uint32_t)load_zp(p.zp, L, n, kb);
                    sc = load_f32(p.scales, n * L.KB + kb, p.scale_dtype);
                }
                dst[kb] = make_entry(z, sc);
            }
        }
    };

    convert(0, 0);
    __syncthreads();
    if (tid == 0) issue_raw(kRawSlots);  // row-tile 0's raw slot is free again

    // Blocks are powers of two >= 16 depths, i.e. 2^spb_log k-steps.
    const int spb_log = SPB_LOG >= 0 ? SPB_LOG : __ffs(L.bs / 16) - 1;
    const int spb_mask = (1 << spb_log) - 1;
    bool bad = false;
    int q = 0, slot = 0;
    uint32_t parity = 0;  // consumption position in the weight ring
    for (int i = 0; i < my_tiles; ++i) {
        const int64_t rt = blockIdx.x + (int64_t)i * gridDim.x;
        const int buf = geo.stage_bufs == 2 ? (i & 1) : 0;
        const StageEntry* st_g = stage + buf * stage_stride + g * kbs;
        const StageEntry* st_g8 = st_g + 8 * kbs;

        uint64_t acc_g = 0, acc_g8 = 0;  // (even, odd) partial sums of the current block
        uint64_t y_g = 0, y_g8 = 0;
        int S = (int)(kt_begin * U::kStepsPerTile);  // k-step index inside the row
        uint64_t cg = 0, cg8 = 0, sg = 0, sg8 = 0;
        bool first = true;

        for (int c = 0; c < nch; ++c, ++q) {
            if (!bad) bad = !mbar_wait(&wbars[slot], parity, p.status);
            if (!bad) {
                const int64_t kt = kt_begin + (int64_t)c * kChunkTiles;
                const int ntile = (int)imin64(kChunkTiles, kt_end - kt);
                uint4 wv[kChunkTiles];
                const uint8_t* sbase = wring + slot * kChunkBytes;
#pragma unroll
                for (int tl = 0; tl < kChunkTiles; ++tl)
                    if (tl < ntile) wv[tl] = reinterpret_cast<const uint4*>(sbase + tl * kTileBytes)[lane];
#pragma unroll
                for (int tl = 0; tl < kChunkTiles; ++tl) {
                    if (tl >= ntile) break;
                    const uint32_t* w = reinterpret_cast<const uint32_t*>(&wv[tl]);
#pragma unroll
                    for (int s = 0; s < U::kStepsPerTile; ++s) {
                        const int ks = tl * U::kStepsPerTile + s;  // k-step inside the chunk
                        const bool block_start = SPB_LOG >= 0 ? ((ks & ((1 << (SPB_LOG < 0 ? 0 : SPB_LOG)) - 1)) == 0)
                                                              : (first || ((S + ks) & spb_mask) == 0);
                        if (block_start) {
                            first = false;
                            const int kb = (S + ks) >> spb_log;
                            const uint4 eg = *reinterpret_cast<const uint4*>(st_g + kb);
                            const uint4 eg8 = *reinterpret_cast<const uint4*>(st_g8 + kb);
                            cg = pack2u(eg.x, eg.y);
                            sg = pack2u(eg.z, eg.w);
                            cg8 = pack2u(eg8.x, eg8.y);
                            sg8 = pack2u(eg8.z, eg8.w);
                        }
                        const float4 xv = reinterpret_cast<const float4*>(xs)[(S + ks) * 4 + t];
                        const uint64_t p1 = pack2(xv.x, xv.y), p2 = pack2(xv.z, xv.w);
                        uint64_t d[4];
                        U::kstep(w, s, cg, cg8, d);
                        acc_g = ffma2(p1, d[0], acc_g);
                        acc_g8 = ffma2(p1, d[1], acc_g8);
                        acc_g = ffma2(p2, d[2], acc_g);
                        acc_g8 = ffma2(p2, d[3], acc_g8);
                        const bool block_end = SPB_LOG >= 0
                                                   ? (((ks + 1) & ((1 << (SPB_LOG < 0 ? 0 : SPB_LOG)) - 1)) == 0)
                                                   : (((S + ks + 1) & spb_mask) == 0);
                        if (block_end) {
                            y_g = ffma2(sg, acc_g, y_g);
                            y_g8 = ffma2(sg8, acc_g8, y_g8);
                            acc_g = 0;
                            acc_g8 = 0;
                        }
                    }
                }
                S += kChunkTiles * U::kStepsPerTile;
                // Refill this slot with the next chunk.  Every lane has used the
                // values it loaded from the slot, so the slot's reads are done
                // before the bulk copy overwrites it.
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
        // Flush a block cut by the end of this warp's slice.
        y_g = ffma2(sg, acc_g, y_g);
        y_g8 = ffma2(sg8, acc_g8, y_g8);
        const float2 yg = unpack2(y_g), yg8 = unpack2(y_g8);
        float vg = yg.x + yg.y, vg8 = yg8.x + yg8.y;
        vg += __shfl_xor_sync(0xffffffffu, vg, 1);
        vg8 += __shfl_xor_sync(0xffffffffu, vg8, 1);
        vg += __shfl_xor_sync(0xffffffffu, vg, 2);
        vg8 += __shfl_xor_sync(0xffffffffu, vg8, 2);
        float* rb = red + (i & 1) * kWarps * 16;
        if (t == 0) {
            rb[warp * 16 + g] = vg;
            rb[warp * 16 + g + 8] = vg8;
        }
        if (i + 1 < my_tiles) {
            if (geo.stage_bufs == 1) __syncthreads();  // every warp is done with the only stage buffer
            convert(i + 1, geo.stage_bufs == 2 ? (buf ^ 1) : 0);
        }
        __syncthreads();
        if (tid == 0) issue_raw(i + 1 + kRawSlots);
        if (warp == (i % kWarps) && lane < 16) {
            float v = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < kWarps; ++w2) v += rb[w2 * 16 + lane];
            const int64_t n = rt * 16 + lane;
            if (n < L.N) {
                if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
                store_f32(p.y, n, v, p.out_dtype);
            }
        }
    }
    // After a timed-out wait, give copies still in flight a bounded chance to
    // land before the CTA exits.
    if (bad && lane == 0) {
        for (int qq = q; qq < issued; ++qq) {
            const int sl = qq % S_SLOTS;
            const uint32_t ph = (uint32_t)((qq / S_SLOTS) & 1);
            for (int it = 0; it < (1 << 16); ++it)
                if (mbar_try_wait(&wbars[sl], ph)) break;
        }
    }
}

}  // namespace

bool gemv_supported(const MatmulParams& p) {
    if (p.M != 1 || p.g_idx != nullptr) return false;
    const size_t limit = device_info().smem_optin;
    const GemvGeom g = gemv_geom(p.L, p.scale_dtype, p.zp != nullptr, limit);
    return g.total_bytes <= limit;
}

template <int BITS, int SPB_LOG>
static cudaError_t launch_one(const MatmulParams& p, const GemvGeom& geo, int64_t grid, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<BITS, SPB_LOG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)geo.total_bytes);
    if (e != cudaSuccess) return e;
    gemv_kernel<BITS, SPB_LOG><<<(unsigned)grid, kThreads, geo.total_bytes, s>>>(p, geo);
    return cudaGetLastError();
}

// The static block structure needs blocks that tile every chunk: k-steps per
// block dividing the k-steps of a chunk (warp slices are whole chunks).
template <int BITS>
static cudaError_t launch_bits(const MatmulParams& p, const GemvGeom& geo, int64_t grid, cudaStream_t s) {
    constexpr int steps_per_chunk = kChunkTiles * (256 / BITS) / 16;
    const int spb = p.L.bs / 16;
    if (spb <= steps_per_chunk) {
        switch (spb) {
            case 1: return launch_one<BITS, 0>(p, geo, grid, s);
            case 2: return launch_one<BITS, 1>(p, geo, grid, s);
            case 4: return launch_one<BITS, 2>(p, geo, grid, s);
            case 8: return launch_one<BITS, 3>(p, geo, grid, s);
            default: break;
        }
    }
    return launch_one<BITS, -1>(p, geo, grid, s);
}

cudaError_t launch_gemv(const MatmulParams& p, cudaStream_t s) {
    const DeviceInfo& di = device_info();
    const GemvGeom geo = gemv_geom(p.L, p.scale_dtype, p.zp != nullptr, di.smem_optin);
    const int64_t grid = imin64(p.L.NT, di.sm_count);
    switch (p.L.bits) {
        case 2: return launch_bits<2>(p, geo, grid, s);
        case 4: return launch_bits<4>(p, geo, grid, s);
        case 8: return launch_bits<8>(p, geo, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
