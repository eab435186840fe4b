// int8-activation path (accuracy level 4), 1 <= M <= 16:
//   s_a[m, kb] = max_k |x[m, k]| / 127,  qa[m, k] = clamp(round(x[m, k] / s_a), -127, 127)
//   Y[m, n]    = sum_kb dot_i32(m, n, kb) * fl32(s_w[n, kb] * s_a[m, kb])   (+ bias[n])
//   dot_i32    = sum_{k in kb} qa[m, k] * (q[n, k] - zp[n, kb])   (exact integers)
//
// The operation follows onnx-runtime-ep-cpu 0.1.0-dev.5, src/kernels/
// matmul_nbits.rs: the accuracy-level-4 path quantises each K-block of the
// activations symmetrically to int8 (fn quantize_activation_signed), takes an
// exact integer dot per block against the weight codes (fn int8_row,
// fn int4_dot_row_scalar) and rescales once by weight scale * activation
// scale.  The rounding is half away from zero (rlx-cpu's quantize thunk uses
// f32::round).
//
// Two kernels on one stream:
//   1. quant_act_kernel: one warp per (m, kb) writes qa [M, KB*bs] (zero past
//      K) and s_a [M, KB] f32 into the caller's workspace.
//   2. gemv_i8_kernel: the same work decomposition as the float decode GEMV
//      (one CTA of 8 warps per 16-row tile and K-split, every weight load of a
//      warp issued first, K-splits of a row tile summed in a cluster through
//      distributed shared memory).  The packed layout gives lane (g, t) the
//      codes of rows g and g+8 at depths {2t, 2t+1, 2t+8, 2t+9} of each
//      16-deep k-step; the CTA stages its activations as int8 words in the
//      same byte order, so one dp4a (unsigned codes x signed activations)
//      takes four products per row.  The zero point enters once per block as
//      zp * sum(qa), whose partial sums come from a dp4a against 0x01010101.
//      The second kernel is launched as a programmatic dependent of the first:
//      it streams its weights while the activations are being quantised and
//      waits (griddepcontrol.wait) only before reading the workspace.
//
// Integer dots are exact; the per-block rescale and the sums across lanes,
// warps and K-splits are f32 in a fixed order, so results are bit-identical
// run to run.
#pragma once

#include <cstdlib>

#include "mnb_internal.h"

namespace mnb {
namespace gi8 {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxTPW = 8;      // k-tiles per warp per round
constexpr int kMaxCluster = 8;  // portable cluster size

struct Geom {
    int C;           // K-splits = cluster size
    int tiles_cta;   // k-tiles per CTA
    int tpw;         // k-tiles per warp per round
    int rounds;      // rounds per warp
    int kb_cta;      // blocks per CTA
    size_t act_bytes, sa_bytes, stage_bytes, red_bytes, part_bytes, total_bytes;
};

struct __align__(8) Entry {
    int32_t z;  // zero point
    float s;    // weight scale
};

// Workspace: qa [M, KB*bs] int8 at offset 0, s_a [M, KB] f32 after it.
__host__ __device__ inline size_t qa_bytes(int64_t M, const Layout& L) {
    return ((size_t)M * (size_t)L.Kpad + 255) & ~size_t(255);
}
__host__ __device__ inline size_t workspace_bytes(int64_t M, const Layout& L) {
    return qa_bytes(M, L) + (size_t)M * (size_t)L.KB * sizeof(float);
}

__device__ __forceinline__ int32_t dp4a_u_s(uint32_t codes, uint32_t acts, int32_t c) {
    int32_t d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(codes), "r"(acts), "r"(c));
    return d;
}

inline int env_or(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

// Same K decomposition as the float decode GEMV: each warp takes up to
// kMaxTPW k-tiles per round, the K-splits of a row tile form a cluster.
// MNB_I8_TPW overrides the tiles per warp (1..8).
inline Geom make_geom(const Layout& L, int64_t M, int MT) {
    Geom g{};
    const int64_t KTL = L.KTILES;
    int tpw = env_or("MNB_I8_TPW", 0);
    if (tpw < 1 || tpw > kMaxTPW) {
        tpw = (int)((KTL + kWarps - 1) / kWarps);
        if (tpw > kMaxTPW) tpw = kMaxTPW;
        if (tpw < 1) tpw = 1;
    }
    const int64_t per_round = (int64_t)kWarps * tpw;
    const int64_t rounds_total = (KTL + per_round - 1) / per_round;
    int C = (int)(rounds_total < kMaxCluster ? rounds_total : kMaxCluster);
    if (C < 1) C = 1;
    g.C = C;
    g.tpw = tpw;
    g.rounds = (int)((rounds_total + C - 1) / C);
    g.tiles_cta = (int)(per_round * g.rounds);
    g.kb_cta = (int)((g.tiles_cta * L.KT + L.bs - 1) / L.bs);
    const int kbs = g.kb_cta | 1;
    g.act_bytes = (size_t)M * g.tiles_cta * L.KT;
    g.sa_bytes = round16((size_t)M * kbs * sizeof(float));
    g.stage_bytes = (size_t)16 * kbs * sizeof(Entry);
    g.red_bytes = (size_t)kWarps * 16 * MT * 4;
    g.part_bytes = (size_t)16 * MT * 4;
    g.total_bytes = g.act_bytes + g.sa_bytes + g.stage_bytes + g.red_bytes + g.part_bytes;
    return g;
}

// Activation words of a lane, per 32-deep unit (two k-steps e = 2j, o = 2j+1
// of the unit), from the unit's 32 int8 values v[0..7] (v[i] = depths 4i..4i+3):
//   4-bit: one word per k-step, bytes at depths {2t, 2t+8, 2t+1, 2t+9}
//          (the order of the code bytes (word & 0x0F0F0F0F) and ((word >> 4) & ...));
//   8-bit: one word per k-step, depths {2t, 2t+1, 2t+8, 2t+9};
//   2-bit: word A0 = {e 2t, o 2t, e 2t+1, o 2t+1}, A2 = the same at +8
//          (the order of the fields ((word >> 2i) & 0x03030303)).
template <int BITS>
__device__ __forceinline__ void act_words(const uint32_t (&v)[8], int t, uint32_t& w0, uint32_t& w1) {
    const uint32_t c = 2u * (uint32_t)(t & 1);
    const int h = t >> 1;
    if constexpr (BITS == 8) {
        const uint32_t sel = c | ((c + 1) << 4) | ((c + 4) << 8) | ((c + 5) << 12);
        w0 = prmt(v[h], v[2 + h], sel);
        w1 = prmt(v[4 + h], v[6 + h], sel);
    } else if constexpr (BITS == 4) {
        const uint32_t sel = c | ((c + 4) << 4) | ((c + 1) << 8) | ((c + 5) << 12);
        w0 = prmt(v[h], v[2 + h], sel);
        w1 = prmt(v[4 + h], v[6 + h], sel);
    } else {
        const uint32_t sel = c | ((c + 4) << 4) | ((c + 1) << 8) | ((c + 5) << 12);
        w0 = prmt(v[h], v[4 + h], sel);
        w1 = prmt(v[2 + h], v[6 + h], sel);
    }
}

// Zero points and weight scales of a CTA's 16 rows x kb_cta blocks into the
// entry table (entry (r, j) at r * kbs + j).  Each thread issues the loads of
// all its entries (up to kPer per pass, consecutive threads on consecutive
// blocks) before it decodes any, so a pass costs one memory latency rather
// than one per entry.  SC is the stored scale type (float, or the 16-bit
// pattern of f16 / bf16).
template <typename SC>
__device__ __forceinline__ void stage_entries(const MatmulParams& p, const Layout& L, int64_t rt, int64_t kb0,
                                              int kb_cta, int kbs, Entry* stage) {
    constexpr int kPer = 4;
    const int tid = threadIdx.x;
    const int total = 16 * kb_cta;
    const SC* sc = static_cast<const SC*>(p.scales);
    for (int base = 0; base < total; base += kPer * kThreads) {
        SC raw[kPer];
        int zq[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int it = base + q * kThreads + tid;
            const int r = it / kb_cta, j = it - r * kb_cta;
            const int64_t n = rt * 16 + r, kb = kb0 + j;
            const bool ok = it < total && n < L.N && kb < L.KB;
            raw[q] = ok ? __ldg(sc + n * L.KB + kb) : SC(0);
            zq[q] = ok ? load_zp(p.zp, L, n, kb) : 0;
        }
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int it = base + q * kThreads + tid;
            if (it < total) {
                const int r = it / kb_cta, j = it - r * kb_cta;
                float sv;
                if constexpr (sizeof(SC) == 4) sv = raw[q];
                else if (p.scale_dtype == kF16) sv = __half2float(__ushort_as_half(raw[q]));
                else sv = __uint_as_float(static_cast<uint32_t>(raw[q]) << 16);
                stage[r * kbs + j] = Entry{zq[q], sv};
            }
        }
    }
}

// ---- 2. the GEMV ----
// SPB_LOG >= 0: blocks of 2^SPB_LOG k-steps and every warp slice starts on a
// block boundary (static block ends); -1: run-time block ends.
template <int BITS, int MT, int SPB_LOG>
__global__ void __launch_bounds__(kThreads, MT == 1 ? 3 : 1)
    gemv_i8_kernel(MatmulParams p, Geom geo, const int8_t* qa, const float* sa, int pdl) {
    constexpr int SPT = 16 / BITS;                   // k-steps per tile
    constexpr int PW = BITS == 8 ? 2 : 4;            // activation words loaded together
    constexpr int KT = 256 / BITS;
    constexpr int UNITS_PER_TILE = KT / 32;
    // 2-bit codes of one 32-bit field group span two k-steps; with 16-deep
    // blocks each k-step's activations are masked to their own bytes.
    constexpr bool kSplit2 = BITS == 2 && SPB_LOG == 0;
    const Layout& L = p.L;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* act = smem;
    float* sa_s = reinterpret_cast<float*>(smem + geo.act_bytes);
    Entry* stage = reinterpret_cast<Entry*>(smem + geo.act_bytes + geo.sa_bytes);
    float* red = reinterpret_cast<float*>(smem + geo.act_bytes + geo.sa_bytes + geo.stage_bytes);
    float* part = red + kWarps * 16 * MT;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = (int)p.M;
    const int C = geo.C;
    const int64_t rt = blockIdx.x / C;
    const int split = (int)(blockIdx.x - rt * C);
    const int64_t cta_t0 = (int64_t)split * geo.tiles_cta;
    const int64_t cta_t1 = imin64(cta_t0 + geo.tiles_cta, L.KTILES);
    const int tpw = geo.tpw;
    const int64_t k_cta0 = cta_t0 * KT;
    const int kb_cta = geo.kb_cta;
    const int kbs = kb_cta | 1;
    const int64_t kb0 = k_cta0 / L.bs;

    // ---- weight loads first ----
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

    // ---- zero points and weight scales of the CTA's (row, block)s ----
    if (p.scale_dtype == kF32) stage_entries<float>(p, L, rt, kb0, kb_cta, kbs, stage);
    else stage_entries<uint16_t>(p, L, rt, kb0, kb_cta, kbs, stage);

    griddep_wait();  // the workspace is written by the quantisation kernel
    if (pdl) griddep_launch_dependents();  // after the wait: at most two chained kernels overlap

    // ---- activation scales and int8 words of this CTA's depths ----
    for (int it = tid; it < M * kb_cta; it += kThreads) {
        const int m = it / kb_cta, j = it - m * kb_cta;
        const int64_t kb = kb0 + j;
        sa_s[m * kbs + j] = kb < L.KB ? __ldg(sa + m * L.KB + kb) : 0.f;
    }
    {
        const int units = geo.tiles_cta * UNITS_PER_TILE;
        for (int it = tid; it < M * units; it += kThreads) {
            const int m = it / units, u = it - m * units;
            const int64_t k = k_cta0 + 32 * (int64_t)u;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
            const int8_t* src = qa + m * L.Kpad + k;
            if (k < L.Kpad) lo = __ldg(reinterpret_cast<const uint4*>(src));
            if (k + 16 < L.Kpad) hi = __ldg(reinterpret_cast<const uint4*>(src + 16));
            const uint32_t v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            const int tl = u / UNITS_PER_TILE, pos = 2 * (u % UNITS_PER_TILE);
            uint8_t* chunk = act + ((int64_t)(m * geo.tiles_cta + tl) * 4) * (KT / 4) + pos * 4;
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                uint32_t w0, w1;
                act_words<BITS>(v, tt, w0, w1);
                *reinterpret_cast<uint2*>(chunk + tt * (KT / 4)) = make_uint2(w0, w1);
            }
        }
    }
    __syncthreads();

    // ---- contraction ----
    const uint32_t act_lane = smem_u32(act) + (uint32_t)t * (KT / 4);
    const uint32_t m_stride = (uint32_t)geo.tiles_cta * KT;
    const int spb_log = SPB_LOG >= 0 ? SPB_LOG : __ffs(L.bs / 16) - 1;
    const int spb_mask = (1 << spb_log) - 1;
    constexpr int kStaticMask = SPB_LOG >= 0 ? (1 << (SPB_LOG >= 0 ? SPB_LOG : 0)) - 1 : 0;
    const Entry* st_g = stage + g * kbs;
    const Entry* st_g8 = stage + (g + 8) * kbs;

    int32_t dq[MT], dq8[MT], da[MT];
    float yg[MT], yg8[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) dq[m] = dq8[m] = da[m] = 0, yg[m] = yg8[m] = 0.f;
    bool fresh = true;
    int last_kb = 0;

    auto flush = [&](int kbl) {
        const Entry eg = st_g[kbl], eg8 = st_g8[kbl];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                const float sam = sa_s[m * kbs + kbl];
                yg[m] = fmaf((float)(dq[m] - eg.z * da[m]), eg.s * sam, yg[m]);
                yg8[m] = fmaf((float)(dq8[m] - eg8.z * da[m]), eg8.s * sam, yg8[m]);
            }
            dq[m] = dq8[m] = da[m] = 0;
        }
        fresh = true;
    };
    auto lds4 = [](uint32_t addr) {
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(addr));
        return v;
    };
    auto lds2 = [](uint32_t addr) {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
        return v;
    };

    for (int round = 0; round < geo.rounds; ++round) {
        const int64_t t0 = warp_tile0(round);
        if (round > 0) load_round(round);
        const int ntile = (int)imin64(tpw, cta_t1 - t0);
        const int tl0 = (int)(t0 - cta_t0);
#pragma unroll
        for (int j = 0; j < kMaxTPW; ++j) {
            if (j < ntile) {
                const uint32_t w[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
                const uint32_t tile_addr = act_lane + (uint32_t)(tl0 + j) * KT;
#pragma unroll
                for (int part0 = 0; part0 < SPT; part0 += (BITS == 8 ? 2 : 4)) {
                    uint32_t a[MT][PW];
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < M) {
                            const uint32_t addr = tile_addr + (uint32_t)m * m_stride + (uint32_t)part0 * 4u;
                            if constexpr (PW == 4) {
                                const uint4 q = lds4(addr);
                                a[m][0] = q.x; a[m][1] = q.y; a[m][2] = q.z; a[m][3] = q.w;
                            } else {
                                const uint2 q = lds2(addr);
                                a[m][0] = q.x; a[m][1] = q.y;
                            }
                        }
                    }
#pragma unroll
                    for (int si = 0; si < PW; ++si) {
                        const int s = part0 + si;               // k-step inside the tile
                        const int ks = j * SPT + s;             // k-step inside the warp's slice
                        const int Sk = tl0 * SPT + ks;          // k-step inside the CTA
                        if constexpr (BITS == 4) {
                            const uint32_t cg = w[s] & 0x0F0F0F0Fu, cg8 = (w[s] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                if (m < M) {
                                    dq[m] = dp4a_u_s(cg, a[m][si], dq[m]);
                                    dq8[m] = dp4a_u_s(cg8, a[m][si], dq8[m]);
                                    da[m] = dp4a_u_s(0x01010101u, a[m][si], da[m]);
                                }
                            }
                        } else if constexpr (BITS == 8) {
                            const uint32_t cg = prmt(w[2 * s], w[2 * s + 1], 0x5410u);
                            const uint32_t cg8 = prmt(w[2 * s], w[2 * s + 1], 0x7632u);
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                if (m < M) {
                                    dq[m] = dp4a_u_s(cg, a[m][si], dq[m]);
                                    dq8[m] = dp4a_u_s(cg8, a[m][si], dq8[m]);
                                    da[m] = dp4a_u_s(0x01010101u, a[m][si], da[m]);
                                }
                            }
                        } else {
                            // code word s / 2 holds k-steps s & ~1 and s | 1; activation
                            // words (2 (s/2) + h) % 4 of this part for field halves h.
                            const int cw = s >> 1, odd = s & 1;
                            if (kSplit2 || !odd) {
                                const uint32_t word = w[cw];
                                const uint32_t c0 = word & 0x03030303u, c0h = (word >> 2) & 0x03030303u;
                                const uint32_t c2 = (word >> 4) & 0x03030303u, c2h = (word >> 6) & 0x03030303u;
                                const int i0 = (2 * cw) % 4, i2 = i0 + 1;
                                const uint32_t mk = kSplit2 ? (odd ? 0xFF00FF00u : 0x00FF00FFu) : 0xFFFFFFFFu;
#pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    if (m < M) {
                                        const uint32_t A0 = a[m][i0] & mk, A2 = a[m][i2] & mk;
                                        dq[m] = dp4a_u_s(c2, A2, dp4a_u_s(c0, A0, dq[m]));
                                        dq8[m] = dp4a_u_s(c2h, A2, dp4a_u_s(c0h, A0, dq8[m]));
                                        da[m] = dp4a_u_s(0x01010101u, A2, dp4a_u_s(0x01010101u, A0, da[m]));
                                    }
                                }
                            }
                        }
                        fresh = false;
                        // for 2-bit without the split, blocks hold whole field groups (>= 2 k-steps)
                        const bool block_end =
                            SPB_LOG >= 0 ? (((ks + 1) & kStaticMask) == 0) : (((Sk + 1) & spb_mask) == 0);
                        last_kb = Sk >> spb_log;
                        if (block_end) flush(last_kb);
                    }
                }
            }
        }
        if (!fresh) flush(last_kb);  // a block cut by the end of this warp's tiles
    }

    // ---- reduce: the 4 lanes of a row (fixed pairing), the warps, the cluster ----
    float* mine = red + warp * 16 * MT;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < M) {
            float v0 = yg[m], v1 = yg8[m];
            v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 1);
            v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 1);
            v0 += __shfl_xor_sync(0xFFFFFFFFu, v0, 2);
            v1 += __shfl_xor_sync(0xFFFFFFFFu, v1, 2);
            if (t == 0) {
                mine[g * MT + m] = v0;
                mine[(g + 8) * MT + m] = v1;
            }
        }
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
        cluster_sync();
    }
    if (split == 0 && owner) {
        const int64_t n = rt * 16 + row;
        if (n < L.N) {
            if (p.bias) v += load_f32(p.bias, n, p.bias_dtype);
            store_f32(p.y, (int64_t)m * L.N + n, v, p.out_dtype);
        }
    }
    if (blockIdx.x == 0 && tid == 0) verify_header(p.packed_hdr, L, p.status);
}

template <int BITS, int MT, int SPB_LOG>
cudaError_t launch_variant(const MatmulParams& p, const Geom& geo, const int8_t* qa, const float* sa,
                           cudaStream_t s) {
    const int pdl = (p.flags & kFlagPDL) ? 1 : 0;
    auto kern = gemv_i8_kernel<BITS, MT, SPB_LOG>;
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
    // always a programmatic dependent of the quantisation kernel before it
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p, geo, qa, sa, pdl);
}

template <int BITS, int MT>
cudaError_t launch_spb(const MatmulParams& p, const Geom& geo, const int8_t* qa, const float* sa, cudaStream_t s) {
    const int spb = p.L.bs / 16;
    const int steps_per_warp = geo.tpw * (16 / BITS);
    if (steps_per_warp % spb == 0) {
        switch (spb) {
            case 1: return launch_variant<BITS, MT, 0>(p, geo, qa, sa, s);
            case 2: return launch_variant<BITS, MT, 1>(p, geo, qa, sa, s);
            case 4: return launch_variant<BITS, MT, 2>(p, geo, qa, sa, s);
            case 8: return launch_variant<BITS, MT, 3>(p, geo, qa, sa, s);
            default: break;
        }
    }
    // 2-bit codes with 16-deep blocks need the static per-k-step split
    if (BITS == 2 && spb == 1) return cudaErrorNotSupported;
    return launch_variant<BITS, MT, -1>(p, geo, qa, sa, s);
}

template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const Geom& geo, const int8_t* qa, const float* sa,
                        cudaStream_t s) {
    if (p.M == 1) return launch_spb<BITS, 1>(p, geo, qa, sa, s);
    return launch_spb<BITS, 16>(p, geo, qa, sa, s);
}

}  // namespace gi8
}  // namespace mnb
