// Grouped (mixture-of-experts) small-batch GEMV: for every token t and
// expert slot s,
//   Y[t, s, :] = X_row(t, s) . dequant(B_e)^T,   e = ids[t, s],
// with X_row(t, s) = X[t] (one activation row shared by a token's slots) or
// X[t, s] (one row per slot).  This is ggml's MUL_MAT_ID as the SpacemiT
// backend computes it (toy 0.8.0, data/vendor/ggml/src/ggml-cpu/spacemit/
// ime.cpp, forward_mul_mat_id: the (slot, token) rows are grouped by the
// expert they select, in ascending token-then-slot order, and each group is
// one product with that expert's matrix), and rlx's grouped dequant matmul
// when every row selects one expert, S = 1 (rlx-cpu 0.2.13,
// src/thunk/ops/quant.rs, exec_dequant_grouped_mat_mul_gguf).
//
// One launch covers every expert with no host round trip.  CTA (x, y) owns
// row tile x / C (K-split x % C) of a set of experts.  It finds the experts
// present in ids once; then, for the y-th, (y + G)-th, ... of them in
// ascending order (G = gridDim.y, chosen on the host so the grid fills the
// GPU about twice), it runs the decode GEMV tile of gemv_mma.cuh on that
// expert's (t, s) pairs, a chunk of pairs per pass.  A chunk is at most the
// MMA's 8 or 16 rows, fewer when the staged activation rows would not fit
// three CTAs per SM.  The pairs are gathered, in order, into shared memory
// inside the first pass, after its weight loads are issued, so the
// gathering hides under the load latency.  Only active experts' weights are
// read.  Pairs whose expert id is out of range belong to no group: their Y
// rows are not written and the device status word reports
// MNB_ERR_INVALID_ARG.
#pragma once

#include "gemv_mma.cuh"

namespace mnb {
namespace gmoe {

using gmma::kThreads;
using gmma::kWarps;

constexpr int kMaxExperts = 1024;  // presence bitmap in shared memory
constexpr int kMaxPairs = 4096;    // T * S: the pair list of one expert in shared memory

struct MoeArgs {
    const int32_t* ids;        // [T, S] expert of each (token, slot)
    int pairs;                 // T * S
    int S;
    int E;
    int x_per_slot;            // 0: X [T, K]; 1: X [T, S, K]
    int bitmap_words;          // ceil(E / 32)
    int chunk;                 // pairs per tile pass (<= MT; the staged X rows)
    size_t extra_off;          // shared-memory offset of the bitmap and pair list
    size_t expert_bytes;       // packed bytes per expert (header included)
    size_t expert_scale_bytes; // N * KB * sizeof(scale)
    size_t expert_zp_bytes;    // N * zp_row
};

// Rows of one tile pass over an expert's pairs: local row m is pair
// list[c0 + m] = t * S + s.  prepare() (called by the tile once its weight
// loads are in flight) gathers the expert's pairs on the first pass.
struct GroupRows {
    int M;                  // rows of this pass, set by prepare()
    int32_t* list;          // the expert's pairs, ascending (shared memory)
    int* count;             // number of the expert's pairs (shared memory)
    int* hits;              // per-warp hit counts (shared memory, kWarps)
    const int32_t* ids;
    int pairs, expert, c0, chunk, S, x_per_slot;

    // Ascending compaction of the pairs whose id is `expert`: each warp
    // takes a contiguous segment of ids, counts its hits, then writes them
    // after the hits of the warps before it.
    __device__ __forceinline__ void prepare() {
        if (c0 == 0) {
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            const int seg = (pairs + kWarps - 1) / kWarps;
            const int b0 = min(pairs, warp * seg), b1 = min(pairs, b0 + seg);
            int h = 0;
            for (int i0 = b0; i0 < b1; i0 += 32) {
                const int i = i0 + lane;
                h += __popc(__ballot_sync(0xFFFFFFFFu, i < b1 && ids[i] == expert));
            }
            if (lane == 0) hits[warp] = h;
            __syncthreads();
            int base = 0, total = 0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                base += w < warp ? hits[w] : 0;
                total += hits[w];
            }
            for (int i0 = b0; i0 < b1; i0 += 32) {
                const int i = i0 + lane;
                const bool hit = i < b1 && ids[i] == expert;
                const uint32_t mask = __ballot_sync(0xFFFFFFFFu, hit);
                if (hit) list[base + __popc(mask & ((1u << lane) - 1u))] = i;
                base += __popc(mask);
            }
            if (threadIdx.x == 0) *count = total;
            __syncthreads();
        }
        M = min(chunk, *count - c0);
    }
    __device__ __forceinline__ int64_t x_row(int m) const {
        return x_per_slot ? list[c0 + m] : list[c0 + m] / S;
    }
    __device__ __forceinline__ int64_t y_row(int m) const { return list[c0 + m]; }
};

__device__ __forceinline__ int nth_set_bit(uint32_t bits, int n) {
    for (int i = 0; i < n; ++i) bits &= bits - 1u;
    return __ffs((int)bits) - 1;
}

template <int BITS, bool BF16X, int MT, int SPB_LOG>
__global__ void __launch_bounds__(kThreads, BITS == 8 ? 4 : 3) gemv_moe_kernel(MatmulParams p, gmma::Geom geo,
                                                                              MoeArgs g) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t* present = reinterpret_cast<uint32_t*>(smem + g.extra_off);
    int32_t* list = reinterpret_cast<int32_t*>(present + g.bitmap_words);
    __shared__ int s_expert, s_count;
    __shared__ int s_hits[kWarps];
    const int tid = threadIdx.x;
    const int TS = g.pairs;

    // ---- 1. experts present in ids ----
    for (int i = tid; i < g.bitmap_words; i += kThreads) present[i] = 0u;
    __syncthreads();
    bool bad = false;
    for (int i = tid; i < TS; i += kThreads) {
        const int32_t e = g.ids[i];
        if (e >= 0 && e < g.E) atomicOr(&present[e >> 5], 1u << (e & 31));
        else bad = true;
    }
    if (bad && blockIdx.x == 0 && blockIdx.y == 0) set_status(p.status, 1 /* MNB_ERR_INVALID_ARG */);
    __syncthreads();

    // ---- 2. every G-th present expert, ascending, from the blockIdx.y-th ----
    int active = 0;
    for (int w = 0; w < g.bitmap_words; ++w) active += __popc(present[w]);
    for (int j = (int)blockIdx.y; j < active; j += (int)gridDim.y) {
        if (tid == 0) {
            int want = j, found = -1;
            for (int w = 0; w < g.bitmap_words && found < 0; ++w) {
                const uint32_t bits = present[w];
                const int c = __popc(bits);
                if (want < c) found = 32 * w + nth_set_bit(bits, want);
                else want -= c;
            }
            s_expert = found;
        }
        __syncthreads();
        const int e = s_expert;

        // ---- 3. the expert's weights; its pairs are gathered inside the first
        //         tile pass, while that pass's weight loads are in flight ----
        MatmulParams q = p;
        const uint8_t* hdr = static_cast<const uint8_t*>(p.packed_hdr) + (size_t)e * g.expert_bytes;
        q.packed_hdr = hdr;
        q.packed = hdr + kHeaderBytes;
        q.scales = static_cast<const uint8_t*>(p.scales) + (size_t)e * g.expert_scale_bytes;
        q.zp = p.zp ? p.zp + (size_t)e * g.expert_zp_bytes : nullptr;
        const int64_t rt = blockIdx.x / geo.C;
        const int split = (int)(blockIdx.x - rt * geo.C);
        int c0 = 0;
        do {
            GroupRows rows{0, list, &s_count, s_hits, g.ids, TS, e, c0, g.chunk, g.S, g.x_per_slot};
            gmma::gemv_tile<BITS, BF16X, MT, SPB_LOG>(q, geo, 0, rt, split, rows, smem);
            c0 += g.chunk;
        } while (c0 < s_count);
        // each expert's header is checked by the first CTA that reads its weights
        if (blockIdx.x == 0 && tid == 0) verify_header(hdr, p.L, p.status);
        __syncthreads();  // the list, s_expert and s_count are rewritten for the next expert
    }
}

template <int BITS, bool BF16X, int MT, int SPB_LOG>
cudaError_t launch_variant(const MatmulParams& p, const gmma::Geom& geo, const MoeArgs& g, unsigned groups,
                           size_t smem_bytes, cudaStream_t s) {
    auto kern = gemv_moe_kernel<BITS, BF16X, MT, SPB_LOG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.L.NT * geo.C), groups);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)geo.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, geo, g);
}

// Static block structure when every warp slice starts on a block boundary
// (as for the plain GEMV).
template <int BITS, bool BF16X, int MT>
cudaError_t launch_spb(const MatmulParams& p, const gmma::Geom& geo, const MoeArgs& g, unsigned groups,
                       size_t smem_bytes, cudaStream_t s) {
    const int spb = p.L.bs / 16;
    const int steps_per_warp = geo.tpw * (16 / BITS);
    if (steps_per_warp % spb == 0) {
        switch (spb) {
            case 1: return launch_variant<BITS, BF16X, MT, 0>(p, geo, g, groups, smem_bytes, s);
            case 2: return launch_variant<BITS, BF16X, MT, 1>(p, geo, g, groups, smem_bytes, s);
            case 4: return launch_variant<BITS, BF16X, MT, 2>(p, geo, g, groups, smem_bytes, s);
            case 8: return launch_variant<BITS, BF16X, MT, 3>(p, geo, g, groups, smem_bytes, s);
            default: break;
        }
    }
    return launch_variant<BITS, BF16X, MT, -1>(p, geo, g, groups, smem_bytes, s);
}

// MT = 8 when no expert can own more than 8 pairs, else 16.
template <int BITS>
cudaError_t launch_bits(const MatmulParams& p, const gmma::Geom& geo, const MoeArgs& g, unsigned groups,
                        size_t smem_bytes, cudaStream_t s) {
    const bool bf = p.act_dtype == kBF16;
    if (g.pairs <= 8)
        return bf ? launch_spb<BITS, true, 8>(p, geo, g, groups, smem_bytes, s)
                  : launch_spb<BITS, false, 8>(p, geo, g, groups, smem_bytes, s);
    return bf ? launch_spb<BITS, true, 16>(p, geo, g, groups, smem_bytes, s)
              : launch_spb<BITS, false, 16>(p, geo, g, groups, smem_bytes, s);
}

}  // namespace gmoe
}  // namespace mnb
