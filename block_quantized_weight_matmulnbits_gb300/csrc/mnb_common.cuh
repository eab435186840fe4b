// Shared device/host helpers of libmnb (CUDA side only).
//
// Packed weight layout
// --------------------
// The ORT MatMulNBits weight B is uint8 [N, KB, blob], codes least-significant
// bits first (onnx-runtime-ep-cpu 0.1.0-dev.5, src/kernels/matmul_nbits.rs,
// module doc and fn dequantize_nbits_value).  mnb_pack_weights re-tiles the
// codes, unchanged, into 512-byte tiles:
//
//   tile (nt, kt) = rows [16 nt, 16 nt + 16) x depths [KT kt, KT kt + KT),
//   KT = 256 / bits (64 for 4-bit, 128 for 2-bit, 32 for 8-bit),
//   tiles ordered row-tile major: all KTILES tiles of row-tile 0, then 1, ...
//
// Inside a tile, lane l = 4 g + t (g = l / 4, t = l % 4) of a warp owns 16
// contiguous bytes, so one warp-wide 16-byte load reads a whole tile.  Lane l
// holds the depths {2t, 2t+1, 2t+8, 2t+9} of every 16-deep k-step for rows g
// and g+8 of the tile: exactly the A-operand fragment a warp-level
// m16n8k16 MMA wants when W rows are the MMA's M dimension.  Per k-step the
// eight codes are named by fragment register r (0: row g, depths 2t/2t+1;
// 1: row g+8, 2t/2t+1; 2: row g, 2t+8/2t+9; 3: row g+8, 2t+8/2t+9) and pair
// element e (0 = even depth, 1 = odd depth):
//   4-bit: k-step s is 32-bit word s; (r, e) is nibble slot r + 4e.  So
//          ((word >> 4r) & 0x000F000F) holds the (even, odd) pair of register
//          r in its two 16-bit halves.
//   2-bit: k-steps 2j, 2j+1 share word j; field i + 8e with i = 4 (s & 1) + r.
//          ((word >> 2i) & 0x00030003) holds the pair.
//   8-bit: k-step s occupies words 2s (depths 2t/2t+1) and 2s+1 (2t+8/2t+9);
//          byte 2 hi + e of the word, hi = row g+8.
// Rows are zero-padded to a multiple of 16 and depths from KB*bs up to a
// multiple of KT; codes of depths [K, KB*bs) are copied as they are.
// A 256-byte header precedes the tiles.
#pragma once

#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace mnb {

constexpr uint32_t kMagic = 0x50424E4Du;  // "MNBP"
constexpr uint32_t kLayoutVersion = 1;
constexpr int64_t kHeaderBytes = 256;
constexpr int kTileBytes = 512;

struct PackedHeader {
    uint32_t magic;
    uint32_t version;
    int64_t N;
    int64_t K;
    int32_t bits;
    int32_t block_size;
    int32_t format;  // 0: MatMulNBits integer codes; else a floating-point weight format (WFormat)
    int32_t kperm;   // 1: depths stored in g_idx group order, the permutation after the tiles (act-order pack)
};

// Weight formats of a packed buffer.  kWfInt: MatMulNBits codes (ORT source
// [N, KB, blob]).  The floating-point formats of rlx-cpu 0.2.13,
// src/thunk/ops/quant.rs (dequant_matmul_fp8, dequant_matmul_nvfp4) come from
// a [K, N] source: FP8 one byte per weight at k * N + n (bits 8), NVFP4 one
// nibble per weight at flat index k * N + n, low nibble first (bits 4).
enum WFormat : int { kWfInt = 0, kWfE4M3 = 1, kWfE5M2 = 2, kWfNVFP4 = 3 };

struct Layout {
    int bits;
    int bs;
    int64_t N, K;
    int64_t KB;      // ceil(K / bs)
    int64_t Kpad;    // KB * bs (the ORT padded depth)
    int64_t KT;      // depths per tile = 256 / bits
    int64_t KTILES;  // tiles per row-tile
    int64_t NT;      // row-tiles = ceil(N / 16)
    int64_t blob;    // bs * bits / 8
    int64_t zp_row;  // ceil(KB * bits / 8)

    __host__ __device__ void init(int64_t n, int64_t k, int b, int blk) {
        bits = b;
        bs = blk;
        N = n;
        K = k;
        KB = (k + blk - 1) / blk;
        Kpad = KB * blk;
        KT = 256 / b;
        KTILES = (Kpad + KT - 1) / KT;
        NT = (n + 15) / 16;
        blob = (int64_t)blk * b / 8;
        zp_row = (KB * b + 7) / 8;
    }
    __host__ __device__ size_t data_bytes() const { return (size_t)NT * KTILES * kTileBytes; }
    __host__ __device__ size_t total_bytes() const { return (size_t)kHeaderBytes + data_bytes(); }

    // Bit index (from the start of the tile data) of code (n, k).
    __host__ __device__ int64_t bit_of(int64_t n, int64_t k) const {
        const int64_t nt = n >> 4;
        const int r16 = (int)(n & 15);
        const int g = r16 & 7, hi = r16 >> 3;
        const int64_t kt = k / KT;
        const int kk = (int)(k - kt * KT);
        const int s = kk >> 4, c = kk & 15;
        const int t = (c & 7) >> 1, e = c & 1, half = c >> 3;
        const int lane = g * 4 + t;
        const int r = half * 2 + hi;
        int bitpos;
        if (bits == 4) {
            bitpos = s * 32 + (r + 4 * e) * 4;
        } else if (bits == 2) {
            const int i = (s & 1) * 4 + r;
            bitpos = (s >> 1) * 32 + (i + 8 * e) * 2;
        } else {
            bitpos = (2 * s + half) * 32 + (hi * 2 + e) * 8;
        }
        return (((nt * KTILES + kt) * 32 + lane) * 128) + bitpos;
    }

    // Inverse of bit_of for one field: tile (nt, kt), lane, 32-bit word j of
    // the lane's 16 bytes and field f inside the word (f < 32 / bits).
    __host__ __device__ void field_coords(int64_t nt, int64_t kt, int lane, int j, int f, int64_t* n,
                                          int64_t* k) const {
        int s, r, e, hi, half;
        if (bits == 4) {
            r = f & 3;
            e = f >> 2;
            s = j;
            hi = r & 1;
            half = r >> 1;
        } else if (bits == 2) {
            e = f >> 3;
            const int i = f & 7;
            s = 2 * j + (i >> 2);
            r = i & 3;
            hi = r & 1;
            half = r >> 1;
        } else {
            hi = f >> 1;
            e = f & 1;
            s = j >> 1;
            half = j & 1;
        }
        const int g = lane >> 2, t = lane & 3;
        *n = nt * 16 + g + 8 * hi;
        *k = kt * KT + 16 * s + 2 * t + 8 * half + e;
    }
};

__host__ __device__ inline int code_mask(int bits) { return bits == 8 ? 0xFF : ((1 << bits) - 1); }

// ---- dtype helpers -------------------------------------------------------

enum : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

__device__ __forceinline__ float load_f32(const void* p, int64_t i, int dt) {
    if (dt == kF32) return __ldg(reinterpret_cast<const float*>(p) + i);
    const uint16_t u = __ldg(reinterpret_cast<const unsigned short*>(p) + i);
    if (dt == kF16) return __half2float(__ushort_as_half(u));
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

__device__ __forceinline__ void store_f32(void* p, int64_t i, float v, int dt) {
    if (dt == kF32) {
        reinterpret_cast<float*>(p)[i] = v;
    } else if (dt == kF16) {
        reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
    } else {
        reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    }
}

__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Zero point of (row n, group g) from the ORT zero-point tensor; NULL => 2^(bits-1).
__device__ __forceinline__ int load_zp(const uint8_t* zp, const Layout& L, int64_t n, int64_t g) {
    if (zp == nullptr) return 1 << (L.bits - 1);
    const int64_t bit = g * L.bits;
    return (__ldg(zp + n * L.zp_row + (bit >> 3)) >> (bit & 7)) & code_mask(L.bits);
}

// ---- PTX wrappers: shared-memory barriers and bulk copies -----------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or the hint (nanoseconds) elapses, instead of polling the barrier.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase of an mbarrier: retries of a suspending try_wait
// (up to kWaitHintNs each), about two seconds in all.  Returns false (and
// records MNB_ERR_TIMEOUT) when the limit runs out.
constexpr uint32_t kWaitHintNs = 100000;
constexpr uint32_t kWaitLimit = 20000;
constexpr uint32_t kWaitPoll = 0xFFFFFFFFu;  // hint value meaning: poll with test_wait, never suspend

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same with the call's limits: `limit` tries, each a suspending try_wait
// with hint_ns (kWaitPoll: test_wait polling, 0: try_wait without a hint).
__device__ __forceinline__ bool mbar_wait_lim(uint64_t* bar, uint32_t parity, int* status, uint32_t limit,
                                              uint32_t hint_ns) {
    for (uint32_t i = 0; i < limit; ++i) {
        const bool ok = hint_ns == kWaitPoll ? mbar_test_wait(bar, parity)
                        : hint_ns          ? mbar_try_wait_sleep(bar, parity, hint_ns)
                                           : mbar_try_wait(bar, parity);
        if (ok) return true;
    }
    set_status(status, 5 /* MNB_ERR_TIMEOUT */);
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if (mbar_try_wait_sleep(bar, parity, kWaitHintNs)) return true;
    }
    set_status(status, 5 /* MNB_ERR_TIMEOUT */);
    return false;
}

// Compare the header mnb_pack_weights wrote at the start of a packed buffer
// with the call's shape; a mismatch sets MNB_ERR_LAYOUT_MISMATCH.  Kernels run
// it from one thread, after their main work, so it costs one 32-byte read.
__device__ __forceinline__ void verify_header(const void* packed_hdr, const Layout& L, int* status,
                                              int format = kWfInt, int kperm = 0) {
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed_hdr);
    if (h->magic != kMagic || h->version != kLayoutVersion || h->N != L.N || h->K != L.K || h->bits != L.bits ||
        h->block_size != L.bs || h->format != format || h->kperm != kperm)
        set_status(status, 6 /* MNB_ERR_LAYOUT_MISMATCH */);
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes: multiple
// of 16; both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
    uint32_t d;
    // (a & mask) | orv
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ---- streaming loads, dependent launch, clusters ------------------------

// 16-byte load that bypasses L1 (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch: wait for the preceding kernel's completion
// (and memory) / allow the next kernel to be scheduled.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ---- small arithmetic helpers ----------------------------------------------

__host__ __device__ inline size_t round16(size_t v) { return (v + 15) & ~size_t(15); }

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ uint64_t pack2u(uint32_t a, uint32_t b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

}  // namespace mnb
