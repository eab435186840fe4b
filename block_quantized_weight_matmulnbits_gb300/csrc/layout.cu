// Weight re-tiling (pack / unpack) and the f32 dequantisation export.
//
// The packed layout is documented in mnb_common.cuh.  Packing moves codes and
// never changes them, so unpack(pack(B)) == B byte for byte.  The export
// computes w = (f32(q) - f32(zp)) * f32(scale) with one f32 rounding, the
// definition of onnx-runtime-ep-cpu 0.1.0-dev.5, src/kernels/matmul_nbits.rs,
// fn dequantize_nbits_value.
#include "mnb_internal.h"

namespace mnb {
namespace {

__device__ __forceinline__ int ort_code(const uint8_t* b, const Layout& L, int64_t n, int64_t k) {
    const int64_t kb = k / L.bs;
    const int64_t bit = (k - kb * L.bs) * L.bits;
    return (b[(n * L.KB + kb) * L.blob + (bit >> 3)] >> (bit & 7)) & code_mask(L.bits);
}

__device__ __forceinline__ int packed_code(const uint8_t* packed, const Layout& L, int64_t n, int64_t k) {
    const int64_t bit = L.bit_of(n, k);
    return (packed[bit >> 3] >> (bit & 7)) & code_mask(L.bits);
}

// Code (n, k) of a [K, N] floating-point weight source (k < K, n < N).
__device__ __forceinline__ int kn_code(const uint8_t* w, const Layout& L, int fmt, int64_t n, int64_t k) {
    const int64_t f = k * L.N + n;
    if (fmt == kWfNVFP4) return (w[f >> 1] >> ((f & 1) * 4)) & 0xF;
    return w[f];
}

// One thread per 32-bit word of tile data.  fmt kWfInt reads ORT codes (the
// padded depths [K, KB*bs) included); the floating-point formats read the
// [K, N] source and zero-fill depths past K (a zero code decodes to +0).
// perm (act-order pack): stored depth j holds the code of depth perm[j].
__global__ void pack_kernel(const uint8_t* __restrict__ b_ort, uint32_t* __restrict__ out, Layout L,
                            int64_t words, int fmt, const int32_t* __restrict__ perm) {
    const int64_t wi = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (wi >= words) return;
    const int64_t tile = wi >> 7;  // 128 words per tile
    const int lane = (int)((wi >> 2) & 31);
    const int j = (int)(wi & 3);
    const int64_t nt = tile / L.KTILES, kt = tile - nt * L.KTILES;
    const int fields = 32 / L.bits;
    uint32_t word = 0;
    for (int f = 0; f < fields; ++f) {
        int64_t n, k;
        L.field_coords(nt, kt, lane, j, f, &n, &k);
        if (fmt == kWfInt) {
            if (perm != nullptr && k < L.Kpad) {
                const int64_t src = perm[k];
                k = src < 0 ? 0 : (src >= L.Kpad ? L.Kpad - 1 : src);  // a bad g_idx sets the status word
            }
            if (n < L.N && k < L.Kpad) word |= (uint32_t)ort_code(b_ort, L, n, k) << (f * L.bits);
        } else if (n < L.N && k < L.K) {
            word |= (uint32_t)kn_code(b_ort, L, fmt, n, k) << (f * L.bits);
        }
    }
    out[wi] = word;
}

__global__ void header_kernel(uint8_t* hdr, Layout L, int fmt, int kperm) {
    const int i = threadIdx.x;
    if (i < kHeaderBytes / 4) reinterpret_cast<uint32_t*>(hdr)[i] = 0;
    __syncthreads();
    if (i == 0) {
        PackedHeader* h = reinterpret_cast<PackedHeader*>(hdr);
        h->magic = kMagic;
        h->version = kLayoutVersion;
        h->N = L.N;
        h->K = L.K;
        h->bits = L.bits;
        h->block_size = L.bs;
        h->format = fmt;
        h->kperm = kperm;
    }
}

// Act-order pack: the depths sorted by their g_idx group (stable), so that
// group g occupies stored depths [g * bs, g * bs + size_g).  One thread per
// original depth k: its rank among the earlier depths of its group gives its
// stored position g * bs + rank, and perm[position] = k.  The
// groups must have the block sizes (bs, the last one K - (KB - 1) * bs), as
// MatMulNBits' g_idx describes a permutation of whole blocks; a value outside
// [0, KB) or a group with too many depths sets MNB_ERR_INVALID_ARG in the
// device status word (so every group then has exactly its size).  Depths
// [K, Kpad) keep their place.
__global__ void gidx_perm_kernel(const int32_t* __restrict__ g_idx, int32_t* __restrict__ perm, Layout L,
                                 int* status) {
    const int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (k >= L.Kpad) return;
    if (k >= L.K) {
        perm[k] = (int32_t)k;
        return;
    }
    const int32_t g = g_idx[k];
    if (g < 0 || g >= L.KB) {
        set_status(status, 1 /* MNB_ERR_INVALID_ARG */);
        return;
    }
    int64_t rank = 0;
    for (int64_t j = 0; j < k; ++j) rank += g_idx[j] == g ? 1 : 0;
    const int64_t size = L.K - (int64_t)g * L.bs < L.bs ? L.K - (int64_t)g * L.bs : L.bs;
    if (rank >= size) {
        set_status(status, 1 /* MNB_ERR_INVALID_ARG */);
        return;
    }
    perm[(int64_t)g * L.bs + rank] = (int32_t)k;
}

// One thread per ORT byte.
__global__ void unpack_kernel(const uint8_t* __restrict__ packed, uint8_t* __restrict__ b_ort, Layout L,
                              int64_t nbytes, int* status) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i == 0) verify_header(packed - kHeaderBytes, L, status);
    if (i >= nbytes) return;
    const int64_t row_bytes = L.KB * L.blob;
    const int64_t n = i / row_bytes;
    const int64_t rem = i - n * row_bytes;
    const int64_t kb = rem / L.blob;
    const int64_t byte_in_blob = rem - kb * L.blob;
    const int per_byte = 8 / L.bits;
    uint32_t v = 0;
    for (int f = 0; f < per_byte; ++f) {
        const int64_t k = kb * L.bs + byte_in_blob * per_byte + f;
        v |= (uint32_t)packed_code(packed, L, n, k) << (f * L.bits);
    }
    b_ort[i] = (uint8_t)v;
}

// One thread per (n, k).
__global__ void dequant_kernel(const uint8_t* __restrict__ packed, const void* __restrict__ scales, int sdt,
                               const uint8_t* __restrict__ zp, float* __restrict__ w, Layout L, int* status) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i == 0) verify_header(packed - kHeaderBytes, L, status);
    if (i >= L.N * L.K) return;
    const int64_t n = i / L.K, k = i - n * L.K;
    const int64_t kb = k / L.bs;
    const int q = packed_code(packed, L, n, k);
    const int z = load_zp(zp, L, n, kb);
    const float s = load_f32(scales, n * L.KB + kb, sdt);
    w[i] = __fmul_rn(__fsub_rn((float)q, (float)z), s);
}

// Act-order prefill: X's depths put in the packed buffer's order, xp[m, j] = x[m, perm[j]] (16-bit
// activations), so that the tensor-core GEMM reads contiguous quantisation blocks.  A CTA takes rows in a
// grid-stride loop: the row is copied into shared memory with 16-byte loads, then each thread gathers 8 stored
// depths from there and writes them with one 16-byte store.  The permutation belongs to the packed weights, so
// a thread's first 8 entries are read once, before the dependency wait, and serve every row; X is read after it.
__device__ __forceinline__ void load_perm8(const int32_t* perm, int64_t i, int64_t K, int (&pk)[8]) {
    const int4 p0 = reinterpret_cast<const int4*>(perm)[2 * i];  // the permutation is 256-byte aligned
    const int4 p1 = reinterpret_cast<const int4*>(perm)[2 * i + 1];
    const int v[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) pk[e] = v[e] < 0 ? 0 : (v[e] >= K ? (int)K - 1 : v[e]);  // a bad pack reads in X
}

__device__ __forceinline__ uint4 gather8(const uint16_t* row, const int (&pk)[8]) {
    uint32_t h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = row[pk[e]];
    return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

__global__ void gather_kperm_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                    uint16_t* __restrict__ xp, int64_t M, int64_t K) {
    extern __shared__ __align__(16) uint16_t row[];
    const int64_t k8 = K / 8;
    const int64_t i0 = threadIdx.x;
    int pk0[8];
    if (i0 < k8) load_perm8(perm, i0, K, pk0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4* src = reinterpret_cast<const uint4*>(x + m * K);
        for (int64_t i = i0; i < k8; i += blockDim.x) reinterpret_cast<uint4*>(row)[i] = src[i];
        __syncthreads();
        uint4* dst = reinterpret_cast<uint4*>(xp + m * K);
        if (i0 < k8) dst[i0] = gather8(row, pk0);
        for (int64_t i = i0 + blockDim.x; i < k8; i += blockDim.x) {
            int pk[8];
            load_perm8(perm, i, K, pk);
            dst[i] = gather8(row, pk);
        }
        __syncthreads();  // the row buffer is reused
    }
}

unsigned blocks_for(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_pack(const uint8_t* b_ort, uint8_t* packed_hdr, const Layout& L, cudaStream_t s, int fmt) {
    header_kernel<<<1, 64, 0, s>>>(packed_hdr, L, fmt, 0);
    const int64_t words = (int64_t)(L.data_bytes() / 4);
    if (words > 0)
        pack_kernel<<<blocks_for(words, 256), 256, 0, s>>>(
            b_ort, reinterpret_cast<uint32_t*>(packed_hdr + kHeaderBytes), L, words, fmt, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_pack_gidx(const uint8_t* b_ort, const int32_t* g_idx, uint8_t* packed_hdr, const Layout& L,
                             cudaStream_t s) {
    int32_t* perm = reinterpret_cast<int32_t*>(packed_hdr + kHeaderBytes + L.data_bytes());
    header_kernel<<<1, 64, 0, s>>>(packed_hdr, L, kWfInt, 1);
    if (L.Kpad > 0) gidx_perm_kernel<<<blocks_for(L.Kpad, 256), 256, 0, s>>>(g_idx, perm, L, device_status_word());
    const int64_t words = (int64_t)(L.data_bytes() / 4);
    if (words > 0)
        pack_kernel<<<blocks_for(words, 256), 256, 0, s>>>(
            b_ort, reinterpret_cast<uint32_t*>(packed_hdr + kHeaderBytes), L, words, kWfInt, perm);
    return cudaGetLastError();
}

cudaError_t launch_gather_kperm(const void* x, const int32_t* perm, void* xp, int64_t M, const Layout& L,
                                bool pdl, cudaStream_t s) {
    if (M <= 0 || L.K <= 0) return cudaSuccess;
    const size_t smem = (size_t)L.K * 2;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(gather_kperm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    // one 16-byte output per thread for K <= 8192: 32..1024 threads
    const int64_t k8 = L.K / 8;
    const unsigned threads = (unsigned)(k8 >= 1024 ? 1024 : ((k8 + 31) / 32) * 32);
    cfg.gridDim = dim3((unsigned)(M < 65535 ? M : 65535));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gather_kperm_kernel, static_cast<const uint16_t*>(x), perm,
                              static_cast<uint16_t*>(xp), M, L.K);
}

cudaError_t launch_unpack(const uint8_t* packed, uint8_t* b_ort, const Layout& L, cudaStream_t s) {
    const int64_t nbytes = L.N * L.KB * L.blob;
    if (nbytes > 0) unpack_kernel<<<blocks_for(nbytes, 256), 256, 0, s>>>(packed, b_ort, L, nbytes, device_status_word());
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t* packed, const void* scales, int scale_dtype, const uint8_t* zp,
                           float* w, const Layout& L, cudaStream_t s) {
    const int64_t n = L.N * L.K;
    if (n > 0) dequant_kernel<<<blocks_for(n, 256), 256, 0, s>>>(packed, scales, scale_dtype, zp, w, L,
                                                                  device_status_word());
    return cudaGetLastError();
}

}  // namespace mnb
