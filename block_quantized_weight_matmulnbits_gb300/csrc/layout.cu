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
__global__ void pack_kernel(const uint8_t* __restrict__ b_ort, uint32_t* __restrict__ out, Layout L,
                            int64_t words, int fmt) {
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
            if (n < L.N && k < L.Kpad) word |= (uint32_t)ort_code(b_ort, L, n, k) << (f * L.bits);
        } else if (n < L.N && k < L.K) {
            word |= (uint32_t)kn_code(b_ort, L, fmt, n, k) << (f * L.bits);
        }
    }
    out[wi] = word;
}

__global__ void header_kernel(uint8_t* hdr, Layout L, int fmt) {
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
    }
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

unsigned blocks_for(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_pack(const uint8_t* b_ort, uint8_t* packed_hdr, const Layout& L, cudaStream_t s, int fmt) {
    header_kernel<<<1, 64, 0, s>>>(packed_hdr, L, fmt);
    const int64_t words = (int64_t)(L.data_bytes() / 4);
    if (words > 0)
        pack_kernel<<<blocks_for(words, 256), 256, 0, s>>>(
            b_ort, reinterpret_cast<uint32_t*>(packed_hdr + kHeaderBytes), L, words, fmt);
    return cudaGetLastError();
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
