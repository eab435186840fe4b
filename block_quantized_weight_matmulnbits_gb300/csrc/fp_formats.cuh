// Floating-point weight formats of rlx-cpu 0.2.13, src/thunk/ops/quant.rs
// (dequant_matmul_fp8, dequant_matmul_nvfp4; fp8_e4m3_to_f32,
// fp8_e5m2_to_f32), decoded exactly from their bit fields:
//   * FP8 E4M3 as the page decodes it: bias 7, exponent 0 subnormal
//     (m * 2^-9), exponent 15 infinity for a zero mantissa and NaN otherwise
//     (the page's IEEE-style rule, not the OCP "fn" variant);
//   * FP8 E5M2: bias 15, subnormals m * 2^-16, exponent 31 infinity / NaN;
//   * the NVFP4 block scale: OCP E4M3 ("fn": exponent 15 is a normal binade,
//     only 0x7F / 0xFF are NaN; the page calls a scale decoder it does not
//     print);
//   * the NVFP4 weight: OCP E2M1 (2 exponent bits, bias 1, 1 mantissa bit;
//     magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; the page calls a decoder it does
//     not print).
#pragma once

#include <cstdint>
#include <cmath>

namespace mnb {
namespace fpf {

__device__ __forceinline__ float make_f32(uint32_t sign, int exp2, uint32_t frac23) {
    // normal f32 with unbiased exponent exp2 (within the normal range) and 23-bit fraction
    return __uint_as_float((sign << 31) | ((uint32_t)(exp2 + 127) << 23) | frac23);
}

// FP8 E4M3 as the page decodes it.
__device__ __forceinline__ float e4m3_page(uint32_t c) {
    const uint32_t s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
    if (e == 15u) return m ? __uint_as_float(0x7FC00000u) : __uint_as_float((s << 31) | 0x7F800000u);
    if (e == 0u) {
        const float v = (float)m * 0.001953125f;  // m * 2^-9, exact
        return s ? -v : v;
    }
    return make_f32(s, (int)e - 7, m << 20);
}

// FP8 E5M2.
__device__ __forceinline__ float e5m2(uint32_t c) {
    const uint32_t s = (c >> 7) & 1u, e = (c >> 2) & 31u, m = c & 3u;
    if (e == 31u) return m ? __uint_as_float(0x7FC00000u) : __uint_as_float((s << 31) | 0x7F800000u);
    if (e == 0u) {
        const float v = (float)m * 1.52587890625e-05f;  // m * 2^-16, exact
        return s ? -v : v;
    }
    return make_f32(s, (int)e - 15, m << 21);
}

// OCP E4M3 ("fn") block scale of NVFP4.
__device__ __forceinline__ float e4m3fn(uint32_t c) {
    const uint32_t s = (c >> 7) & 1u, e = (c >> 3) & 15u, m = c & 7u;
    if (e == 15u && m == 7u) return __uint_as_float(0x7FC00000u);
    if (e == 0u) {
        const float v = (float)m * 0.001953125f;
        return s ? -v : v;
    }
    return make_f32(s, (int)e - 7, m << 20);
}

// OCP E2M1 weight nibble.
__device__ __forceinline__ float e2m1(uint32_t c) {
    const uint32_t s = (c >> 3) & 1u, e = (c >> 1) & 3u, m = c & 1u;
    if (e == 0u) {
        const float v = m ? 0.5f : 0.f;
        return s ? -v : v;
    }
    return make_f32(s, (int)e - 1, m << 22);
}

}  // namespace fpf
}  // namespace mnb
