/*
 * CPU oracle for block-quantized weight-only matmul (MatMulNBits).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the bench use it.  It shares no code, header, table or helper with the CUDA
 * library.  It is deliberately plain and slow: element-by-element unpacking,
 * dequantisation in f32 exactly as the operator defines it, and accumulation
 * in f64.  The only parallelism is an OpenMP loop over independent outputs,
 * which does not change any result.
 *
 * Sources followed (page title, function):
 *  - onnx-runtime-ep-cpu 0.1.0-dev.5, src/kernels/matmul_nbits.rs:
 *      module doc (B is [N, ceil(K/bs), bs*bits/8], least-significant bits
 *      first), `MatMulNBitsFactory::create` (bits in {2,4,8}, bs a power of
 *      two >= 16), `MatMulNBitsKernel::execute` (shapes of scales,
 *      zero_points [N, ceil(KB*bits/8)], g_idx [K] or [KB*bs], bias [N] added
 *      after the product), `dequantize_nbits_value` (code and zero-point
 *      extraction, default zero point 2^(bits-1), w = (q - zp) * scale in
 *      f32), `MatMulNBitsKernel::dequantize_weight` (grouped path: the code
 *      stays at its block position, scale and zero point follow g_idx),
 *      `quantize_activation_signed` (per-K-block symmetric int8 activations,
 *      scale = max|x| / 127, round to nearest), `int4_dot_row_scalar` and
 *      `int8_row` (exact integer block dot, then one f32 rescale by
 *      weight scale * activation scale).
 *  - rlx-cpu 0.2.13, src/thunk/ops/quant.rs: `dequant_matmul_int4`
 *      ((nibble - z) * s, low nibble first) corroborates the dequant form;
 *      the per-channel quantize thunk rounds with Rust's f32::round (half
 *      away from zero), which is the rounding used for int8 activations;
 *      `fp8_e4m3_to_f32`, `fp8_e5m2_to_f32`, `dequant_matmul_fp8` and
 *      `dequant_matmul_nvfp4` define the FP8 and NVFP4 weight formats.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- the storage layout, one element at a time ------------------------- */

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Code q[n, k] of B stored as [N, KB, bs*bits/8] bytes, LSB first.
 * The element at position i inside block kb sits at bit i*bits of the
 * block's blob; byte = blob[(i*bits)/8], shift = (i*bits)%8. */
int oracle_code(const uint8_t* b, int64_t N, int64_t K, int bits, int bs, int64_t n, int64_t k) {
    (void)N;
    int64_t kblocks = ceil_div(K, bs);
    int64_t blob = (int64_t)bs * bits / 8;
    int64_t kb = k / bs;
    int64_t within = k % bs;
    int64_t bit = within * bits;
    uint8_t byte = b[(n * kblocks + kb) * blob + bit / 8];
    int mask = (bits == 8) ? 0xFF : ((1 << bits) - 1);
    return (byte >> (bit % 8)) & mask;
}

/* Zero point of (n, group g): packed at `bits` width, LSB first, in a row of
 * ceil(KB*bits/8) bytes; absent => 2^(bits-1). */
int oracle_zero_point(const uint8_t* zp, int64_t N, int64_t K, int bits, int bs, int64_t n, int64_t g) {
    (void)N;
    if (zp == NULL) return 1 << (bits - 1);
    int64_t kblocks = ceil_div(K, bs);
    int64_t row_bytes = ceil_div(kblocks * bits, 8);
    int64_t bit = g * bits;
    int mask = (bits == 8) ? 0xFF : ((1 << bits) - 1);
    return (zp[n * row_bytes + bit / 8] >> (bit % 8)) & mask;
}

/* Group (scale / zero-point column) of depth k: g_idx[k] when given,
 * else the block k / bs. */
static int64_t group_of(const int32_t* g_idx, int bs, int64_t k) {
    return g_idx ? (int64_t)g_idx[k] : k / bs;
}

/* w[n, k] = fl32( (f32(q) - f32(zp)) * f32(scale) ), one f32 rounding
 * (the subtraction of two small integers is exact).  Scales arrive already
 * widened to f32 ([N, KB] row-major).  g_idx may be NULL. */
float oracle_weight(const uint8_t* b, const float* scales, const uint8_t* zp, const int32_t* g_idx,
                    int64_t N, int64_t K, int bits, int bs, int64_t n, int64_t k) {
    int64_t kblocks = ceil_div(K, bs);
    int64_t g = group_of(g_idx, bs, k);
    int q = oracle_code(b, N, K, bits, bs, n, k);
    int z = oracle_zero_point(zp, N, K, bits, bs, n, g);
    volatile float diff = (float)q - (float)z;
    volatile float w = diff * scales[n * kblocks + g];
    return w;
}

/* Full dequantised weight in [N, K] row-major f32. */
void oracle_dequantize(const uint8_t* b, const float* scales, const uint8_t* zp, const int32_t* g_idx,
                       int64_t N, int64_t K, int bits, int bs, float* w) {
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = oracle_weight(b, scales, zp, g_idx, N, K, bits, bs, n, k);
}

/* One output: y = sum_k f64(x[m,k]) * f64(w[n,k]) (+ bias[n]); also returns
 * sum_k |x[m,k] * w[n,k]|, the scale of the accumulation error bound. */
static void one_output(const double* x, const uint8_t* b, const float* scales, const uint8_t* zp,
                       const int32_t* g_idx, const double* bias, int64_t N, int64_t K, int bits, int bs,
                       int64_t m, int64_t n, double* y, double* absdot) {
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double w = (double)oracle_weight(b, scales, zp, g_idx, N, K, bits, bs, n, k);
        double p = x[m * K + k] * w;
        acc += p;
        mag += fabs(p);
    }
    if (bias) {
        acc += bias[n];
        mag += fabs(bias[n]);
    }
    *y = acc;
    if (absdot) *absdot = mag;
}

/* Y[M, N] in f64.  x is [M, K] already widened (exactly) to f64; bias is
 * [N] widened to f64 or NULL. */
void oracle_matmul(const double* x, const uint8_t* b, const float* scales, const uint8_t* zp,
                   const int32_t* g_idx, const double* bias, int64_t M, int64_t N, int64_t K, int bits,
                   int bs, double* y, double* absdot) {
    int64_t n;
#pragma omp parallel for schedule(dynamic, 4)
    for (n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m)
            one_output(x, b, scales, zp, g_idx, bias, N, K, bits, bs, m, n, &y[m * N + n],
                       absdot ? &absdot[m * N + n] : NULL);
}

/* Selected outputs (ms[i], ns[i]), i < P, for sampled checks at full size. */
void oracle_matmul_points(const double* x, const uint8_t* b, const float* scales, const uint8_t* zp,
                          const int32_t* g_idx, const double* bias, int64_t M, int64_t N, int64_t K,
                          int bits, int bs, const int64_t* ms, const int64_t* ns, int64_t P, double* y,
                          double* absdot) {
    (void)M;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 8)
    for (i = 0; i < P; ++i)
        one_output(x, b, scales, zp, g_idx, bias, N, K, bits, bs, ms[i], ns[i], &y[i],
                   absdot ? &absdot[i] : NULL);
}

/* ---- int8-activation variant ------------------------------------------- */

/* Per (m, K-block) symmetric int8 quantisation of f32 activations:
 * amax = max |x| over the block's valid depths, s_a = amax / 127 (f32),
 * qa = clamp(round_half_away(x / s_a), -127, 127) computed in f32.
 * An all-zero block gets s_a = 0 and codes 0.  Depths past K (the padded
 * tail of the last block) get code 0.  qa is [M, KB*bs], sa is [M, KB]. */
void oracle_quantize_act(const float* x, int64_t M, int64_t K, int bs, int8_t* qa, float* sa) {
    int64_t kblocks = ceil_div(K, bs);
    int64_t kpad = kblocks * bs;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < kblocks; ++kb) {
            int64_t k0 = kb * bs;
            int64_t k1 = k0 + bs < K ? k0 + bs : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                float a = fabsf(x[m * K + k]);
                if (a > amax) amax = a;
            }
            volatile float s = amax / 127.0f;
            sa[m * kblocks + kb] = s;
            for (int64_t k = k0; k < k0 + bs; ++k) {
                int8_t code = 0;
                if (k < K && amax > 0.0f) {
                    volatile float r = x[m * K + k] / s;
                    float rr = roundf(r);
                    if (rr > 127.0f) rr = 127.0f;
                    if (rr < -127.0f) rr = -127.0f;
                    code = (int8_t)rr;
                }
                qa[m * kpad + k] = code;
            }
        }
    }
}

/* y[m, n] = sum_kb f64(dot_i32) * f64(fl32(s_w * s_a)) (+ bias[n]), with
 * dot_i32 = sum over the block of qa * (q - zp) in exact integers.
 * absdot[m, n] = sum_k |x_hat * w| with x_hat = qa * s_a (the magnitude of the
 * products of the quantised activations).  Only plain blocks (no g_idx). */
void oracle_matmul_a8(const int8_t* qa, const float* sa, const uint8_t* b, const float* scales,
                      const uint8_t* zp, const double* bias, int64_t M, int64_t N, int64_t K, int bits,
                      int bs, double* y, double* absdot) {
    int64_t kblocks = ceil_div(K, bs);
    int64_t kpad = kblocks * bs;
    int64_t n;
#pragma omp parallel for schedule(dynamic, 4)
    for (n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, mag = 0.0;
            for (int64_t kb = 0; kb < kblocks; ++kb) {
                int z = oracle_zero_point(zp, N, K, bits, bs, n, kb);
                int64_t dot = 0;
                int64_t absint = 0;
                for (int64_t k = kb * bs; k < kb * bs + bs && k < K; ++k) {
                    int q = oracle_code(b, N, K, bits, bs, n, k);
                    int64_t t = (int64_t)qa[m * kpad + k] * (int64_t)(q - z);
                    dot += t;
                    absint += t < 0 ? -t : t;
                }
                volatile float sw = scales[n * kblocks + kb];
                volatile float sprod = sw * sa[m * kblocks + kb];
                acc += (double)(int32_t)dot * (double)sprod;
                mag += (double)absint * fabs((double)sa[m * kblocks + kb] * (double)sw);
            }
            if (bias) {
                acc += bias[n];
                mag += fabs(bias[n]);
            }
            y[m * N + n] = acc;
            if (absdot) absdot[m * N + n] = mag;
        }
    }
}

/* ---- other weight formats: FP8 and NVFP4 ---------------------------------
 * rlx-cpu 0.2.13, src/thunk/ops/quant.rs: fp8_e4m3_to_f32, fp8_e5m2_to_f32,
 * dequant_matmul_fp8, dequant_matmul_nvfp4.  Weights are stored [K, N]
 * (element (p, j) at flat index p * N + j). */

/* A minifloat with `ebits` exponent bits (bias 2^(ebits-1) - 1) and `mbits`
 * mantissa bits, as the page decodes FP8: exponent 0 is subnormal
 * (mant * 2^(1 - bias - mbits)); the all-ones exponent is infinity for a zero
 * mantissa and NaN otherwise (IEEE style). */
static float ieee_minifloat(unsigned code, int ebits, int mbits) {
    unsigned sign = (code >> (ebits + mbits)) & 1u;
    unsigned e = (code >> mbits) & ((1u << ebits) - 1u);
    unsigned m = code & ((1u << mbits) - 1u);
    int bias = (1 << (ebits - 1)) - 1;
    double v;
    if (e == 0) {
        v = ldexp((double)m, 1 - bias - mbits);
    } else if (e == (1u << ebits) - 1u) {
        if (m != 0) return NAN;
        v = INFINITY;
    } else {
        v = ldexp(1.0 + ldexp((double)m, -mbits), (int)e - bias);
    }
    return (float)(sign ? -v : v);
}

/* fp8_e4m3_to_f32 as the page defines it (exponent 15 is inf / NaN). */
float oracle_fp8_e4m3(int code) { return ieee_minifloat((unsigned)code & 0xFFu, 4, 3); }

/* fp8_e5m2_to_f32 as the page defines it. */
float oracle_fp8_e5m2(int code) { return ieee_minifloat((unsigned)code & 0xFFu, 5, 2); }

/* NVFP4 block scale.  The page calls fp8_e4m3_scale_to_f32 without printing
 * it; read as the OCP E4M3 format NVFP4 scales are stored in ("fn": no
 * infinity, exponent 15 is a normal binade except mantissa 7, which is NaN;
 * largest value 448). */
float oracle_e4m3fn_scale(int code) {
    unsigned c = (unsigned)code & 0xFFu;
    unsigned e = (c >> 3) & 0xFu, m = c & 7u;
    if (e == 15u && m == 7u) return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, (int)e - 7);
    return (float)((c & 0x80u) ? -v : v);
}

/* FP4 E2M1 weight code.  The page calls fp4_e2m1_to_f32 without printing it;
 * read as OCP E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit, no
 * infinity or NaN: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
float oracle_e2m1(int nibble) {
    unsigned c = (unsigned)nibble & 0xFu;
    unsigned e = (c >> 1) & 3u, m = c & 1u;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)e - 1);
    return (float)((c & 8u) ? -v : v);
}

/* dequant_matmul_fp8: y[i, j] = sum_p x[i, p] * w(p, j) * s[j], w the FP8 code
 * at w8[p * N + j] decoded as e4m3 (e5m2 = 0) or e5m2, s[j] = scales[j] or 1
 * when scales is NULL (the page's missing-scale default).  f64 accumulation;
 * absdot = sum_p |x * w * s|. */
void oracle_matmul_fp8(const double* x, const uint8_t* w8, const float* scales, int64_t M, int64_t K, int64_t N,
                       int e5m2, double* y, double* absdot) {
    int64_t j;
#pragma omp parallel for schedule(dynamic, 4)
    for (j = 0; j < N; ++j) {
        double s = scales ? (double)scales[j] : 1.0;
        for (int64_t i = 0; i < M; ++i) {
            double acc = 0.0, mag = 0.0;
            for (int64_t p = 0; p < K; ++p) {
                int code = w8[p * N + j];
                double w = e5m2 ? oracle_fp8_e5m2(code) : oracle_fp8_e4m3(code);
                double t = x[i * K + p] * w * s;
                acc += t;
                mag += fabs(t);
            }
            y[i * N + j] = acc;
            if (absdot) absdot[i * N + j] = mag;
        }
    }
}

/* The NVFP4 weight (p, j), formed in f32 as the page forms it:
 * e2m1(nibble) * e4m3(block scale) * global_scale, with the nibble at flat
 * index f = p * N + j (byte f / 2, low nibble when f is even) and the block
 * scale at scale8[(p / 16) * N + j]. */
float oracle_nvfp4_weight(const uint8_t* w4, const uint8_t* scale8, float global_scale, int64_t N, int64_t p,
                          int64_t j) {
    int64_t f = p * N + j;
    int nibble = (f & 1) ? (w4[f / 2] >> 4) : (w4[f / 2] & 0x0F);
    volatile float a = oracle_e2m1(nibble) * oracle_e4m3fn_scale(scale8[(p / 16) * N + j]);
    volatile float w = a * global_scale;
    return w;
}

/* dequant_matmul_nvfp4: y[i, j] = sum_p x[i, p] * w(p, j), f64 accumulation;
 * absdot = sum_p |x * w|. */
void oracle_matmul_nvfp4(const double* x, const uint8_t* w4, const uint8_t* scale8, float global_scale, int64_t M,
                         int64_t K, int64_t N, double* y, double* absdot) {
    int64_t j;
#pragma omp parallel for schedule(dynamic, 4)
    for (j = 0; j < N; ++j) {
        for (int64_t i = 0; i < M; ++i) {
            double acc = 0.0, mag = 0.0;
            for (int64_t p = 0; p < K; ++p) {
                double t = x[i * K + p] * (double)oracle_nvfp4_weight(w4, scale8, global_scale, N, p, j);
                acc += t;
                mag += fabs(t);
            }
            y[i * N + j] = acc;
            if (absdot) absdot[i * N + j] = mag;
        }
    }
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}
