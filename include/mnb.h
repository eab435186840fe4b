/*
 * mnb.h -- C ABI of libmnb, block-quantized weight-only matmul (MatMulNBits)
 * for NVIDIA GB300 (sm_103a).
 *
 *     Y[M, N] = X[M, K] . dequant(B)^T
 *
 * The operation and its storage format are those of the ONNX Runtime
 * com.microsoft::MatMulNBits operator as restated by onnx-runtime-ep-cpu
 * 0.1.0-dev.5, src/kernels/matmul_nbits.rs (module doc; MatMulNBitsFactory::
 * create; MatMulNBitsKernel::execute; fn dequantize_nbits_value):
 *
 *   - B is uint8 [N, KB, blob] with KB = ceil(K / block_size) and
 *     blob = block_size * bits / 8.  Codes are packed least-significant bits
 *     first: element i of block kb of row n sits at bit i*bits of that blob.
 *   - scales is [N, KB] (f32, f16 or bf16), one per (row, K-block).
 *   - zero_points is uint8 [N, ceil(KB * bits / 8)], packed at `bits` width,
 *     least-significant bits first, or NULL, in which case every zero point
 *     is 2^(bits-1) (8 for 4-bit, 128 for 8-bit, 2 for 2-bit).
 *   - w[n, k] = (q[n, k] - zp[n, k / bs]) * scale[n, k / bs], evaluated in f32.
 *   - bits is 2, 4 or 8; block_size is a power of two >= 16.
 *   - When K is not a multiple of block_size the last block is partial; its
 *     codes past K are ignored.
 *
 * Conventions shared by every entry point:
 *   - Pointers documented as "device" must point to memory the current CUDA
 *     device can access (cudaMalloc, or a torch CUDA tensor's data_ptr()).
 *     The caller owns every buffer; the library allocates no device memory
 *     and keeps no state between calls other than a per-device status word
 *     and the file-scope device arrays of mnb_matmul_a8_static and
 *     mnb_matmul_host_io.
 *   - All work is enqueued on `stream` (NULL = the legacy default stream) and
 *     is asynchronous.  A returned MNB_OK means the arguments were valid and
 *     the launch was accepted; faults during execution surface at the
 *     caller's next synchronisation, and kernel-detected problems (a packed
 *     buffer whose header does not match, a bounded wait that ran out) are
 *     recorded in the device status word read by mnb_get_device_error().
 *   - Arguments are validated on the host before anything is launched.  A
 *     non-OK status means nothing was enqueued.  The library never aborts,
 *     exits or prints unless MNB_LOG=1 is set in the environment.
 *   - Device pointers must be 16-byte aligned unless stated otherwise.
 */
#ifndef MNB_H_
#define MNB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MNB_ABI_VERSION 1

/* Symbols of the shared library; everything else in it is hidden. */
#if defined(__GNUC__)
#define MNB_API __attribute__((visibility("default")))
#else
#define MNB_API
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA headers. */
typedef struct CUstream_st* mnb_stream_t;

typedef enum mnb_status {
    MNB_OK = 0,
    MNB_ERR_INVALID_ARG = 1,      /* a pointer, size, dtype or alignment is invalid */
    MNB_ERR_UNSUPPORTED = 2,      /* valid for the operator, but no kernel here handles it */
    MNB_ERR_CUDA = 3,             /* a CUDA runtime call failed (launch, attribute query) */
    MNB_ERR_NO_MEM = 4,           /* a caller-provided buffer is too small */
    MNB_ERR_TIMEOUT = 5,          /* (device status) a bounded wait inside a kernel ran out */
    MNB_ERR_LAYOUT_MISMATCH = 6   /* (device status) packed buffer header does not match N, K, bits, bs */
} mnb_status;

typedef enum mnb_dtype { MNB_F32 = 0, MNB_F16 = 1, MNB_BF16 = 2 } mnb_dtype;

/* Kernel families.  MNB_KERNEL_AUTO lets the library choose from M, dtypes and
 * accuracy level; the others force one (tests and benchmarks).  Forcing a
 * kernel that cannot handle the call returns MNB_ERR_UNSUPPORTED. */
typedef enum mnb_kernel {
    MNB_KERNEL_AUTO = 0,
    MNB_KERNEL_GEMV = 1,      /* M == 1 decode GEMV, any X dtype, CUDA cores, TMA-streamed weights */
    MNB_KERNEL_GEMV_MMA = 2,  /* 1 <= M <= 16, bf16/f16 X, warp-level tensor-core MMA on registers,
                                 TMA-streamed weights (the decode default for bf16/f16 X) */
    MNB_KERNEL_GEMM_TC = 3,   /* M >= 1 prefill GEMM, bf16/f16 X, tcgen05 + TMEM + TMA */
    MNB_KERNEL_GENERIC = 4,   /* any shape and dtype, CUDA cores, shared-memory tiles */
    MNB_KERNEL_GEMV_I8 = 5    /* int8-activation path (accuracy_level 4), integer dot products */
} mnb_kernel;

/* Flags of mnb_matmul_args.flags. */
/* MNB_FLAG_PDL: launch with programmatic dependent launch.  The kernel starts
 * streaming the weights, scales, zero points and bias before the preceding
 * kernel on the stream has finished (its X and Y accesses still wait for it),
 * and lets the next kernel start as its own blocks retire.  Use it only when
 * the preceding kernel does not write packed_b, scales, zero_points or bias
 * (true for constant model weights).  Honoured by MNB_KERNEL_GEMV_MMA,
 * MNB_KERNEL_GEMV_I8 and the FP8 / NVFP4 decode GEMVs (mnb_matmul_fp_ex);
 * other kernels ignore it. */
#define MNB_FLAG_PDL 1
/* MNB_FLAG_KPERM: packed_b comes from mnb_pack_weights_gidx (act-order); the
 * permutation stored in it replaces g_idx, which must be NULL.  Not with
 * accuracy_level 4 (MNB_ERR_UNSUPPORTED). */
#define MNB_FLAG_KPERM 2

/* ---- weight layout (one-time re-tiling) -------------------------------- */

/* Bytes of the packed weight buffer for (N, K, bits, block_size), or 0 if the
 * arguments are invalid.  The buffer is a 256-byte header followed by the
 * codes of B re-tiled into 512-byte tiles of 16 rows, each tile holding one
 * 16-byte slice per lane of a 32-lane warp; the code values are unchanged,
 * so packing is a pure permutation (plus zero padding of the row count to a
 * multiple of 16 and of the padded K to a multiple of 256/bits). */
MNB_API size_t mnb_packed_size(int64_t N, int64_t K, int bits, int block_size);

/* Re-tile B (ORT layout, device, [N, KB, blob] uint8, any alignment) into
 * packed_b (device, 256-byte aligned, packed_bytes >= mnb_packed_size()).
 * Writes the header and every byte of the buffer.  MNB_ERR_NO_MEM if
 * packed_bytes is too small.  Follows the storage rule of
 * onnx-runtime-ep-cpu matmul_nbits.rs (module doc, fn dequantize_nbits_value). */
MNB_API mnb_status mnb_pack_weights(const uint8_t* b_ort, void* packed_b, size_t packed_bytes,
                            int64_t N, int64_t K, int bits, int block_size, mnb_stream_t stream);

/* Act-order (g_idx) weights.  MatMulNBits' g_idx[k] names the quantisation
 * block (scale and zero-point column) of depth k while the code keeps its
 * place (onnx-runtime-ep-cpu matmul_nbits.rs, MatMulNBitsKernel::
 * dequantize_weight).  mnb_pack_weights_gidx re-tiles B with its depths sorted
 * by group (stable), so that group g occupies the stored depths of block g,
 * and stores that permutation (int32, one entry per padded depth) after the
 * tiles.  A call with MNB_FLAG_KPERM then runs the decode GEMV on it, gathering
 * X through the permutation (M <= 8), the tensor-core prefill GEMM after a
 * gather of X into the workspace (M > 8, see mnb_workspace_size_ex), or the
 * generic kernel for other shapes, with no g_idx argument.
 *   g_idx   device int32 [K] (4-byte aligned), values in [0, KB), each block
 *           holding exactly its depths (bs, the last K - (KB - 1) * bs): a
 *           permutation of whole blocks, as act-order quantisers write it.
 *           Another g_idx sets MNB_ERR_INVALID_ARG in the device status word
 *           (the buffer is then unusable); it stays usable with the plain
 *           mnb_pack_weights and g_idx in mnb_matmul_ex (generic kernel).
 * The size is mnb_packed_size_gidx(); unpack and dequantize take only buffers
 * from mnb_pack_weights.  The header records the act-order pack, so a call
 * whose MNB_FLAG_KPERM does not match it sets MNB_ERR_LAYOUT_MISMATCH. */
MNB_API size_t mnb_packed_size_gidx(int64_t N, int64_t K, int bits, int block_size);
MNB_API mnb_status mnb_pack_weights_gidx(const uint8_t* b_ort, const int32_t* g_idx, void* packed_b,
                                 size_t packed_bytes, int64_t N, int64_t K, int bits, int block_size,
                                 mnb_stream_t stream);

/* Inverse of mnb_pack_weights: write the ORT-layout bytes of B (device,
 * [N, KB, blob] uint8) back from packed_b.  pack followed by unpack returns
 * the original bytes exactly, padding codes of a partial last block included. */
MNB_API mnb_status mnb_unpack_codes(const void* packed_b, uint8_t* b_ort, int64_t N, int64_t K, int bits,
                            int block_size, mnb_stream_t stream);

/* Dequantised weight w_nk (device, [N, K] f32, row-major, 4-byte aligned):
 * w = (f32(q) - f32(zp)) * f32(scale), one f32 rounding, bit-identical to
 * onnx-runtime-ep-cpu matmul_nbits.rs fn dequantize_nbits_value.  scales is
 * device [N, KB] of scale_dtype (natural alignment); zero_points may be NULL. */
MNB_API mnb_status mnb_dequantize(const void* packed_b, const void* scales, const uint8_t* zero_points,
                          float* w_nk, int64_t N, int64_t K, int bits, int block_size,
                          mnb_dtype scale_dtype, mnb_stream_t stream);

/* ---- the matmul -------------------------------------------------------- */

/* Y = X . dequant(B)^T.
 *   x           device [M, K] act_dtype, row-major (16-byte aligned)
 *   packed_b    device, written by mnb_pack_weights for the same N, K, bits, block_size
 *   scales      device [N, KB] scale_dtype (natural alignment)
 *   zero_points device [N, ceil(KB*bits/8)] uint8, or NULL (=> 2^(bits-1))
 *   y           device [M, N] out_dtype, row-major (16-byte aligned)
 * Accumulation is in f32 (fp32 accumulator, f32 or exact-integer partial
 * products); the result is rounded once to out_dtype with round-to-nearest-even.
 * The reduction order is fixed for a given launch configuration, so repeated
 * calls give bit-identical results.  M == 0 is a no-op. */
MNB_API mnb_status mnb_matmul(const void* x, const void* packed_b, const void* scales,
                      const uint8_t* zero_points, void* y, int64_t M, int64_t N, int64_t K, int bits,
                      int block_size, mnb_dtype act_dtype, mnb_dtype out_dtype, mnb_dtype scale_dtype,
                      mnb_stream_t stream);

/* Extended call: everything of mnb_matmul plus
 *   g_idx          device int32 [K] or NULL: group (scale/zero-point column) of
 *                  each depth, each in [0, KB) (onnx-runtime-ep-cpu matmul_nbits.rs,
 *                  MatMulNBitsKernel::dequantize_weight, grouped path).  The kernel
 *                  checks every value: a depth whose group is outside [0, KB)
 *                  sets MNB_ERR_INVALID_ARG in the device status word and the call
 *                  writes no element of Y.  Only MNB_KERNEL_GENERIC handles g_idx.
 *   bias           device [N] of bias_dtype or NULL, added after the product
 *                  (MatMulNBitsKernel::execute).
 *   accuracy_level 0..3: float path.  4: activations quantised per K-block to
 *                  int8 (scale = max|x|/127, round half away from zero), exact
 *                  integer block dot, then one f32 rescale by
 *                  f32(scale * s_a) (fn quantize_activation_signed, fn int8_row,
 *                  int8_matmul_amx).  M <= 16 runs the int8 GEMV (exact integer
 *                  block dots); larger M the tensor-core GEMM in tf32 over the
 *                  quantised activations code * s_a and the weights (q - zp) *
 *                  scale, each rounded to tf32 (relative error <= 2^-11 per
 *                  operand, inside the per-element bound).  Needs workspace.
 *   workspace      device scratch of at least mnb_workspace_size() bytes
 *                  (256-byte aligned) or NULL when that size is 0.
 *   kernel         MNB_KERNEL_AUTO or a forced family.
 *   flags          MNB_FLAG_* (0 for none). */
typedef struct mnb_matmul_args {
    const void* x;
    const void* packed_b;
    const void* scales;
    const uint8_t* zero_points;
    const int32_t* g_idx;
    const void* bias;
    void* y;
    int64_t M, N, K;
    int bits;
    int block_size;
    mnb_dtype act_dtype;
    mnb_dtype out_dtype;
    mnb_dtype scale_dtype;
    mnb_dtype bias_dtype;
    int accuracy_level;
    void* workspace;
    size_t workspace_bytes;
    mnb_kernel kernel;
    mnb_stream_t stream;
    int flags;  /* MNB_FLAG_* */
} mnb_matmul_args;

MNB_API mnb_status mnb_matmul_ex(const mnb_matmul_args* args);

/* Scratch bytes mnb_matmul_ex needs for this call (0 for the float path). */
MNB_API size_t mnb_workspace_size(int64_t M, int64_t N, int64_t K, int bits, int block_size, int accuracy_level);

/* The same for a call with these MNB_FLAG_* flags: with MNB_FLAG_KPERM and
 * M > 8 the act-order prefill needs X in the pack's depth order,
 * ceil256(M * K * 2) bytes (bf16 / f16 X).  Given that workspace, such a call
 * gathers X into it and runs the tensor-core prefill GEMM; without it, the
 * generic kernel (a forced MNB_KERNEL_GEMM_TC returns MNB_ERR_NO_MEM).  The
 * gather holds one row of X in shared memory, so K * 2 bytes must fit in a
 * CTA's opt-in shared memory (K up to about 116000 on this part); longer rows
 * take the generic kernel (a forced MNB_KERNEL_GEMM_TC returns
 * MNB_ERR_UNSUPPORTED). */
MNB_API size_t mnb_workspace_size_ex(int64_t M, int64_t N, int64_t K, int bits, int block_size,
                             int accuracy_level, int flags);

/* Per-(row, K-block) int8 activation quantisation on its own (the first step
 * of accuracy_level 4): qa device int8 [M, KB*bs] (tail past K zero), sa
 * device f32 [M, KB].  Bit-identical to the definition in the mnb_matmul_ex
 * comment above. */
MNB_API mnb_status mnb_quantize_activations(const void* x, int8_t* qa, float* sa, int64_t M, int64_t K,
                                    int block_size, mnb_dtype act_dtype, mnb_stream_t stream);

/* int8-activation matmul (accuracy level 4) that allocates nothing and takes
 * no workspace: for callers that cannot call cudaMalloc.  No counterpart on
 * the pages; an addition to the boundary.  Arguments as mnb_matmul (device
 * pointers, ORT layouts); zero_points may be NULL.
 *   Scratch: a file-scope device array of MNB_A8_STATIC_SCRATCH_BYTES (1 MiB)
 *   per device holds the quantised activations and their block scales
 *   (mnb_workspace_size(M, N, K, bits, block_size, 4) bytes).  Calls that
 *   need more return MNB_ERR_NO_MEM without launching.  Nothing in it needs
 *   to start at zero: the quantisation kernel writes every byte the GEMV
 *   reads.
 *   Set-up: the first call in a CUDA context (that is, on a device, with
 *   that device current) looks the array's device address up with
 *   cudaGetSymbolAddress and caches it for that context; make that first
 *   call outside stream capture.  A context created later (after a device
 *   reset, say) gets its own lookup.
 *   Concurrency: calls that overlap on the same device (different streams,
 *   threads or graphs in flight together) share the array and race; calls
 *   ordered on one stream are safe.
 * Returns the statuses of mnb_matmul_ex with accuracy_level 4. */
#define MNB_A8_STATIC_SCRATCH_BYTES (1u << 20)
MNB_API mnb_status mnb_matmul_a8_static(const void* x, const void* packed_b, const void* scales,
                                        const uint8_t* zero_points, void* y, int64_t M, int64_t N, int64_t K,
                                        int bits, int block_size, mnb_dtype act_dtype, mnb_dtype out_dtype,
                                        mnb_dtype scale_dtype, mnb_stream_t stream);

/* Grouped (mixture-of-experts) MatMulNBits, one launch over all experts:
 *   Y[t, s, :] = X_row(t, s) . dequant(B_{ids[t, s]})^T   (0 <= t < T, 0 <= s < S)
 * This is ggml's MUL_MAT_ID as the SpacemiT backend computes it (toy 0.8.0,
 * data/vendor/ggml/src/ggml-cpu/spacemit/ime.cpp, forward_mul_mat_id:
 * (slot, token) rows grouped by the expert they select, in ascending
 * token-then-slot order, each group one product with that expert's matrix)
 * and rlx's grouped dequant matmul (rlx-cpu 0.2.13, src/thunk/ops/quant.rs,
 * exec_dequant_grouped_mat_mul_gguf: one expert per row, S = 1).
 *   x           device [T, K] (x_per_slot = 0: one activation row per token,
 *               shared by its S slots) or [T, S, K] (x_per_slot = 1), bf16
 *               or f16 (f32 is MNB_ERR_UNSUPPORTED), 16-byte aligned.
 *   ids         device int32 [T, S]: the expert of each (token, slot).
 *   packed_b    device, 256-byte aligned: E packed weights back to back, each
 *               mnb_packed_size(N, K, bits, block_size) bytes as written by
 *               mnb_pack_weights from that expert's ORT bytes.
 *   scales      device [E, N, KB] of scale_dtype.
 *   zero_points device uint8 [E, N, ceil(KB*bits/8)] or NULL (default
 *               2^(bits-1) for every expert).
 *   y           device [T, S, N] of out_dtype, 16-byte aligned.
 * Calls with T*S <= 8 run the K-chunk decode schedule over the selected
 * experts' row tiles end to end; larger calls the per-tile kernel.
 * The weights of experts that no pair selects are not read.  Limits:
 * E <= 1024 and T*S <= 4096 (MNB_ERR_UNSUPPORTED beyond).  An id outside
 * [0, E) is not checked on the host (ids live on the device): its Y row is
 * left unwritten and the device status word becomes MNB_ERR_INVALID_ARG
 * (read it with mnb_get_device_error).  T == 0 returns MNB_OK. */
MNB_API mnb_status mnb_matmul_grouped(const void* x, const int32_t* ids, const void* packed_b, const void* scales,
                                      const uint8_t* zero_points, void* y, int64_t T, int64_t S, int64_t E,
                                      int x_per_slot, int64_t N, int64_t K, int bits, int block_size,
                                      mnb_dtype act_dtype, mnb_dtype out_dtype, mnb_dtype scale_dtype,
                                      mnb_stream_t stream);

/* mnb_matmul_ex with X and Y in page-locked HOST memory: the call moves the
 * activations in and the result out itself, with no copy-engine transfers.
 * No counterpart on the pages; an addition to the boundary.
 *   args->x  host [M, K] of act_dtype, 16-byte aligned, page-locked
 *            (cudaHostAlloc / cudaMallocHost, or cudaHostRegister'ed).
 *   args->y  host [M, N] of out_dtype, 16-byte aligned, page-locked.
 *   Everything else is as mnb_matmul_ex (device weights, scales, workspace).
 * Steps, all on args->stream: one small kernel reads X over the host link
 * into one of two file-scope device arrays of MNB_HOST_IO_X_BYTES (8 MiB)
 * per device (alternate calls use alternate arrays); the matmul runs as its
 * programmatic dependent (its weight stream starts while X is in flight) and
 * stores Y straight into the host buffer.  With MNB_FLAG_PDL the X read also
 * starts before the preceding kernel on the stream has finished (the
 * preceding kernel must then not write x either); every call's Y stores stay
 * ordered after the preceding kernel's completion.  Y is complete when the
 * stream's work is (synchronise before reading it).
 *   Pointer check: outside stream capture every call checks with
 *   cudaPointerGetAttributes that x and y are page-locked host memory (or
 *   device memory) and uses the device address that reports; pageable
 *   memory is MNB_ERR_INVALID_ARG and nothing is launched.  During capture
 *   the addresses are used as given: under unified addressing the device
 *   address of page-locked memory is its host address.
 *   Limits: M*K*sizeof(act) > MNB_HOST_IO_X_BYTES returns MNB_ERR_NO_MEM
 *   without launching.  The first call in a CUDA context looks the arrays'
 *   device address up (cudaGetSymbolAddress) and caches it for that
 *   context; make that first call outside stream capture.  Calls that
 *   overlap on one device (different streams, graphs in flight together)
 *   share the arrays and race; calls ordered on one stream are safe.
 * Returns the statuses of mnb_matmul_ex. */
#define MNB_HOST_IO_X_BYTES (8u << 20)
MNB_API mnb_status mnb_matmul_host_io(const mnb_matmul_args* args);

/* ---- floating-point weight formats --------------------------------------
 * dequant_matmul_fp8 and dequant_matmul_nvfp4 of rlx-cpu 0.2.13,
 * src/thunk/ops/quant.rs: Y[m, n] = sum_k X[m, k] * w(k, n) with
 *   FP8:   w(k, n) = fp8(W[k, n]) * s[n]   (s = 1 when scales is NULL), one f32
 *          rounding; E4M3 as that page decodes it (bias 7, exponent 15 is
 *          infinity for a zero mantissa and NaN otherwise), or E5M2;
 *   NVFP4: w(k, n) = f32(f32(e2m1(W[k, n]) * e4m3(S[k / 16, n])) * global_scale),
 *          OCP E2M1 codes and OCP E4M3 ("fn") block scales, two f32 roundings.
 * The weights are re-tiled once like the integer codes (the same 512-byte
 * tiles: FP8 as 8-bit codes, NVFP4 as 4-bit codes); the products are
 * accumulated in f32 and the result rounded once to out_dtype.  Non-finite
 * weights propagate as IEEE arithmetic does. */

typedef enum mnb_wformat { MNB_WF_E4M3 = 1, MNB_WF_E5M2 = 2, MNB_WF_NVFP4 = 3 } mnb_wformat;

/* Bytes of the packed buffer for an N x K weight of `format`, or 0 if the
 * arguments are invalid. */
MNB_API size_t mnb_fp_packed_size(int64_t N, int64_t K, mnb_wformat format);

/* Re-tile a [K, N] weight (device, any alignment; FP8: K*N bytes, row-major,
 * element (k, n) at k*N + n; NVFP4: ceil(K*N/2) bytes, element (k, n) is the
 * nibble of flat index k*N + n, low nibble first) into packed (device,
 * 256-byte aligned, packed_bytes >= mnb_fp_packed_size()).  Codes are moved,
 * never changed; depths past K are zero codes (+0).  MNB_ERR_NO_MEM if
 * packed_bytes is too small. */
MNB_API mnb_status mnb_pack_fp_weights(const uint8_t* w_kn, void* packed, size_t packed_bytes, int64_t N,
                               int64_t K, mnb_wformat format, mnb_stream_t stream);

/* Y = X . W with the weight packed by mnb_pack_fp_weights for the same N, K
 * and format.
 *   x        device [M, K] act_dtype, row-major (16-byte aligned)
 *   scales   FP8: device f32 [N] (4-byte aligned) or NULL;
 *            NVFP4: device uint8 [ceil(K/16), N] E4M3 block scales (required)
 *   global_scale  NVFP4 only (ignored for FP8)
 *   y        device [M, N] out_dtype, row-major (16-byte aligned)
 * A header that does not match (N, K, format) sets MNB_ERR_LAYOUT_MISMATCH in
 * the device status word.  M == 0 is a no-op. */
MNB_API mnb_status mnb_matmul_fp(const void* x, const void* packed, const void* scales, float global_scale,
                         void* y, int64_t M, int64_t N, int64_t K, mnb_wformat format, mnb_dtype act_dtype,
                         mnb_dtype out_dtype, mnb_stream_t stream);

/* mnb_matmul_fp with MNB_FLAG_* flags (0 for none; an unknown bit is
 * MNB_ERR_INVALID_ARG).  With MNB_FLAG_PDL the decode GEMVs read the weights
 * and the NVFP4 block scales before the preceding kernel on the stream has
 * finished; X and Y wait for it. */
MNB_API mnb_status mnb_matmul_fp_ex(const void* x, const void* packed, const void* scales, float global_scale,
                            void* y, int64_t M, int64_t N, int64_t K, mnb_wformat format,
                            mnb_dtype act_dtype, mnb_dtype out_dtype, mnb_stream_t stream, int flags);

/* ---- diagnostics ------------------------------------------------------- */

/* Environment overrides, read at each call (none changes a result beyond
 * rounding order; none is needed for normal use):
 *   MNB_LOG=1              print the kernel family chosen for each call
 *   MNB_PROFILE=1          an NVTX range around each mnb_matmul_ex /
 *                          mnb_matmul_fp call and each pack, and per
 *                          kernel family ("pack" for the packs) the
 *                          host time in the call and the device time between
 *                          CUDA events recorded around its launches (none
 *                          under graph capture), printed on stderr every
 *                          MNB_PROFILE_EVERY calls (default 512).  The events
 *                          cost the calls their programmatic-launch overlap.
 *   MNB_GEMV_MAX_M         largest M routed to the decode GEMV (default 16)
 *   MNB_GEMV_SCHED=ks|tile|pers|stream|xr
 *                          force one schedule of the tensor-core decode GEMV
 *                          (default: the K-chunk schedule where it applies,
 *                          else one CTA per row tile)
 *   MNB_GEMV_PERS=0|1      per-tile or persistent decode GEMV when no
 *                          schedule is forced
 *   MNB_MMA_TPW, MNB_I8_TPW  k-tiles per warp of the decode / int8 GEMV (1..8)
 *   MNB_TC_KERNEL=bs       prefill GEMM for bf16 X with per-block partial sums
 *                          instead of the hi/lo weight split
 *   MNB_TC_BT=32|64|128    token tile of the block-scaled prefill GEMM
 *   MNB_TC_SPLITK=1|2      K split over a 2-CTA cluster in the hi/lo GEMM
 *                          (1: never, 2: always)
 *   MNB_WAIT_MODE=0|1|2    bounded mbarrier waits: suspend with a time hint,
 *                          try_wait without a hint (the default), or
 *                          test_wait polling
 *   MNB_WAIT_LIMIT=n       test hook: n tries per bounded wait (then
 *                          MNB_ERR_TIMEOUT in the status word)
 *   MNB_GEMV_STAGE_BUFS, MNB_GEMV_MAX_SLOTS  ring shape of the f32 GEMV
 *   MNB_A8_HILO=0          accuracy level 4 with M <= 4: the int8 dp4a GEMV
 *                          instead of hi / lo bf16 activation rows
 *   MNB_A8_HILO=2          the same with the hi / lo rows written to the
 *                          workspace by a separate quantiser (same bits)
 *   MNB_FP_KERNEL=generic  FP8 / NVFP4: the exact generic kernel
 *   MNB_FP_KERNEL=lut      NVFP4 decode: the CUDA-core table GEMV instead
 *                          of the tensor-core one
 *   MNB_MOE_SCHED=tile     mnb_matmul_grouped with at most 8 pairs on the
 *                          per-tile kernel instead of the K-chunk schedule
 *   MNB_MOE_SETS           expert sets per row tile of the per-tile grouped kernel
 *   MNB_FAIL_LAUNCH=1      test hook: every launch reports MNB_ERR_CUDA
 *                          without launching */

/* The family mnb_matmul_ex would run with kernel == MNB_KERNEL_AUTO (host
 * only, no GPU needed).  Thresholds: MNB_GEMV_MAX_M (default 16) and the
 * environment override of the same name. */
MNB_API mnb_kernel mnb_select_kernel(int64_t M, int64_t N, int64_t K, int bits, int block_size,
                             mnb_dtype act_dtype, int accuracy_level);

/* Read and clear the current device's status word (an mnb_status value set
 * by a kernel; MNB_OK if none).  Synchronises the device. */
MNB_API mnb_status mnb_get_device_error(int* code);

MNB_API const char* mnb_status_string(mnb_status s);
MNB_API const char* mnb_kernel_name(mnb_kernel k);
MNB_API int mnb_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MNB_H_ */
