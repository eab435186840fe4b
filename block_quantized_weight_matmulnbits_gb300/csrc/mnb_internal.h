// Internal launch interface between the C ABI (capi.cu) and the kernel files.
// Every launcher enqueues on `stream` and returns the cudaError_t of the launch.
#pragma once

#include <cstdint>
#include <cstddef>
#include <mutex>
#include <cuda_runtime.h>
#include <utility>

#include "mnb_common.cuh"

namespace mnb {

struct MatmulParams {
    const void* x;
    const uint8_t* packed;   // tile data (header already skipped)
    const void* packed_hdr;  // start of the packed buffer (header)
    const void* scales;
    const uint8_t* zp;
    const int32_t* g_idx;
    const int32_t* kperm;    // act-order pack (MNB_FLAG_KPERM): original depth of each stored depth, or null
    const void* bias;
    void* y;
    int64_t M;
    Layout L;
    int act_dtype, out_dtype, scale_dtype, bias_dtype;
    int* status;             // device status word
    void* workspace;
    size_t workspace_bytes;
    int flags;               // MNB_FLAG_* of the call
    uint32_t wait_limit;     // bounded mbarrier waits: tries before MNB_ERR_TIMEOUT
    uint32_t wait_hint_ns;   // suspend hint of each try (0: poll)
};

// Wait limits of the call: kWaitLimit x kWaitHintNs (about two seconds), or
// MNB_WAIT_LIMIT=n polls of 0 ns (a test hook that makes a kernel's first
// wait that is not already satisfied run out).
void wait_limits(uint32_t* limit, uint32_t* hint_ns);

constexpr int kFlagPDL = 1;    // == MNB_FLAG_PDL
constexpr int kFlagKPerm = 2;  // == MNB_FLAG_KPERM

// A matmul with a floating-point weight format (WFormat kWfE4M3, kWfE5M2,
// kWfNVFP4): FP8 scales are f32 [N] or null, NVFP4 scales are E4M3 bytes
// [ceil(K / 16), N] times global_scale.
struct FpParams {
    const void* x;
    const uint8_t* packed;   // tile data (header already skipped)
    const void* packed_hdr;
    const void* scales;
    float global_scale;
    void* y;
    int64_t M;
    Layout L;
    int fmt;
    int act_dtype, out_dtype;
    int* status;
    int flags;
};

// The packed layout of a floating-point format: FP8 as 8-bit codes with
// 128-deep tiling blocks, NVFP4 as 4-bit codes with its 16-deep scale blocks.
inline void fp_layout(Layout* L, int64_t N, int64_t K, int fmt) {
    if (fmt == kWfNVFP4) L->init(N, K, 4, 16);
    else L->init(N, K, 8, 128);
}

cudaError_t launch_fp_generic(const FpParams& p, cudaStream_t s);
bool gemv_fp_supported(const FpParams& p);
bool gemv_nv_selected(const FpParams& p);
cudaError_t launch_gemv_fp(const FpParams& p, cudaStream_t s);

// Accuracy level 4 on the prefill GEMM: workspace = the quantised
// activations code * s_a rounded to tf32, f32 [M, Kpad] (zeros past K).
inline size_t a8_gemm_workspace_bytes(int64_t M, const Layout& L) {
    return ((size_t)M * (size_t)L.Kpad * 4 + 255) & ~size_t(255);
}
cudaError_t launch_quant_act_tf32(const void* x, int act_dtype, float* xq, int64_t M, const Layout& L, bool pdl,
                                  cudaStream_t s);
bool gemm_a8_supported(const MatmulParams& p);
cudaError_t launch_gemm_a8(const MatmulParams& p, cudaStream_t s);

cudaError_t launch_pack(const uint8_t* b_ort, uint8_t* packed_hdr, const Layout& L, cudaStream_t s,
                        int fmt = kWfInt);
// Act-order pack: depths in g_idx group order, the int32 permutation (Kpad entries) after the tiles.
cudaError_t launch_pack_gidx(const uint8_t* b_ort, const int32_t* g_idx, uint8_t* packed_hdr, const Layout& L,
                             cudaStream_t s);
inline size_t kperm_bytes(const Layout& L) { return ((size_t)L.Kpad * 4 + 255) & ~size_t(255); }
// Act-order prefill: X's depths in the pack's order (16-bit activations, K % 8 == 0) into xp [M, K].
cudaError_t launch_gather_kperm(const void* x, const int32_t* perm, void* xp, int64_t M, const Layout& L,
                                bool pdl, cudaStream_t s);
inline size_t kperm_gemm_workspace_bytes(int64_t M, const Layout& L) {
    return ((size_t)M * (size_t)L.K * 2 + 255) & ~size_t(255);
}
cudaError_t launch_unpack(const uint8_t* packed, uint8_t* b_ort, const Layout& L, cudaStream_t s);
cudaError_t launch_dequant(const uint8_t* packed, const void* scales, int scale_dtype, const uint8_t* zp,
                           float* w, const Layout& L, cudaStream_t s);

cudaError_t launch_generic(const MatmulParams& p, cudaStream_t s);

// Decode GEMV (M == 1).  Returns cudaErrorNotSupported when the shape is
// outside what the kernel handles (the caller then reports UNSUPPORTED).
bool gemv_supported(const MatmulParams& p);
cudaError_t launch_gemv(const MatmulParams& p, cudaStream_t s);

bool gemv_mma_supported(const MatmulParams& p);
cudaError_t launch_gemv_mma(const MatmulParams& p, cudaStream_t s);
// act-order pack (p.kperm set): the K-chunk decode GEMV gathering X through the permutation
bool gemv_ks_kperm_supported(const MatmulParams& p);
cudaError_t launch_gemv_ks_kperm(const MatmulParams& p, cudaStream_t s);

bool gemm_tc_supported(const MatmulParams& p);
cudaError_t launch_gemm_tc(const MatmulParams& p, cudaStream_t s);

size_t i8_workspace_bytes(int64_t M, const Layout& L);
bool gemv_i8_supported(const MatmulParams& p);
cudaError_t launch_quant_act(const void* x, int act_dtype, int8_t* qa, float* sa, int64_t M, const Layout& L,
                             cudaStream_t s);
cudaError_t launch_gemv_i8(const MatmulParams& p, cudaStream_t s);

// Device properties of the current device (cached per device).
struct DeviceInfo {
    int device;
    int sm_count;
    int major, minor;
    size_t smem_optin;
};
const DeviceInfo& device_info();

// Device address of the current device's status word (see mnb_get_device_error).
int* device_status_word();

// MNB_FAIL_LAUNCH=1: entry points report MNB_ERR_CUDA instead of launching.
bool inject_launch_failure();

// MNB_PROFILE=1 (read on every call): an NVTX range around the entry point and
// per-kernel-family host and device timers, reported on stderr every
// MNB_PROFILE_EVERY calls (default 512).  A scope does nothing when disabled.
bool profile_enabled();
class ProfileScope {
public:
    ProfileScope(const char* range, cudaStream_t s);
    ~ProfileScope();
    void done(const char* kernel);  // the call launched its work under this family name
    ProfileScope(const ProfileScope&) = delete;
    ProfileScope& operator=(const ProfileScope&) = delete;

private:
    bool on_ = false, done_ = false;
    cudaStream_t stream_ = nullptr;
    double t0_ = 0;
    std::pair<cudaEvent_t, cudaEvent_t> ev_{nullptr, nullptr};
};

// Identifier of the CUDA context current on the calling thread (the driver's
// context id, unique for the life of the process, so a context created after
// a device reset never matches an older one).  False when no context is
// current or the driver cannot say.
bool current_context_id(unsigned long long* id);

// Device address of a file-scope __device__ array, cached per CUDA context.
// `lookup` (defined in the .cu file that owns the array) calls
// cudaGetSymbolAddress on it.  The first call in a context performs the
// lookup, which may load the module: make it outside stream capture.
struct SymbolCache {
    static constexpr int kSlots = 32;
    std::mutex mu;
    unsigned long long ctx[kSlots] = {};
    void* addr[kSlots] = {};
    int used = 0;
};
cudaError_t cached_symbol_address(SymbolCache& cache, cudaError_t (*lookup)(void**), void** out);

}  // namespace mnb
