// C ABI of libmnb: host-side validation, kernel selection and launch on the
// caller's stream.  See include/mnb.h for the contract of each entry point.
//
// Validation follows the operator's own checks (onnx-runtime-ep-cpu
// 0.1.0-dev.5, src/kernels/matmul_nbits.rs, MatMulNBitsFactory::create:
// bits in {2, 4, 8}, block_size a power of two >= 16, K and N > 0;
// MatMulNBitsKernel::execute: tensor shapes).  Nothing is launched unless
// every check passes.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "mnb.h"
#include "mnb_internal.h"

namespace mnb {
namespace {

bool log_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("MNB_LOG");
        return v && v[0] == '1';
    }();
    return on;
}

int64_t env_int(const char* name, int64_t dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    char* end = nullptr;
    const long long r = std::strtoll(v, &end, 10);
    return (end && *end == 0) ? (int64_t)r : dflt;
}

// One status word per device, in device memory owned by the library.
__device__ int g_status_word;

cudaError_t lookup_status_word(void** p) { return cudaGetSymbolAddress(p, g_status_word); }
SymbolCache g_status_cache;

struct PerDevice {
    bool init = false;
    DeviceInfo info{};
    int* status = nullptr;  // device address of g_status_word in the current context
};

std::mutex g_mu;
std::vector<PerDevice> g_dev;

PerDevice* per_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
    PerDevice& pd = g_dev[dev];
    if (!pd.init) {
        DeviceInfo di{};
        di.device = dev;
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
        di.sm_count = v;
        cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return nullptr;
        di.smem_optin = (size_t)v;
        pd.info = di;
        pd.init = true;
    }
    // The address belongs to the current context, not to the device index:
    // after a device reset the array may live elsewhere.
    void* addr = nullptr;
    if (cached_symbol_address(g_status_cache, lookup_status_word, &addr) != cudaSuccess) return nullptr;
    pd.status = static_cast<int*>(addr);
    return &pd;
}

bool valid_dtype(int d) { return d == kF32 || d == kF16 || d == kBF16; }
size_t dtype_bytes(int d) { return d == kF32 ? 4 : 2; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

bool valid_shape(int64_t N, int64_t K, int bits, int bs) {
    if (N <= 0 || K <= 0) return false;
    if (bits != 2 && bits != 4 && bits != 8) return false;
    if (bs < 16 || !pow2(bs)) return false;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 31)) return false;
    return true;
}

mnb_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MNB_OK;
    cudaGetLastError();  // clear a sticky launch error so the next call starts clean
    if (log_enabled()) std::fprintf(stderr, "[mnb] CUDA error: %s\n", cudaGetErrorString(e));
    return MNB_ERR_CUDA;
}

}  // namespace

bool current_context_id(unsigned long long* id) {
    // cuCtxGetCurrent / cuCtxGetId through the runtime's driver entry points,
    // so the library needs no link-time dependency on libcuda.
    typedef int (*GetCurrentFn)(void**);
    typedef int (*GetIdFn)(void*, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(f);
        cudaGetLastError();
    });
    if (!get_current || !get_id) return false;
    void* ctx = nullptr;
    if (get_current(&ctx) != 0 || ctx == nullptr) return false;
    return get_id(ctx, id) == 0;
}

cudaError_t cached_symbol_address(SymbolCache& cache, cudaError_t (*lookup)(void**), void** out) {
    unsigned long long id = 0;
    if (!current_context_id(&id)) {
        // No context yet: the lookup creates the primary context.
        void* p = nullptr;
        const cudaError_t e = lookup(&p);
        if (e != cudaSuccess) return e;
        if (!current_context_id(&id)) {  // cannot key the cache: use the fresh address
            *out = p;
            return cudaSuccess;
        }
    }
    std::lock_guard<std::mutex> lk(cache.mu);
    for (int i = 0; i < cache.used; ++i) {
        if (cache.ctx[i] == id) {
            *out = cache.addr[i];
            return cudaSuccess;
        }
    }
    void* p = nullptr;
    const cudaError_t e = lookup(&p);
    if (e != cudaSuccess) return e;
    const int slot = cache.used < SymbolCache::kSlots ? cache.used++ : (int)(id % SymbolCache::kSlots);
    cache.ctx[slot] = id;
    cache.addr[slot] = p;
    *out = p;
    return cudaSuccess;
}

void wait_limits(uint32_t* limit, uint32_t* hint_ns) {
    const int64_t n = env_int("MNB_WAIT_LIMIT", 0);
    if (n > 0) {
        *limit = (uint32_t)n;
        *hint_ns = 0;
        return;
    }
    // MNB_WAIT_MODE (tuning): 0 suspend with a time hint, 1 try_wait without a
    // hint, 2 busy polling with test_wait; the limits keep every mode near two seconds.
    switch (env_int("MNB_WAIT_MODE", 1)) {
        case 0: *limit = kWaitLimit; *hint_ns = kWaitHintNs; break;
        case 2: *limit = 1u << 26; *hint_ns = kWaitPoll; break;
        default: *limit = 1u << 24; *hint_ns = 0; break;  // measured fastest on the tcgen05 GEMMs
    }
}

// Test hook: MNB_FAIL_LAUNCH=1 makes every launch report a CUDA error without
// launching anything (exercises the error path on the host, no GPU fault).
bool inject_launch_failure() { return env_int("MNB_FAIL_LAUNCH", 0) == 1; }

const DeviceInfo& device_info() {
    static DeviceInfo empty{};
    PerDevice* pd = per_device();
    return pd ? pd->info : empty;
}

int* device_status_word() {
    PerDevice* pd = per_device();
    return pd ? pd->status : nullptr;
}

}  // namespace mnb

using namespace mnb;

extern "C" {

int mnb_abi_version(void) { return MNB_ABI_VERSION; }

const char* mnb_status_string(mnb_status s) {
    switch (s) {
        case MNB_OK: return "ok";
        case MNB_ERR_INVALID_ARG: return "invalid argument";
        case MNB_ERR_UNSUPPORTED: return "unsupported configuration";
        case MNB_ERR_CUDA: return "CUDA runtime error";
        case MNB_ERR_NO_MEM: return "buffer too small";
        case MNB_ERR_TIMEOUT: return "bounded wait inside a kernel ran out";
        case MNB_ERR_LAYOUT_MISMATCH: return "packed buffer header does not match the call";
    }
    return "unknown status";
}

const char* mnb_kernel_name(mnb_kernel k) {
    switch (k) {
        case MNB_KERNEL_AUTO: return "auto";
        case MNB_KERNEL_GEMV: return "gemv";
        case MNB_KERNEL_GEMV_MMA: return "gemv_mma";
        case MNB_KERNEL_GEMM_TC: return "gemm_tc";
        case MNB_KERNEL_GENERIC: return "generic";
        case MNB_KERNEL_GEMV_I8: return "gemv_i8";
    }
    return "unknown";
}

size_t mnb_packed_size(int64_t N, int64_t K, int bits, int block_size) {
    if (!valid_shape(N, K, bits, block_size)) return 0;
    Layout L;
    L.init(N, K, bits, block_size);
    return L.total_bytes();
}

size_t mnb_packed_size_gidx(int64_t N, int64_t K, int bits, int block_size) {
    if (!valid_shape(N, K, bits, block_size)) return 0;
    Layout L;
    L.init(N, K, bits, block_size);
    return L.total_bytes() + kperm_bytes(L);
}

mnb_status mnb_pack_weights_gidx(const uint8_t* b_ort, const int32_t* g_idx, void* packed_b, size_t packed_bytes,
                                 int64_t N, int64_t K, int bits, int block_size, mnb_stream_t stream) {
    if (!valid_shape(N, K, bits, block_size) || !b_ort || !g_idx || !packed_b) return MNB_ERR_INVALID_ARG;
    if (!aligned(packed_b, 256) || !aligned(g_idx, 4)) return MNB_ERR_INVALID_ARG;
    Layout L;
    L.init(N, K, bits, block_size);
    if (packed_bytes < L.total_bytes() + kperm_bytes(L)) return MNB_ERR_NO_MEM;
    if (!per_device()) return from_cuda(cudaGetLastError());
    if (inject_launch_failure()) return MNB_ERR_CUDA;
    ProfileScope prof("mnb_pack_weights_gidx", (cudaStream_t)stream);
    const cudaError_t e = launch_pack_gidx(b_ort, g_idx, static_cast<uint8_t*>(packed_b), L, (cudaStream_t)stream);
    if (e == cudaSuccess) prof.done("pack_gidx");
    return from_cuda(e);
}

mnb_status mnb_pack_weights(const uint8_t* b_ort, void* packed_b, size_t packed_bytes, int64_t N, int64_t K,
                            int bits, int block_size, mnb_stream_t stream) {
    if (!valid_shape(N, K, bits, block_size) || !b_ort || !packed_b) return MNB_ERR_INVALID_ARG;
    if (!aligned(packed_b, 256)) return MNB_ERR_INVALID_ARG;
    Layout L;
    L.init(N, K, bits, block_size);
    if (packed_bytes < L.total_bytes()) return MNB_ERR_NO_MEM;
    if (inject_launch_failure()) return MNB_ERR_CUDA;
    ProfileScope prof("mnb_pack_weights", (cudaStream_t)stream);
    const cudaError_t e = launch_pack(b_ort, static_cast<uint8_t*>(packed_b), L, (cudaStream_t)stream);
    if (e == cudaSuccess) prof.done("pack");
    return from_cuda(e);
}

mnb_status mnb_unpack_codes(const void* packed_b, uint8_t* b_ort, int64_t N, int64_t K, int bits,
                            int block_size, mnb_stream_t stream) {
    if (!valid_shape(N, K, bits, block_size) || !b_ort || !packed_b) return MNB_ERR_INVALID_ARG;
    if (!aligned(packed_b, 256)) return MNB_ERR_INVALID_ARG;
    Layout L;
    L.init(N, K, bits, block_size);
    if (inject_launch_failure()) return MNB_ERR_CUDA;
    return from_cuda(launch_unpack(static_cast<const uint8_t*>(packed_b) + kHeaderBytes, b_ort, L,
                                   (cudaStream_t)stream));
}

mnb_status mnb_dequantize(const void* packed_b, const void* scales, const uint8_t* zero_points, float* w_nk,
                          int64_t N, int64_t K, int bits, int block_size, mnb_dtype scale_dtype,
                          mnb_stream_t stream) {
    if (!valid_shape(N, K, bits, block_size) || !packed_b || !scales || !w_nk) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(scale_dtype) || !aligned(packed_b, 256) || !aligned(w_nk, 4) ||
        !aligned(scales, dtype_bytes(scale_dtype)))
        return MNB_ERR_INVALID_ARG;
    Layout L;
    L.init(N, K, bits, block_size);
    if (inject_launch_failure()) return MNB_ERR_CUDA;
    return from_cuda(launch_dequant(static_cast<const uint8_t*>(packed_b) + kHeaderBytes, scales, scale_dtype,
                                    zero_points, w_nk, L, (cudaStream_t)stream));
}

static_assert((int)MNB_WF_E4M3 == kWfE4M3 && (int)MNB_WF_E5M2 == kWfE5M2 && (int)MNB_WF_NVFP4 == kWfNVFP4,
              "weight format codes of the C API and the kernels agree");

static bool valid_fp(int64_t N, int64_t K, int format) {
    return N > 0 && K > 0 && N <= (int64_t(1) << 31) && K <= (int64_t(1) << 31) &&
           (format == MNB_WF_E4M3 || format == MNB_WF_E5M2 || format == MNB_WF_NVFP4);
}

size_t mnb_fp_packed_size(int64_t N, int64_t K, mnb_wformat format) {
    if (!valid_fp(N, K, format)) return 0;
    Layout L;
    fp_layout(&L, N, K, format);
    return L.total_bytes();
}

mnb_status mnb_pack_fp_weights(const uint8_t* w_kn, void* packed, size_t packed_bytes, int64_t N, int64_t K,
                               mnb_wformat format, mnb_stream_t stream) {
    if (!valid_fp(N, K, format) || !w_kn || !packed || !aligned(packed, 256)) return MNB_ERR_INVALID_ARG;
    Layout L;
    fp_layout(&L, N, K, format);
    if (packed_bytes < L.total_bytes()) return MNB_ERR_NO_MEM;
    if (inject_launch_failure()) return MNB_ERR_CUDA;
    ProfileScope prof("mnb_pack_fp_weights", (cudaStream_t)stream);
    const cudaError_t e = launch_pack(w_kn, static_cast<uint8_t*>(packed), L, (cudaStream_t)stream, format);
    if (e == cudaSuccess) prof.done("pack_fp");
    return from_cuda(e);
}

mnb_status mnb_matmul_fp(const void* x, const void* packed, const void* scales, float global_scale, void* y,
                         int64_t M, int64_t N, int64_t K, mnb_wformat format, mnb_dtype act_dtype,
                         mnb_dtype out_dtype, mnb_stream_t stream) {
    return mnb_matmul_fp_ex(x, packed, scales, global_scale, y, M, N, K, format, act_dtype, out_dtype, stream, 0);
}

mnb_status mnb_matmul_fp_ex(const void* x, const void* packed, const void* scales, float global_scale, void* y,
                            int64_t M, int64_t N, int64_t K, mnb_wformat format, mnb_dtype act_dtype,
                            mnb_dtype out_dtype, mnb_stream_t stream, int flags) {
    if (!valid_fp(N, K, format) || M < 0 || !valid_dtype(act_dtype) || !valid_dtype(out_dtype) ||
        (flags & ~MNB_FLAG_PDL) != 0)
        return MNB_ERR_INVALID_ARG;
    if (M == 0) return MNB_OK;
    if (!x || !packed || !y || (format == MNB_WF_NVFP4 && !scales)) return MNB_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(packed, 256) ||
        (format != MNB_WF_NVFP4 && scales && !aligned(scales, 4)))
        return MNB_ERR_INVALID_ARG;
    PerDevice* pd = per_device();
    if (!pd) return from_cuda(cudaGetLastError());
    FpParams p{};
    p.x = x;
    p.packed_hdr = packed;
    p.packed = static_cast<const uint8_t*>(packed) + kHeaderBytes;
    p.scales = scales;
    p.global_scale = global_scale;
    p.y = y;
    p.M = M;
    fp_layout(&p.L, N, K, format);
    p.fmt = format;
    p.act_dtype = act_dtype;
    p.out_dtype = out_dtype;
    p.status = pd->status;
    p.flags = flags;
    if (inject_launch_failure()) return MNB_ERR_CUDA;
    const bool fast = gemv_fp_supported(p);
    const char* kname = fast ? (gemv_nv_selected(p) ? "gemv_nv" : "gemv_fp") : "fp_generic";
    if (log_enabled())
        std::fprintf(stderr, "[mnb] matmul_fp M=%lld N=%lld K=%lld format=%d kernel=%s\n", (long long)M,
                     (long long)N, (long long)K, (int)format, kname);
    ProfileScope prof("mnb_matmul_fp", (cudaStream_t)stream);
    const cudaError_t e = fast ? launch_gemv_fp(p, (cudaStream_t)stream) : launch_fp_generic(p, (cudaStream_t)stream);
    if (e == cudaSuccess) prof.done(kname);
    return from_cuda(e);
}

size_t mnb_workspace_size_ex(int64_t M, int64_t N, int64_t K, int bits, int block_size, int accuracy_level,
                             int flags) {
    const size_t base = mnb_workspace_size(M, N, K, bits, block_size, accuracy_level);
    if (!(flags & kFlagKPerm) || accuracy_level == 4 || !valid_shape(N, K, bits, block_size) || M <= 8) return base;
    Layout L;
    L.init(N, K, bits, block_size);
    const size_t g = kperm_gemm_workspace_bytes(M, L);  // the act-order prefill's X in the pack's order
    return g > base ? g : base;
}

size_t mnb_workspace_size(int64_t M, int64_t N, int64_t K, int bits, int block_size, int accuracy_level) {
    if (!valid_shape(N, K, bits, block_size) || M < 0) return 0;
    if (accuracy_level != 4) return 0;
    Layout L;
    L.init(N, K, bits, block_size);
    const size_t i8 = i8_workspace_bytes(M, L);
    if (M <= 16) return i8;  // the int8 GEMV
    const size_t g = a8_gemm_workspace_bytes(M, L);  // the prefill GEMM (bf16 activation codes)
    return g > i8 ? g : i8;
}

mnb_kernel mnb_select_kernel(int64_t M, int64_t N, int64_t K, int bits, int block_size, mnb_dtype act_dtype,
                             int accuracy_level) {
    (void)N;
    (void)K;
    (void)bits;
    (void)block_size;
    const int64_t gemv_max_m = env_int("MNB_GEMV_MAX_M", 16);
    if (accuracy_level == 4) return M <= 16 ? MNB_KERNEL_GEMV_I8 : MNB_KERNEL_GEMM_TC;
    if (act_dtype == MNB_F32) return M == 1 ? MNB_KERNEL_GEMV : MNB_KERNEL_GENERIC;
    if (M <= gemv_max_m) return MNB_KERNEL_GEMV_MMA;
    return MNB_KERNEL_GEMM_TC;
}

}  // extern "C"

namespace {

// The body of mnb_matmul_ex; on a launch, *family names the kernel family that ran.
mnb_status matmul_ex_impl(const mnb_matmul_args* a, const char** family) {
    if (!a) return MNB_ERR_INVALID_ARG;
    if (!valid_shape(a->N, a->K, a->bits, a->block_size) || a->M < 0) return MNB_ERR_INVALID_ARG;
    if (!valid_dtype(a->act_dtype) || !valid_dtype(a->out_dtype) || !valid_dtype(a->scale_dtype))
        return MNB_ERR_INVALID_ARG;
    if (a->bias && !valid_dtype(a->bias_dtype)) return MNB_ERR_INVALID_ARG;
    if (a->accuracy_level < 0 || a->accuracy_level > 4) return MNB_ERR_INVALID_ARG;
    if (a->M == 0) return MNB_OK;
    if (!a->x || !a->packed_b || !a->scales || !a->y) return MNB_ERR_INVALID_ARG;
    if (!aligned(a->x, 16) || !aligned(a->y, 16) || !aligned(a->packed_b, 256) ||
        !aligned(a->scales, dtype_bytes(a->scale_dtype)) || (a->g_idx && !aligned(a->g_idx, 4)) ||
        (a->bias && !aligned(a->bias, dtype_bytes(a->bias_dtype))))
        return MNB_ERR_INVALID_ARG;
    PerDevice* pd = per_device();
    if (!pd) return from_cuda(cudaGetLastError());

    MatmulParams p{};
    p.x = a->x;
    p.packed_hdr = a->packed_b;
    p.packed = static_cast<const uint8_t*>(a->packed_b) + kHeaderBytes;
    p.scales = a->scales;
    p.zp = a->zero_points;
    p.g_idx = a->g_idx;
    p.bias = a->bias;
    p.y = a->y;
    p.M = a->M;
    p.L.init(a->N, a->K, a->bits, a->block_size);
    p.act_dtype = a->act_dtype;
    p.out_dtype = a->out_dtype;
    p.scale_dtype = a->scale_dtype;
    p.bias_dtype = a->bias_dtype;
    p.status = pd->status;
    p.workspace = a->workspace;
    p.workspace_bytes = a->workspace_bytes;
    p.flags = a->flags;
    wait_limits(&p.wait_limit, &p.wait_hint_ns);

    if (a->flags & kFlagKPerm) {
        // act-order pack: the buffer's own permutation replaces g_idx; the K-chunk decode GEMV
        // (X gathered while it is staged) or the generic kernel
        if (a->g_idx) return MNB_ERR_INVALID_ARG;
        if (a->accuracy_level == 4) return MNB_ERR_UNSUPPORTED;
        p.kperm = reinterpret_cast<const int32_t*>(p.packed + p.L.data_bytes());
        // prefill: X put in the pack's depth order in the workspace, then the tensor-core GEMM
        const bool gemm_ok = (a->act_dtype == MNB_BF16 || a->act_dtype == MNB_F16) && a->K % 8 == 0 &&
                             (size_t)a->K * 2 <= device_info().smem_optin && gemm_tc_supported(p);
        const size_t gneed = kperm_gemm_workspace_bytes(a->M, p.L);
        const bool ws_ok = a->workspace && a->workspace_bytes >= gneed && aligned(a->workspace, 256);
        mnb_kernel kk = a->kernel;
        if (kk == MNB_KERNEL_AUTO)
            kk = gemv_ks_kperm_supported(p) ? MNB_KERNEL_GEMV_MMA
                 : (a->M > 8 && gemm_ok && ws_ok) ? MNB_KERNEL_GEMM_TC : MNB_KERNEL_GENERIC;
        cudaError_t ek;
        if (kk == MNB_KERNEL_GEMV_MMA) {
            if (!gemv_ks_kperm_supported(p)) return MNB_ERR_UNSUPPORTED;
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            ek = launch_gemv_ks_kperm(p, (cudaStream_t)a->stream);
        } else if (kk == MNB_KERNEL_GEMM_TC) {
            if (!gemm_ok) return MNB_ERR_UNSUPPORTED;
            if (!a->workspace || a->workspace_bytes < gneed) return MNB_ERR_NO_MEM;
            if (!aligned(a->workspace, 256)) return MNB_ERR_INVALID_ARG;
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            ek = launch_gather_kperm(a->x, p.kperm, a->workspace, a->M, p.L, (a->flags & kFlagPDL) != 0,
                                     (cudaStream_t)a->stream);
            if (ek == cudaSuccess) {
                MatmulParams q = p;
                q.x = a->workspace;  // X in the pack's depth order; q.kperm stays set for the header check
                q.flags |= kFlagPDL;  // the GEMM's weight stream overlaps the gather
                ek = launch_gemm_tc(q, (cudaStream_t)a->stream);
            }
        } else if (kk == MNB_KERNEL_GENERIC) {
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            ek = launch_generic(p, (cudaStream_t)a->stream);
        } else {
            return MNB_ERR_UNSUPPORTED;
        }
        if (log_enabled())
            std::fprintf(stderr, "[mnb] matmul M=%lld N=%lld K=%lld bits=%d bs=%d kernel=%s (act-order pack)\n",
                         (long long)a->M, (long long)a->N, (long long)a->K, a->bits, a->block_size,
                         mnb_kernel_name(kk));
        *family = kk == MNB_KERNEL_GEMV_MMA ? "gemv_mma/act-order"
                  : kk == MNB_KERNEL_GEMM_TC ? "gemm_tc/act-order" : "generic/act-order";
        return from_cuda(ek);
    }

    mnb_kernel k = a->kernel;
    if (k == MNB_KERNEL_AUTO && a->accuracy_level == 4) {
        k = a->M <= 16 && gemv_i8_supported(p) ? MNB_KERNEL_GEMV_I8 : MNB_KERNEL_GEMM_TC;
    } else if (k == MNB_KERNEL_AUTO) {
        k = mnb_select_kernel(a->M, a->N, a->K, a->bits, a->block_size, a->act_dtype, a->accuracy_level);
        // The specialised kernels decline what they cannot do; the generic
        // kernel takes every float-path call.
        if (a->g_idx && a->accuracy_level != 4) k = MNB_KERNEL_GENERIC;
        if (k == MNB_KERNEL_GEMV && !gemv_supported(p)) k = MNB_KERNEL_GENERIC;
        if (k == MNB_KERNEL_GEMV_MMA && !gemv_mma_supported(p)) k = a->M == 1 ? MNB_KERNEL_GEMV : MNB_KERNEL_GEMM_TC;
        if (k == MNB_KERNEL_GEMV && !gemv_supported(p)) k = MNB_KERNEL_GENERIC;
        if (k == MNB_KERNEL_GEMM_TC && !gemm_tc_supported(p)) k = MNB_KERNEL_GENERIC;
    }
    if (a->accuracy_level == 4 && k != MNB_KERNEL_GEMV_I8 && k != MNB_KERNEL_GEMM_TC) return MNB_ERR_UNSUPPORTED;
    if (a->accuracy_level != 4 && k == MNB_KERNEL_GEMV_I8) return MNB_ERR_UNSUPPORTED;

    cudaStream_t s = (cudaStream_t)a->stream;
    cudaError_t e = cudaSuccess;
    switch (k) {
        case MNB_KERNEL_GENERIC:
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            e = launch_generic(p, s);
            break;
        case MNB_KERNEL_GEMV:
            if (!gemv_supported(p)) return MNB_ERR_UNSUPPORTED;
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            e = launch_gemv(p, s);
            break;
        case MNB_KERNEL_GEMV_MMA:
            if (a->g_idx || !gemv_mma_supported(p)) return MNB_ERR_UNSUPPORTED;
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            e = launch_gemv_mma(p, s);
            break;
        case MNB_KERNEL_GEMM_TC:
            if (a->accuracy_level == 4) {
                if (a->g_idx || !gemm_a8_supported(p)) return MNB_ERR_UNSUPPORTED;
                const size_t need = a8_gemm_workspace_bytes(a->M, p.L);
                if (a->workspace_bytes < need || !a->workspace) return MNB_ERR_NO_MEM;
                if (!aligned(a->workspace, 256)) return MNB_ERR_INVALID_ARG;
                if (inject_launch_failure()) return MNB_ERR_CUDA;
                e = launch_gemm_a8(p, s);
                break;
            }
            if (a->g_idx || !gemm_tc_supported(p)) return MNB_ERR_UNSUPPORTED;
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            e = launch_gemm_tc(p, s);
            break;
        case MNB_KERNEL_GEMV_I8: {
            if (a->g_idx || !gemv_i8_supported(p)) return MNB_ERR_UNSUPPORTED;
            const size_t need = i8_workspace_bytes(a->M, p.L);
            if (a->workspace_bytes < need || (need && !a->workspace)) return MNB_ERR_NO_MEM;
            if (a->workspace && !aligned(a->workspace, 256)) return MNB_ERR_INVALID_ARG;
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            e = launch_gemv_i8(p, s);
            break;
        }
        default:
            return MNB_ERR_INVALID_ARG;
    }
    if (log_enabled())
        std::fprintf(stderr, "[mnb] matmul M=%lld N=%lld K=%lld bits=%d bs=%d kernel=%s\n", (long long)a->M,
                     (long long)a->N, (long long)a->K, a->bits, a->block_size, mnb_kernel_name(k));
    *family = a->accuracy_level == 4 ? (k == MNB_KERNEL_GEMV_I8 ? "gemv_i8/acc4" : "gemm_tc/acc4") : mnb_kernel_name(k);
    return from_cuda(e);
}

}  // namespace

extern "C" {

mnb_status mnb_matmul_ex(const mnb_matmul_args* a) {
    ProfileScope prof("mnb_matmul_ex", a ? (cudaStream_t)a->stream : nullptr);
    const char* family = nullptr;
    const mnb_status st = matmul_ex_impl(a, &family);
    if (st == MNB_OK && family) prof.done(family);
    return st;
}

mnb_status mnb_matmul(const void* x, const void* packed_b, const void* scales, const uint8_t* zero_points,
                      void* y, int64_t M, int64_t N, int64_t K, int bits, int block_size, mnb_dtype act_dtype,
                      mnb_dtype out_dtype, mnb_dtype scale_dtype, mnb_stream_t stream) {
    mnb_matmul_args a;
    std::memset(&a, 0, sizeof(a));
    a.x = x;
    a.packed_b = packed_b;
    a.scales = scales;
    a.zero_points = zero_points;
    a.y = y;
    a.M = M;
    a.N = N;
    a.K = K;
    a.bits = bits;
    a.block_size = block_size;
    a.act_dtype = act_dtype;
    a.out_dtype = out_dtype;
    a.scale_dtype = scale_dtype;
    a.bias_dtype = MNB_F32;
    a.accuracy_level = 0;
    a.kernel = MNB_KERNEL_AUTO;
    a.stream = stream;
    return mnb_matmul_ex(&a);
}

mnb_status mnb_quantize_activations(const void* x, int8_t* qa, float* sa, int64_t M, int64_t K, int block_size,
                                    mnb_dtype act_dtype, mnb_stream_t stream) {
    if (!valid_shape(1, K, 4, block_size) || M < 0 || !valid_dtype(act_dtype)) return MNB_ERR_INVALID_ARG;
    if (M == 0) return MNB_OK;
    if (!x || !qa || !sa || !aligned(x, 16) || !aligned(qa, 16) || !aligned(sa, 4)) return MNB_ERR_INVALID_ARG;
    Layout L;
    L.init(1, K, 4, block_size);
    if (inject_launch_failure()) return MNB_ERR_CUDA;
    return from_cuda(launch_quant_act(x, act_dtype, qa, sa, M, L, (cudaStream_t)stream));
}

mnb_status mnb_get_device_error(int* code) {
    PerDevice* pd = per_device();
    if (!pd) return from_cuda(cudaGetLastError());
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int));
    if (e != cudaSuccess) return from_cuda(e);
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
    if (e != cudaSuccess) return from_cuda(e);
    if (code) *code = v;
    return MNB_OK;
}

}  // extern "C"
