// mnb_matmul_host_io: the matmul with activations and result in page-locked
// host memory.  On a Grace-Blackwell node the GPU addresses host memory
// directly over NVLink-C2C, so the transfers are done by kernels rather than
// by copy-engine operations (each of which costs a few microseconds of
// dependency latency per call):
//   1. fetch_kernel reads X from the host into one of two file-scope device
//      arrays (alternate calls use alternate arrays) and immediately allows
//      its programmatic dependent to launch; with MNB_FLAG_PDL it is itself a
//      programmatic dependent of the preceding kernel;
//   2. the matmul (mnb_matmul_ex with MNB_FLAG_PDL) starts its weight stream
//      while X is in flight, waits for the fetch before it reads X, and
//      stores Y straight into the host buffer.
// The library allocates nothing.
#include <cstring>
#include <mutex>

#include "mnb.h"
#include "mnb_internal.h"

namespace {

constexpr size_t kXBytes = MNB_HOST_IO_X_BYTES;
constexpr int kMaxDevices = 64;
constexpr int kFetchThreads = 256;

// Two staging buffers per device (a __device__ variable exists once in every
// context), used by alternate calls: the fetch of call i+1 may run while the
// matmul of call i still reads its X.
static __device__ __align__(256) uint8_t g_host_x[2][kXBytes];

std::mutex g_mu;
unsigned g_calls[kMaxDevices] = {};

cudaError_t lookup_x(void** p) { return cudaGetSymbolAddress(p, g_host_x); }
mnb::SymbolCache g_x_cache;

// The staging buffer of this call: the two alternate call by call.  The
// arrays' address is looked up per context (see mnb::cached_symbol_address).
cudaError_t x_buffer_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* base = nullptr;
    e = mnb::cached_symbol_address(g_x_cache, lookup_x, &base);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    *out = static_cast<uint8_t*>(base) + (size_t)(g_calls[dev]++ & 1u) * kXBytes;
    return cudaSuccess;
}

// Copy n16 16-byte words, then `tail` trailing bytes, from host-resident src
// to device dst.  Loads use the "fetch again" cache operator: host memory
// is written by the CPU between calls.  Launched as a programmatic dependent
// (MNB_FLAG_PDL) it copies while the preceding kernel still runs and
// finishes only after that kernel has: the matmul that waits on this fetch
// is then ordered after the preceding call's matmul as well.
__global__ void __launch_bounds__(kFetchThreads) fetch_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                             int64_t n16, int tail) {
    mnb::griddep_launch_dependents();  // the matmul may start streaming its weights now
    const int64_t stride = (int64_t)gridDim.x * kFetchThreads;
    for (int64_t i = (int64_t)blockIdx.x * kFetchThreads + threadIdx.x; i < n16; i += stride) dst[i] = __ldcv(src + i);
    if (blockIdx.x == 0 && (int)threadIdx.x < tail) {
        const uint8_t* s8 = reinterpret_cast<const uint8_t*>(src + n16);
        uint8_t* d8 = reinterpret_cast<uint8_t*>(dst + n16);
        d8[threadIdx.x] = __ldcv(s8 + threadIdx.x);
    }
    mnb::griddep_wait();  // no-op unless launched as a programmatic dependent
}

// Device address of a caller pointer that must be page-locked host memory
// or device memory.  nullptr when it is neither (pageable memory).
const void* device_alias(const void* p) {
    cudaPointerAttributes a;
    std::memset(&a, 0, sizeof(a));
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    switch (a.type) {
        case cudaMemoryTypeHost: return a.devicePointer;
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged: return p;
        default: return nullptr;
    }
}

}  // namespace

extern "C" {

mnb_status mnb_matmul_host_io(const mnb_matmul_args* args) {
    if (!args) return MNB_ERR_INVALID_ARG;
    const mnb_matmul_args& a = *args;
    const bool dt_ok = (a.act_dtype == MNB_F32 || a.act_dtype == MNB_F16 || a.act_dtype == MNB_BF16);
    if (!dt_ok || a.M < 0 || mnb_packed_size(a.N, a.K, a.bits, a.block_size) == 0) return MNB_ERR_INVALID_ARG;
    if (a.M == 0) return mnb_matmul_ex(args);
    if (!a.x || !a.y) return MNB_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a.x) & 15) || (reinterpret_cast<uintptr_t>(a.y) & 15))
        return MNB_ERR_INVALID_ARG;
    const size_t elt = a.act_dtype == MNB_F32 ? 4 : 2;
    if ((uint64_t)a.M > kXBytes || (uint64_t)a.K > kXBytes || (size_t)a.M * (size_t)a.K * elt > kXBytes)
        return MNB_ERR_NO_MEM;
    const size_t x_bytes = (size_t)a.M * (size_t)a.K * elt;

    cudaStream_t s = (cudaStream_t)a.stream;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        cudaGetLastError();
        return MNB_ERR_CUDA;
    }
    const void* x_dev = a.x;
    void* y_dev = a.y;
    if (cap == cudaStreamCaptureStatusNone) {
        x_dev = device_alias(a.x);
        y_dev = const_cast<void*>(device_alias(a.y));
        if (!x_dev || !y_dev) return MNB_ERR_INVALID_ARG;
    }
    void* xbuf = nullptr;
    if (x_buffer_for_current_device(&xbuf) != cudaSuccess) {
        cudaGetLastError();
        return MNB_ERR_CUDA;
    }
    if (mnb::inject_launch_failure()) return MNB_ERR_CUDA;

    const int64_t n16 = (int64_t)(x_bytes / 16);
    const int tail = (int)(x_bytes % 16);
    int sms = mnb::device_info().sm_count;
    if (sms <= 0) sms = 1;
    int64_t grid = (n16 + kFetchThreads - 1) / kFetchThreads;
    if (grid > 2 * (int64_t)sms) grid = 2 * (int64_t)sms;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kFetchThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (a.flags & MNB_FLAG_PDL) ? 1 : 0;
    const uint4* src = static_cast<const uint4*>(x_dev);
    uint4* dst = static_cast<uint4*>(xbuf);
    if (cudaLaunchKernelEx(&cfg, fetch_kernel, src, dst, n16, tail) != cudaSuccess) {
        cudaGetLastError();
        return MNB_ERR_CUDA;
    }

    mnb_matmul_args b = a;
    b.x = xbuf;
    b.y = y_dev;
    b.flags |= MNB_FLAG_PDL;
    return mnb_matmul_ex(&b);
}

}  // extern "C"
