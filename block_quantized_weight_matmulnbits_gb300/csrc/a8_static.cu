// int8-activation matmul without a caller workspace (mnb_matmul_a8_static):
// the quantised activations and block scales go to a file-scope device array
// instead of memory the caller allocates.  The library allocates nothing.
#include <cstring>
#include <mutex>

#include "mnb.h"
#include "mnb_internal.h"

namespace {

constexpr size_t kScratchBytes = MNB_A8_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// One per device (a __device__ variable exists once in every context).
static __device__ __align__(256) uint8_t g_a8_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Address of this device's array, looked up once per device.
cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_a8_scratch);
        if (e != cudaSuccess) return e;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

mnb_status mnb_matmul_a8_static(const void* x, const void* packed_b, const void* scales,
                                const uint8_t* zero_points, void* y, int64_t M, int64_t N, int64_t K, int bits,
                                int block_size, mnb_dtype act_dtype, mnb_dtype out_dtype, mnb_dtype scale_dtype,
                                mnb_stream_t stream) {
    if (mnb_workspace_size(M, N, K, bits, block_size, 4) > kScratchBytes) return MNB_ERR_NO_MEM;
    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MNB_ERR_CUDA;
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
    a.accuracy_level = 4;
    a.workspace = scratch;
    a.workspace_bytes = kScratchBytes;
    a.kernel = MNB_KERNEL_AUTO;
    a.stream = stream;
    return mnb_matmul_ex(&a);
}

}  // extern "C"
