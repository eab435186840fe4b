// int8-activation matmul without a caller workspace (mnb_matmul_a8_static):
// the quantised activations and block scales go to a file-scope device array
// instead of memory the caller allocates.  The library allocates nothing.
#include <cstring>

#include "mnb.h"
#include "mnb_internal.h"

namespace {

constexpr size_t kScratchBytes = MNB_A8_STATIC_SCRATCH_BYTES;

// One per device (a __device__ variable exists once in every context).
static __device__ __align__(256) uint8_t g_a8_scratch[kScratchBytes];

// In host code g_a8_scratch names a host-side stand-in, not device memory:
// kernels get the device address that cudaGetSymbolAddress reports for the
// current context (the device current at the call).
cudaError_t lookup_scratch(void** p) { return cudaGetSymbolAddress(p, g_a8_scratch); }
mnb::SymbolCache g_scratch_cache;

// Address of the current context's array: looked up on the first call in a
// context (device), then cached per context.
cudaError_t scratch_for_current_device(void** out) {
    return mnb::cached_symbol_address(g_scratch_cache, lookup_scratch, out);
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
