// Kernel families not built yet: they decline every call, so dispatch falls
// back to a kernel that exists and forced calls report MNB_ERR_UNSUPPORTED.
#include "mnb_internal.h"

namespace mnb {

size_t i8_workspace_bytes(int64_t, const Layout&) { return 0; }
bool gemv_i8_supported(const MatmulParams&) { return false; }
cudaError_t launch_quant_act(const void*, int, int8_t*, float*, int64_t, const Layout&, cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_gemv_i8(const MatmulParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace mnb
