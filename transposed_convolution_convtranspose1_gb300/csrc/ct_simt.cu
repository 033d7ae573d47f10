// ct_simt.cu -- fp32 stride-phase implicit GEMM on CUDA cores.
#include "ct_routes.h"

namespace ct {

bool simt_supports(const Problem&) { return false; }
bool simt_preferred(const Problem&) { return false; }
size_t simt_workspace_bytes(const Problem&) { return 0; }
cudaError_t launch_simt(const Problem&, const void*, const void*, const void*, void*, void*,
                        cudaStream_t, Profile*) {
    return cudaErrorNotSupported;
}

}  // namespace ct
