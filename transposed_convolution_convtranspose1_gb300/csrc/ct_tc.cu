// ct_tc.cu -- tensor-core (tcgen05) stride-phase implicit GEMM route.
#include "ct_routes.h"

namespace ct {

// Error word written by bounded device-side waits (0 = none).
__device__ unsigned int g_device_error = 0;

bool tc_supports(const Problem&) { return false; }
bool tc_preferred(const Problem&) { return false; }
size_t tc_workspace_bytes(const Problem&) { return 0; }
cudaError_t launch_tc(const Problem&, const void*, const void*, const void*, void*, void*,
                      cudaStream_t, Profile*) {
    return cudaErrorNotSupported;
}

}  // namespace ct

extern "C" int ct_device_status(int clear, unsigned int* code) {
    unsigned int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, ct::g_device_error, sizeof(v));
    if (e == cudaSuccess && clear && v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(ct::g_device_error, &zero, sizeof(zero));
    }
    if (code) *code = v;
    if (e != cudaSuccess) return CT_ERR_CUDA;
    return v ? CT_ERR_DEVICE_TIMEOUT : CT_OK;
}
