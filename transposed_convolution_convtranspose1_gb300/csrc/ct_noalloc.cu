// ct_noalloc.cu -- the forward transposed convolution for callers that must
// not allocate device memory.
//
// Some callers cannot call cudaMalloc (or cudaMallocAsync) at the point where
// they run the convolution: code that runs while a CUDA graph is being
// captured with allocation forbidden, plugins of inference engines whose
// enqueue step may only use memory the engine handed out, frameworks that own
// the whole device memory budget through their own pool, and real-time
// callers that allow no allocation after start-up.  For them this file keeps
// the scratch space the kernels need (the reordered weights and the
// channels-last copy of x of the tensor-core route) in one statically sized
// device array, so the call itself allocates nothing.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "ct_internal.h"

namespace ct {

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CT_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch for the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
cudaError_t noalloc_scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace ct

extern "C" int ct_conv_transpose_nd_noalloc(const void* x, const void* w, const void* bias, void* y,
                                            int nd, int64_t B, int64_t C_in, int64_t C_out,
                                            const int64_t* in_spatial, const int64_t* k,
                                            const int* stride, const int* pad_lo,
                                            const int* pad_hi, const int* dilation,
                                            const int* output_padding, int groups, int dtype,
                                            void* stream) {
    // Scratch this problem needs on the route the library picks for it
    // (also validates every argument).
    size_t need = 0;
    int rc = ct_conv_transpose_workspace_bytes(nd, B, C_in, C_out, in_spatial, k, stride, pad_lo,
                                               pad_hi, dilation, output_padding, groups, dtype,
                                               &need);
    if (rc != CT_OK) return rc;
    if (need > (size_t)CT_NOALLOC_SCRATCH_BYTES)
        return ct::report_error(CT_ERR_WORKSPACE,
                                "this problem needs %zu bytes of scratch; the no-allocation entry "
                                "point has a fixed %zu bytes (use ct_conv_transpose_nd with a "
                                "workspace instead)",
                                need, (size_t)CT_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    if (need > 0) {
        cudaError_t e = ct::noalloc_scratch_address(&scratch);
        if (e != cudaSuccess)
            return ct::report_error(CT_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                                    cudaGetErrorString(e));
    }
    // With a workspace supplied, ct_conv_transpose_nd allocates nothing.
    return ct_conv_transpose_nd(x, w, bias, y, scratch, (size_t)CT_NOALLOC_SCRATCH_BYTES, nd, B,
                                C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                                output_padding, groups, dtype, stream);
}
