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

#include <cuda.h>
#include <cudaTypedefs.h>

#include "ct_internal.h"

namespace ct {

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CT_NOALLOC_SCRATCH_BYTES];

namespace {

// Driver entry points naming the current context (no link-time dependency on
// libcuda; the runtime hands them out).
struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 current = nullptr;
    PFN_cuCtxGetId_v12000 id = nullptr;
};

const CtxFns& ctx_fns() {
    static std::once_flag once;
    static CtxFns f;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            f.current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            f.id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    return f;
}

// Device address of g_noalloc_scratch for the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with that device current and cached together with the unique id of the
// device's context.  The look-up runs again whenever that id changes, so a
// cudaDeviceReset (which destroys the context and, with it, the module that
// holds the array) costs one more look-up instead of leaving a dead address.
cudaError_t noalloc_scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    static unsigned long long ctx_id[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    // the device's primary context current (the runtime creates it if needed)
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    const CtxFns& f = ctx_fns();
    unsigned long long id = 0;
    CUcontext ctx = nullptr;
    if (!f.current || !f.id || f.current(&ctx) != CUDA_SUCCESS || !ctx || f.id(ctx, &id) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || ctx_id[dev] != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
        ctx_id[dev] = id;
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
