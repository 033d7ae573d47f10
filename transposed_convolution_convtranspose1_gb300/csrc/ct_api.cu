// ct_api.cu -- host side of the C ABI: validation, output shape, stride-phase
// plan, route choice, workspace sizing and dispatch.  No device code here.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include "ct_internal.h"
#include "ct_routes.h"

namespace ct {
namespace {

thread_local char g_msg[512] = "";

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char* where) {
    return fail(CT_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Output extent of one axis (SKaiNET #1464 Summary "output size", with the
// NKI page's separate low/high pads).
int64_t out_extent(int64_t I, int64_t K, int64_t S, int64_t PL, int64_t PH, int64_t DL,
                   int64_t OP) {
    return (I - 1) * S - PL - PH + DL * (K - 1) + OP + 1;
}

// Checks the per-axis attributes and fills the normalised axis fields.
// The rules are those SKaiNET #1464 lists for its CPU kernel: positive
// stride and dilation, non-negative padding and
// output_padding < max(stride, dilation) per axis.
int fill_axes(Problem* p, int nd, const int64_t* in_spatial, const int64_t* k, const int* stride,
              const int* pad_lo, const int* pad_hi, const int* dilation,
              const int* output_padding) {
    if (nd < 1 || nd > 3) return fail(CT_ERR_RANK, "nd must be 1, 2 or 3 (got %d)", nd);
    if (!in_spatial || !k || !stride || !pad_lo || !pad_hi || !dilation || !output_padding)
        return fail(CT_ERR_NULL, "a per-axis attribute array is NULL");
    p->nd = nd;
    for (int a = 0; a < 3; ++a) {
        p->I[a] = 1; p->K[a] = 1; p->O[a] = 1;
        p->S[a] = 1; p->PL[a] = 0; p->PH[a] = 0; p->DL[a] = 1; p->OP[a] = 0;
    }
    for (int j = 0; j < nd; ++j) {
        const int a = 3 - nd + j;
        if (in_spatial[j] < 0) return fail(CT_ERR_SHAPE, "input extent of axis %d is negative", j);
        if (k[j] < 1) return fail(CT_ERR_PARAM, "kernel size of axis %d must be >= 1", j);
        if (stride[j] < 1) return fail(CT_ERR_PARAM, "stride of axis %d must be >= 1", j);
        if (dilation[j] < 1) return fail(CT_ERR_PARAM, "dilation of axis %d must be >= 1", j);
        if (pad_lo[j] < 0 || pad_hi[j] < 0)
            return fail(CT_ERR_PARAM, "padding of axis %d must be >= 0", j);
        const int lim = stride[j] > dilation[j] ? stride[j] : dilation[j];
        if (output_padding[j] < 0 || output_padding[j] >= lim)
            return fail(CT_ERR_PARAM,
                        "output_padding of axis %d must be in [0, max(stride, dilation)) = [0, %d)",
                        j, lim);
        if (k[j] > kMaxK || stride[j] > kMaxStride)
            return fail(CT_ERR_TOO_LARGE, "axis %d: kernel size <= %d and stride <= %d supported", j,
                        kMaxK, kMaxStride);
        if (in_spatial[j] > (1ll << 30) || dilation[j] > (1 << 20) || pad_lo[j] > (1 << 30) ||
            pad_hi[j] > (1 << 30))
            return fail(CT_ERR_TOO_LARGE, "axis %d: size or attribute too large", j);
        p->I[a] = in_spatial[j]; p->K[a] = k[j]; p->S[a] = stride[j];
        p->PL[a] = pad_lo[j]; p->PH[a] = pad_hi[j]; p->DL[a] = dilation[j];
        p->OP[a] = output_padding[j];
        p->O[a] = out_extent(p->I[a], p->K[a], p->S[a], p->PL[a], p->PH[a], p->DL[a], p->OP[a]);
        if (p->O[a] < 1)
            return fail(CT_ERR_SHAPE, "output extent of axis %d would be %lld (< 1)", j,
                        (long long)p->O[a]);
        if (p->O[a] > (1ll << 31) - 1)
            return fail(CT_ERR_TOO_LARGE, "output extent of axis %d exceeds 2^31-1", j);
    }
    return CT_OK;
}

int validate(Problem* p, int nd, int64_t B, int64_t C_in, int64_t C_out, const int64_t* in_spatial,
             const int64_t* k, const int* stride, const int* pad_lo, const int* pad_hi,
             const int* dilation, const int* output_padding, int groups, int dtype) {
    *p = Problem{};
    int rc = fill_axes(p, nd, in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding);
    if (rc != CT_OK) return rc;
    if (dtype != CT_F32 && dtype != CT_F16 && dtype != CT_BF16)
        return fail(CT_ERR_DTYPE,
                    "dtype %d is not a supported floating type (CT_F32, CT_F16, CT_BF16)", dtype);
    if (B < 0 || C_in < 0 || C_out < 0) return fail(CT_ERR_SHAPE, "B, C_in and C_out must be >= 0");
    if (groups < 1) return fail(CT_ERR_GROUPS, "groups must be >= 1 (got %d)", groups);
    if (C_in % groups != 0 || C_out % groups != 0)
        return fail(CT_ERR_GROUPS, "groups=%d must divide C_in=%lld and C_out=%lld", groups,
                    (long long)C_in, (long long)C_out);
    if (C_in > (1 << 24) || C_out > (1 << 24) || B > (1ll << 31))
        return fail(CT_ERR_TOO_LARGE, "B, C_in or C_out too large");
    p->B = B; p->C_in = C_in; p->C_out = C_out; p->G = groups;
    p->Cig = (int)(C_in / groups); p->Cog = (int)(C_out / groups);
    p->dtype = (ct_dtype)dtype;
    const double xe = (double)B * C_in * p->in_spatial();
    const double ye = (double)B * C_out * p->out_spatial();
    const double we = (double)C_in * p->Cog * p->taps();
    if (xe > 4e18 || ye > 4e18 || we > 4e18) return fail(CT_ERR_TOO_LARGE, "tensor too large");
    return CT_OK;
}

bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

bool route_supports(const Problem& p, int route) {
    const bool empty_out = p.y_elems() == 0;
    const bool no_input = p.C_in == 0 || p.in_spatial() == 0;
    switch (route) {
        case CT_ROUTE_NONE: return empty_out;
        case CT_ROUTE_BIAS_FILL: return !empty_out && no_input;
        case CT_ROUTE_GATHER: return !empty_out && !no_input;
        case CT_ROUTE_GROUPED: return !empty_out && !no_input && grouped_supports(p);
        case CT_ROUTE_SIMT_GEMM: return !empty_out && !no_input && simt_supports(p);
        case CT_ROUTE_TC_GEMM: return !empty_out && !no_input && tc_supports(p);
        case CT_ROUTE_TC32_GEMM: return !empty_out && !no_input && tc32_supports(p);
        default: return false;
    }
}

int choose_route(const Problem& p) {
    if (p.y_elems() == 0) return CT_ROUTE_NONE;
    if (p.C_in == 0 || p.in_spatial() == 0) return CT_ROUTE_BIAS_FILL;
    if (route_supports(p, CT_ROUTE_TC_GEMM) && tc_preferred(p)) return CT_ROUTE_TC_GEMM;
    if (route_supports(p, CT_ROUTE_TC32_GEMM) && tc32_preferred(p)) return CT_ROUTE_TC32_GEMM;
    if (route_supports(p, CT_ROUTE_SIMT_GEMM) && simt_preferred(p)) return CT_ROUTE_SIMT_GEMM;
    if (route_supports(p, CT_ROUTE_GROUPED) && grouped_preferred(p)) return CT_ROUTE_GROUPED;
    return CT_ROUTE_GATHER;
}

size_t route_workspace(const Problem& p, int route) {
    switch (route) {
        case CT_ROUTE_SIMT_GEMM: return simt_workspace_bytes(p);
        case CT_ROUTE_TC_GEMM: return tc_workspace_bytes(p);
        case CT_ROUTE_TC32_GEMM: return tc32_workspace_bytes(p);
        default: return 0;
    }
}

int run(const Problem& p, int route, const void* x, const void* w, const void* bias, void* y,
        void* workspace, size_t workspace_bytes, cudaStream_t stream, Profile* prof) {
    const size_t need = route_workspace(p, route);
    void* ws = workspace;
    bool owned = false;
    if (need > 0) {
        if (ws) {
            if (workspace_bytes < need)
                return fail(CT_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                            workspace_bytes, need);
            if (!aligned(ws, 256)) return fail(CT_ERR_ALIGN, "workspace must be 256-byte aligned");
        } else {
            cudaError_t e = cudaMallocAsync(&ws, need, stream);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
            owned = true;
        }
    }
    cudaError_t e = cudaSuccess;
    bool act_done = false;
    switch (route) {
        case CT_ROUTE_NONE: break;
        case CT_ROUTE_BIAS_FILL: e = launch_bias_fill(p, bias, y, stream, prof); break;
        case CT_ROUTE_GATHER: e = launch_gather(p, x, w, bias, y, stream, prof); break;
        case CT_ROUTE_GROUPED: e = launch_grouped(p, x, w, bias, y, stream, prof, &act_done); break;
        case CT_ROUTE_SIMT_GEMM: e = launch_simt(p, x, w, bias, y, ws, stream, prof); break;
        case CT_ROUTE_TC_GEMM: e = launch_tc(p, x, w, bias, y, ws, stream, prof); break;
        case CT_ROUTE_TC32_GEMM: e = launch_tc32(p, x, w, bias, y, ws, stream, prof); break;
        default: e = cudaErrorInvalidValue; break;
    }
    // the CUDA-core routes without a fused activation apply it as a second
    // pass over y (the tcgen05 routes, the bias fill and the grouped warp
    // kernel fuse it into their epilogues)
    if (e == cudaSuccess && p.act != 0 && !act_done &&
        (route == CT_ROUTE_GATHER || route == CT_ROUTE_GROUPED || route == CT_ROUTE_SIMT_GEMM))
        e = launch_activation(p, y, stream, prof);
    if (owned) {
        cudaError_t e2 = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return CT_OK;
}

// Resources of the host-buffer entry point, one set per device, created on
// first use and kept until process exit: a stream-ordered memory pool that
// keeps its memory between calls (no re-mapping per call; returned by
// ct_host_buffers_release), two non-blocking side streams (input and output
// copies) and the events that order the pipeline.
constexpr size_t kHostPipelineMinBytes = 8u << 20;  // smaller calls run as one chunk
constexpr int kHostMaxChunks = 8;

struct HostRes {
    std::mutex mu;
    cudaMemPool_t pool = nullptr;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_done_in = nullptr, ev_done_out = nullptr;
    cudaEvent_t ev_in[kHostMaxChunks] = {}, ev_comp[kHostMaxChunks] = {};
};

cudaError_t host_resources(HostRes** out) {
    static std::mutex mu;
    static HostRes* res[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (res[dev]) {
        *out = res[dev];
        return cudaSuccess;
    }
    HostRes* R = new HostRes();
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    e = cudaMemPoolCreate(&R->pool, &props);
    if (e == cudaSuccess) {
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(R->pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&R->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&R->s_out, cudaStreamNonBlocking);
    cudaEvent_t* evs[3] = {&R->ev_start, &R->ev_done_in, &R->ev_done_out};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
    for (int i = 0; i < kHostMaxChunks && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&R->ev_in[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&R->ev_comp[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return e;  // leaks the partial set; the device is unusable anyway
    res[dev] = R;
    *out = R;
    return cudaSuccess;
}

int check_pointers(const Problem& p, const void* x, const void* w, const void* bias, const void* y) {
    if (p.x_elems() > 0 && !x) return fail(CT_ERR_NULL, "x is NULL");
    if (p.w_elems() > 0 && !w) return fail(CT_ERR_NULL, "w is NULL");
    if (p.y_elems() > 0 && !y) return fail(CT_ERR_NULL, "y is NULL");
    const size_t eb = p.elem_bytes();
    if (!aligned(x, eb) || !aligned(w, eb) || !aligned(y, eb) || !aligned(bias, eb))
        return fail(CT_ERR_ALIGN, "pointers must be aligned to the element size (%zu bytes)", eb);
    return CT_OK;
}

}  // namespace

int report_error(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return status;
}

void plan_axis(const Problem& p, int axis, AxisPlan* out) {
    const int s = p.S[axis];
    out->s = s;
    for (int r = 0; r < s; ++r) {
        out->q_extent[r] = (r < p.O[axis]) ? (p.O[axis] - r + s - 1) / s : 0;
        int n = 0;
        // Walk taps from high to low so that input offsets come out increasing.
        for (int t = (int)p.K[axis] - 1; t >= 0; --t) {
            const int64_t v = (int64_t)r + p.PL[axis] - (int64_t)t * p.DL[axis];
            const int64_t m = ((v % s) + s) % s;
            if (m != 0) continue;
            out->tap[r][n] = t;
            out->off[r][n] = (int)(v / s);  // exact: v is a multiple of s
            ++n;
        }
        out->ntaps[r] = n;
    }
}

namespace {
std::atomic<uint64_t> g_wait_limit_ns{CT_WAIT_LIMIT_DEFAULT_NS};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

cudaError_t device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && have[dev]) {
        *out = cache[dev];
        return cudaSuccess;
    }
    DeviceInfo d{};
    d.device = dev;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) return e;
    int optin = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    d.smem_optin = (size_t)optin;
    if (dev >= 0 && dev < 64) {
        cache[dev] = d;
        have[dev] = true;
    }
    *out = d;
    return cudaSuccess;
}

}  // namespace ct

using namespace ct;

extern "C" {

int ct_version(void) { return 100; }

unsigned long long ct_set_wait_limit_ns(unsigned long long ns) {
    return g_wait_limit_ns.exchange(ns);
}

const char* ct_last_error(void) { return g_msg; }

const char* ct_status_string(int status) {
    switch (status) {
        case CT_OK: return "CT_OK";
        case CT_ERR_NULL: return "CT_ERR_NULL";
        case CT_ERR_RANK: return "CT_ERR_RANK";
        case CT_ERR_SHAPE: return "CT_ERR_SHAPE";
        case CT_ERR_PARAM: return "CT_ERR_PARAM";
        case CT_ERR_GROUPS: return "CT_ERR_GROUPS";
        case CT_ERR_BIAS: return "CT_ERR_BIAS";
        case CT_ERR_DTYPE: return "CT_ERR_DTYPE";
        case CT_ERR_CUDA: return "CT_ERR_CUDA";
        case CT_ERR_DEVICE_TIMEOUT: return "CT_ERR_DEVICE_TIMEOUT";
        case CT_ERR_WORKSPACE: return "CT_ERR_WORKSPACE";
        case CT_ERR_ALIGN: return "CT_ERR_ALIGN";
        case CT_ERR_ROUTE: return "CT_ERR_ROUTE";
        case CT_ERR_TOO_LARGE: return "CT_ERR_TOO_LARGE";
        default: return "unknown status";
    }
}

int ct_conv_transpose_out_shape(int nd, const int64_t* in_spatial, const int64_t* k,
                                const int* stride, const int* pad_lo, const int* pad_hi,
                                const int* dilation, const int* output_padding,
                                int64_t* out_spatial) {
    Problem p;
    p = Problem{};
    int rc = fill_axes(&p, nd, in_spatial, k, stride, pad_lo, pad_hi, dilation, output_padding);
    if (rc != CT_OK) return rc;
    if (!out_spatial) return fail(CT_ERR_NULL, "out_spatial is NULL");
    for (int j = 0; j < nd; ++j) out_spatial[j] = p.O[3 - nd + j];
    return CT_OK;
}

int ct_conv_transpose_route(int nd, int64_t B, int64_t C_in, int64_t C_out,
                            const int64_t* in_spatial, const int64_t* k, const int* stride,
                            const int* pad_lo, const int* pad_hi, const int* dilation,
                            const int* output_padding, int groups, int dtype, int* route) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    if (!route) return fail(CT_ERR_NULL, "route is NULL");
    *route = choose_route(p);
    return CT_OK;
}

int ct_conv_transpose_kernel(int nd, int64_t B, int64_t C_in, int64_t C_out,
                             const int64_t* in_spatial, const int64_t* k, const int* stride,
                             const int* pad_lo, const int* pad_hi, const int* dilation,
                             const int* output_padding, int groups, int dtype, const char** name) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    if (!name) return fail(CT_ERR_NULL, "name is NULL");
    switch (choose_route(p)) {
        case CT_ROUTE_TC_GEMM: *name = "tc_phase_gemm"; break;
        case CT_ROUTE_TC32_GEMM: *name = "tc32_phase_gemm"; break;
        case CT_ROUTE_SIMT_GEMM: *name = "simt_phase_gemm"; break;
        case CT_ROUTE_GROUPED: *name = grouped_kernel_name(p); break;
        case CT_ROUTE_GATHER: *name = "gather_kernel"; break;
        case CT_ROUTE_BIAS_FILL: *name = "bias_fill_kernel"; break;
        default: *name = ""; break;
    }
    return CT_OK;
}

int ct_conv_transpose_route_workspace_bytes(int nd, int64_t B, int64_t C_in, int64_t C_out,
                                            const int64_t* in_spatial, const int64_t* k,
                                            const int* stride, const int* pad_lo,
                                            const int* pad_hi, const int* dilation,
                                            const int* output_padding, int groups, int dtype,
                                            int route, size_t* bytes) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    if (!bytes) return fail(CT_ERR_NULL, "bytes is NULL");
    if (route == CT_ROUTE_AUTO) route = choose_route(p);
    if (!route_supports(p, route)) return fail(CT_ERR_ROUTE, "route %d cannot run this problem", route);
    *bytes = route_workspace(p, route);
    return CT_OK;
}

int ct_conv_transpose_workspace_bytes(int nd, int64_t B, int64_t C_in, int64_t C_out,
                                      const int64_t* in_spatial, const int64_t* k,
                                      const int* stride, const int* pad_lo, const int* pad_hi,
                                      const int* dilation, const int* output_padding, int groups,
                                      int dtype, size_t* bytes) {
    return ct_conv_transpose_route_workspace_bytes(nd, B, C_in, C_out, in_spatial, k, stride,
                                                   pad_lo, pad_hi, dilation, output_padding,
                                                   groups, dtype, CT_ROUTE_AUTO, bytes);
}

int ct_conv_transpose_nd_profiled(const void* x, const void* w, const void* bias, void* y,
                                  void* workspace, size_t workspace_bytes, int nd, int64_t B,
                                  int64_t C_in, int64_t C_out, const int64_t* in_spatial,
                                  const int64_t* k, const int* stride, const int* pad_lo,
                                  const int* pad_hi, const int* dilation,
                                  const int* output_padding, int groups, int dtype, int route,
                                  void* stream, void* main_start, void* main_stop, int* launches,
                                  int* route_taken) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    rc = check_pointers(p, x, w, bias, y);
    if (rc != CT_OK) return rc;
    if (route == CT_ROUTE_AUTO) {
        route = choose_route(p);
    } else if (!route_supports(p, route)) {
        return fail(CT_ERR_ROUTE, "route %d cannot run this problem", route);
    }
    Profile prof;
    prof.main_start = (cudaEvent_t)main_start;
    prof.main_stop = (cudaEvent_t)main_stop;
    rc = run(p, route, x, w, bias, y, workspace, workspace_bytes, (cudaStream_t)stream, &prof);
    if (launches) *launches = prof.launches;
    if (route_taken) *route_taken = route;
    return rc;
}

int ct_conv_transpose_nd_route(const void* x, const void* w, const void* bias, void* y,
                               void* workspace, size_t workspace_bytes, int nd, int64_t B,
                               int64_t C_in, int64_t C_out, const int64_t* in_spatial,
                               const int64_t* k, const int* stride, const int* pad_lo,
                               const int* pad_hi, const int* dilation, const int* output_padding,
                               int groups, int dtype, int route, void* stream) {
    return ct_conv_transpose_nd_profiled(x, w, bias, y, workspace, workspace_bytes, nd, B, C_in,
                                         C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                                         output_padding, groups, dtype, route, stream, nullptr,
                                         nullptr, nullptr, nullptr);
}

int ct_conv_transpose_nd(const void* x, const void* w, const void* bias, void* y, void* workspace,
                         size_t workspace_bytes, int nd, int64_t B, int64_t C_in, int64_t C_out,
                         const int64_t* in_spatial, const int64_t* k, const int* stride,
                         const int* pad_lo, const int* pad_hi, const int* dilation,
                         const int* output_padding, int groups, int dtype, void* stream) {
    return ct_conv_transpose_nd_route(x, w, bias, y, workspace, workspace_bytes, nd, B, C_in, C_out,
                                      in_spatial, k, stride, pad_lo, pad_hi, dilation,
                                      output_padding, groups, dtype, CT_ROUTE_AUTO, stream);
}

int ct_conv_transpose_nd_host(const void* x, const void* w, const void* bias, void* y, int nd,
                              int64_t B, int64_t C_in, int64_t C_out, const int64_t* in_spatial,
                              const int64_t* k, const int* stride, const int* pad_lo,
                              const int* pad_hi, const int* dilation, const int* output_padding,
                              int groups, int dtype, void* stream) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    rc = check_pointers(p, x, w, bias, y);
    if (rc != CT_OK) return rc;
    HostRes* R = nullptr;
    cudaError_t e = host_resources(&R);
    if (e != cudaSuccess) return cuda_fail(e, "host call resources");
    std::lock_guard<std::mutex> lock(R->mu);  // the side streams and events are shared
    cudaStream_t s = (cudaStream_t)stream;
    const size_t eb = p.elem_bytes();
    const size_t wb = (size_t)p.w_elems() * eb;
    const size_t bb = bias ? (size_t)p.C_out * eb : 0;
    // batch chunks: chunk c's input copy, compute and output copy run on
    // three streams, so that copies in both directions overlap the compute
    const size_t xb_all = (size_t)p.x_elems() * eb, yb_all = (size_t)p.y_elems() * eb;
    int64_t nchunk = 1;
    if (p.B > 1 && xb_all + yb_all >= kHostPipelineMinBytes)
        nchunk = std::min<int64_t>(p.B, kHostMaxChunks);
    const int64_t bc = (p.B + nchunk - 1) / nchunk;  // batch elements per chunk
    nchunk = p.B > 0 ? (p.B + bc - 1) / bc : 1;
    const size_t xb1 = (size_t)(p.x_elems() / std::max<int64_t>(p.B, 1)) * eb;  // per batch element
    const size_t yb1 = (size_t)(p.y_elems() / std::max<int64_t>(p.B, 1)) * eb;
    Problem pc = p;  // the largest and the last chunk size the workspace
    pc.B = std::min<int64_t>(bc, p.B);
    size_t ws = route_workspace(pc, choose_route(pc));
    pc.B = p.B - (nchunk - 1) * bc;
    if (pc.B > 0) ws = std::max(ws, route_workspace(pc, choose_route(pc)));
    auto round = [](size_t n) { return (n + 255) / 256 * 256; };
    const size_t total = round(xb_all) + round(wb) + round(bb) + round(yb_all) + round(ws);
    char* base = nullptr;
    if (total > 0) {
        e = cudaMallocFromPoolAsync((void**)&base, total, R->pool, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync(host call buffers)");
    }
    char* dx = base;
    char* dw = dx + round(xb_all);
    char* db = dw + round(wb);
    char* dy = db + round(bb);
    char* dws = dy + round(yb_all);
    rc = CT_OK;
    // the side streams start after everything already queued on `stream`
    e = cudaEventRecord(R->ev_start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(R->s_in, R->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(R->s_out, R->ev_start, 0);
    if (e == cudaSuccess && wb) e = cudaMemcpyAsync(dw, w, wb, cudaMemcpyHostToDevice, R->s_in);
    if (e == cudaSuccess && bb) e = cudaMemcpyAsync(db, bias, bb, cudaMemcpyHostToDevice, R->s_in);
    if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync(host to device)");
    for (int64_t c = 0; c < nchunk && rc == CT_OK; ++c) {
        const int64_t b0 = c * bc, nb = std::min(bc, p.B - b0);
        const size_t xo = (size_t)b0 * xb1, yo = (size_t)b0 * yb1;
        if (nb > 0 && xb1 > 0)
            e = cudaMemcpyAsync(dx + xo, static_cast<const char*>(x) + xo, nb * xb1,
                                cudaMemcpyHostToDevice, R->s_in);
        if (e == cudaSuccess) e = cudaEventRecord(R->ev_in[c], R->s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, R->ev_in[c], 0);
        if (e != cudaSuccess) {
            rc = cuda_fail(e, "cudaMemcpyAsync(host to device)");
            break;
        }
        rc = ct_conv_transpose_nd(dx + xo, dw, bias ? db : nullptr, dy + yo, ws ? dws : nullptr, ws,
                                  nd, nb, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi,
                                  dilation, output_padding, groups, dtype, stream);
        if (rc != CT_OK) break;
        e = cudaEventRecord(R->ev_comp[c], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(R->s_out, R->ev_comp[c], 0);
        if (e == cudaSuccess && nb > 0 && yb1 > 0)
            e = cudaMemcpyAsync(static_cast<char*>(y) + yo, dy + yo, nb * yb1, cudaMemcpyDeviceToHost,
                                R->s_out);
        if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync(device to host)");
    }
    // `stream` waits for both side streams before the buffers go back to the pool
    cudaError_t e2 = cudaEventRecord(R->ev_done_in, R->s_in);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, R->ev_done_in, 0);
    if (e2 == cudaSuccess) e2 = cudaEventRecord(R->ev_done_out, R->s_out);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, R->ev_done_out, 0);
    if (base) cudaFreeAsync(base, s);
    e = cudaStreamSynchronize(s);
    if (rc == CT_OK && e2 != cudaSuccess) rc = cuda_fail(e2, "ordering the host call's streams");
    if (rc == CT_OK && e != cudaSuccess) rc = cuda_fail(e, "cudaStreamSynchronize");
    return rc;
}

// Options of the extended call: weight layout (0 PyTorch, 1 [k...][C_in][C_out],
// 2 [k...][C_out][C_in]; 1 and 2 need groups == 1), taps stored reversed,
// epilogue activation code (0..6) and its parameter.
static int ex_options(Problem* p, int w_layout, int taps_flipped, int activation,
                      float activation_alpha) {
    if (w_layout < 0 || w_layout > 2) return fail(CT_ERR_PARAM, "w_layout must be 0, 1 or 2 (got %d)", w_layout);
    if (w_layout != 0 && p->G != 1)
        return fail(CT_ERR_GROUPS, "weight layouts 1 and 2 are defined for groups == 1 only");
    if (taps_flipped != 0 && taps_flipped != 1) return fail(CT_ERR_PARAM, "taps_flipped must be 0 or 1");
    if (activation < CT_ACT_NONE || activation > CT_ACT_SIGMOID)
        return fail(CT_ERR_PARAM, "unknown activation %d", activation);
    p->act = activation;
    p->act_alpha = activation_alpha;
    return CT_OK;
}

int ct_conv_transpose_ex_workspace_bytes(int nd, int64_t B, int64_t C_in, int64_t C_out,
                                         const int64_t* in_spatial, const int64_t* k,
                                         const int* stride, const int* pad_lo, const int* pad_hi,
                                         const int* dilation, const int* output_padding,
                                         int groups, int dtype, int w_layout, int taps_flipped,
                                         size_t* bytes) {
    if (!bytes) return fail(CT_ERR_NULL, "bytes is NULL");
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    rc = ex_options(&p, w_layout, taps_flipped, CT_ACT_NONE, 0.f);
    if (rc != CT_OK) return rc;
    const bool conv = w_layout != 0 || taps_flipped != 0;
    const size_t wb = conv ? ((size_t)p.w_elems() * p.elem_bytes() + 255) / 256 * 256 : 0;
    *bytes = wb + route_workspace(p, choose_route(p));
    return CT_OK;
}

int ct_conv_transpose_nd_ex(const void* x, const void* w, const void* bias, void* y,
                            void* workspace, size_t workspace_bytes, int nd, int64_t B,
                            int64_t C_in, int64_t C_out, const int64_t* in_spatial,
                            const int64_t* k, const int* stride, const int* pad_lo,
                            const int* pad_hi, const int* dilation, const int* output_padding,
                            int groups, int dtype, int w_layout, int taps_flipped, int activation,
                            float activation_alpha, void* stream) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    rc = ex_options(&p, w_layout, taps_flipped, activation, activation_alpha);
    if (rc != CT_OK) return rc;
    rc = check_pointers(p, x, w, bias, y);
    if (rc != CT_OK) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const int route = choose_route(p);
    const bool conv = w_layout != 0 || taps_flipped != 0;
    if (!conv) return run(p, route, x, w, bias, y, workspace, workspace_bytes, s, nullptr);
    // the weights in the PyTorch layout first, in the workspace's head
    const size_t wb = ((size_t)p.w_elems() * p.elem_bytes() + 255) / 256 * 256;
    const size_t need = wb + route_workspace(p, route);
    char* ws = static_cast<char*>(workspace);
    bool owned = false;
    if (ws) {
        if (workspace_bytes < need)
            return fail(CT_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                        workspace_bytes, need);
        if (!aligned(ws, 256)) return fail(CT_ERR_ALIGN, "workspace must be 256-byte aligned");
    } else if (need > 0) {
        cudaError_t e = cudaMallocAsync((void**)&ws, need, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
        owned = true;
    }
    cudaError_t e = launch_weight_to_torch_layout(p, w, ws, w_layout, taps_flipped, s);
    if (e != cudaSuccess) rc = cuda_fail(e, "weight layout kernel");
    if (rc == CT_OK)
        rc = run(p, route, x, ws, bias, y, need > wb ? ws + wb : nullptr, need - wb, s, nullptr);
    if (owned) {
        e = cudaFreeAsync(ws, s);
        if (rc == CT_OK && e != cudaSuccess) rc = cuda_fail(e, "cudaFreeAsync(workspace)");
    }
    return rc;
}

int ct_conv_transpose_backward_workspace_bytes(int nd, int64_t B, int64_t C_in, int64_t C_out,
                                               const int64_t* in_spatial, const int64_t* k,
                                               const int* stride, const int* pad_lo,
                                               const int* pad_hi, const int* dilation,
                                               const int* output_padding, int groups, int dtype,
                                               size_t* bytes) {
    if (!bytes) return fail(CT_ERR_NULL, "bytes is NULL");
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    if (!backward_supported(p))
        return fail(CT_ERR_TOO_LARGE, "backward: %lld taps per input channel block exceed the staged slab",
                    (long long)p.taps());
    *bytes = backward_workspace_bytes(p);
    return CT_OK;
}

int ct_conv_transpose_backward_kernels(int nd, int64_t B, int64_t C_in, int64_t C_out,
                                       const int64_t* in_spatial, const int64_t* k, const int* stride,
                                       const int* pad_lo, const int* pad_hi, const int* dilation,
                                       const int* output_padding, int groups, int dtype,
                                       const char** dx_kernel, const char** dw_kernel) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    if (!dx_kernel || !dw_kernel) return fail(CT_ERR_NULL, "kernel name pointers must not be NULL");
    if (!backward_supported(p))
        return fail(CT_ERR_TOO_LARGE, "backward: %lld taps per input channel block exceed the staged slab",
                    (long long)p.taps());
    *dx_kernel = backward_dx_kernel_name(p);
    *dw_kernel = backward_dw_kernel_name(p);
    return CT_OK;
}

int ct_conv_transpose_backward_nd(const void* x, const void* w, const void* dy, void* dx, void* dw,
                                  void* db, void* workspace, size_t workspace_bytes, int nd,
                                  int64_t B, int64_t C_in, int64_t C_out,
                                  const int64_t* in_spatial, const int64_t* k, const int* stride,
                                  const int* pad_lo, const int* pad_hi, const int* dilation,
                                  const int* output_padding, int groups, int dtype, void* stream) {
    Problem p;
    int rc = validate(&p, nd, B, C_in, C_out, in_spatial, k, stride, pad_lo, pad_hi, dilation,
                      output_padding, groups, dtype);
    if (rc != CT_OK) return rc;
    const bool need_dy = dx || dw || db;
    if ((need_dy && p.y_elems() > 0 && !dy) || (dx && p.x_elems() > 0 && !w) ||
        (dw && p.w_elems() > 0 && p.x_elems() > 0 && !x))
        return fail(CT_ERR_NULL, "backward: dy (and w for dx, x for dw) must not be NULL");
    const size_t eb = p.elem_bytes();
    for (const void* q : {x, w, dy, (const void*)dx, (const void*)dw, (const void*)db})
        if (q && !aligned(q, eb)) return fail(CT_ERR_ALIGN, "pointers must be aligned to the element size (%zu bytes)", eb);
    if (!backward_supported(p))
        return fail(CT_ERR_TOO_LARGE, "backward: %lld taps per input channel block exceed the staged slab",
                    (long long)p.taps());
    cudaStream_t s = (cudaStream_t)stream;
    const size_t need = backward_workspace_bytes(p, dx != nullptr, dw != nullptr, db != nullptr);
    void* ws = workspace;
    bool owned = false;
    if (need > 0) {
        if (ws) {
            if (workspace_bytes < need)
                return fail(CT_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                            workspace_bytes, need);
            if (!aligned(ws, 256)) return fail(CT_ERR_ALIGN, "workspace must be 256-byte aligned");
        } else {
            cudaError_t e = cudaMallocAsync(&ws, need, s);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(backward workspace)");
            owned = true;
        }
    }
    cudaError_t e = launch_backward(p, x, w, dy, dx, dw, db, ws, s, nullptr);
    if (owned) {
        cudaError_t e2 = cudaFreeAsync(ws, s);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e, "backward kernel launch");
    return CT_OK;
}

int ct_host_buffers_release(void) {
    HostRes* R = nullptr;
    cudaError_t e = host_resources(&R);
    if (e != cudaSuccess) return cuda_fail(e, "host call resources");
    std::lock_guard<std::mutex> lock(R->mu);
    e = cudaMemPoolTrimTo(R->pool, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolTrimTo");
    return CT_OK;
}

}  // extern "C"

extern "C" int ct_device_status(int clear, unsigned int* code) {
    unsigned int a = 0, b = 0, c = 0, d = 0, f = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = ct::tc_error_word(&a, clear != 0);
    if (e == cudaSuccess) e = ct::tc32_error_word(&b, clear != 0);
    if (e == cudaSuccess) e = ct::grouped_tma_error_word(&c, clear != 0);
    if (e == cudaSuccess) e = ct::grouped_warp_error_word(&d, clear != 0);
    if (e == cudaSuccess) e = ct::backward_error_word(&f, clear != 0);
    const unsigned int all = a | b | c | d | f;
    if (code) *code = all;
    if (e != cudaSuccess) return ct::report_error(CT_ERR_CUDA, "%s", cudaGetErrorString(e));
    return all ? CT_ERR_DEVICE_TIMEOUT : CT_OK;
}
