// ct_internal.h -- shared declarations of the CUDA library behind include/ct.h.
//
// Every problem is normalised to three spatial axes (0 = D, 1 = H, 2 = W);
// the unused leading axes of a 1-D or 2-D problem have extent 1, kernel 1,
// stride 1, no padding and dilation 1, which leaves the result unchanged.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "ct.h"

namespace ct {

// Per-axis limits the planner and kernels rely on.
constexpr int kMaxK = 32;        // kernel taps per axis
constexpr int kMaxStride = 32;   // stride per axis
constexpr int kMaxPhaseTaps = 32;

struct Problem {
    int nd;
    int64_t B, C_in, C_out;
    int G, Cig, Cog;
    int64_t I[3], K[3], O[3];
    int S[3], PL[3], PH[3], DL[3], OP[3];
    ct_dtype dtype;
    // activation applied after the bias (ct_activation codes; 0 = none) and
    // its parameter: fused by the tcgen05 routes and the bias fill, a second
    // pass over y (launch_activation) on the CUDA-core routes
    int act = 0;
    float act_alpha = 0.f;

    int64_t in_spatial() const { return I[0] * I[1] * I[2]; }
    int64_t out_spatial() const { return O[0] * O[1] * O[2]; }
    int64_t taps() const { return K[0] * K[1] * K[2]; }
    int64_t x_elems() const { return B * C_in * in_spatial(); }
    int64_t y_elems() const { return B * C_out * out_spatial(); }
    int64_t w_elems() const { return C_in * (int64_t)Cog * taps(); }
    size_t elem_bytes() const { return dtype == CT_F32 ? 4 : 2; }
};

// Stride-phase plan of one axis.  Output o = r + s*q (residue r in [0, s))
// receives tap t exactly when (r + pad_lo - t*d) is a multiple of s; that tap
// then reads input i = q + off with off = (r + pad_lo - t*d) / s.  Taps are
// listed in increasing input offset, i.e. in reversed tap order.
struct AxisPlan {
    int s;                              // number of residues (= stride)
    int64_t q_extent[kMaxStride];       // #q with r + s*q < O, per residue
    int ntaps[kMaxStride];
    int tap[kMaxStride][kMaxPhaseTaps];
    int off[kMaxStride][kMaxPhaseTaps];
};

void plan_axis(const Problem& p, int axis, AxisPlan* out);

// Records a message for ct_last_error() on this thread and returns `status`.
int report_error(int status, const char* fmt, ...);

// Limit of every bounded device-side wait in later launches (ns; process-wide,
// set by ct_set_wait_limit_ns, 2 s by default; 0 = give up at the first
// incomplete probe).
uint64_t wait_limit_ns();

// Device properties cached per device.
struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;
};
cudaError_t device_info(DeviceInfo* out);

// Optional per-call profiling: events recorded on the launching stream just
// before and just after the route's dominant kernel, and a count of the
// kernels the call launched.
struct Profile {
    cudaEvent_t main_start = nullptr;
    cudaEvent_t main_stop = nullptr;
    int launches = 0;
};

// Brackets the dominant kernel's launch with the profile events (if any).
inline void prof_begin(Profile* pr, cudaStream_t s) {
    if (pr && pr->main_start) cudaEventRecord(pr->main_start, s);
}
inline void prof_end(Profile* pr, cudaStream_t s) {
    if (pr && pr->main_stop) cudaEventRecord(pr->main_stop, s);
}
inline void prof_count(Profile* pr, int n = 1) {
    if (pr) pr->launches += n;
}

// Launchers.  Each returns the first CUDA error it met (cudaSuccess if none).
cudaError_t launch_bias_fill(const Problem& p, const void* bias, void* y,
                             cudaStream_t stream, Profile* prof);
cudaError_t launch_gather(const Problem& p, const void* x, const void* w,
                          const void* bias, void* y, cudaStream_t stream, Profile* prof);
// y = act(y) in place (Problem.act), for the routes without a fused one.
cudaError_t launch_activation(const Problem& p, void* y, cudaStream_t stream, Profile* prof);
// w in layout 1 ([k...][C_in][C_out]), 2 ([k...][C_out][C_in]) or 0 (the
// PyTorch layout), taps reversed when `flipped` -> wp in the PyTorch layout.
cudaError_t launch_weight_to_torch_layout(const Problem& p, const void* w, void* wp, int layout,
                                          int flipped, cudaStream_t stream);

}  // namespace ct
