// ct_gather.cu -- the generic CUDA-core gather route and the bias-fill edge path.
//
// Gather form of the operation: output o receives tap t from input
// i = (o + pad_lo - t*d) / s exactly when that quotient is exact and inside
// [0, I) on every axis -- the scatter of SKaiNET #1464 (Summary, DefaultCpuOps)
// with its index map inverted, so that each thread owns its outputs and no two
// threads add into the same element (no atomics).  One thread owns one
// output position and a block of OCB output channels of one group, as in
// the ONNX page's grouped stride-phase variant: each input value it reads is
// used for all OCB channels, and the block keeps the group's weights in
// shared memory, loaded a single time.  This kernel serves every shape and
// dtype and is the reference route the specialised routes are tested beside.
#include <algorithm>

#include "ct_internal.h"
#include "ct_types.cuh"

namespace ct {
namespace {

struct GatherArgs {
    const void* x;
    const void* w;
    const void* bias;
    void* y;
    int64_t C_in, C_out;
    int G, Cig, Cog, n_ocb;
    int I[3], K[3], O[3], S[3], PL[3], DL[3];
    int64_t In, On;
    int Kn;
    int64_t n_rows;  // B * G * n_ocb
};

// Shared-memory weight slab layout: [tap][ic_g][j] (j = oc within the block).
template <typename T, int OCB, bool SMEM>
__global__ void __launch_bounds__(128) gather_kernel(const GatherArgs a) {
    extern __shared__ float slab[];
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ w = static_cast<const T*>(a.w);
    const T* __restrict__ bias = static_cast<const T*>(a.bias);
    T* __restrict__ y = static_cast<T*>(a.y);

    const int64_t row = (int64_t)blockIdx.y + (int64_t)blockIdx.z * gridDim.y;
    if (row >= a.n_rows) return;  // uniform per block: before any barrier
    const int ocb = (int)(row % a.n_ocb);
    const int64_t bg = row / a.n_ocb;
    const int g = (int)(bg % a.G);
    const int64_t b = bg / a.G;
    const int oc0 = ocb * OCB;
    const int nvalid = min(OCB, a.Cog - oc0);

    if (SMEM) {
        const int total = a.Kn * a.Cig * OCB;
        for (int e = threadIdx.x; e < total; e += blockDim.x) {
            const int j = e % OCB;
            const int ic = (e / OCB) % a.Cig;
            const int t = e / (OCB * a.Cig);
            float v = 0.f;
            if (j < nvalid) v = to_f32(w[((int64_t)(g * a.Cig + ic) * a.Cog + oc0 + j) * a.Kn + t]);
            slab[e] = v;
        }
        __syncthreads();
    }

    float bv[OCB];
#pragma unroll
    for (int j = 0; j < OCB; ++j)
        bv[j] = (bias != nullptr && j < nvalid) ? to_f32(bias[g * a.Cog + oc0 + j]) : 0.f;

    const T* xg = x + (b * a.C_in + (int64_t)g * a.Cig) * a.In;
    const int64_t ybase = (b * a.C_out + (int64_t)g * a.Cog + oc0) * a.On;

    for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < a.On;
         o += (int64_t)gridDim.x * blockDim.x) {
        const int ow = (int)(o % a.O[2]);
        const int oh = (int)((o / a.O[2]) % a.O[1]);
        const int od = (int)(o / ((int64_t)a.O[2] * a.O[1]));
        float acc[OCB];
#pragma unroll
        for (int j = 0; j < OCB; ++j) acc[j] = 0.f;

        for (int t0 = 0; t0 < a.K[0]; ++t0) {
            const int v0 = od + a.PL[0] - t0 * a.DL[0];
            if (v0 < 0 || v0 % a.S[0] != 0) continue;
            const int i0 = v0 / a.S[0];
            if (i0 >= a.I[0]) continue;
            for (int t1 = 0; t1 < a.K[1]; ++t1) {
                const int v1 = oh + a.PL[1] - t1 * a.DL[1];
                if (v1 < 0 || v1 % a.S[1] != 0) continue;
                const int i1 = v1 / a.S[1];
                if (i1 >= a.I[1]) continue;
                for (int t2 = 0; t2 < a.K[2]; ++t2) {
                    const int v2 = ow + a.PL[2] - t2 * a.DL[2];
                    if (v2 < 0 || v2 % a.S[2] != 0) continue;
                    const int i2 = v2 / a.S[2];
                    if (i2 >= a.I[2]) continue;
                    const int tap = (t0 * a.K[1] + t1) * a.K[2] + t2;
                    const T* xp = xg + ((int64_t)i0 * a.I[1] + i1) * a.I[2] + i2;
                    for (int ic = 0; ic < a.Cig; ++ic) {
                        const float xv = to_f32(xp[(int64_t)ic * a.In]);
                        if (SMEM) {
                            const float* wr = slab + ((int64_t)tap * a.Cig + ic) * OCB;
#pragma unroll
                            for (int j = 0; j < OCB; ++j) acc[j] = fmaf(xv, wr[j], acc[j]);
                        } else {
                            const T* wr = w + ((int64_t)(g * a.Cig + ic) * a.Cog + oc0) * a.Kn + tap;
#pragma unroll
                            for (int j = 0; j < OCB; ++j)
                                if (j < nvalid) acc[j] = fmaf(xv, to_f32(wr[(int64_t)j * a.Kn]), acc[j]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < OCB; ++j)
            if (j < nvalid) y[ybase + (int64_t)j * a.On + o] = from_f32<T>(acc[j] + bv[j]);
    }
}

template <typename T>
__global__ void bias_fill_kernel(const T* __restrict__ bias, T* __restrict__ y, int64_t C_out,
                                 int64_t On, int64_t total, int act, float act_alpha) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t c = (i / On) % C_out;
        const float v = bias ? to_f32(bias[c]) : 0.f;
        y[i] = from_f32<T>(act_f32(v, act, act_alpha));
    }
}

template <typename T, int OCB>
cudaError_t launch_gather_t(const GatherArgs& a, cudaStream_t stream, int sm_count,
                            size_t smem_optin, Profile* prof) {
    const size_t slab = (size_t)a.Kn * a.Cig * OCB * sizeof(float);
    const bool use_smem = slab <= 48 * 1024 || slab <= smem_optin / 2;
    const int threads = 128;
    int64_t gx = (a.On + threads - 1) / threads;
    // enough blocks to fill the GPU many times over; the loop strides the rest
    const int64_t rows = a.n_rows;
    const int64_t want = (int64_t)sm_count * 16;
    if (gx * rows > want) gx = std::max<int64_t>(1, (want + rows - 1) / rows);
    const int64_t gy = std::min<int64_t>(rows, 65535);
    const int64_t gz = (rows + gy - 1) / gy;
    if (gz > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)gz);
    if (use_smem) {
        if (slab > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(gather_kernel<T, OCB, true>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)slab);
            if (e != cudaSuccess) return e;
        }
        prof_begin(prof, stream);
        gather_kernel<T, OCB, true><<<grid, threads, slab, stream>>>(a);
    } else {
        prof_begin(prof, stream);
        gather_kernel<T, OCB, false><<<grid, threads, 0, stream>>>(a);
    }
    prof_end(prof, stream);
    prof_count(prof);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_gather_dtype(const Problem& p, GatherArgs a, cudaStream_t stream,
                                Profile* prof) {
    DeviceInfo d;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    int ocb = 16;
    if (p.Cog <= 1) ocb = 1;
    else if (p.Cog <= 2) ocb = 2;
    else if (p.Cog <= 4) ocb = 4;
    else if (p.Cog <= 8) ocb = 8;
    a.n_ocb = (p.Cog + ocb - 1) / ocb;
    a.n_rows = p.B * (int64_t)p.G * a.n_ocb;
    switch (ocb) {
        case 1: return launch_gather_t<T, 1>(a, stream, d.sm_count, d.smem_optin, prof);
        case 2: return launch_gather_t<T, 2>(a, stream, d.sm_count, d.smem_optin, prof);
        case 4: return launch_gather_t<T, 4>(a, stream, d.sm_count, d.smem_optin, prof);
        case 8: return launch_gather_t<T, 8>(a, stream, d.sm_count, d.smem_optin, prof);
        default: return launch_gather_t<T, 16>(a, stream, d.sm_count, d.smem_optin, prof);
    }
}

}  // namespace

cudaError_t launch_gather(const Problem& p, const void* x, const void* w, const void* bias, void* y,
                          cudaStream_t stream, Profile* prof) {
    GatherArgs a{};
    a.x = x; a.w = w; a.bias = bias; a.y = y;
    a.C_in = p.C_in; a.C_out = p.C_out;
    a.G = p.G; a.Cig = p.Cig; a.Cog = p.Cog;
    for (int i = 0; i < 3; ++i) {
        a.I[i] = (int)p.I[i]; a.K[i] = (int)p.K[i]; a.O[i] = (int)p.O[i];
        a.S[i] = p.S[i]; a.PL[i] = p.PL[i]; a.DL[i] = p.DL[i];
    }
    a.In = p.in_spatial();
    a.On = p.out_spatial();
    a.Kn = (int)p.taps();
    switch (p.dtype) {
        case CT_F32: return launch_gather_dtype<float>(p, a, stream, prof);
        case CT_F16: return launch_gather_dtype<__half>(p, a, stream, prof);
        default: return launch_gather_dtype<__nv_bfloat16>(p, a, stream, prof);
    }
}

cudaError_t launch_bias_fill(const Problem& p, const void* bias, void* y, cudaStream_t stream,
                             Profile* prof) {
    const int64_t total = p.y_elems();
    if (total == 0) return cudaSuccess;
    DeviceInfo d;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    blocks = std::min<int64_t>(blocks, (int64_t)d.sm_count * 8);
    const int64_t On = p.out_spatial();
    prof_begin(prof, stream);
    switch (p.dtype) {
        case CT_F32:
            bias_fill_kernel<float><<<(unsigned)blocks, threads, 0, stream>>>(
                (const float*)bias, (float*)y, p.C_out, On, total, p.act, p.act_alpha);
            break;
        case CT_F16:
            bias_fill_kernel<__half><<<(unsigned)blocks, threads, 0, stream>>>(
                (const __half*)bias, (__half*)y, p.C_out, On, total, p.act, p.act_alpha);
            break;
        default:
            bias_fill_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, stream>>>(
                (const __nv_bfloat16*)bias, (__nv_bfloat16*)y, p.C_out, On, total, p.act, p.act_alpha);
            break;
    }
    prof_end(prof, stream);
    prof_count(prof);
    return cudaGetLastError();
}

// w in another layout -> w' in the PyTorch layout [C_in][C_out/groups][k...]
// (the NKI page's filter_shape and flip_filter_taps_in_kernel, conv3d_transpose
// parameters): layout 1 = [k...][C_in][C_out], layout 2 = [k...][C_out][C_in]
// (groups 1), layout 0 = the PyTorch one; `flipped` means the stored taps are
// reversed along every spatial axis.  One thread per element of w'.
template <typename T>
__global__ void weight_to_torch_layout(const T* __restrict__ w, T* __restrict__ wp, int64_t C_in,
                                       int64_t Cog, int K0, int K1, int K2, int layout, int flipped,
                                       int64_t total) {
    const int64_t Kn = (int64_t)K0 * K1 * K2;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = e % Kn;
        const int64_t oc = (e / Kn) % Cog;
        const int64_t ic = e / (Kn * Cog);
        int t2 = (int)(t % K2), t1 = (int)((t / K2) % K1), t0 = (int)(t / ((int64_t)K2 * K1));
        if (flipped) {
            t0 = K0 - 1 - t0;
            t1 = K1 - 1 - t1;
            t2 = K2 - 1 - t2;
        }
        const int64_t ts = ((int64_t)t0 * K1 + t1) * K2 + t2;
        int64_t src;
        if (layout == 1) src = (ts * C_in + ic) * Cog + oc;
        else if (layout == 2) src = (ts * Cog + oc) * C_in + ic;
        else src = (ic * Cog + oc) * Kn + ts;
        wp[e] = w[src];
    }
}

cudaError_t launch_weight_to_torch_layout(const Problem& p, const void* w, void* wp, int layout,
                                          int flipped, cudaStream_t stream) {
    const int64_t total = p.w_elems();
    if (total == 0) return cudaSuccess;
    DeviceInfo d;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((total + threads - 1) / threads, (int64_t)d.sm_count * 8);
    const int K0 = (int)p.K[0], K1 = (int)p.K[1], K2 = (int)p.K[2];
    switch (p.dtype) {
        case CT_F32:
            weight_to_torch_layout<float><<<(unsigned)blocks, threads, 0, stream>>>(
                (const float*)w, (float*)wp, p.C_in, p.Cog, K0, K1, K2, layout, flipped, total);
            break;
        case CT_F16:
            weight_to_torch_layout<__half><<<(unsigned)blocks, threads, 0, stream>>>(
                (const __half*)w, (__half*)wp, p.C_in, p.Cog, K0, K1, K2, layout, flipped, total);
            break;
        default:
            weight_to_torch_layout<__nv_bfloat16><<<(unsigned)blocks, threads, 0, stream>>>(
                (const __nv_bfloat16*)w, (__nv_bfloat16*)wp, p.C_in, p.Cog, K0, K1, K2, layout,
                flipped, total);
            break;
    }
    return cudaGetLastError();
}

// y = act(y) in place: the activation of the CUDA-core routes (gather,
// grouped, SIMT), whose unrolled epilogues would carry the activation's code
// at every store site; it runs as a second pass over y (16-bit outputs are
// then rounded twice).
template <typename T>
__global__ void activation_kernel(T* __restrict__ y, int64_t n, int act, float alpha) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        y[i] = from_f32<T>(act_f32(to_f32(y[i]), act, alpha));
}

cudaError_t launch_activation(const Problem& p, void* y, cudaStream_t stream, Profile* prof) {
    const int64_t n = p.y_elems();
    if (n == 0 || p.act == 0) return cudaSuccess;
    DeviceInfo d;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    const int threads = 256;
    const int64_t blocks = std::min<int64_t>((n + threads - 1) / threads, (int64_t)d.sm_count * 16);
    switch (p.dtype) {
        case CT_F32:
            activation_kernel<float><<<(unsigned)blocks, threads, 0, stream>>>((float*)y, n, p.act, p.act_alpha);
            break;
        case CT_F16:
            activation_kernel<__half><<<(unsigned)blocks, threads, 0, stream>>>((__half*)y, n, p.act, p.act_alpha);
            break;
        default:
            activation_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, stream>>>(
                (__nv_bfloat16*)y, n, p.act, p.act_alpha);
            break;
    }
    prof_count(prof);
    return cudaGetLastError();
}

}  // namespace ct
