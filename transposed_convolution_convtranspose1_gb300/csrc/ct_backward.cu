// ct_backward.cu -- gradients of the transposed convolution on CUDA cores.
//
// The backward pass of "feat(ops): implement convTranspose2d -- CPU kernel,
// backward and StableHLO lowering" (SKaiNET #1464, Summary:
// convTranspose2dBackward, the adjoint giving input, weight and bias
// gradients), generalised like the forward pass to 1-D/3-D, groups,
// asymmetric padding and output_padding.  Every forward product
//     y[b, oc, o] += x[b, ic, i] * w[ic, oc_g, t],  o_a = i_a*s_a - pad_lo_a + t_a*d_a
// (o inside the output, ic in oc's group g) gives
//     dx[b, ic, i]    = sum over oc_g, t of  w[ic, oc_g, t]  * dy[b, g*Cog + oc_g, o(i, t)]
//     dw[ic, oc_g, t] = sum over b, i of     x[b, ic, i]     * dy[b, g*Cog + oc_g, o(i, t)]
//     db[oc]          = sum over b, o of     dy[b, oc, o]
// so dx is a strided correlation of dy with w (each input position gathers
// the K outputs its taps wrote), dw a reduction over batch and positions,
// db a per-channel sum.  Kernels (fp32 accumulation, one rounding to the
// tensor dtype, no atomics: every result is summed in a fixed order, so runs
// are bit-reproducible):
//   bwd_db_kernel   one block per output channel; each thread sums a strided
//                   share of the channel in four compensated (Kahan) fp32
//                   sums, then a fixed shared-memory tree.
//   bwd_dx_kernel   one thread per input position and ICB input channels of
//                   a group; the group's weights for a chunk of output
//                   channels are staged in shared memory ([oc][tap][ICB]) and
//                   read as broadcasts; per tap the thread finds the output
//                   position its input fed (or none) once, then walks the
//                   chunk's output channels.
//   bwd_dw_kernel   per (group, tile of 64 input channels, tile of 64
//                   (output channel, tap) pairs, K slice): the slice's
//                   positions are staged 32 at a time, a thread loading 8
//                   rows of one column (x rows and the dy values each (oc,
//                   tap) pair reads, zero where the tap falls outside the
//                   output) before storing any; 256 threads, each a 4 x 4
//                   register tile.  Slices write fp32
//                   partials; bwd_dw_reduce adds them in slice order and
//                   rounds once.
#include <algorithm>
#include <cstring>

#include "ct_internal.h"
#include "ct_types.cuh"

namespace ct {
namespace {

struct BwdArgs {
    const void* x;
    const void* w;
    const void* dy;
    void* dx;
    void* dw;
    void* db;
    float* part;            // dw partials [n_ks][C_in][Cog][taps]
    int64_t B, C_in, C_out;
    int G, Cig, Cog;
    int I[3], K[3], O[3], S[3], PL[3], DL[3];
    int64_t In, On;
    int Kn;
    int n_ks;               // K slices of dw
    int64_t ks_len;         // positions (over batch x input) per slice
    int occ;                // output channels per staged dx weight chunk
};

// ---------------------------------------------------------------------------
// db
// ---------------------------------------------------------------------------

constexpr int kDbThreads = 512;

template <typename T>
__global__ void __launch_bounds__(kDbThreads) bwd_db_kernel(const __grid_constant__ BwdArgs a) {
    __shared__ float red[kDbThreads];
    const int64_t oc = blockIdx.x;
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    // four independent compensated (Kahan) sums per thread, so that four
    // loads are in flight; comp holds each sum's lost low-order part
    float sum[4] = {0.f, 0.f, 0.f, 0.f}, comp[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t b = 0; b < a.B; ++b) {
        const T* p = dy + (b * a.C_out + oc) * a.On;
        for (int64_t o = threadIdx.x; o < a.On; o += 4 * kDbThreads) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t ou = o + (int64_t)u * kDbThreads;
                v[u] = ou < a.On ? to_f32(p[ou]) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float y = v[u] - comp[u];
                const float t = sum[u] + y;
                comp[u] = (t - sum[u]) - y;
                sum[u] = t;
            }
        }
    }
    red[threadIdx.x] = (sum[0] + sum[1]) + (sum[2] + sum[3]);
    __syncthreads();
    for (int h = kDbThreads / 2; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h) red[threadIdx.x] += red[threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0) static_cast<T*>(a.db)[oc] = from_f32<T>(red[0]);
}

// ---------------------------------------------------------------------------
// dx
// ---------------------------------------------------------------------------

constexpr int kDxThreads = 128;

template <typename T, int ICB>
__global__ void __launch_bounds__(kDxThreads) bwd_dx_kernel(const __grid_constant__ BwdArgs a,
                                                             int n_icb) {
    extern __shared__ __align__(16) float wsm[];  // [oc in chunk][tap][ICB]
    const T* __restrict__ w = static_cast<const T*>(a.w);
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    T* __restrict__ dx = static_cast<T*>(a.dx);

    // blockIdx.y: (b, g, input-channel block); blockIdx.x: positions
    const int64_t row = blockIdx.y + (int64_t)blockIdx.z * gridDim.y;
    const int icb = (int)(row % n_icb);
    const int64_t bg = row / n_icb;
    const int g = (int)(bg % a.G);
    const int64_t b = bg / a.G;
    const int ic0 = icb * ICB;
    const int nic = min(ICB, a.Cig - ic0);
    const int64_t i = (int64_t)blockIdx.x * kDxThreads + threadIdx.x;
    const bool live = i < a.In;
    int i0 = 0, i1 = 0, i2 = 0;
    if (live) {
        i2 = (int)(i % a.I[2]);
        i1 = (int)((i / a.I[2]) % a.I[1]);
        i0 = (int)(i / ((int64_t)a.I[2] * a.I[1]));
    }
    float acc[ICB];
#pragma unroll
    for (int c = 0; c < ICB; ++c) acc[c] = 0.f;
    const T* dyg = dy + (b * a.C_out + (int64_t)g * a.Cog) * a.On;

    for (int oc0 = 0; oc0 < a.Cog; oc0 += a.occ) {
        const int noc = min(a.occ, a.Cog - oc0);
        __syncthreads();  // the previous chunk's weights are no longer read
        const int n = noc * a.Kn * ICB;
        for (int e = threadIdx.x; e < n; e += kDxThreads) {
            const int c = e % ICB;
            const int t = (e / ICB) % a.Kn;
            const int oc = e / (ICB * a.Kn);
            wsm[e] = c < nic ? to_f32(w[((int64_t)(g * a.Cig + ic0 + c) * a.Cog + oc0 + oc) * a.Kn + t])
                             : 0.f;
        }
        __syncthreads();
        if (!live) continue;
        for (int t0 = 0; t0 < a.K[0]; ++t0) {
            const int o0 = i0 * a.S[0] - a.PL[0] + t0 * a.DL[0];
            if (o0 < 0 || o0 >= a.O[0]) continue;
            for (int t1 = 0; t1 < a.K[1]; ++t1) {
                const int o1 = i1 * a.S[1] - a.PL[1] + t1 * a.DL[1];
                if (o1 < 0 || o1 >= a.O[1]) continue;
                for (int t2 = 0; t2 < a.K[2]; ++t2) {
                    const int o2 = i2 * a.S[2] - a.PL[2] + t2 * a.DL[2];
                    if (o2 < 0 || o2 >= a.O[2]) continue;
                    const int t = (t0 * a.K[1] + t1) * a.K[2] + t2;
                    const T* dp = dyg + (int64_t)oc0 * a.On + ((int64_t)o0 * a.O[1] + o1) * a.O[2] + o2;
                    const float* wp = wsm + (int64_t)t * ICB;
                    for (int oc = 0; oc < noc; ++oc, dp += a.On, wp += a.Kn * ICB) {
                        const float v = to_f32(*dp);
#pragma unroll
                        for (int c = 0; c < ICB; ++c) acc[c] = fmaf(v, wp[c], acc[c]);
                    }
                }
            }
        }
    }
    if (!live) return;
    T* dxp = dx + (b * a.C_in + (int64_t)g * a.Cig + ic0) * a.In + i;
#pragma unroll
    for (int c = 0; c < ICB; ++c)
        if (c < nic) dxp[(int64_t)c * a.In] = from_f32<T>(acc[c]);
}

// ---------------------------------------------------------------------------
// dw
// ---------------------------------------------------------------------------

constexpr int kDwTM = 64;     // input channels per tile
constexpr int kDwTN = 64;     // (output channel, tap) pairs per tile
constexpr int kDwTK = 32;     // positions staged per step
constexpr int kDwThreads = 256;
constexpr int kDwRows = 8;    // staged rows per thread (of x and of dy)

template <typename T>
__global__ void __launch_bounds__(kDwThreads) bwd_dw_kernel(const __grid_constant__ BwdArgs a,
                                                             int n_mt, int n_nt) {
    __shared__ __align__(16) float xs[kDwTM][kDwTK + 4];
    __shared__ __align__(16) float ds[kDwTN][kDwTK + 4];
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ dy = static_cast<const T*>(a.dy);

    int64_t blk = blockIdx.x;
    const int mt = (int)(blk % n_mt); blk /= n_mt;
    const int nt = (int)(blk % n_nt); blk /= n_nt;
    const int g = (int)(blk % a.G);
    const int ks = (int)(blk / a.G);
    const int m0 = mt * kDwTM, n0 = nt * kDwTN;
    const int NN = a.Cog * a.Kn;  // (oc_g, tap) pairs of the group
    const int64_t k_begin = (int64_t)ks * a.ks_len;
    const int64_t k_end = min((int64_t)(ks + 1) * a.ks_len, a.B * a.In);

    // compute: this thread's 4 x 4 outputs, rows tm * 4 .., columns tn * 4 ..
    const int tm = threadIdx.x / 16, tn = threadIdx.x % 16;
    // staging: column kk of the step, rows r0 .. r0 + kDwRows - 1
    const int kk = threadIdx.x % kDwTK, r0 = (threadIdx.x / kDwTK) * kDwRows;
    // the (oc_g, tap) pairs of this thread's staged dy rows
    int n_oc[kDwRows], n_t[kDwRows][3];
#pragma unroll
    for (int r = 0; r < kDwRows; ++r) {
        const int n = min(n0 + r0 + r, NN - 1);
        const int t = n % a.Kn;
        n_oc[r] = n / a.Kn;
        n_t[r][2] = t % a.K[2];
        n_t[r][1] = (t / a.K[2]) % a.K[1];
        n_t[r][0] = t / (a.K[2] * a.K[1]);
    }
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;

    for (int64_t k0 = k_begin; k0 < k_end; k0 += kDwTK) {
        // load this thread's staged values (all loads before any store)
        const int64_t k = k0 + kk;
        const bool kok = k < k_end;
        int64_t b = 0, i = 0;
        int i0 = 0, i1 = 0, i2 = 0;
        if (kok) {
            b = k / a.In;
            i = k - b * a.In;
            i2 = (int)(i % a.I[2]);
            i1 = (int)((i / a.I[2]) % a.I[1]);
            i0 = (int)(i / ((int64_t)a.I[2] * a.I[1]));
        }
        float xv[kDwRows], dv[kDwRows];
        const T* xp = x + (b * a.C_in + (int64_t)g * a.Cig + m0 + r0) * a.In + i;
        const T* dyb = dy + (b * a.C_out + (int64_t)g * a.Cog) * a.On;
#pragma unroll
        for (int r = 0; r < kDwRows; ++r) {
            xv[r] = (kok && m0 + r0 + r < a.Cig) ? to_f32(xp[(int64_t)r * a.In]) : 0.f;
            float v = 0.f;
            if (kok && n0 + r0 + r < NN) {
                const int o0 = i0 * a.S[0] - a.PL[0] + n_t[r][0] * a.DL[0];
                const int o1 = i1 * a.S[1] - a.PL[1] + n_t[r][1] * a.DL[1];
                const int o2 = i2 * a.S[2] - a.PL[2] + n_t[r][2] * a.DL[2];
                if (o0 >= 0 && o0 < a.O[0] && o1 >= 0 && o1 < a.O[1] && o2 >= 0 && o2 < a.O[2])
                    v = to_f32(dyb[(int64_t)n_oc[r] * a.On + ((int64_t)o0 * a.O[1] + o1) * a.O[2] + o2]);
            }
            dv[r] = v;
        }
        __syncthreads();  // the previous step's tiles are no longer read
#pragma unroll
        for (int r = 0; r < kDwRows; ++r) {
            xs[r0 + r][kk] = xv[r];
            ds[r0 + r][kk] = dv[r];
        }
        __syncthreads();
#pragma unroll 2
        for (int q = 0; q < kDwTK; q += 4) {
            float4 xa[4], da[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) xa[r] = *reinterpret_cast<const float4*>(&xs[tm * 4 + r][q]);
#pragma unroll
            for (int c = 0; c < 4; ++c) da[c] = *reinterpret_cast<const float4*>(&ds[tn * 4 + c][q]);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    acc[r][c] = fmaf(xa[r].x, da[c].x, acc[r][c]);
                    acc[r][c] = fmaf(xa[r].y, da[c].y, acc[r][c]);
                    acc[r][c] = fmaf(xa[r].z, da[c].z, acc[r][c]);
                    acc[r][c] = fmaf(xa[r].w, da[c].w, acc[r][c]);
                }
        }
    }
    // partials [ks][C_in][Cog * taps]
    float* part = a.part + ((int64_t)ks * a.C_in + (int64_t)g * a.Cig) * NN;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int m = m0 + tm * 4 + r;
        if (m >= a.Cig) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int n = n0 + tn * 4 + c;
            if (n < NN) part[(int64_t)m * NN + n] = acc[r][c];
        }
    }
}

// dw[e] = sum over slices (in slice order) of part[ks][e], rounded once.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dw_reduce(const float* __restrict__ part, T* __restrict__ dw,
                                                     int64_t n, int n_ks) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int k = 0; k < n_ks; ++k) s += part[(int64_t)k * n + e];
        dw[e] = from_f32<T>(s);
    }
}

// ---------------------------------------------------------------------------
// host planning and launches
// ---------------------------------------------------------------------------

constexpr size_t kDxSmemMax = 96 * 1024;  // staged dx weight chunk

struct BwdPlan {
    int icb, n_icb, occ;
    size_t dx_smem;
    int n_mt, n_nt, n_ks;
    int64_t ks_len;
    size_t part_bytes;
};

bool bwd_plan(const Problem& p, int sm_count, BwdPlan* pl) {
    const int64_t Kn = p.taps();
    int icb = p.Cig >= 16 ? 16 : p.Cig >= 8 ? 8 : p.Cig >= 4 ? 4 : p.Cig >= 2 ? 2 : 1;
    while (icb > 1 && (size_t)Kn * icb * sizeof(float) > kDxSmemMax) icb /= 2;
    if ((size_t)Kn * icb * sizeof(float) > kDxSmemMax) return false;
    pl->icb = icb;
    pl->n_icb = (int)std::max<int64_t>(1, (p.Cig + icb - 1) / icb);
    const int64_t occ = std::max<int64_t>(1, std::min<int64_t>(p.Cog, (int64_t)(kDxSmemMax / ((size_t)Kn * icb * sizeof(float)))));
    pl->occ = (int)std::min<int64_t>(occ, 64);
    pl->dx_smem = (size_t)pl->occ * Kn * icb * sizeof(float);
    pl->n_mt = (int)((p.Cig + kDwTM - 1) / kDwTM);
    const int64_t NN = (int64_t)p.Cog * Kn;
    if (NN >= (1ll << 31)) return false;
    pl->n_nt = (int)((NN + kDwTN - 1) / kDwTN);
    const int64_t tiles = (int64_t)p.G * pl->n_mt * pl->n_nt;
    const int64_t Ktot = p.B * p.in_spatial();
    int64_t ks = tiles > 0 ? (4ll * sm_count + tiles - 1) / tiles : 1;
    ks = std::max<int64_t>(1, std::min<int64_t>(ks, 64));
    ks = std::max<int64_t>(1, std::min<int64_t>(ks, (Ktot + 255) / 256));
    pl->n_ks = (int)ks;
    pl->ks_len = (Ktot + ks - 1) / ks;
    pl->part_bytes = (size_t)ks * (size_t)p.C_in * (size_t)NN * sizeof(float);
    return true;
}

void fill_args(const Problem& p, BwdArgs* a) {
    std::memset(a, 0, sizeof(*a));
    a->B = p.B;
    a->C_in = p.C_in;
    a->C_out = p.C_out;
    a->G = p.G;
    a->Cig = p.Cig;
    a->Cog = p.Cog;
    for (int ax = 0; ax < 3; ++ax) {
        a->I[ax] = (int)p.I[ax];
        a->K[ax] = (int)p.K[ax];
        a->O[ax] = (int)p.O[ax];
        a->S[ax] = p.S[ax];
        a->PL[ax] = p.PL[ax];
        a->DL[ax] = p.DL[ax];
    }
    a->In = p.in_spatial();
    a->On = p.out_spatial();
    a->Kn = (int)p.taps();
}

template <typename T, int ICB>
cudaError_t launch_dx_t(const BwdArgs& a, const BwdPlan& pl, cudaStream_t stream) {
    const int64_t rows = a.B * (int64_t)a.G * pl.n_icb;
    const int64_t gx = (a.In + kDxThreads - 1) / kDxThreads;
    if (rows == 0 || gx == 0) return cudaSuccess;
    if (gx >= (1ll << 31)) return cudaErrorInvalidConfiguration;
    const int64_t gy = std::min<int64_t>(rows, 65535);
    const int64_t gz = (rows + gy - 1) / gy;
    if (gz > 65535) return cudaErrorInvalidConfiguration;
    if (pl.dx_smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(bwd_dx_kernel<T, ICB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)pl.dx_smem);
        if (e != cudaSuccess) return e;
    }
    bwd_dx_kernel<T, ICB><<<dim3((unsigned)gx, (unsigned)gy, (unsigned)gz), kDxThreads, pl.dx_smem, stream>>>(
        a, pl.n_icb);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_backward_t(const Problem& p, const BwdPlan& pl, BwdArgs a, cudaStream_t stream,
                              int* launches) {
    cudaError_t e = cudaSuccess;
    if (a.db && p.C_out > 0) {
        bwd_db_kernel<T><<<(unsigned)p.C_out, kDbThreads, 0, stream>>>(a);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.dx) {
        switch (pl.icb) {
            case 1: e = launch_dx_t<T, 1>(a, pl, stream); break;
            case 2: e = launch_dx_t<T, 2>(a, pl, stream); break;
            case 4: e = launch_dx_t<T, 4>(a, pl, stream); break;
            case 8: e = launch_dx_t<T, 8>(a, pl, stream); break;
            default: e = launch_dx_t<T, 16>(a, pl, stream); break;
        }
        ++*launches;
        if (e != cudaSuccess) return e;
    }
    const int64_t nw = p.w_elems();
    if (a.dw && nw > 0) {
        const int64_t blocks = (int64_t)p.G * pl.n_mt * pl.n_nt * pl.n_ks;
        if (blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
        bwd_dw_kernel<T><<<(unsigned)blocks, kDwThreads, 0, stream>>>(a, pl.n_mt, pl.n_nt);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int rb = (int)std::min<int64_t>((nw + 255) / 256, 152 * 8);
        bwd_dw_reduce<T><<<rb, 256, 0, stream>>>(a.part, static_cast<T*>(a.dw), nw, pl.n_ks);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

bool backward_supported(const Problem& p) {
    BwdPlan pl;
    return bwd_plan(p, 152, &pl);
}

size_t backward_workspace_bytes(const Problem& p) {
    DeviceInfo d;
    int sm = 152;
    if (device_info(&d) == cudaSuccess) sm = d.sm_count;
    BwdPlan pl;
    if (!bwd_plan(p, sm, &pl)) return 0;
    return (pl.part_bytes + 255) / 256 * 256;
}

cudaError_t launch_backward(const Problem& p, const void* x, const void* w, const void* dy, void* dx,
                            void* dw, void* db, void* workspace, cudaStream_t stream, int* launches) {
    DeviceInfo d;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return e;
    BwdPlan pl;
    if (!bwd_plan(p, d.sm_count, &pl)) return cudaErrorInvalidValue;
    BwdArgs a;
    fill_args(p, &a);
    a.x = x;
    a.w = w;
    a.dy = dy;
    a.dx = dx;
    a.dw = dw;
    a.db = db;
    a.part = static_cast<float*>(workspace);
    a.n_ks = pl.n_ks;
    a.ks_len = pl.ks_len;
    a.occ = pl.occ;
    int n = 0;
    int* cnt = launches ? launches : &n;
    switch (p.dtype) {
        case CT_F32: return launch_backward_t<float>(p, pl, a, stream, cnt);
        case CT_F16: return launch_backward_t<__half>(p, pl, a, stream, cnt);
        default: return launch_backward_t<__nv_bfloat16>(p, pl, a, stream, cnt);
    }
}

}  // namespace ct

