// ct_grouped_tma.cu -- fp32 grouped stride-phase gather whose input rows
// arrive by TMA.
//
// The ONNX page's grouped stride-phase variant (ai.onnx.ConvTranspose,
// nchw2d_grouped_stride_phase_blocked) for groups of 5..8 input and output
// channels on 2-D/3-D fp32 outputs.  Same arithmetic as the staged kernel of
// ct_grouped.cu (one fp32 FMA chain per output: D, H, W taps in increasing
// input offset, channels in order, bias added last), with the per-element
// work of staging and of the inner loop taken out:
//   - a block owns (b, g, od, a band of 16 q_h values, a chunk of 64 q_w
//     values); one thread copies the band's input rows for each D tap with
//     one TMA box [8 channels][18 rows][72 columns] (column origin rounded
//     down to a multiple of 4; rows, depths, channels and columns outside the
//     tensor read as zero), while the other threads store the bias-only rows
//     and stage the group's weights duplicated, {w, w};
//   - a warp item is 4 consecutive q_h of one H residue; lane l owns q_w = l
//     and l + 32, so per (tap, input channel) 8 four-byte loads at fixed
//     offsets and 4 broadcast 16-byte weight loads feed 4 rows x 8 output
//     channels x 2 positions = 32 packed two-lane FMAs;
//   - the wait for the copy is bounded (a launch parameter, 2 s by default):
//     past it the kernel records an error in the unit's device error word,
//     waits (bounded) for the copy and goes on.
#include <algorithm>
#include <cstring>

#include "ct_routes.h"
#include "ct_tcgen05.cuh"
#include "ct_types.cuh"

namespace ct {
namespace {

using tcg::smem_u32;

constexpr int kGW = 4;          // warps per block
constexpr int kGR = 4;          // rows (consecutive q_h) per warp item
constexpr int kGQ = 64;         // q_w positions per chunk: lane l owns l and l + 32
constexpr int kGC = 8;          // channels per group, padded (input and output)
constexpr int kGQB = 16;        // q_h per band
constexpr int kGNR = 18;        // staged rows per D tap: a band plus an H offset span of 2
constexpr int kGWB = 72;        // staged columns: 3 (origin rounding) + 64 + W offset span <= 5
constexpr int kGMaxSW = 4;
constexpr int kGMaxSA = 8;
constexpr int kGMaxTaps = 8;
constexpr size_t kGTile = (size_t)kGC * kGNR * kGWB * sizeof(float);  // bytes per D tap
constexpr unsigned kErrGroupedCopy = 1u << 4;

struct GtParams {
    CUtensorMap tmap_x;     // x as 4-D (W, H, D, B * C_in), fp32
    const float* w;
    const float* bias;
    float* y;
    int C_in, C_out, G, Cig, Cog;
    int I[3], O[3], S[3], K[3];
    int ntap[3][kGMaxSA];
    int tap[3][kGMaxSA][kGMaxTaps];
    int off[3][kGMaxSA][kGMaxTaps];
    int qext[3][kGMaxSA];   // #q with r + s*q < O, per axis and residue
    int taps;
    int n_hb, n_qc;         // bands along q_h, chunks along q_w
    int offmin_h, wmin;     // smallest H and W offsets
    int vec2;               // W stride 2, one live W residue, 8-byte aligned rows
    int live_w;             // that residue
    int vecb;               // bias rows: 8-byte aligned rows of even width
    int nd_max;             // most D taps of any D residue
    uint64_t wait_ns;       // limit of the copy's wait (0: give up at the first incomplete probe)
};

// The k-th H residue with (live) or without (dead) taps.
__device__ __forceinline__ int kth_residue(const GtParams& P, int k, bool live, bool d_live) {
    for (int r = 0; r < P.S[1]; ++r) {
        const bool l = d_live && P.ntap[1][r] > 0;
        if (l == live) {
            if (k == 0) return r;
            --k;
        }
    }
    return 0;
}

__global__ void __launch_bounds__(kGW * 32, 4) grouped_tma_kernel(const __grid_constant__ GtParams P) {
    extern __shared__ __align__(128) float sm[];
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;

    int64_t blk = blockIdx.x;
    const int qc = (int)(blk % P.n_qc); blk /= P.n_qc;
    const int hb = (int)(blk % P.n_hb); blk /= P.n_hb;
    const int od = (int)(blk % P.O[0]); blk /= P.O[0];
    const int g = (int)(blk % P.G);
    const int64_t b = blk / P.G;
    const int rd = od % P.S[0], qd = od / P.S[0];
    const int nd_ = P.ntap[0][rd];
    const int qh0 = hb * kGQB, q0 = qc * kGQ;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // shared memory: weights [tap][ic][oc] as {w, w} at the aligned base (so
    // that a float4 of them is one 16-byte load), then the x tiles
    // [jd][ic][row][col] at a multiple of 512 bytes
    float2* w2 = reinterpret_cast<float2*>(sm);
    float* xs = sm + (size_t)P.taps * kGC * kGC * 2;
    const uint32_t bar = smem_u32(&bar_storage);
    const int x_org = (q0 + P.wmin) & ~3;         // column origin, a multiple of 4
    const int sh = q0 + P.wmin - x_org;           // 0..3
    const int Sh = P.S[1], Sw = P.S[2], O1 = P.O[1], O2 = P.O[2];
    int n_live = 0;  // H residues with taps (none when the D residue has none)
    for (int r = 0; r < Sh; ++r) n_live += (nd_ > 0 && P.ntap[1][r] > 0);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        if (n_live > 0) {  // the copy is waited for below exactly when it is issued
            tcg::mbar_init(bar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tcg::mbar_expect_tx(bar, (uint32_t)(nd_ * kGTile));
            const int ch0 = (int)(b * P.C_in) + g * P.Cig;
            for (int jd = 0; jd < nd_; ++jd)
                tcg::tma_load_4d(smem_u32(xs + (size_t)jd * (kGTile / sizeof(float))), &P.tmap_x, bar,
                            x_org, qh0 + P.offmin_h, qd + P.off[0][rd][jd], ch0);
        }
    }

    float bv[kGC];
#pragma unroll
    for (int oc = 0; oc < kGC; ++oc) bv[oc] = (P.bias != nullptr && oc < P.Cog) ? P.bias[g * P.Cog + oc] : 0.f;
    const int64_t out_plane = (int64_t)P.O[0] * O1 * O2;
    float* yb = P.y + (b * P.C_out + (int64_t)g * P.Cog) * out_plane + (int64_t)od * O1 * O2;

    // rows without taps: bias over the chunk's columns, while the copy runs
    for (int it = warp; it < (Sh - n_live) * kGQB; it += kGW) {
        const int rh = kth_residue(P, it / kGQB, false, nd_ > 0);
        const int qh = qh0 + it % kGQB;
        if (qh >= P.qext[1][rh]) continue;
        const int oh = Sh * qh + rh;
        const int c0 = Sw * q0, c1 = min(Sw * (q0 + kGQ), O2);
#pragma unroll
        for (int oc = 0; oc < kGC; ++oc) {
            if (oc >= P.Cog) break;
            float* yr = yb + (int64_t)oc * out_plane + (int64_t)oh * O2;
            if (P.vecb) {
                for (int ow = c0 + 2 * lane; ow < c1; ow += 64)
                    *reinterpret_cast<float2*>(yr + ow) = make_float2(bv[oc], bv[oc]);
            } else {
                for (int ow = c0 + lane; ow < c1; ow += 32) yr[ow] = bv[oc];
            }
        }
    }
    if (n_live == 0) return;  // no copy was issued

    // the group's weights, duplicated
    {
        constexpr int kB = 4;
        const int wn = P.taps * kGC * kGC;
        for (int e0 = threadIdx.x; e0 < wn; e0 += kB * kGW * 32) {
            float v[kB];
#pragma unroll
            for (int k = 0; k < kB; ++k) {
                const int e = e0 + k * kGW * 32;
                const int oc = e % kGC, ic = (e / kGC) % kGC, t = e / (kGC * kGC);
                v[k] = (e < wn && oc < P.Cog && ic < P.Cig)
                           ? P.w[((int64_t)(g * P.Cig + ic) * P.Cog + oc) * P.taps + t] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kB; ++k)
                if (e0 + k * kGW * 32 < wn) w2[e0 + k * kGW * 32] = make_float2(v[k], v[k]);
        }
    }
    __syncthreads();  // weights stored; the barrier's initialisation visible
    if (!tcg::mbar_wait(bar, 0, kErrGroupedCopy, &abort_flag, P.wait_ns)) tcg::mbar_drain(bar, 0);

    const int ngrp = kGQB / kGR;
    for (int it = warp; it < n_live * ngrp; it += kGW) {
        const int rh = kth_residue(P, it / ngrp, true, true);
        const int qhb = qh0 + (it % ngrp) * kGR;
        if (qhb >= P.qext[1][rh]) continue;
        const int nh_ = P.ntap[1][rh];
        for (int r = 0; r < Sw; ++r) {
            if (P.vec2 && r != P.live_w) continue;  // written with the live residue
            const int nw_ = P.ntap[2][r];
            if (nw_ == 0) {
#pragma unroll
                for (int i = 0; i < kGR; ++i) {
                    const int qh = qhb + i;
                    if (qh >= P.qext[1][rh]) break;
                    float* yr = yb + (int64_t)(Sh * qh + rh) * O2 + r;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int q = q0 + lane + 32 * u;
                        if (q >= P.qext[2][r]) continue;
#pragma unroll
                        for (int oc = 0; oc < kGC; ++oc) {
                            if (oc >= P.Cog) break;
                            yr[(int64_t)oc * out_plane + (int64_t)Sw * q] = bv[oc];
                        }
                    }
                }
                continue;
            }
            float2 acc[kGR][kGC];
#pragma unroll
            for (int i = 0; i < kGR; ++i)
#pragma unroll
                for (int oc = 0; oc < kGC; ++oc) acc[i][oc] = make_float2(0.f, 0.f);
            for (int jd = 0; jd < nd_; ++jd) {
                for (int jh = 0; jh < nh_; ++jh) {
                    // row of item row 0 within the tile, column of lane 0 at offset 0
                    const int row0 = (qhb - qh0) + P.off[1][rh][jh] - P.offmin_h;
                    const float* xr = xs + (size_t)jd * (kGTile / sizeof(float)) + row0 * kGWB + sh - P.wmin + lane;
                    const int tdh = (P.tap[0][rd][jd] * P.K[1] + P.tap[1][rh][jh]) * P.K[2];
                    for (int jw = 0; jw < nw_; ++jw) {
                        const float* xp = xr + P.off[2][r][jw];
                        const float4* wp = reinterpret_cast<const float4*>(sm) +
                                           (tdh + P.tap[2][r][jw]) * (kGC * kGC / 2);
#pragma unroll
                        for (int ic = 0; ic < kGC; ++ic) {
                            float2 xv[kGR];
#pragma unroll
                            for (int i = 0; i < kGR; ++i)
                                xv[i] = make_float2(xp[(ic * kGNR + i) * kGWB], xp[(ic * kGNR + i) * kGWB + 32]);
#pragma unroll
                            for (int o2 = 0; o2 < kGC / 2; ++o2) {
                                const float4 wq = wp[ic * (kGC / 2) + o2];
                                const float2 wa = make_float2(wq.x, wq.y), wb = make_float2(wq.z, wq.w);
#pragma unroll
                                for (int i = 0; i < kGR; ++i) {
                                    fma2(acc[i][2 * o2], xv[i], wa);
                                    fma2(acc[i][2 * o2 + 1], xv[i], wb);
                                }
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kGR; ++i) {
                const int qh = qhb + i;
                if (qh >= P.qext[1][rh]) break;
                float* yr = yb + (int64_t)(Sh * qh + rh) * O2;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int q = q0 + lane + 32 * u;
                    if (q >= P.qext[2][r]) continue;
#pragma unroll
                    for (int oc = 0; oc < kGC; ++oc) {
                        if (oc >= P.Cog) break;
                        const float v = (u ? acc[i][oc].y : acc[i][oc].x) + bv[oc];
                        float* yo = yr + (int64_t)oc * out_plane + (int64_t)Sw * q;
                        if (P.vec2) {
                            *reinterpret_cast<float2*>(yo) =
                                r == 0 ? make_float2(v, bv[oc]) : make_float2(bv[oc], v);
                        } else {
                            yo[r] = v;
                        }
                    }
                }
            }
        }
    }
}

struct GtPlan {
    AxisPlan ax[3];
    int offmin_h, wmin, nd_max;
    size_t smem;
};

bool make_gt_plan(const Problem& p, GtPlan* pl) {
    if (p.dtype != CT_F32) return false;
    if (p.Cig < 5 || p.Cig > kGC || p.Cog < 5 || p.Cog > kGC) return false;
    if (p.S[2] > kGMaxSW || p.S[0] > kGMaxSA || p.S[1] > kGMaxSA) return false;
    if (p.I[2] % 4 != 0) return false;  // 16-byte row pitch for the tensor map
    if (p.B * p.C_in >= (1ll << 31) || p.I[0] * p.I[1] * p.I[2] >= (1ll << 31)) return false;
    for (int a = 0; a < 3; ++a) {
        plan_axis(p, a, &pl->ax[a]);
        for (int r = 0; r < p.S[a]; ++r)
            if (pl->ax[a].ntaps[r] > kGMaxTaps) return false;
    }
    if (pl->ax[1].q_extent[0] < 12) return false;  // bands of 16 q_h
    if (p.O[0] * (int64_t)p.O[1] * p.O[2] >= (1ll << 31)) return false;
    int hmin = 1 << 30, hmax = -(1 << 30), wmin = 1 << 30, wmax = -(1 << 30), ndmax = 0;
    for (int r = 0; r < p.S[1]; ++r)
        for (int j = 0; j < pl->ax[1].ntaps[r]; ++j) {
            hmin = std::min(hmin, pl->ax[1].off[r][j]);
            hmax = std::max(hmax, pl->ax[1].off[r][j]);
        }
    for (int r = 0; r < p.S[2]; ++r)
        for (int j = 0; j < pl->ax[2].ntaps[r]; ++j) {
            wmin = std::min(wmin, pl->ax[2].off[r][j]);
            wmax = std::max(wmax, pl->ax[2].off[r][j]);
        }
    for (int r = 0; r < p.S[0]; ++r) ndmax = std::max(ndmax, pl->ax[0].ntaps[r]);
    if (hmin > hmax || wmin > wmax) return false;
    if (kGQB + (hmax - hmin) > kGNR) return false;      // rows of a band fit the box
    if (3 + kGQ + (wmax - wmin) > kGWB) return false;   // columns fit the box
    pl->offmin_h = hmin;
    pl->wmin = wmin;
    pl->nd_max = std::max(ndmax, 1);
    pl->smem = (size_t)pl->nd_max * kGTile + (size_t)p.taps() * kGC * kGC * sizeof(float2);
    return pl->smem <= 200 * 1024;
}

}  // namespace

bool grouped_tma_supports(const Problem& p, const void* x) {
    GtPlan pl;
    return ((uintptr_t)x % 16) == 0 && tcg::encode_fn() != nullptr && make_gt_plan(p, &pl);
}

cudaError_t launch_grouped_tma(const Problem& p, const void* x, const void* w, const void* bias,
                               void* y, cudaStream_t stream) {
    GtPlan pl;
    if (!make_gt_plan(p, &pl) || ((uintptr_t)x % 16) != 0) return cudaErrorInvalidValue;
    auto enc = tcg::encode_fn();
    if (!enc) return cudaErrorNotSupported;
    GtParams P;
    std::memset(&P, 0, sizeof(P));
    {
        const cuuint64_t dims[4] = {(cuuint64_t)p.I[2], (cuuint64_t)p.I[1], (cuuint64_t)p.I[0],
                                    (cuuint64_t)(p.B * p.C_in)};
        const cuuint64_t row = (cuuint64_t)p.I[2] * 4;
        const cuuint64_t strides[3] = {row, row * p.I[1], row * p.I[1] * p.I[0]};
        const cuuint32_t box[4] = {(cuuint32_t)kGWB, (cuuint32_t)kGNR, 1, (cuuint32_t)kGC};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        CUresult r = enc(&P.tmap_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(x), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    P.w = static_cast<const float*>(w);
    P.bias = static_cast<const float*>(bias);
    P.y = static_cast<float*>(y);
    P.C_in = (int)p.C_in;
    P.C_out = (int)p.C_out;
    P.G = p.G;
    P.Cig = p.Cig;
    P.Cog = p.Cog;
    for (int a = 0; a < 3; ++a) {
        P.I[a] = (int)p.I[a];
        P.O[a] = (int)p.O[a];
        P.S[a] = p.S[a];
        P.K[a] = (int)p.K[a];
        for (int r = 0; r < p.S[a]; ++r) {
            P.ntap[a][r] = pl.ax[a].ntaps[r];
            P.qext[a][r] = (int)pl.ax[a].q_extent[r];
            for (int j = 0; j < pl.ax[a].ntaps[r]; ++j) {
                P.tap[a][r][j] = pl.ax[a].tap[r][j];
                P.off[a][r][j] = pl.ax[a].off[r][j];
            }
        }
    }
    P.taps = (int)p.taps();
    P.n_hb = (int)((pl.ax[1].q_extent[0] + kGQB - 1) / kGQB);
    P.n_qc = (int)((pl.ax[2].q_extent[0] + kGQ - 1) / kGQ);
    P.offmin_h = pl.offmin_h;
    P.wmin = pl.wmin;
    P.nd_max = pl.nd_max;
    P.wait_ns = wait_limit_ns();
    const bool y2 = (p.O[2] % 2) == 0 && ((uintptr_t)y % 8) == 0;
    P.vecb = y2;
    int live = -1, n_live_w = 0;
    for (int r = 0; r < p.S[2]; ++r)
        if (pl.ax[2].ntaps[r] > 0) { live = r; ++n_live_w; }
    P.vec2 = y2 && p.S[2] == 2 && n_live_w == 1;
    P.live_w = P.vec2 ? live : 0;
    const int64_t blocks = p.B * (int64_t)p.G * p.O[0] * P.n_hb * P.n_qc;
    if (blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
    const size_t smem = pl.smem;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(grouped_tma_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    grouped_tma_kernel<<<(unsigned)blocks, kGW * 32, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t grouped_tma_error_word(unsigned int* v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_device_error, sizeof(*v));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace ct
