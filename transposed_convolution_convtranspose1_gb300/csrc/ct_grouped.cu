// ct_grouped.cu -- grouped/depthwise stride-phase gather on CUDA cores.
//
// The ONNX page's grouped stride-phase variant (ai.onnx.ConvTranspose,
// nchw2d_grouped_stride_phase_blocked): a thread computes some output
// positions for all output channels of their group, so each input value read
// serves every one of those channels, and a block loads its group's weights
// into shared memory a single time.
// Laid out for GB300:
//   - one warp per output row (b, od, oh), so every lane shares the row's D
//     and H residues and therefore its tap lists (no divergence on them);
//   - each lane owns one q along W and all s_w W residues of it, i.e. the s_w
//     consecutive outputs s_w*q .. s_w*q + s_w - 1, so residues with no taps
//     (bias only) and residues with taps sit in every lane alike;
//   - accumulators for all COG output channels of the group in registers,
//     weights read from the shared-memory slab as broadcasts, input samples
//     read once per (tap, channel) with lanes on consecutive positions;
//   - stores: for each output channel a warp writes 32*s_w consecutive
//     elements of one output row.
// The staged variant (used whenever its shared-memory footprint fits) first
// copies a band's input rows into shared memory; the direct variant reads
// the input through the L1 cache.
#include <algorithm>
#include <cstring>

#include "ct_routes.h"
#include "ct_types.cuh"

namespace ct {
namespace {

constexpr int kGrpMaxS = 4;       // W stride handled by one lane
constexpr int kGrpMaxSA = 8;      // D / H stride
constexpr int kGrpMaxTaps = 8;    // taps per axis and residue
constexpr int kGrpWarps = 8;      // rows per block
constexpr size_t kGrpMaxSlab = 48 * 1024;
constexpr int kGrpStageW = 4;     // staged variant: input width <= 32 * kGrpStageW

// Floats per staged position: CIGP channels, padded so that lanes reading
// consecutive positions with 16-byte loads hit distinct bank groups.
template <int CIGP>
constexpr int xstride() { return CIGP == 4 ? 4 : CIGP + 4; }

struct GroupedParams {
    const void* x;
    const void* w;
    const void* bias;
    void* y;
    int C_in, C_out, G, Cig, Cog;
    int I[3], O[3], S[3], Kdims[3];
    int ntap[3][kGrpMaxSA];
    int tap[3][kGrpMaxSA][kGrpMaxTaps];
    int off[3][kGrpMaxSA][kGrpMaxTaps];
    int qw_ext[kGrpMaxS];
    int n_rowblk;          // ceil(O_d * O_h / kGrpWarps)
    int taps;              // kD * kH * kW
    // staged variant: bands of R output rows of one output depth
    int R, n_band, nr_max, offmin_h;
    int vec2;              // fp32, stride 2 along W: rows 8-byte aligned (float2 stores)
    int cigp;              // staged variant: channels per group padded to 4, 8 or 16
    int ws, base_w;        // staged row: WS positions p, iw = p + base_w
};

// slab layout: [tap][ic][COG] (COG >= Cog, zero padded)
template <typename T, int SW, int COG>
__global__ void __launch_bounds__(kGrpWarps * 32) grouped_kernel(const __grid_constant__ GroupedParams P) {
    extern __shared__ float slab[];
    const T* __restrict__ x = static_cast<const T*>(P.x);
    const T* __restrict__ w = static_cast<const T*>(P.w);
    const T* __restrict__ bias = static_cast<const T*>(P.bias);
    T* __restrict__ y = static_cast<T*>(P.y);

    int64_t blk = blockIdx.x;
    const int rb = (int)(blk % P.n_rowblk); blk /= P.n_rowblk;
    const int g = (int)(blk % P.G);
    const int64_t b = blk / P.G;

    // stage the group's weights: w[g*Cig + ic][oc][tap] -> slab[tap][ic][oc]
    const int slab_n = P.taps * P.Cig * COG;
    for (int e = threadIdx.x; e < slab_n; e += blockDim.x) {
        const int oc = e % COG;
        const int ic = (e / COG) % P.Cig;
        const int t = e / (COG * P.Cig);
        float v = 0.f;
        if (oc < P.Cog) v = to_f32(w[((int64_t)(g * P.Cig + ic) * P.Cog + oc) * P.taps + t]);
        slab[e] = v;
    }
    __syncthreads();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int row = rb * kGrpWarps + warp;
    if (row >= P.O[0] * P.O[1]) return;  // after the only barrier
    const int od = row / P.O[1], oh = row % P.O[1];
    const int rd = od % P.S[0], qd = od / P.S[0];
    const int rh = oh % P.S[1], qh = oh / P.S[1];
    const int nd_ = P.ntap[0][rd], nh_ = P.ntap[1][rh];

    float bv[COG];
#pragma unroll
    for (int oc = 0; oc < COG; ++oc)
        bv[oc] = (bias != nullptr && oc < P.Cog) ? to_f32(bias[g * P.Cog + oc]) : 0.f;

    const int64_t in_plane = (int64_t)P.I[0] * P.I[1] * P.I[2];
    const T* xg = x + (b * P.C_in + (int64_t)g * P.Cig) * in_plane;
    const int64_t out_plane = (int64_t)P.O[0] * P.O[1] * P.O[2];
    T* yrow = y + (b * P.C_out + (int64_t)g * P.Cog) * out_plane +
              ((int64_t)od * P.O[1] + oh) * P.O[2];

    const int nq = P.qw_ext[0];  // residue 0 has the most positions
    for (int q = lane; q - lane < nq; q += 32) {
        float acc[SW][COG];
#pragma unroll
        for (int r = 0; r < SW; ++r)
#pragma unroll
            for (int oc = 0; oc < COG; ++oc) acc[r][oc] = 0.f;

#pragma unroll
        for (int r = 0; r < SW; ++r) {
            const int nw_ = P.ntap[2][r];
            if (q >= P.qw_ext[r]) continue;
            for (int jd = 0; jd < nd_; ++jd) {
                const int id = qd + P.off[0][rd][jd];
                if (id < 0 || id >= P.I[0]) continue;
                for (int jh = 0; jh < nh_; ++jh) {
                    const int ih = qh + P.off[1][rh][jh];
                    if (ih < 0 || ih >= P.I[1]) continue;
                    const T* xr = xg + ((int64_t)id * P.I[1] + ih) * P.I[2];
                    const int tdh = (P.tap[0][rd][jd] * P.Kdims[1] + P.tap[1][rh][jh]) * P.Kdims[2];
                    for (int jw = 0; jw < nw_; ++jw) {
                        const int iw = q + P.off[2][r][jw];
                        if (iw < 0 || iw >= P.I[2]) continue;
                        const float* ws = slab + (int64_t)(tdh + P.tap[2][r][jw]) * P.Cig * COG;
                        const T* xp = xr + iw;
                        for (int ic = 0; ic < P.Cig; ++ic) {
                            const float xv = to_f32(xp[(int64_t)ic * in_plane]);
                            const float* wv = ws + ic * COG;
#pragma unroll
                            for (int oc = 0; oc < COG; ++oc) acc[r][oc] = fmaf(xv, wv[oc], acc[r][oc]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int oc = 0; oc < COG; ++oc) {
            if (oc >= P.Cog) break;
#pragma unroll
            for (int r = 0; r < SW; ++r)
                if (q < P.qw_ext[r])
                    yrow[(int64_t)oc * out_plane + r + (int64_t)SW * q] = from_f32<T>(acc[r][oc] + bv[oc]);
        }
    }
}


// Staged variant: one block per (b, g, od, band of R output rows).  The input
// rows the band reads (every D tap of the depth's phase and the H rows of all
// the band's rows) are first copied into shared memory channels-innermost,
// [row][p][ic] with CIGP channels (zero padded, positions xstride<CIGP>()
// floats apart) and WS positions p covering
// iw = p + base_w for every position slot and tap offset (zeros outside the
// input), so the tap loop needs no bounds checks: for one tap a lane reads
// its CIGP channels with CIGP/4 16-byte loads.  Each lane owns two q
// positions of a row (q and q + 32) and every W residue of them; per tap and
// channel the COG weights are loaded once (broadcast) and used for both
// positions with packed two-lane fp32 FMAs over output-channel pairs.
template <typename T, int SW, int COG, int CIGP>
__global__ void __launch_bounds__(kGrpWarps * 32) grouped_staged_kernel(const __grid_constant__ GroupedParams P) {
    extern __shared__ __align__(16) float sm[];
    const T* __restrict__ x = static_cast<const T*>(P.x);
    const T* __restrict__ w = static_cast<const T*>(P.w);
    const T* __restrict__ bias = static_cast<const T*>(P.bias);
    T* __restrict__ y = static_cast<T*>(P.y);
    constexpr int COGP = COG < 2 ? 2 : COG;   // padded to an even count for f32x2 pairs

    int64_t blk = blockIdx.x;
    const int band = (int)(blk % P.n_band); blk /= P.n_band;
    const int od = (int)(blk % P.O[0]); blk /= P.O[0];
    const int g = (int)(blk % P.G);
    const int64_t b = blk / P.G;
    const int rd = od % P.S[0], qd = od / P.S[0];
    const int nd_ = P.ntap[0][rd];
    const int oh0 = band * P.R;
    const int ih_lo = oh0 / P.S[1] + P.offmin_h;
    const int NR = P.nr_max;
    const int WS = P.ws;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // weights: slab[tap][ic][oc], CIGP x COGP per tap (zero padded)
    float* slab = sm;
    float* xs = sm + P.taps * CIGP * COGP;  // [jd * NR + r][p][CIGP]
    // Loads are issued in batches (every load of a batch in flight before
    // its stores), so that the block waits for global memory a few times
    // rather than once per staged element.
    constexpr int kSlabBatch = 4;
    const int slab_n = P.taps * CIGP * COGP;
    for (int e0 = threadIdx.x; e0 < slab_n; e0 += kSlabBatch * blockDim.x) {
        float v[kSlabBatch];
#pragma unroll
        for (int k = 0; k < kSlabBatch; ++k) {
            const int e = e0 + k * blockDim.x;
            const int oc = e % COGP;
            const int ic = (e / COGP) % CIGP;
            const int t = e / (COGP * CIGP);
            v[k] = (e < slab_n && oc < P.Cog && ic < P.Cig)
                       ? to_f32(w[((int64_t)(g * P.Cig + ic) * P.Cog + oc) * P.taps + t]) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kSlabBatch; ++k)
            if (e0 + k * blockDim.x < slab_n) slab[e0 + k * blockDim.x] = v[k];
    }
    const int64_t in_plane = (int64_t)P.I[0] * P.I[1] * P.I[2];
    const T* xg = x + (b * P.C_in + (int64_t)g * P.Cig) * in_plane;
    // one staged row (jd, r) per warp iteration: all CIGP channels, lanes on p
    for (int rowi = warp; rowi < nd_ * NR; rowi += kGrpWarps) {
        const int jd = rowi / NR, r = rowi - jd * NR;
        const int id = qd + P.off[0][rd][jd];
        const int ih = ih_lo + r;
        const bool row_ok = id >= 0 && id < P.I[0] && ih >= 0 && ih < P.I[1];
        const T* src = xg + ((int64_t)id * P.I[1] + ih) * P.I[2];
        // every slot of the row loaded before any is stored
        float v[kGrpStageW][CIGP];
#pragma unroll
        for (int k = 0; k < kGrpStageW; ++k) {
            const int pp = lane + 32 * k;
            const int iw = pp + P.base_w;
            const bool ok = row_ok && pp < WS && iw >= 0 && iw < P.I[2];
#pragma unroll
            for (int ic = 0; ic < CIGP; ++ic)
                v[k][ic] = (ok && ic < P.Cig) ? to_f32(src[(int64_t)ic * in_plane + iw]) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kGrpStageW; ++k) {
            const int pp = lane + 32 * k;
            if (pp >= WS) break;
            float4* dst = reinterpret_cast<float4*>(xs + ((int64_t)rowi * WS + pp) * xstride<CIGP>());
#pragma unroll
            for (int c4 = 0; c4 < CIGP / 4; ++c4)
                dst[c4] = make_float4(v[k][4 * c4], v[k][4 * c4 + 1], v[k][4 * c4 + 2], v[k][4 * c4 + 3]);
        }
    }
    __syncthreads();

    float bv[COGP];
#pragma unroll
    for (int oc = 0; oc < COGP; ++oc)
        bv[oc] = (bias != nullptr && oc < P.Cog) ? to_f32(bias[g * P.Cog + oc]) : 0.f;
    const int64_t out_plane = (int64_t)P.O[0] * P.O[1] * P.O[2];
    const int nq = P.qw_ext[0];

    const int rows_per_warp = P.R / kGrpWarps;
    for (int i = 0; i < rows_per_warp; ++i) {
        const int row = warp * rows_per_warp + i;  // consecutive rows: mixed H residues
        const int oh = oh0 + row;
        if (oh >= P.O[1]) break;
        const int rh = oh % P.S[1], qh = oh / P.S[1];
        const int nh_ = P.ntap[1][rh];
        T* yrow = y + (b * P.C_out + (int64_t)g * P.Cog) * out_plane +
                  ((int64_t)od * P.O[1] + oh) * P.O[2];
        for (int qb = 0; qb < nq; qb += 64) {
            const int qv0 = qb + lane, qv1 = qb + 32 + lane;
            float2 acc[2][SW][COGP / 2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int r = 0; r < SW; ++r)
#pragma unroll
                    for (int o2 = 0; o2 < COGP / 2; ++o2) acc[u][r][o2] = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < SW; ++r) {
                const int nw_ = P.ntap[2][r];
                for (int jd = 0; jd < nd_; ++jd)
                    for (int jh = 0; jh < nh_; ++jh) {
                        const int lr = jd * NR + qh + P.off[1][rh][jh] - ih_lo;
                        const float* xr = xs + ((int64_t)lr * WS + qv0 - P.base_w) * xstride<CIGP>();
                        const int tdh = (P.tap[0][rd][jd] * P.Kdims[1] + P.tap[1][rh][jh]) * P.Kdims[2];
                        for (int jw = 0; jw < nw_; ++jw) {
                            const float4* x0p =
                                reinterpret_cast<const float4*>(xr + P.off[2][r][jw] * xstride<CIGP>());
                            const float4* x1p = x0p + 32 * xstride<CIGP>() / 4;
                            const float* ws = slab + (tdh + P.tap[2][r][jw]) * CIGP * COGP;
#pragma unroll
                            for (int c4 = 0; c4 < CIGP / 4; ++c4) {
                                const float4 a0 = x0p[c4], a1 = x1p[c4];
                                const float xa[4] = {a0.x, a0.y, a0.z, a0.w};
                                const float xb[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                                for (int ii = 0; ii < 4; ++ii) {
                                    const float* wr = ws + (c4 * 4 + ii) * COGP;
                                    const float2 d0 = make_float2(xa[ii], xa[ii]);
                                    const float2 d1 = make_float2(xb[ii], xb[ii]);
                                    if constexpr (COGP % 4 == 0) {
#pragma unroll
                                        for (int o4 = 0; o4 < COGP / 4; ++o4) {
                                            const float4 wq = *reinterpret_cast<const float4*>(wr + 4 * o4);
                                            const float2 wlo = make_float2(wq.x, wq.y);
                                            const float2 whi = make_float2(wq.z, wq.w);
                                            fma2(acc[0][r][2 * o4], d0, wlo);
                                            fma2(acc[1][r][2 * o4], d1, wlo);
                                            fma2(acc[0][r][2 * o4 + 1], d0, whi);
                                            fma2(acc[1][r][2 * o4 + 1], d1, whi);
                                        }
                                    } else {
#pragma unroll
                                        for (int o2 = 0; o2 < COGP / 2; ++o2) {
                                            const float2 wv = *reinterpret_cast<const float2*>(wr + 2 * o2);
                                            fma2(acc[0][r][o2], d0, wv);
                                            fma2(acc[1][r][o2], d1, wv);
                                        }
                                    }
                                }
                            }
                        }
                    }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int q = u ? qv1 : qv0;
                if (q >= nq) continue;
#pragma unroll
                for (int oc = 0; oc < COG; ++oc) {
                    if (oc >= P.Cog) break;
                    T* yo = yrow + (int64_t)oc * out_plane + (int64_t)SW * q;
                    const float bo = bv[oc];
                    if constexpr (SW == 2 && sizeof(T) == 4) {
                        if (P.vec2 && q < P.qw_ext[1]) {
                            const float v0 = (oc & 1) ? acc[u][0][oc >> 1].y : acc[u][0][oc >> 1].x;
                            const float v1 = (oc & 1) ? acc[u][1][oc >> 1].y : acc[u][1][oc >> 1].x;
                            *reinterpret_cast<float2*>(yo) = make_float2(v0 + bo, v1 + bo);
                            continue;
                        }
                    }
#pragma unroll
                    for (int r = 0; r < SW; ++r) {
                        const float v = (oc & 1) ? acc[u][r][oc >> 1].y : acc[u][r][oc >> 1].x;
                        if (q < P.qw_ext[r]) yo[r] = from_f32<T>(v + bo);
                    }
                }
            }
        }
    }
}

struct GroupedPlan {
    AxisPlan ax[3];
    int cog_pad;
    bool staged;
    int R, nr_max, offmin_h, cigp, ws, base_w;
    size_t smem;
};

constexpr size_t kGrpMaxStaged = 96 * 1024;

int pad_cog(int cog) {
    if (cog <= 1) return 1;
    if (cog <= 2) return 2;
    if (cog <= 4) return 4;
    if (cog <= 8) return 8;
    return 16;
}

bool make_plan(const Problem& p, GroupedPlan* pl) {
    if (p.Cog > 16) return false;
    if (p.S[2] > kGrpMaxS || p.S[0] > kGrpMaxSA || p.S[1] > kGrpMaxSA) return false;
    for (int a = 0; a < 3; ++a) {
        plan_axis(p, a, &pl->ax[a]);
        for (int r = 0; r < p.S[a]; ++r)
            if (pl->ax[a].ntaps[r] > kGrpMaxTaps) return false;
    }
    pl->cog_pad = pad_cog(p.Cog);
    const size_t slab = (size_t)p.taps() * p.Cig * pl->cog_pad * sizeof(float);
    if (slab > kGrpMaxSlab) return false;
    if (p.O[0] * p.O[1] >= (1ll << 30)) return false;
    // staged variant: bands of R rows; the band reads input rows
    // [oh0 / s_h + min_off, (oh0 + R - 1) / s_h + max_off]
    int offmin = 1 << 30, offmax = -(1 << 30), ndmax = 0;
    for (int r = 0; r < p.S[1]; ++r)
        for (int j = 0; j < pl->ax[1].ntaps[r]; ++j) {
            offmin = std::min(offmin, pl->ax[1].off[r][j]);
            offmax = std::max(offmax, pl->ax[1].off[r][j]);
        }
    for (int r = 0; r < p.S[0]; ++r) ndmax = std::max(ndmax, pl->ax[0].ntaps[r]);
    pl->staged = false;
    pl->cigp = p.Cig <= 4 ? 4 : p.Cig <= 8 ? 8 : p.Cig <= 16 ? 16 : 0;
    // W span of the staged rows: position slots q in [0, 64 * ceil(nq / 64))
    // read iw = q + off for every W offset off of every residue
    int wmin = 1 << 30, wmax = -(1 << 30);
    for (int r = 0; r < p.S[2]; ++r)
        for (int j = 0; j < pl->ax[2].ntaps[r]; ++j) {
            wmin = std::min(wmin, pl->ax[2].off[r][j]);
            wmax = std::max(wmax, pl->ax[2].off[r][j]);
        }
    const int64_t nq_slots = (pl->ax[2].q_extent[0] + 63) / 64 * 64;
    if (offmin <= offmax && wmin <= wmax && pl->cigp > 0 &&
        nq_slots + (wmax - wmin) <= 32 * kGrpStageW) {
        pl->ws = (int)(nq_slots + (wmax - wmin));
        pl->base_w = wmin;
        for (int R : {16, 8}) {
            // floor((oh0 + R - 1) / s) - floor(oh0 / s) <= floor((R - 1) / s) + 1
            const int nr = (R - 1) / p.S[1] + 2 + (offmax - offmin);
            const int cogp = pl->cog_pad < 2 ? 2 : pl->cog_pad;
            const size_t wslab = (size_t)p.taps() * pl->cigp * cogp * sizeof(float);
            const int xst = pl->cigp == 4 ? 4 : pl->cigp + 4;  // xstride<CIGP>()
            const size_t sm = wslab + (size_t)std::max(ndmax, 1) * nr * pl->ws * xst * sizeof(float);
            if (sm <= kGrpMaxStaged) {
                pl->staged = true;
                pl->R = R;
                pl->nr_max = nr;
                pl->offmin_h = offmin;
                pl->smem = sm;
                break;
            }
        }
    }
    return true;
}

template <typename T, int SW, int COG, int CIGP>
cudaError_t launch_staged(const GroupedParams& P, int64_t blocks, size_t smem, cudaStream_t stream) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(grouped_staged_kernel<T, SW, COG, CIGP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    grouped_staged_kernel<T, SW, COG, CIGP><<<(unsigned)blocks, kGrpWarps * 32, smem, stream>>>(P);
    return cudaGetLastError();
}

template <typename T, int SW, int COG>
cudaError_t launch_grouped_t(const GroupedParams& P, int64_t blocks, size_t smem, cudaStream_t stream) {
    if (P.R > 0) {
        switch (P.cigp) {
            case 4: return launch_staged<T, SW, COG, 4>(P, blocks, smem, stream);
            case 8: return launch_staged<T, SW, COG, 8>(P, blocks, smem, stream);
            default: return launch_staged<T, SW, COG, 16>(P, blocks, smem, stream);
        }
    } else {
        grouped_kernel<T, SW, COG><<<(unsigned)blocks, kGrpWarps * 32, smem, stream>>>(P);
    }
    return cudaGetLastError();
}

template <typename T, int SW>
cudaError_t dispatch_cog(int cog, const GroupedParams& P, int64_t blocks, size_t slab,
                         cudaStream_t stream) {
    switch (cog) {
        case 1: return launch_grouped_t<T, SW, 1>(P, blocks, slab, stream);
        case 2: return launch_grouped_t<T, SW, 2>(P, blocks, slab, stream);
        case 4: return launch_grouped_t<T, SW, 4>(P, blocks, slab, stream);
        case 8: return launch_grouped_t<T, SW, 8>(P, blocks, slab, stream);
        default: return launch_grouped_t<T, SW, 16>(P, blocks, slab, stream);
    }
}

template <typename T>
cudaError_t dispatch_sw(int sw, int cog, const GroupedParams& P, int64_t blocks, size_t slab,
                        cudaStream_t stream) {
    switch (sw) {
        case 1: return dispatch_cog<T, 1>(cog, P, blocks, slab, stream);
        case 2: return dispatch_cog<T, 2>(cog, P, blocks, slab, stream);
        case 3: return dispatch_cog<T, 3>(cog, P, blocks, slab, stream);
        default: return dispatch_cog<T, 4>(cog, P, blocks, slab, stream);
    }
}

}  // namespace

bool grouped_supports(const Problem& p) {
    GroupedPlan pl;
    return make_plan(p, &pl);
}

bool grouped_preferred(const Problem& p) { return p.Cog <= 16; }

const char* grouped_kernel_name(const Problem& p) {
    GroupedPlan pl;
    if (!make_plan(p, &pl)) return "";
    // asked for an input at a 16-byte aligned address, as device allocations are
    alignas(16) static const char aligned = 0;
    if (grouped_warp_supports(p, &aligned)) return "grouped_warp_kernel";
    if (grouped_tma_supports(p, &aligned)) return "grouped_tma_kernel";
    return pl.staged ? "grouped_staged_kernel" : "grouped_kernel";
}

cudaError_t launch_grouped(const Problem& p, const void* x, const void* w, const void* bias,
                           void* y, cudaStream_t stream, Profile* prof, bool* act_done) {
    GroupedPlan pl;
    *act_done = false;
    if (!make_plan(p, &pl)) return cudaErrorInvalidValue;
    if (grouped_warp_supports(p, x)) {
        prof_begin(prof, stream);
        cudaError_t e = launch_grouped_warp(p, x, w, bias, y, stream);
        prof_end(prof, stream);
        prof_count(prof);
        *act_done = true;
        return e;
    }
    if (grouped_tma_supports(p, x)) {
        prof_begin(prof, stream);
        cudaError_t e = launch_grouped_tma(p, x, w, bias, y, stream);
        prof_end(prof, stream);
        prof_count(prof);
        return e;
    }
    GroupedParams P;
    std::memset(&P, 0, sizeof(P));
    P.x = x;
    P.w = w;
    P.bias = bias;
    P.y = y;
    P.C_in = (int)p.C_in;
    P.C_out = (int)p.C_out;
    P.G = p.G;
    P.Cig = p.Cig;
    P.Cog = p.Cog;
    for (int a = 0; a < 3; ++a) {
        P.I[a] = (int)p.I[a];
        P.O[a] = (int)p.O[a];
        P.S[a] = p.S[a];
        P.Kdims[a] = (int)p.K[a];
        for (int r = 0; r < p.S[a]; ++r) {
            P.ntap[a][r] = pl.ax[a].ntaps[r];
            for (int j = 0; j < pl.ax[a].ntaps[r]; ++j) {
                P.tap[a][r][j] = pl.ax[a].tap[r][j];
                P.off[a][r][j] = pl.ax[a].off[r][j];
            }
        }
    }
    for (int r = 0; r < p.S[2]; ++r) P.qw_ext[r] = (int)pl.ax[2].q_extent[r];
    P.taps = (int)p.taps();
    P.n_rowblk = (int)((p.O[0] * p.O[1] + kGrpWarps - 1) / kGrpWarps);
    int64_t blocks = p.B * (int64_t)p.G * P.n_rowblk;
    size_t slab = (size_t)P.taps * P.Cig * pl.cog_pad * sizeof(float);
    if (pl.staged) {
        P.R = pl.R;
        P.n_band = (int)((p.O[1] + pl.R - 1) / pl.R);
        P.nr_max = pl.nr_max;
        P.offmin_h = pl.offmin_h;
        P.cigp = pl.cigp;
        P.ws = pl.ws;
        P.base_w = pl.base_w;
        P.vec2 = p.dtype == CT_F32 && p.S[2] == 2 && (p.O[2] % 2) == 0 && ((uintptr_t)y % 8) == 0;
        blocks = p.B * (int64_t)p.G * p.O[0] * P.n_band;
        slab = pl.smem;
    }
    if (blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
    prof_begin(prof, stream);
    cudaError_t e;
    switch (p.dtype) {
        case CT_F32: e = dispatch_sw<float>(p.S[2], pl.cog_pad, P, blocks, slab, stream); break;
        case CT_F16: e = dispatch_sw<__half>(p.S[2], pl.cog_pad, P, blocks, slab, stream); break;
        default: e = dispatch_sw<__nv_bfloat16>(p.S[2], pl.cog_pad, P, blocks, slab, stream); break;
    }
    prof_end(prof, stream);
    prof_count(prof);
    return e;
}

}  // namespace ct
