// ct_simt.cu -- fp32 stride-phase implicit GEMM on CUDA cores (FFMA).
//
// Same decomposition as the tensor-core route: outputs are split by their
// residue on every axis, and within one phase each output row
// (b, od, oh) and W residue rw is a dense GEMM
//     Y[oc, q] = sum_{(td,th,tw) in T(rd) x T(rh) x T(rw), ic} W'[t][ic][oc] * X[b, ic, id, ih, q + off_w]
// with id = qd + off_d, ih = qh + off_h -- the stride-phase tiled GEMM the
// ONNX page lists for 1-D and 2-D (conv-transpose1d-phase-tiled,
// conv-transpose2d-phase-gemm-tiled) -- computed here in exact fp32 FMA so
// that fp32 problems keep fp32 accuracy.  Two kernels run:
//   1. simt_weight_reorder : w [C_in, C_out, taps] -> W' [taps][C_in_pad][N_pad]
//   2. simt_phase_gemm     : 128 (oc) x 128 (q) tiles, K in steps of 16,
//      256 threads with 8 x 8 register tiles (packed two-lane fp32 FMAs,
//      fma.rn.f32x2, the same IEEE result as fmaf), both operands staged
//      in a three-stage shared-memory ring through cp.async (weights 16 bytes
//      at a time, the tap-shifted x window 4 bytes at a time since its start
//      is arbitrary, lanes on consecutive elements), one barrier per k-tile,
//      bias added in fp32 at the end.
#include <algorithm>
#include <cstring>

#include "ct_routes.h"
#include "ct_types.cuh"

namespace ct {
namespace {

constexpr int kBM = 128;  // output channels per tile
constexpr int kBN = 128;  // q positions per tile
constexpr int kBK = 16;   // reduction step
constexpr int kStages = 3; // cp.async pipeline depth
constexpr int kSimtThreads = 256;
constexpr int kSimtMaxS = 8;
constexpr int kSimtMaxTaps = 16;

struct SimtParams {
    const float* x;
    const float* wp;  // [taps][C_in_pad][N_pad]
    const float* bias;
    float* y;
    int C_in, C_in_pad, C_out, N_pad;
    int I[3], O[3], S[3], Kdims[3];
    int ntap[3][kSimtMaxS];
    int tap[3][kSimtMaxS][kSimtMaxTaps];
    int off[3][kSimtMaxS][kSimtMaxTaps];
    int qw_ext[kSimtMaxS];
    int n_qblk, n_ocblk;
    int64_t n_blocks;
};

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

// 4-byte copy; src_bytes = 0 writes a zero instead of reading.
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kSimtThreads, 2) simt_phase_gemm(const __grid_constant__ SimtParams P) {
    extern __shared__ __align__(16) float smem_f[];
    // stage s: As[s][k][oc] then Bs[s][k][q]
    auto As = [&](int s, int k) { return smem_f + (size_t)s * 2 * kBK * kBM + (size_t)k * kBM; };
    auto Bs = [&](int s, int k) { return smem_f + (size_t)s * 2 * kBK * kBM + (size_t)(kBK + k) * kBN; };

    // block -> (oc block, q block, W residue, output row (b, od, oh))
    int64_t blk = blockIdx.x;
    const int ocb = (int)(blk % P.n_ocblk); blk /= P.n_ocblk;
    const int qb = (int)(blk % P.n_qblk); blk /= P.n_qblk;
    const int rw = (int)(blk % P.S[2]); blk /= P.S[2];
    const int oh = (int)(blk % P.O[1]); blk /= P.O[1];
    const int od = (int)(blk % P.O[0]);
    const int64_t b = blk / P.O[0];
    const int rd = od % P.S[0], qd = od / P.S[0];
    const int rh = oh % P.S[1], qh = oh / P.S[1];
    const int oc0 = ocb * kBM, q0 = qb * kBN;
    const int qext = P.qw_ext[rw];
    if (q0 >= qext) return;  // uniform per block

    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int warp = tid / 32, lane = tid % 32;

    const int nd_ = P.ntap[0][rd], nh_ = P.ntap[1][rh], nw_ = P.ntap[2][rw];
    const int ntaps = nd_ * nh_ * nw_;
    const int kchunks = P.C_in_pad / kBK;
    const int nk = ntaps * kchunks;

    const int64_t in_plane = (int64_t)P.I[0] * P.I[1] * P.I[2];
    const float* xb = P.x + b * P.C_in * in_plane;

    // A tile: 16 x 128 floats = 512 float4, two per thread (rows warp, warp + 8);
    // B tile: 16 x 128 floats, rows warp and warp + 8, lanes on consecutive floats
    auto load_tile = [&](int kt, int st) {
        const int j = kt / kchunks;
        const int ic0 = (kt % kchunks) * kBK;
        const int jw = j % nw_;
        const int jh = (j / nw_) % nh_;
        const int jd = j / (nw_ * nh_);
        const int tap = (P.tap[0][rd][jd] * P.Kdims[1] + P.tap[1][rh][jh]) * P.Kdims[2] + P.tap[2][rw][jw];
        const int id = qd + P.off[0][rd][jd];
        const int ih = qh + P.off[1][rh][jh];
        const int iwb = q0 + P.off[2][rw][jw];
        const bool dh_ok = id >= 0 && id < P.I[0] && ih >= 0 && ih < P.I[1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = warp + 8 * h;
            cp_async16(As(st, k) + lane * 4,
                       P.wp + ((int64_t)tap * P.C_in_pad + ic0 + k) * P.N_pad + oc0 + lane * 4);
            const int ic = ic0 + k;
            const bool row_ok = dh_ok && ic < P.C_in;
            const float* xr = xb + (int64_t)ic * in_plane + ((int64_t)id * P.I[1] + ih) * P.I[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int col = lane + 32 * i;
                const int iw = iwb + col;
                const bool ok = row_ok && iw >= 0 && iw < P.I[2];
                cp_async4(Bs(st, k) + col, ok ? xr + iw : P.x, ok);
            }
        }
    };

    // acc2[i][jj] holds outputs (oc_i, q_{2jj}) and (oc_i, q_{2jj+1})
    float2 acc2[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc2[i][j] = make_float2(0.f, 0.f);

    if (nk > 0) {
        // prologue: stages 0 .. kStages-2
#pragma unroll
        for (int st = 0; st < kStages - 1; ++st) {
            if (st < nk) load_tile(st, st);
            cp_async_commit();
        }
        for (int kt = 0; kt < nk; ++kt) {
            cp_async_wait<kStages - 2>();  // tile kt has landed
            __syncthreads();               // and every thread is done with tile kt - 1
            {
                const int kn = kt + kStages - 1;
                if (kn < nk) load_tile(kn, kn % kStages);
                cp_async_commit();
            }
            const int st = kt % kStages;
#pragma unroll
            for (int k = 0; k < kBK; ++k) {
                const float4 a0 = *reinterpret_cast<const float4*>(As(st, k) + ty * 4);
                const float4 a1 = *reinterpret_cast<const float4*>(As(st, k) + ty * 4 + 64);
                const float4 b0 = *reinterpret_cast<const float4*>(Bs(st, k) + tx * 4);
                const float4 b1 = *reinterpret_cast<const float4*>(Bs(st, k) + tx * 4 + 64);
                const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const float2 bb[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                      make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 ad = make_float2(a[i], a[i]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) fma2(acc2[i][j], ad, bb[j]);
                }
            }
        }
        cp_async_wait<0>();
    }

    // epilogue: y[b, oc, od, oh, ow = rw + s_w * q] = acc + bias[oc]
    const int64_t plane = (int64_t)P.O[0] * P.O[1] * P.O[2];
    const int64_t row_off = ((int64_t)od * P.O[1] + oh) * P.O[2];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int oc = oc0 + ty * 4 + (i & 3) + (i >> 2) * 64;
        if (oc >= P.C_out) continue;
        const float bv = P.bias ? P.bias[oc] : 0.f;
        float* yr = P.y + (b * P.C_out + oc) * plane + row_off;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int q = q0 + tx * 4 + (j & 3) + (j >> 2) * 64;
            const float a = (j & 1) ? acc2[i][j >> 1].y : acc2[i][j >> 1].x;
            if (q < qext) yr[rw + (int64_t)P.S[2] * q] = a + bv;
        }
    }
}

// W'[t][c][n] = w[c][n][t] for c < C_in, n < C_out; 0 in the padding.
__global__ void simt_weight_reorder(const float* __restrict__ w, float* __restrict__ wp, int C_in,
                                    int C_out, int taps, int C_in_pad, int N_pad) {
    const int64_t total = (int64_t)taps * C_in_pad * N_pad;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int n = (int)(e % N_pad);
        const int c = (int)((e / N_pad) % C_in_pad);
        const int t = (int)(e / ((int64_t)N_pad * C_in_pad));
        wp[e] = (c < C_in && n < C_out) ? w[((int64_t)c * C_out + n) * taps + t] : 0.f;
    }
}

struct SimtPlan {
    int C_in_pad, N_pad;
    AxisPlan ax[3];
};

bool make_plan(const Problem& p, SimtPlan* pl) {
    if (p.dtype != CT_F32 || p.G != 1) return false;
    for (int a = 0; a < 3; ++a) {
        if (p.S[a] > kSimtMaxS) return false;
        plan_axis(p, a, &pl->ax[a]);
        for (int r = 0; r < p.S[a]; ++r)
            if (pl->ax[a].ntaps[r] > kSimtMaxTaps) return false;
    }
    pl->C_in_pad = (int)((p.C_in + kBK - 1) / kBK * kBK);
    pl->N_pad = (int)((p.C_out + kBM - 1) / kBM * kBM);
    return true;
}

}  // namespace

bool simt_supports(const Problem& p) {
    SimtPlan pl;
    return make_plan(p, &pl);
}

bool simt_preferred(const Problem& p) {
    // worth the tile machinery once the reduction and the channel count fill a tile
    return p.C_in >= 32 && p.C_out >= 32;
}

size_t simt_workspace_bytes(const Problem& p) {
    SimtPlan pl;
    if (!make_plan(p, &pl)) return 0;
    return ((size_t)p.taps() * pl.C_in_pad * pl.N_pad * 4 + 255) / 256 * 256;
}

cudaError_t launch_simt(const Problem& p, const void* x, const void* w, const void* bias, void* y,
                        void* workspace, cudaStream_t stream, Profile* prof) {
    SimtPlan pl;
    if (!make_plan(p, &pl)) return cudaErrorInvalidValue;
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    float* wp = static_cast<float*>(workspace);
    {
        const int64_t tot = p.taps() * pl.C_in_pad * pl.N_pad;
        const int blocks = (int)std::min<int64_t>((tot + 255) / 256, (int64_t)dev.sm_count * 8);
        simt_weight_reorder<<<blocks, 256, 0, stream>>>(static_cast<const float*>(w), wp,
                                                        (int)p.C_in, (int)p.C_out, (int)p.taps(),
                                                        pl.C_in_pad, pl.N_pad);
        prof_count(prof);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    SimtParams P;
    std::memset(&P, 0, sizeof(P));
    P.x = static_cast<const float*>(x);
    P.wp = wp;
    P.bias = static_cast<const float*>(bias);
    P.y = static_cast<float*>(y);
    P.C_in = (int)p.C_in;
    P.C_in_pad = pl.C_in_pad;
    P.C_out = (int)p.C_out;
    P.N_pad = pl.N_pad;
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
    P.n_qblk = (int)((pl.ax[2].q_extent[0] + kBN - 1) / kBN);
    P.n_ocblk = pl.N_pad / kBM;
    const int64_t blocks =
        p.B * p.O[0] * p.O[1] * (int64_t)p.S[2] * P.n_qblk * (int64_t)P.n_ocblk;
    if (blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
    P.n_blocks = blocks;
    const size_t smem = (size_t)kStages * 2 * kBK * kBM * sizeof(float);
    e = cudaFuncSetAttribute(simt_phase_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_begin(prof, stream);
    simt_phase_gemm<<<(unsigned)blocks, kSimtThreads, smem, stream>>>(P);
    prof_end(prof, stream);
    prof_count(prof);
    return cudaGetLastError();
}

}  // namespace ct
