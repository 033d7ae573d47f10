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
//   bwd_db_partial  a block per (output channel, run of its On positions, all
//                   batch elements); each thread sums 8-value vectors in four
//                   compensated (Kahan) fp32 sums, then a fixed shared-memory
//                   tree; bwd_db_final adds a channel's segments in order.
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
//   bwd_dw_grouped_kernel   dw of small groups (at most 8 input and 8 output
//                   channels, at most 27 taps): persistent blocks, each a
//                   contiguous run of bands of 4 input rows; a band's x rows
//                   and the dy rows its taps reach are staged in shared
//                   memory (fp32: 16-byte copies of whole spans, the next
//                   band while this one is summed) and every thread sums one
//                   output channel's taps for its input channels over its
//                   positions.  Partials per (column, run segment) and
//                   bwd_dw_reduce as above.
#include <algorithm>
#include <climits>
#include <cstring>
#include <type_traits>

#include "ct_internal.h"
#include "ct_routes.h"
#include "ct_tcgen05.cuh"
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
    uint64_t wait_ns;       // limit of the bounded waits on staged copies
};

// ---------------------------------------------------------------------------
// db
// ---------------------------------------------------------------------------

constexpr int kDbThreads = 256;

// db in two passes.  Pass 1: block (oc, k) sums channel oc over every batch
// element and the k-th run [k seg, (k+1) seg) of its On positions (seg a
// multiple of 8), each thread in four compensated (Kahan) sums over 8-value
// vectors, a vector of every batch element before the next vector (one 16-byte load for 16-bit types, two for fp32, when On is a
// multiple of 8 and dy is 16-byte aligned), then a fixed shared-memory tree;
// the block writes part[oc][k].  Pass 2 adds each channel's partials in order
// (compensated) and rounds once.
template <typename T>
__global__ void __launch_bounds__(kDbThreads) bwd_db_partial(const __grid_constant__ BwdArgs a, float* part,
                                                             int n_seg, int64_t seg, bool vec) {
    __shared__ float red[kDbThreads];
    const int64_t oc = blockIdx.x / n_seg;
    const int k = (int)(blockIdx.x % n_seg);
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const int64_t o0 = (int64_t)k * seg, o1 = min(a.On, o0 + seg);
    float sum[4] = {0.f, 0.f, 0.f, 0.f}, comp[4] = {0.f, 0.f, 0.f, 0.f};
    auto add = [&](int u, float v) {
        const float y = v - comp[u];
        const float t = sum[u] + y;
        comp[u] = (t - sum[u]) - y;
        sum[u] = t;
    };
    // a thread's position vector of every batch element in turn: B independent
    // loads per vector, so several are in flight
    const T* chan = dy + oc * a.On;
    const int64_t bstride = a.C_out * a.On;
    if (vec) {
        for (int64_t o = o0 + 8 * (int64_t)threadIdx.x; o < o1; o += 8 * kDbThreads) {
#pragma unroll 4
            for (int64_t b = 0; b < a.B; ++b) {
                const T* q = chan + b * bstride + o;
                float v[8];
                if constexpr (sizeof(T) == 2) {
                    const uint4 u = *reinterpret_cast<const uint4*>(q);
                    const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = to_f32(h[j]);
                } else {
                    const float4 q0 = reinterpret_cast<const float4*>(q)[0];
                    const float4 q1 = reinterpret_cast<const float4*>(q)[1];
                    v[0] = q0.x; v[1] = q0.y; v[2] = q0.z; v[3] = q0.w;
                    v[4] = q1.x; v[5] = q1.y; v[6] = q1.z; v[7] = q1.w;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) add(j & 3, v[j]);
            }
        }
    } else {
        for (int64_t o = o0 + threadIdx.x; o < o1; o += kDbThreads)
#pragma unroll 4
            for (int64_t b = 0; b < a.B; ++b) add((int)(b & 3), to_f32(chan[b * bstride + o]));
    }
    red[threadIdx.x] = (sum[0] + sum[1]) + (sum[2] + sum[3]);
    __syncthreads();
    for (int h = kDbThreads / 2; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h) red[threadIdx.x] += red[threadIdx.x + h];
        __syncthreads();
    }
    if (threadIdx.x == 0) part[oc * n_seg + k] = red[0];
}

template <typename T>
__global__ void __launch_bounds__(256) bwd_db_final(const float* __restrict__ part, T* __restrict__ db, int64_t C_out,
                                                    int n_seg) {
    const int64_t oc = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (oc >= C_out) return;
    float sum = 0.f, comp = 0.f;
    for (int k = 0; k < n_seg; ++k) {
        const float y = part[oc * n_seg + k] - comp;
        const float t = sum + y;
        comp = (t - sum) - y;
        sum = t;
    }
    db[oc] = from_f32<T>(sum);
}

// Position runs of each channel for bwd_db_partial: about eight resident
// 256-thread blocks per SM in all, each run at least 2048 positions.
void db_split(const Problem& p, int sm_count, int* n_seg, int64_t* seg) {
    const int64_t n = p.out_spatial();
    const int64_t want = std::max<int64_t>(1, 8ll * std::max(1, sm_count) / std::max<int64_t>(1, p.C_out));
    const int64_t k = std::max<int64_t>(1, std::min<int64_t>(want, (n + 2047) / 2048));
    int64_t s = (n + k - 1) / k;
    s = (s + 7) / 8 * 8;
    *seg = std::max<int64_t>(8, s);
    *n_seg = (int)std::max<int64_t>(1, (n + *seg - 1) / *seg);
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

// dw for small groups (Cig, Cog <= 8, taps <= 27).  A column is (batch
// element, input depth, group); its input rows are cut into bands of kDwgR.
// A band needs its x rows and the RD dy rows its taps reach (dy zero outside
// the output, so interior products need no range check).  Partials:
// part[(b, input depth, segment)][g*Cig + ic][oc*taps + t], one per run of a
// column's bands that one block sums, zeros in the slots no block uses.
constexpr int kDwgR = 4;       // input rows per band
constexpr int kDwgC = 8;       // channels per group, at most
constexpr unsigned kErrDwCopy = 1u << 7;  // a staged copy of the grouped dw kernel timed out

struct DwgGeom {
    int n_band;               // bands of kDwgR input rows along H
    int n_blocks;             // persistent blocks: block k takes bands [k T / n_blocks, (k+1) T / n_blocks)
    int n_seg;                // partial slots per column (segments of a column's bands, at most)
    int RD, CD;               // staged dy rows (per jd) and columns
    int ow_min;               // output column of the first staged column (-pad_lo of W)
    int stage_floats;         // one staging buffer
    // element copies (16-bit types): x [ic][r][w], dy [oc][jd][rr][W phase][column / S_W]
    int rp;                   // staged dy row pitch (floats)
    int CDH;                  // columns per W phase
    int xs_plane, ds_off, ds_oc, ds_jd;
    int toff[27];             // per tap: offset of its dy value from the position's base
    // span copies (fp32): per input channel its band rows, per (oc, jd) the RD
    // dy rows as one grid of pitch O_W; offset tables; zeros for channels past Cig
    int xslot;                // floats per x channel slot
    int gslot;                // floats per dy grid slot
    int xs_tab, g_tab;        // offsets of the x / grid origin tables (ints) in a buffer
    int gpad;                 // extra offset of odd output channels' grids (bank spread)
    int zero_off, zero_len;   // zeros for channels past Cig (after both buffers)
    int red_off;              // lane totals of the second position half (after the zeros)
    int w_a, w_b;             // input columns [w_a, w_b) read only columns inside y for every tap
    int tjd[27];              // per tap: its depth tap (grid)
    int tgo[27];              // per tap: offset in the grid from (r * S_H) * O_W + w * S_W
    int tnew[27];             // per tap: 1 where the depth tap changes
    int tcol[27];             // per tap: output column of input column 0, tw * d_W - pad_lo
};

// Stage one band by element copies (16-bit types): x rows [ic][r][w] (zero
// for ic >= Cig) and the dy region the band's taps read, [oc][jd][rr][W
// phase][column / S_W] (zero outside y), so that neighbouring input columns
// read neighbouring words for every tap.  A warp takes one staged row at a
// time, its lanes 32 consecutive columns.
template <typename T>
__device__ __forceinline__ void dwg_stage(const BwdArgs& a, const DwgGeom& G, float* buf, int64_t b, int g, int id,
                                          int i0) {
    const T* __restrict__ x = static_cast<const T*>(a.x);
    const T* __restrict__ dy = static_cast<const T*>(a.dy);
    const int IW = a.I[2];
    const int rows = min(kDwgR, a.I[1] - i0);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, n_warps = blockDim.x / 32;
    const T* xb = x + ((b * a.C_in + (int64_t)g * a.Cig) * a.I[0] + id) * (int64_t)a.I[1] * IW + (int64_t)i0 * IW;
    const int64_t x_chan = (int64_t)a.I[0] * a.I[1] * IW;
    for (int row = warp; row < kDwgC * rows; row += n_warps) {
        const int ic = row / rows, r = row - ic * rows;
        const bool ok = ic < a.Cig;
        const T* src = xb + (ok ? ic * x_chan + (int64_t)r * IW : 0);
        float* dst = buf + ic * G.xs_plane + r * IW;
        for (int w = lane; w < IW; w += 32) dst[w] = ok ? to_f32(src[w]) : 0.f;
    }
    const int KD = a.K[0], S2 = a.S[2], RD = G.RD;
    const int oh0 = i0 * a.S[1] - a.PL[1], ow0 = G.ow_min;
    const int64_t o_plane = (int64_t)a.O[1] * a.O[2];
    const T* dyb = dy + (b * a.C_out + (int64_t)g * a.Cog) * a.O[0] * o_plane;
    // this lane's first column in (W phase, column / S_W) form, and the step of 32 columns
    const int ph0 = lane % S2, q0 = lane / S2, dph = 32 % S2, dq = 32 / S2;
    float* ds = buf + G.ds_off;
    for (int row = warp; row < a.Cog * KD * RD; row += n_warps) {
        const int rr = row % RD, jd = (row / RD) % KD, oc = row / (RD * KD);
        const int od = id * a.S[0] - a.PL[0] + jd * a.DL[0], oh = oh0 + rr;
        const bool row_ok = od >= 0 && od < a.O[0] && oh >= 0 && oh < a.O[1];
        const T* src = dyb + (row_ok ? ((int64_t)oc * a.O[0] + od) * o_plane + (int64_t)oh * a.O[2] : 0);
        float* dst = ds + oc * G.ds_oc + jd * G.ds_jd + rr * G.rp;
        int ph = ph0, q = q0;
        for (int cc = lane; cc < G.CD; cc += 32) {
            const int ow = ow0 + cc;
            dst[ph * G.CDH + q] = row_ok && ow >= 0 && ow < a.O[2] ? to_f32(src[ow]) : 0.f;
            ph += dph;
            q += dq;
            if (ph >= S2) { ph -= S2; ++q; }
        }
    }
}

// Stage one band by span copies (fp32; every thread takes part): per input
// channel its band rows (contiguous in x) into its slot, per (oc, jd) the dy
// rows of the band that lie inside y (contiguous, full width) into its grid,
// each span widened to 16-byte boundaries and moved in 16-byte cp.async
// pieces (span j by warp j mod warps, its lanes taking every 32nd piece).  A
// grid's origin is shifted by 0..3 floats so that the copy's destination is
// 16-byte aligned; the tables record where element 0 of each x channel and
// row 0 / column 0 of each grid landed; channels past Cig point at zeros.
// Odd output channels' grids sit gpad floats further on, so that the two
// output channels a warp reads at once fall in different banks.  Each thread
// then arrives on the buffer's mbarrier (initialised for the
// whole block) once its own pieces have landed.
__device__ __forceinline__ void dwg_issue_spans(const BwdArgs& a, const DwgGeom& G, float* sm, int buf_off,
                                                uint32_t bar, int64_t b, int g, int id, int i0) {
    const float* __restrict__ x = static_cast<const float*>(a.x);
    const float* __restrict__ dy = static_cast<const float*>(a.dy);
    const int IW = a.I[2], KD = a.K[0], RD = G.RD, OW = a.O[2];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, n_warps = blockDim.x / 32;
    const int rows = min(kDwgR, a.I[1] - i0);
    const int n_items = a.Cig + a.Cog * KD;
    const int oh0 = i0 * a.S[1] - a.PL[1];
    const int rr_lo = max(0, -oh0), rr_hi = min(RD - 1, a.O[1] - 1 - oh0);  // grid rows inside y
    int* xtab = reinterpret_cast<int*>(sm + buf_off + G.xs_tab);
    int* gtab = reinterpret_cast<int*>(sm + buf_off + G.g_tab);
    for (int k = warp; k < n_items; k += n_warps) {
        const float* src = nullptr;
        int n = 0, dst = 0;
        if (k < a.Cig) {
            src = x + ((b * a.C_in + (int64_t)g * a.Cig + k) * a.I[0] + id) * (int64_t)a.I[1] * IW + (int64_t)i0 * IW;
            n = rows * IW;
            const int slot = buf_off + k * G.xslot;  // a multiple of 4 floats
            const int lead = (int)((reinterpret_cast<uintptr_t>(src) & 15) / 4);
            dst = slot;
            if (lane == 0) xtab[k] = slot + lead;
        } else {
            const int kk = k - a.Cig, jd = kk % KD, oc = kk / KD;
            const int od = id * a.S[0] - a.PL[0] + jd * a.DL[0];
            const int slot = buf_off + G.xslot * a.Cig + kk * G.gslot + (oc & 1) * G.gpad;
            int origin = slot + 4;
            if (od >= 0 && od < a.O[0] && rr_lo <= rr_hi) {
                src = dy + (((b * a.C_out + (int64_t)g * a.Cog + oc) * a.O[0] + od) * a.O[1] + oh0 + rr_lo) *
                               (int64_t)OW;
                n = (rr_hi - rr_lo + 1) * OW;
                // grid origin = slot + 4 + delta; the copy lands at origin + rr_lo * O_W - lead
                const int lead = (int)((reinterpret_cast<uintptr_t>(src) & 15) / 4);
                origin += ((lead - rr_lo * OW) % 4 + 4) % 4;
                dst = origin + rr_lo * OW - lead;
            }
            if (lane == 0) gtab[kk] = origin;
        }
        if (n > 0) {
            const uintptr_t s0 = reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15);
            const uintptr_t s1 = (reinterpret_cast<uintptr_t>(src + n) + 15) & ~uintptr_t(15);
            const int pieces = (int)((s1 - s0) / 16);
            const uint32_t d0 = tcg::smem_u32(sm + dst);
            for (int c = lane; c < pieces; c += 32)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d0 + 16u * c),
                             "l"(reinterpret_cast<const void*>(s0 + 16u * c))
                             : "memory");
        }
    }
    if (threadIdx.x < kDwgC - a.Cig) xtab[a.Cig + threadIdx.x] = G.zero_off;
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for an mbarrier phase by one thread, which sleeps in the
// try_wait (suspend hint) instead of spinning; the others wait at the block
// barrier that follows.  A limit of 0 gives up at once.  Records kErrDwCopy
// and returns false on giving up.
__device__ __forceinline__ bool dwg_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (limit_ns == 0) {
        atomicOr(&g_device_error, kErrDwCopy);
        return false;
    }
    const uint64_t t0 = tcg::globaltimer_ns();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(100000u)
            : "memory");
        if (ok) return true;
        if (tcg::globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_device_error, kErrDwCopy);
            return false;
        }
    }
}

// Zero the grid rows of this buffer that lie outside y (no copy wrote them,
// or a copy's widening did): per depth tap, all RD rows when its depth lies
// outside y, else the rows before rr_lo and after rr_hi; a warp per row.
// Returns whether the band has such rows (the same answer in every thread).
__device__ __forceinline__ bool dwg_zero_rows(const BwdArgs& a, const DwgGeom& G, const float* buf, float* sm, int id,
                                              int i0) {
    const int KD = a.K[0], RD = G.RD, OW = a.O[2];
    const int oh0 = i0 * a.S[1] - a.PL[1];
    const int rr_lo = max(0, -oh0), rr_hi = min(RD - 1, a.O[1] - 1 - oh0);
    const int od0 = id * a.S[0] - a.PL[0];
    const bool depth_ok = od0 >= 0 && od0 + (KD - 1) * a.DL[0] < a.O[0];
    if (rr_lo == 0 && rr_hi == RD - 1 && depth_ok) return false;
    const int* gtab = reinterpret_cast<const int*>(buf + G.g_tab);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, n_warps = blockDim.x / 32;
    int row = warp, rr = warp % RD, kk = warp / RD;  // row = kk * RD + rr, kk = oc * KD + jd
    for (; row < a.Cog * KD * RD; row += n_warps) {
        const int jd = kk % KD;
        const int od = od0 + jd * a.DL[0];
        if (od < 0 || od >= a.O[0] || rr < rr_lo || rr > rr_hi) {
            float* dst = sm + gtab[kk] + rr * OW;
            for (int c = lane; c < OW; c += 32) dst[c] = 0.f;
        }
        rr += n_warps;
        while (rr >= RD) { rr -= RD; ++kk; }
    }
    return true;
}

// One butterfly step over lanes OFF apart: a lane keeps the half of its OFF
// * 2 values that its OFF bit selects and adds its partner's copy of them.
template <int OFF, int N>
__device__ __forceinline__ void butterfly_step(float (&v)[N], int lane) {
    const bool upper = (lane & OFF) != 0;
#pragma unroll
    for (int j = 0; j < OFF; ++j) {
        const float send = upper ? v[j] : v[j + OFF];
        const float keep = upper ? v[j + OFF] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
    }
}

// Sum each of N values (N = 32 or 16) over the N lanes of the warp (or of
// its half) that hold them, by a fixed butterfly, so the order is the same on
// every run; lane l returns the total of v[l mod N].
template <int N>
__device__ __forceinline__ float lane_totals(float (&v)[N], int lane) {
    if constexpr (N == 32) butterfly_step<16>(v, lane);
    butterfly_step<8>(v, lane);
    butterfly_step<4>(v, lane);
    butterfly_step<2>(v, lane);
    butterfly_step<1>(v, lane);
    return v[0];
}

// dw of groups with at most 8 input and 8 output channels.  The work is cut
// into units -- (group, batch element, input depth, run of bpb bands of
// kDwgR input rows) -- and each persistent block takes units blockIdx.x,
// blockIdx.x + gridDim.x, ... in turn.  Each thread keeps ICT x KN fp32 sums
// (input channels x taps, in channel pairs for the packed FMA) of one output
// channel.
//   fp32 (ROWS): bands are staged by span copies (16-byte cp.async), the
//   block's next band (of this unit or the next) while this one is summed
//   (two buffers, an mbarrier each).  Warp (oc pair, ic group, position half)
//   splits its lanes into two halves of 16, one per output channel of the
//   pair, both walking the same 16 consecutive positions: x reads are
//   broadcasts and the two halves' dy reads fall in different banks.  Chunks
//   of 16 positions alternate between the two position halves.  After a
//   unit's last band each half-warp sums its lanes (butterfly), the second
//   position half hands its totals over in shared memory and the first adds
//   them and writes the unit's partial.
//   16-bit types: element copies into the phase-split layout (one buffer);
//   warp (oc, ic group), lane l the positions l, l + 32, ...; lane totals
//   over the whole warp.
// bwd_dw_reduce adds the band groups' partials in order.  A span copy that
// does not arrive within the wait limit sets kErrDwCopy; the block then
// drains its copies and stops.
template <typename T, int ICT, int KN, bool ROWS>
__global__ void __launch_bounds__(kDwgC * (kDwgC / ICT) * 32, ICT == 8 ? 2 : 1)
    bwd_dw_grouped_kernel(const __grid_constant__ BwdArgs a, const __grid_constant__ DwgGeom G) {
    extern __shared__ __align__(128) float sm_raw[];
    __shared__ __align__(8) uint64_t bar[2];
    __shared__ int abort_flag;
    float* sm = sm_raw + ((128u - (tcg::smem_u32(sm_raw) & 127u)) & 127u) / 4;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr int NIG = kDwgC / ICT;  // input channel groups
    // ROWS: warp = (oc pair, ic group, position half), lane = (oc of the pair, position)
    // else: warp = (oc, ic group), lane = position
    const int oc = ROWS ? 2 * (warp % 4) + lane / 16 : warp % kDwgC;
    const int icb = ROWS ? ((warp / 4) % NIG) * ICT : (warp / kDwgC) * ICT;
    const int half = ROWS ? warp / (4 * NIG) : 0;
    const int j16 = lane % 16;
    const bool live = oc < a.Cog && icb < a.Cig;
    const int IW = a.I[2], S1 = a.S[1], S2 = a.S[2];

    // band z of all T = columns x n_band, column c = ((b * I_D) + id) * G + g
    struct Band {
        int64_t b;
        int g, id, band;
        int64_t col;
    };
    auto band_of = [&](int64_t z) {
        Band w;
        w.col = z / G.n_band;
        w.band = (int)(z - w.col * G.n_band);
        w.g = (int)(w.col % a.G);
        const int64_t bd = w.col / a.G;
        w.id = (int)(bd % a.I[0]);
        w.b = bd / a.I[0];
        return w;
    };
    const int64_t TB = (int64_t)a.G * a.B * a.I[0] * G.n_band;
    const int64_t z_lo = (int64_t)blockIdx.x * TB / G.n_blocks, z_hi = (int64_t)(blockIdx.x + 1) * TB / G.n_blocks;
    // the block holding band z: the largest k with floor(k TB / n_blocks) <= z
    auto block_of = [&](int64_t zz) { return ((zz + 1) * G.n_blocks + TB - 1) / TB - 1; };
    if (z_lo >= z_hi) return;

    // sums of input channel pairs (icb + 2m, icb + 2m + 1), per tap
    float2 acc[ICT / 2][KN];
#pragma unroll
    for (int m = 0; m < ICT / 2; ++m)
#pragma unroll
        for (int t = 0; t < KN; ++t) acc[m][t] = make_float2(0.f, 0.f);

    int64_t z = z_lo;
    Band cu = band_of(z);
    int n_issued = 0, n_done = 0;  // bands staged by span copies, and (thread 0) waited for
    if constexpr (ROWS) {
        if (threadIdx.x == 0) {
            abort_flag = 0;
            tcg::mbar_init(tcg::smem_u32(&bar[0]), blockDim.x);  // every thread arrives once per band
            tcg::mbar_init(tcg::smem_u32(&bar[1]), blockDim.x);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        for (int e = threadIdx.x; e < G.zero_len; e += blockDim.x) sm[G.zero_off + e] = 0.f;
        __syncthreads();
        dwg_issue_spans(a, G, sm, 0, tcg::smem_u32(&bar[0]), cu.b, cu.g, cu.id, cu.band * kDwgR);
        n_issued = 1;
    }
    bool ok = true;
    for (int k = 0;; ++k) {
        const bool more = z + 1 < z_hi;
        const Band nx = more ? band_of(z + 1) : cu;
        float* buf = sm + (ROWS ? (k & 1) : 0) * G.stage_floats;
        if constexpr (ROWS) {
            if (more) {
                dwg_issue_spans(a, G, sm, ((k + 1) & 1) * G.stage_floats, tcg::smem_u32(&bar[(k + 1) & 1]), nx.b,
                                nx.g, nx.id, nx.band * kDwgR);
                ++n_issued;
            }

            // band k of the block is buffer k & 1's (k >> 1)-th copy
            if (threadIdx.x == 0) {
                if (dwg_wait(tcg::smem_u32(&bar[k & 1]), (k >> 1) & 1, a.wait_ns))
                    ++n_done;
                else
                    abort_flag = 1;
            }
            __syncthreads();
            if (abort_flag) { ok = false; break; }
            if (dwg_zero_rows(a, G, buf, sm, cu.id, cu.band * kDwgR)) __syncthreads();
        } else {
            dwg_stage<T>(a, G, buf, cu.b, cu.g, cu.id, cu.band * kDwgR);
            __syncthreads();
        }
        if (live) {
            const int rows = min(kDwgR, a.I[1] - cu.band * kDwgR);
            if constexpr (ROWS) {
                const int* xtab = reinterpret_cast<const int*>(buf + G.xs_tab);
                const int* gtab = reinterpret_cast<const int*>(buf + G.g_tab) + oc * a.K[0];
                const int OW = a.O[2];
                int xo[ICT];
#pragma unroll
                for (int i = 0; i < ICT; ++i) xo[i] = xtab[icb + i];
                // dy of tap t at goff(t) + pos: offsets in registers up to 16 taps, looked up beyond
                constexpr int NG = KN <= 16 ? KN : 1;
                int gt[NG];
#pragma unroll
                for (int t = 0; t < NG; ++t) gt[t] = gtab[G.tjd[t]] + G.tgo[t];
                auto goff = [&](int t) { return KN <= 16 ? gt[t < NG ? t : 0] : gtab[G.tjd[t]] + G.tgo[t]; };
                // positions: first the columns [w_a, w_b), whose taps all read dy
                // columns inside y, then the others, whose taps outside y add
                // nothing (masked); this half-warp takes position q = 16 c + j16
                // of chunks c = half, half + 2, ... (the interior walked
                // incrementally: 32 positions between a half's chunks)
                const int nwi = G.w_b - G.w_a, nwe = IW - nwi;
                const int n_int = rows * nwi, n_all = rows * IW;
                int ri = 0, wi = G.w_a + 16 * half + j16;
                if (nwi > 0)
                    while (wi >= G.w_b) { wi -= nwi; ++ri; }
                for (int q0 = 16 * half; q0 < n_all; q0 += 32) {
                    const int q = q0 + j16;
                    int r = ri, w = wi;
                    if (q >= n_int && q < n_all) {
                        const int e = q - n_int, re = e / nwe, c = e - re * nwe;
                        r = re;
                        w = c < G.w_a ? c : G.w_b + (c - G.w_a);
                    }
                    if (q0 + 16 <= n_int) {
                        float2 xp[ICT / 2];
                        const int p = r * IW + w;
#pragma unroll
                        for (int m = 0; m < ICT / 2; ++m) xp[m] = make_float2(sm[xo[2 * m] + p], sm[xo[2 * m + 1] + p]);
                        const int pos = r * S1 * OW + w * S2;
#pragma unroll
                        for (int t = 0; t < KN; ++t) {
                            const float dv = sm[goff(t) + pos];
                            const float2 d2 = make_float2(dv, dv);
#pragma unroll
                            for (int m = 0; m < ICT / 2; ++m) acc[m][t] = __ffma2_rn(xp[m], d2, acc[m][t]);
                        }
                    } else if (q < n_all) {
                        float2 xp[ICT / 2];
                        const int p = r * IW + w;
#pragma unroll
                        for (int m = 0; m < ICT / 2; ++m) xp[m] = make_float2(sm[xo[2 * m] + p], sm[xo[2 * m + 1] + p]);
                        const int pos = r * S1 * OW + w * S2;
#pragma unroll
                        for (int t = 0; t < KN; ++t) {
                            const unsigned ow = (unsigned)(w * S2 + G.tcol[t]);
                            const float dv = ow < (unsigned)OW ? sm[goff(t) + pos] : 0.f;
                            const float2 d2 = make_float2(dv, dv);
#pragma unroll
                            for (int m = 0; m < ICT / 2; ++m) acc[m][t] = __ffma2_rn(xp[m], d2, acc[m][t]);
                        }
                    }
                    if (nwi > 0) {
                        wi += 32;
                        while (wi >= G.w_b) { wi -= nwi; ++ri; }
                    }
                }
            } else {
                const float* xs = buf + icb * G.xs_plane;
                const float* ds = buf + G.ds_off + oc * G.ds_oc;
                for (int p = lane; p < rows * IW; p += 32) {
                    const int r = p / IW, w = p - r * IW;
                    float xv[ICT];
#pragma unroll
                    for (int i = 0; i < ICT; ++i) xv[i] = xs[i * G.xs_plane + p];
                    const float* dp = ds + r * S1 * G.rp + w;
#pragma unroll
                    for (int t = 0; t < KN; ++t) {
                        const float dv = dp[G.toff[t]];
#pragma unroll
                        for (int m = 0; m < ICT / 2; ++m) {
                            acc[m][t].x = fmaf(xv[2 * m], dv, acc[m][t].x);
                            acc[m][t].y = fmaf(xv[2 * m + 1], dv, acc[m][t].y);
                        }
                    }
                }
            }
        }
        __syncthreads();  // the buffer is staged again
        if (!more || nx.col != cu.col) {
            // the block's segment of this column is done: its partial goes to slot s
            // (the number of block boundaries inside the column before it); the
            // column's last segment also zeroes the slots no block uses
            const int64_t col0 = cu.col * G.n_band;
            const int s_here = (int)(blockIdx.x - block_of(col0));
            const int s_end = z + 1 == col0 + G.n_band ? G.n_seg : s_here + 1;
            const int NN = a.Cog * a.Kn;
            const int64_t chunk = (cu.b * a.I[0] + cu.id) * G.n_seg + s_here;
            float* part = a.part + (chunk * a.C_in + (int64_t)cu.g * a.Cig) * NN;
            for (int s2 = s_here + 1; s2 < s_end; ++s2) {
                float* zp = a.part + (((cu.b * a.I[0] + cu.id) * G.n_seg + s2) * a.C_in + (int64_t)cu.g * a.Cig) * NN;
                for (int e = threadIdx.x; e < a.Cig * NN; e += blockDim.x) zp[e] = 0.f;
            }
            constexpr int N = ROWS ? 16 : 32;
            constexpr int NC = (ICT * KN + N - 1) / N;  // chunks of N sums
            float mine[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float v[N];
#pragma unroll
                for (int jj = 0; jj < N; ++jj) {
                    const int kk = c * N + jj, i = kk / KN, t = kk % KN;
                    v[jj] = kk < ICT * KN ? (i % 2 ? acc[i / 2][t].y : acc[i / 2][t].x) : 0.f;
                }
                mine[c] = lane_totals<N>(v, lane);
            }
            if constexpr (ROWS) {
                // the second position half hands its totals to the first: [oc pair][ic group][chunk][lane]
                float* red = sm + G.red_off + ((warp % 4) * NIG + (warp / 4) % NIG) * NC * 32;
                if (half == 1)
#pragma unroll
                    for (int c = 0; c < NC; ++c) red[c * 32 + lane] = mine[c];
                __syncthreads();
                if (half == 0)
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const int kk = c * N + j16;
                        const float tot = mine[c] + red[c * 32 + lane];
                        if (live && kk < ICT * KN) {
                            const int ic = icb + kk / KN, t = kk % KN;
                            if (ic < a.Cig && t < a.Kn) part[(int64_t)ic * NN + oc * a.Kn + t] = tot;
                        }
                    }
            } else {
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const int kk = c * N + lane;
                    if (live && kk < ICT * KN) {
                        const int ic = icb + kk / KN, t = kk % KN;
                        if (ic < a.Cig && t < a.Kn) part[(int64_t)ic * NN + oc * a.Kn + t] = mine[c];
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < ICT / 2; ++m)
#pragma unroll
                for (int t = 0; t < KN; ++t) acc[m][t] = make_float2(0.f, 0.f);
        }
        if (!more) break;
        ++z;
        cu = nx;
    }
    if constexpr (ROWS) {
        if (!ok && threadIdx.x == 0)  // copies issued and not waited for complete before the block leaves
            for (int k = n_done; k < n_issued; ++k) tcg::mbar_drain(tcg::smem_u32(&bar[k & 1]), (k >> 1) & 1);
    }
}

// dw[e] = sum over slices (in slice order) of part[ks][e], rounded once.
template <typename T>
__global__ void __launch_bounds__(256) bwd_dw_reduce(const float* __restrict__ part, T* __restrict__ dw,
                                                     int64_t n, int n_ks) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
#pragma unroll 8
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
    bool dwg;           // dw by bwd_dw_grouped_kernel
    int dwg_kn;         // its tap-count instantiation
    int dwg_ict;        // input channels per warp
    int dwg_threads;
    size_t dwg_smem;    // element-copy staging
    DwgGeom geom;
    bool dwg_rows;      // fp32 row-copy staging fits
    size_t dwg_smem_rows;
    DwgGeom geom_rows;
    int sm_count;       // the SM count the plan was made for
};

// The small-group dw kernel's geometry, when it applies: at most 8 input and
// 8 output channels per group, at most 27 taps, staging within 110 KB (two
// blocks per SM).  fp32 takes the row-copy layout when it fits, everything
// else the element-copy layout; the band grouping (and so the partials) does
// not depend on the layout.
bool dwg_plan(const Problem& p, int sm_count, BwdPlan* pl) {
    const int64_t taps = p.taps();
    if (p.Cig > kDwgC || p.Cog > kDwgC || taps > 27) return false;
    if (p.I[2] > 4096 || p.I[1] > (1 << 24) || p.S[2] > 64 || p.PL[2] > 4096) return false;
    DwgGeom G;
    std::memset(&G, 0, sizeof(G));
    const int rows = (int)std::min<int64_t>(kDwgR, p.I[1]);
    const int IW = (int)p.I[2], KD = (int)p.K[0];
    G.n_band = (int)((p.I[1] + kDwgR - 1) / kDwgR);
    G.RD = (int)(p.S[1] * (rows - 1) + p.DL[1] * (p.K[1] - 1) + 1);
    G.CD = (int)(p.S[2] * (IW - 1) + p.DL[2] * (p.K[2] - 1) + 1);
    G.ow_min = -p.PL[2];
    pl->dwg_kn = taps <= 4 ? 4 : taps <= 9 ? 9 : taps <= 16 ? 16 : 27;
    pl->dwg_ict = pl->dwg_kn <= 9 ? 8 : 4;
    pl->dwg_threads = kDwgC * (kDwgC / pl->dwg_ict) * 32;
    // persistent blocks (two per SM with 256 threads, one with 512), each a
    // contiguous run of the T = G B I_D n_band bands; a column's bands are cut
    // into at most n_seg runs (the runs are at least T / n_blocks long)
    const int64_t TB = (int64_t)p.G * p.B * p.I[0] * G.n_band;
    const int64_t nb = std::max<int64_t>(1, std::min<int64_t>(TB, (pl->dwg_threads == 256 ? 2 : 1) *
                                                                      (int64_t)std::max(1, sm_count)));
    G.n_blocks = (int)nb;
    const int64_t gap = std::max<int64_t>(1, TB / nb);
    G.n_seg = (int)std::min<int64_t>(G.n_band, (G.n_band - 1) / gap + 2);
    const size_t kMax = 115000;  // two blocks per SM
    // element copies: x [ic][r][w], dy [oc][jd][rr][W phase][column / S_W]
    {
        DwgGeom& C = pl->geom;
        C = G;
        C.CDH = (G.CD + p.S[2] - 1) / p.S[2];
        C.rp = C.CDH * p.S[2];
        C.xs_plane = (rows * IW + 3) / 4 * 4;
        C.ds_off = kDwgC * C.xs_plane;
        C.ds_jd = G.RD * C.rp;
        C.ds_oc = (KD * C.ds_jd + 3) / 4 * 4;
        C.stage_floats = C.ds_off + kDwgC * C.ds_oc;
        for (int t = 0; t < 27; ++t) {
            const int u = t < taps ? t : 0;  // padding taps read tap 0's word
            const int tw = (int)(u % p.K[2]), th = (int)((u / p.K[2]) % p.K[1]), td = (int)(u / (p.K[2] * p.K[1]));
            const int cw = tw * p.DL[2];
            C.toff[t] = td * C.ds_jd + th * p.DL[1] * C.rp + (cw % p.S[2]) * C.CDH + cw / p.S[2];
        }
        const size_t smem = (size_t)C.stage_floats * sizeof(float) + 128;
        if (smem > kMax) return false;
        pl->dwg_smem = smem;
    }
    // span copies: x channel slots, dy grids of RD rows x O_W (4 + 0..3 floats
    // before the origin, widening room after), tables, zeros
    {
        DwgGeom& R = pl->geom_rows;
        R = G;
        const int OW = (int)p.O[2];
        const int64_t grid = (int64_t)G.RD * OW;
        R.xslot = (kDwgR * IW + 8 + 3) / 4 * 4;
        R.gslot = (int)std::min<int64_t>((grid + 16 + 31) / 32 * 32, 1 << 24);
        // odd output channels' grids gpad further: the two halves of a warp read
        // 16 consecutive positions (columns S_W apart) of two grids; pick the
        // shift that spreads those 32 words over the most banks
        {
            int best = 33;
            for (int d = 0; d < 32; d += 4) {
                int cnt[32] = {0}, worst = 0;
                for (int jj = 0; jj < 16; ++jj) {
                    worst = std::max(worst, ++cnt[(jj * p.S[2]) % 32]);
                    worst = std::max(worst, ++cnt[(d + jj * p.S[2]) % 32]);
                }
                if (worst < best) {
                    best = worst;
                    R.gpad = d;
                }
            }
        }
        R.xs_tab = p.Cig * R.xslot + p.Cog * KD * R.gslot + R.gpad;
        R.g_tab = R.xs_tab + kDwgC;
        R.stage_floats = (R.g_tab + p.Cog * KD + 31) / 32 * 32;
        R.zero_off = 2 * R.stage_floats;
        R.zero_len = (kDwgR * IW + 3) / 4 * 4;
        R.red_off = R.zero_off + R.zero_len;
        const int red_len = 4 * (kDwgC / pl->dwg_ict) * ((pl->dwg_ict * pl->dwg_kn + 15) / 16) * 32;
        // interior input columns: 0 <= w * S_W - pad_lo + tw * d_W <= O_W - 1 for every tw
        const int span = p.DL[2] * (int)(p.K[2] - 1);
        R.w_a = std::min(IW, (std::max(0, p.PL[2]) + p.S[2] - 1) / p.S[2]);
        const int last = OW - 1 + p.PL[2] - span;  // w * S_W <= last
        R.w_b = last < 0 ? 0 : std::min(IW, last / p.S[2] + 1);
        if (R.w_b < R.w_a) R.w_b = R.w_a;
        for (int t = 0; t < 27; ++t) {
            const int u = t < taps ? t : 0;
            const int tw = (int)(u % p.K[2]), th = (int)((u / p.K[2]) % p.K[1]), td = (int)(u / (p.K[2] * p.K[1]));
            R.tjd[t] = td;
            R.tcol[t] = G.ow_min + tw * p.DL[2];
            R.tgo[t] = th * p.DL[1] * OW + R.tcol[t];
            R.tnew[t] = t == 0 || R.tjd[t] != R.tjd[t - 1] || t >= taps;
        }
        const size_t smem = ((size_t)R.red_off + red_len) * sizeof(float) + 128;
        pl->dwg_rows = p.dtype == CT_F32 && grid < (1 << 22) && smem <= kMax;
        pl->dwg_smem_rows = smem;
    }
    const int64_t chunks = p.B * p.I[0] * G.n_seg;
    if (chunks * p.G >= (1ll << 31) || chunks >= (1ll << 31)) return false;
    pl->n_ks = (int)chunks;
    pl->part_bytes = (size_t)chunks * (size_t)p.C_in * (size_t)p.Cog * taps * sizeof(float);
    return true;
}

bool bwd_plan(const Problem& p, int sm_count, BwdPlan* pl) {
    pl->sm_count = sm_count;
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
    pl->dwg = dwg_plan(p, sm_count, pl);  // replaces n_ks and part_bytes when it applies
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

// Persistent launch of the planned blocks (their band runs fix the partial
// slots, so the grid is part of the plan).
template <typename T, int ICT, int KN, bool ROWS>
cudaError_t launch_dwg_v(const BwdArgs& a, const DwgGeom& G, size_t smem, cudaStream_t stream) {
    auto k = bwd_dw_grouped_kernel<T, ICT, KN, ROWS>;
    constexpr int threads = kDwgC * (kDwgC / ICT) * 32;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    k<<<(unsigned)G.n_blocks, threads, smem, stream>>>(a, G);
    return cudaGetLastError();
}

// The grouped dw kernel: row copies for fp32 when they fit, element copies
// otherwise.
template <typename T, int ICT, int KN>
cudaError_t launch_dwg_t(const BwdArgs& a, const BwdPlan& pl, int64_t units, cudaStream_t stream) {
    if (units == 0) return cudaSuccess;
    if constexpr (std::is_same<T, float>::value) {
        if (pl.dwg_rows) return launch_dwg_v<T, ICT, KN, true>(a, pl.geom_rows, pl.dwg_smem_rows, stream);
    }
    return launch_dwg_v<T, ICT, KN, false>(a, pl.geom, pl.dwg_smem, stream);
}

template <typename T>
cudaError_t launch_backward_t(const Problem& p, const BwdPlan& pl, BwdArgs a, cudaStream_t stream,
                              int* launches) {
    cudaError_t e = cudaSuccess;
    if (a.db && p.C_out > 0) {
        // the partials use the workspace before dx and dw do (same stream)
        int n_seg;
        int64_t seg;
        db_split(p, pl.sm_count, &n_seg, &seg);
        float* part = a.part;
        const bool vec = p.out_spatial() % 8 == 0 && (uintptr_t)a.dy % 16 == 0;
        const int64_t blocks = p.C_out * n_seg;
        if (blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
        bwd_db_partial<T><<<(unsigned)blocks, kDbThreads, 0, stream>>>(a, part, n_seg, seg, vec);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        bwd_db_final<T><<<(unsigned)((p.C_out + 255) / 256), 256, 0, stream>>>(part, static_cast<T*>(a.db), p.C_out,
                                                                          n_seg);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.dx && p.x_elems() > 0 && tc_dx_supports(p)) {
        // tensor cores: dy's channels-last copy (with the gathered weights) in
        // the workspace, then the GEMM; dw, if asked for, reuses the workspace
        // after them on the same stream
        e = launch_tc_dx(p, a.dy, a.w, a.dx, a.part, stream);
        *launches += 2;
        if (e != cudaSuccess) return e;
    } else if (a.dx && p.x_elems() > 0 && tc32_dx_supports(p)) {
        // fp32: the same mapping on the error-compensated TF32 GEMM
        e = launch_tc32_dx(p, a.dy, a.w, a.dx, a.part, stream);
        *launches += 2;
        if (e != cudaSuccess) return e;
    } else if (a.dx) {
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
    if (a.dw && nw > 0 && p.B * p.in_spatial() > 0 && tc_dw_supports(p) && (uintptr_t)a.x % 16 == 0) {
        // tensor cores: dy's channels-last copy and the split partials in the
        // workspace, then the GEMM and the reduction of the splits
        e = launch_tc_dw(p, a.x, a.dy, a.dw, a.part, stream);
        *launches += 3;
        if (e != cudaSuccess) return e;
    } else if (a.dw && nw > 0 && pl.dwg) {
        const int64_t blocks = (int64_t)p.G * pl.n_ks;
        switch (pl.dwg_kn) {
            case 4: e = launch_dwg_t<T, 8, 4>(a, pl, blocks, stream); break;
            case 9: e = launch_dwg_t<T, 8, 9>(a, pl, blocks, stream); break;
            case 16: e = launch_dwg_t<T, 4, 16>(a, pl, blocks, stream); break;
            default: e = launch_dwg_t<T, 4, 27>(a, pl, blocks, stream); break;
        }
        ++*launches;
        if (e != cudaSuccess) return e;
        const int rb = (int)std::min<int64_t>((nw + 255) / 256, 152 * 8);
        bwd_dw_reduce<T><<<rb, 256, 0, stream>>>(a.part, static_cast<T*>(a.dw), nw, pl.n_ks);
        ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    } else if (a.dw && nw > 0) {
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

cudaError_t backward_error_word(unsigned int* v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_device_error, sizeof(*v));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    return e;
}

const char* backward_dx_kernel_name(const Problem& p) {
    if (p.x_elems() == 0) return "";
    if (tc_dx_supports(p)) return "tc_phase_gemm";
    return tc32_dx_supports(p) ? "tc32_phase_gemm" : "bwd_dx_kernel";
}

const char* backward_dw_kernel_name(const Problem& p) {
    if (p.w_elems() == 0) return "";
    DeviceInfo d;
    int sm = 152;
    if (device_info(&d) == cudaSuccess) sm = d.sm_count;
    BwdPlan pl;
    if (!bwd_plan(p, sm, &pl)) return "";
    if (tc_dw_supports(p) && p.B * p.in_spatial() > 0) return "tc_dw_gemm";
    return pl.dwg ? "bwd_dw_grouped_kernel" : "bwd_dw_kernel";
}

bool backward_supported(const Problem& p) {
    BwdPlan pl;
    return bwd_plan(p, 152, &pl);
}

size_t backward_workspace_bytes(const Problem& p, bool dx, bool dw, bool db) {
    DeviceInfo d;
    int sm = 152;
    if (device_info(&d) == cudaSuccess) sm = d.sm_count;
    BwdPlan pl;
    if (!bwd_plan(p, sm, &pl)) return 0;
    size_t need = dw ? (pl.part_bytes + 255) / 256 * 256 : 0;
    if (db && p.C_out > 0) {
        int n_seg;
        int64_t seg;
        db_split(p, sm, &n_seg, &seg);
        need = std::max(need, ((size_t)p.C_out * n_seg * sizeof(float) + 255) / 256 * 256);
    }
    if (dw && p.w_elems() > 0 && tc_dw_supports(p)) need = std::max(need, tc_dw_workspace_bytes(p));
    if (dx && p.x_elems() > 0 && tc_dx_supports(p)) need = std::max(need, tc_dx_workspace_bytes(p));
    if (dx && p.x_elems() > 0 && tc32_dx_supports(p)) need = std::max(need, tc32_dx_workspace_bytes(p));
    return need;
}

size_t backward_workspace_bytes(const Problem& p) { return backward_workspace_bytes(p, true, true, true); }

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
    a.wait_ns = wait_limit_ns();
    int n = 0;
    int* cnt = launches ? launches : &n;
    switch (p.dtype) {
        case CT_F32: return launch_backward_t<float>(p, pl, a, stream, cnt);
        case CT_F16: return launch_backward_t<__half>(p, pl, a, stream, cnt);
        default: return launch_backward_t<__nv_bfloat16>(p, pl, a, stream, cnt);
    }
}

}  // namespace ct

