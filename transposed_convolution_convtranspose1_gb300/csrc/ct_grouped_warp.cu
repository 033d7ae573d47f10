// ct_grouped_warp.cu -- fp32 grouped stride-phase gather on persistent pairs
// of warps: a compute warp and a memory warp per pair.
//
// The ONNX page's grouped stride-phase variant (ai.onnx.ConvTranspose,
// Implementation variants, nchw2d_grouped_stride_phase_blocked) for groups of
// 5..8 input and output channels on 2-D/3-D fp32 outputs: a thread's outputs
// cover every output channel of their group and the group's weights sit in
// shared memory.  The arithmetic is that of the other grouped kernels: one
// fp32 FMA chain per output over the D, H and W taps in increasing input
// offset and the input channels in order, the bias added last.
//
// Work split.  An item is (b, g, od, 3 consecutive q_h, a chunk of at most 61
// consecutive q_w).  The items are cut into equal contiguous ranges, one per
// warp pair of a persistent grid (one CTA of up to 8 pairs per SM), so every
// pair runs about the same number of items and consecutive items of a pair
// share their group.  Each pair owns two buffers in shared memory.
//   - The memory warp stages each item's weights and tap table in a buffer and
//     copies the item's input rows into it with one TMA box
//     [8 channels][3 + H offset span rows][64 columns] per D tap (column
//     origin rounded down to a multiple of 4, the copy's alignment rule; rows,
//     columns, depths and channels outside x read as zero), two items ahead.
//     While the compute warp works on an item, it writes the item's output
//     rows that no tap reaches (bias only); once the compute warp has left the
//     item's sums in the buffer, it takes them into registers, refills the
//     buffer with the next item but one, and stores the sums with the bias
//     and activation added.
//   - The compute warp computes, for lane l, q_w = q0 + l and q0 + l + 32 of
//     the 3 rows for all 8 output channels: 24 accumulators, each a pair of
//     output channels updated by one packed two-lane FMA (the input value used
//     twice, the pair's two weights as they lie in shared memory); per (tap,
//     input channel) 6 four-byte input loads and 2 broadcast 16-byte weight
//     loads feed 24 packed FMAs.  The taps come from the item's table of
//     (input offset, weight offset) pairs.  It leaves the raw sums over the
//     input it has just consumed.  An item is one (H, W) phase of a cell, so
//     cells with several live phases are several items.
//   - With a W stride of 2 and one live W residue, a live output and its
//     bias-only neighbour form one 8-byte store; when moreover one H residue
//     is live and a chunk spans the row, every row of a cell is written whole
//     with such stores.
// Waits are bounded (the limit is a launch parameter): a warp whose wait gives
// up records an error in this file's device word and raises its pair's abort
// flag; the memory warp lets the copies it issued land (bounded) and both
// stop.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "ct_routes.h"
#include "ct_tcgen05.cuh"
#include "ct_types.cuh"

namespace ct {
namespace {

using tcg::smem_u32;

constexpr int kWC = 8;          // channels per group, padded (input and output)
constexpr int kWRows = 3;       // q_h rows per item
constexpr int kWBW = 64;        // staged columns per row (TMA box width)
constexpr int kWPad = 32;       // floats after each buffer: reads of lanes past the chunk
constexpr int kWMaxPairs = 8;
constexpr int kWMinPairs = 4;
constexpr int kWMaxSW = 4;
constexpr int kWMaxSA = 8;
constexpr int kWMaxTaps = 8;
constexpr unsigned kErrWarpCopy = 1u << 5;     // a compute warp's wait for its input
constexpr unsigned kErrWarpResult = 1u << 6;   // a memory warp's wait for results

struct GwParams {
    CUtensorMap tmap_x;     // x as 4-D (W, H, D, B * C_in), fp32
    const float* w;
    const float* bias;
    float* y;
    int C_in, C_out, G, Cig, Cog;
    int O[3], S[3], K[3];
    int ntap[3][kWMaxSA];
    int tap[3][kWMaxSA][kWMaxTaps];
    int off[3][kWMaxSA][kWMaxTaps];
    int qext[3][kWMaxSA];   // #q with r + s*q < O, per axis and residue
    int taps;
    int Q;                  // q_w per chunk (<= 61 - W offset span)
    int n_band, n_chunk;    // bands of 3 q_h, chunks of Q q_w
    int offmin_h, wmin;     // smallest H and W input offsets
    int n_lh, n_lw;         // H and W residues with taps
    int live_h[kWMaxSA], live_w[kWMaxSW];
    int vec2;               // W stride 2, one live W residue, even O_w, 8-byte aligned y
    int dense;              // vec2, one live H residue and one chunk per row: whole rows
                            // of (bias | value, bias | value) pairs per item
    int64_t n_items;        // cells x n_lh x n_lw
    uint32_t box_floats;    // one TMA box
    uint32_t in_floats;     // a buffer's input part: nd_box boxes + kWPad (>= an item's results)
    uint32_t buf_floats;    // a buffer: input, weights [tap][ic][oc], tap table
    uint64_t wait_ns;       // limit of each wait (0: give up at once)
    int act;                // activation after the bias (ACT instantiations only)
    float act_alpha;
};

// An item: a cell (b, g, od, 3 consecutive q_h, a chunk of q_w) and one of its
// (H, W) phases (ph = index over the live H residues x live W residues).
struct Item {
    int64_t b;
    int g, od, band, chunk, ph;
    int rd, qd, nd, qa, q0, rh, rw;
};

__device__ __forceinline__ void finish(const GwParams& P, Item& m) {
    m.rd = m.od % P.S[0];
    m.qd = m.od / P.S[0];
    m.nd = P.ntap[0][m.rd];
    m.qa = m.band * kWRows;
    m.q0 = m.chunk * P.Q;
    m.rh = P.live_h[m.ph / P.n_lw];
    m.rw = P.live_w[m.ph % P.n_lw];
}

// Item `it` in the order (b, g, od, band, chunk, ph), ph fastest.
__device__ __forceinline__ Item decode(const GwParams& P, int64_t it) {
    Item m;
    const int nph = P.n_lh * P.n_lw;
    m.ph = (int)(it % nph);
    it /= nph;
    m.chunk = (int)(it % P.n_chunk);
    it /= P.n_chunk;
    m.band = (int)(it % P.n_band);
    it /= P.n_band;
    m.od = (int)(it % P.O[0]);
    it /= P.O[0];
    m.g = (int)(it % P.G);
    m.b = it / P.G;
    finish(P, m);
    return m;
}

// The item after m, without divisions.
__device__ __forceinline__ void advance(const GwParams& P, Item& m) {
    if (++m.ph == P.n_lh * P.n_lw) {
        m.ph = 0;
        if (++m.chunk == P.n_chunk) {
            m.chunk = 0;
            if (++m.band == P.n_band) {
                m.band = 0;
                if (++m.od == P.O[0]) {
                    m.od = 0;
                    if (++m.g == P.G) {
                        m.g = 0;
                        ++m.b;
                    }
                }
            }
        }
    }
    finish(P, m);
}

// Whether the item has work: a D tap reaches its depth and a row of its band
// lies in its H residue.
__device__ __forceinline__ bool live(const GwParams& P, const Item& m) {
    return m.nd > 0 && m.qa < P.qext[1][m.rh];
}

// Bounded wait of one lane (as tcg::mbar_wait, checking the pair's abort
// flag and the clock after every probe): false when it ran past limit_ns
// (recording `code` and raising *abort) or the flag rose; a limit of 0 gives
// up at once.
__device__ __forceinline__ bool wait_lane(uint32_t bar, uint32_t parity, unsigned code, volatile int* abort,
                                          uint64_t limit_ns) {
    if (limit_ns == 0) {
        atomicOr(&g_device_error, code);
        *abort = 1;
        return false;
    }
    const uint64_t t0 = tcg::globaltimer_ns();
    for (;;) {
        if (tcg::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (tcg::globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_device_error, code);
            *abort = 1;
            return false;
        }
    }
}

// All lanes wait; false when the wait gave up (or the pair's abort flag rose).
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, unsigned code, volatile int* abort,
                                         uint64_t limit) {
    return __all_sync(0xffffffffu, wait_lane(bar, parity, code, abort, limit));
}

// v over p[0 .. n): head scalars up to a 16-byte boundary, 16-byte body, tail.
__device__ __forceinline__ void fill_span(float* p, int n, float v, int lane) {
    const int mis = (int)(((uint32_t)(uintptr_t)p >> 2) & 3u);
    const int head = min((4 - mis) & 3, n);
    const int n4 = (n - head) >> 2;
    const int t0 = head + 4 * n4;
    if (lane < head) p[lane] = v;
    float4* q = reinterpret_cast<float4*>(p + head);
    const float4 v4 = make_float4(v, v, v, v);
    if (lane < n4) q[lane] = v4;
#pragma unroll 1
    for (int k = lane + 32; k < n4; k += 32) q[k] = v4;  // rows wider than 128 floats
    if (t0 + lane < n) p[t0 + lane] = v;
}

template <bool ACT>
__device__ __forceinline__ float gw_act(float v, const GwParams& P) {
    if constexpr (ACT) return act_f32(v, P.act, P.act_alpha);
    else return v;
}

__device__ __forceinline__ float* out_base(const GwParams& P, const Item& m, int64_t plane) {
    return P.y + (m.b * P.C_out + (int64_t)m.g * P.Cog) * plane + (int64_t)m.od * P.O[1] * P.O[2];
}

// The memory warp: for each live item, in order, the item's buffer receives
// the group's weights (when another group's are there), the phase's tap table
// and the input copy; the outputs no tap reaches are written up front; each
// item's results are stored (bias and activation added) as soon as the
// compute warp has left them in the buffer, and the buffer is refilled.
template <int BR, bool ACT>
__device__ __forceinline__ void memory_warp(const GwParams& P, int64_t i0, int64_t i1, float* buf0,
                                            float* buf1, uint32_t bc0, uint32_t bc1, uint32_t bf0,
                                            uint32_t bf1, volatile int* abort, int lane) {
    const int S1 = P.S[1], S2 = P.S[2], O1 = P.O[1], O2 = P.O[2];
    const int64_t plane = (int64_t)P.O[0] * O1 * O2;
    int wg_buf[2] = {-1, -1};  // group whose weights each buffer holds
    uint32_t issued[2] = {0, 0};

    // prepares live item m in buffer x and starts its copy
    auto prepare = [&](const Item& m, int x) {
        float* bx = x ? buf1 : buf0;
        float* wsm = bx + P.in_floats;
        int2* tab = reinterpret_cast<int2*>(wsm + (size_t)P.taps * kWC * kWC);
        if (m.g != wg_buf[x]) {
            const int wn = P.taps * kWC * kWC;
            constexpr int kB = 18;  // 9 taps: every load of a lane in flight at once
            for (int e0 = lane; e0 < wn; e0 += kB * 32) {
                float v[kB];
#pragma unroll
                for (int j = 0; j < kB; ++j) {
                    const int e = e0 + j * 32;
                    const int oc = e % kWC, ic = (e / kWC) % kWC, t = e / (kWC * kWC);
                    v[j] = (e < wn && oc < P.Cog && ic < P.Cig)
                               ? __ldg(&P.w[((int64_t)(m.g * P.Cig + ic) * P.Cog + oc) * P.taps + t])
                               : 0.f;
                }
#pragma unroll
                for (int j = 0; j < kB; ++j)
                    if (e0 + j * 32 < wn) wsm[e0 + j * 32] = v[j];
            }
            wg_buf[x] = m.g;
        }
        // taps in D, H, W order as (offset in the buffer from the lane's
        // column, weight offset in float4)
        const int nh = P.ntap[1][m.rh], nw = P.ntap[2][m.rw];
        const int nt = m.nd * nh * nw;
        const int sh = m.q0 + P.wmin - ((m.q0 + P.wmin) & ~3);
        for (int t = lane; t < nt; t += 32) {
            const int jw = t % nw, jh = (t / nw) % nh, jd = t / (nw * nh);
            const int tap = (P.tap[0][m.rd][jd] * P.K[1] + P.tap[1][m.rh][jh]) * P.K[2] + P.tap[2][m.rw][jw];
            tab[t] = make_int2(jd * (int)P.box_floats + (P.off[1][m.rh][jh] - P.offmin_h) * kWBW +
                                   P.off[2][m.rw][jw] - P.wmin + sh,
                               tap * (kWC * kWC / 4));
        }
        // the stores above are released by the arrive that expects the copy
        __syncwarp();
        if (lane == 0) {
            const uint32_t bar = x ? bc1 : bc0;
            tcg::mbar_expect_tx(bar, (uint32_t)m.nd * P.box_floats * 4u);
            const int x_org = (m.q0 + P.wmin) & ~3;  // a multiple of 4 (floor for negatives too)
            const int ch0 = (int)(m.b * P.C_in) + m.g * P.Cig;
            for (int jd = 0; jd < m.nd; ++jd)
                tcg::tma_load_4d(smem_u32(bx + (size_t)jd * P.box_floats), &P.tmap_x, bar, x_org,
                                 m.qa + P.offmin_h, m.qd + P.off[0][m.rd][jd], ch0);
        }
        ++issued[x];
    };
    int64_t next = i0;  // next item to consider for preparing, and that item
    Item nm = decode(P, i0);
    auto prepare_next = [&](int x) {
        for (; next < i1; ++next, advance(P, nm))
            if (live(P, nm)) {
                prepare(nm, x);
                ++next;
                advance(P, nm);
                return;
            }
    };
    prepare_next(0);
    prepare_next(1);
    int bg = -1;
    float bv[kWC], bd[kWC];
    auto load_bias = [&](int g) {
        if (g == bg) return;
#pragma unroll
        for (int oc = 0; oc < kWC; ++oc) {
            bv[oc] = (P.bias != nullptr && oc < P.Cog) ? __ldg(&P.bias[g * P.Cog + oc]) : 0.f;
            bd[oc] = gw_act<ACT>(bv[oc], P);  // outputs no tap reaches hold act(bias)
        }
        bg = g;
    };

    // Dense geometry: every output row of the item's cell, a float2 (the two
    // outputs of a W residue pair) per lane step, a lane owning the pairs
    // j = lane and lane + 32.  Rows that no tap reaches (bias) in one pass; the
    // live rows (value, bias) in the other, from values r[i][u][oc] the lane
    // holds in registers.
    const int half = O2 >> 1;
    const int64_t plane2 = plane >> 1;  // O_w even
    auto dense_dead = [&](const Item& c) {
        float2* yb = reinterpret_cast<float2*>(out_base(P, c, plane));
        for (int i = 0; i < kWRows; ++i) {
            const int qh = c.qa + i;
            for (int rh = 0; rh < S1; ++rh) {
                const int oh = S1 * qh + rh;
                if (oh >= O1) break;
                if (c.nd > 0 && rh == P.live_h[0]) continue;
                float2* yr = yb + (int64_t)oh * (O2 >> 1);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int j = lane + 32 * u;
                    if (j >= half) continue;
#pragma unroll
                    for (int oc = 0; oc < kWC; ++oc)
                        if (oc < P.Cog) yr[oc * plane2 + j] = make_float2(bd[oc], bd[oc]);
                }
            }
        }
    };
    auto dense_live = [&](const Item& c, const float (&r)[kWRows][2][kWC], auto act) {
        float2* yb = reinterpret_cast<float2*>(out_base(P, c, plane));
        const int lw = P.live_w[0];
#pragma unroll
        for (int i = 0; i < kWRows; ++i) {
            const int oh = S1 * (c.qa + i) + P.live_h[0];
            if (oh >= O1) break;
            float2* yr = yb + (int64_t)oh * (O2 >> 1);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int j = lane + 32 * u;
                if (j >= half) continue;
#pragma unroll
                for (int oc = 0; oc < kWC; ++oc) {
                    if (oc >= P.Cog) continue;
                    const float v = act(r[i][u][oc] + bv[oc]);
                    yr[oc * plane2 + j] = lw == 0 ? make_float2(v, bd[oc]) : make_float2(bd[oc], v);
                }
            }
        }
    };

    // per item: the outputs of its cell that no tap reaches (at the cell's first
    // item, while the compute warp works on this item), then its results and
    // the buffer's next item
    int k = 0;  // live items seen
    Item m = decode(P, i0);
    for (int64_t it = i0; it < i1; ++it, advance(P, m)) {
        if (P.dense) {
            load_bias(m.g);
            dense_dead(m);
            if (!live(P, m)) continue;
            const int x = k & 1;
            if (!wait_all(x ? bf1 : bf0, (uint32_t)(k >> 1) & 1u, kErrWarpResult, abort, P.wait_ns)) {
                for (int y = 0; y < 2; ++y)
                    if (issued[y] > 0) tcg::mbar_drain(y ? bc1 : bc0, (issued[y] - 1) & 1u);
                return;
            }
            const float* res = x ? buf1 : buf0;  // [i][oc][64]
            // the results into registers, the buffer refilled at once, then the stores
            float r[kWRows][2][kWC];
#pragma unroll
            for (int i = 0; i < kWRows; ++i)
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int oc = 0; oc < kWC; ++oc) r[i][u][oc] = res[(i * kWC + oc) * kWBW + lane + 32 * u];
            __syncwarp();
            if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            prepare_next(x);
            if constexpr (ACT) {
                // one dispatch on the activation, then its code at every store
                switch (P.act) {
                    case 1: dense_live(m, r, [&](float v) { return act_fixed<1>(v, P.act_alpha); }); break;
                    case 2: dense_live(m, r, [&](float v) { return act_fixed<2>(v, P.act_alpha); }); break;
                    case 3: dense_live(m, r, [&](float v) { return act_fixed<3>(v, P.act_alpha); }); break;
                    case 4: dense_live(m, r, [&](float v) { return act_fixed<4>(v, P.act_alpha); }); break;
                    case 5: dense_live(m, r, [&](float v) { return act_fixed<5>(v, P.act_alpha); }); break;
                    case 6: dense_live(m, r, [&](float v) { return act_fixed<6>(v, P.act_alpha); }); break;
                    default: dense_live(m, r, [](float v) { return v; }); break;
                }
            } else {
                dense_live(m, r, [](float v) { return v; });
            }
            ++k;
            continue;
        }
        if (m.ph == 0) {  // each cell once, by the pair that owns its first item
            load_bias(m.g);
            float* yb = out_base(P, m, plane);
            const int c0 = S2 * m.q0, c1 = min(S2 * (m.q0 + P.Q), O2);
            for (int i = 0; i < kWRows; ++i) {
                const int qh = m.qa + i;
                for (int rh = 0; rh < S1; ++rh) {
                    const int oh = S1 * qh + rh;
                    if (oh >= O1) continue;
                    if (m.nd == 0 || P.ntap[1][rh] == 0) {
#pragma unroll
                        for (int oc = 0; oc < kWC; ++oc)
                            if (oc < P.Cog) fill_span(yb + oc * plane + (int64_t)oh * O2 + c0, c1 - c0, bd[oc], lane);
                    } else if (!P.vec2) {
                        // W residues without taps in a live row
                        for (int rw = 0; rw < S2; ++rw) {
                            if (P.ntap[2][rw] > 0) continue;
                            for (int u = 0; u < 2; ++u) {
                                const int q = m.q0 + lane + 32 * u;
                                if (lane + 32 * u >= P.Q || q >= P.qext[2][rw]) continue;
#pragma unroll
                                for (int oc = 0; oc < kWC; ++oc)
                                    if (oc < P.Cog) yb[oc * plane + (int64_t)oh * O2 + S2 * q + rw] = bd[oc];
                            }
                        }
                    }
                }
            }
        }
        if (!live(P, m)) continue;
        const int x = k & 1;
        const float* res = x ? buf1 : buf0;  // [i][oc][64]
        if (!wait_all(x ? bf1 : bf0, (uint32_t)(k >> 1) & 1u, kErrWarpResult, abort, P.wait_ns)) {
            // gave up (or the compute warp did): let the copies issued land, stop
            for (int y = 0; y < 2; ++y)
                if (issued[y] > 0) tcg::mbar_drain(y ? bc1 : bc0, (issued[y] - 1) & 1u);
            return;
        }
        load_bias(m.g);
        float* yb = out_base(P, m, plane);
#pragma unroll
        for (int i = 0; i < kWRows; ++i) {
            const int qh = m.qa + i;
            if (qh >= P.qext[1][m.rh]) break;
            float* yr = yb + (int64_t)(S1 * qh + m.rh) * O2;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int q = m.q0 + lane + 32 * u;
                if (lane + 32 * u >= P.Q || q >= P.qext[2][m.rw]) continue;
                float* yq = yr + S2 * q;
#pragma unroll
                for (int oc = 0; oc < kWC; ++oc) {
                    if (oc >= P.Cog) continue;
                    const float v = gw_act<ACT>(res[(i * kWC + oc) * kWBW + lane + 32 * u] + bv[oc], P);
                    float* yo = yq + oc * plane;
                    if (P.vec2)
                        *reinterpret_cast<float2*>(yo) = m.rw == 0 ? make_float2(v, bd[oc]) : make_float2(bd[oc], v);
                    else
                        yo[m.rw] = v;
                }
            }
        }
        __syncwarp();
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        prepare_next(x);
        ++k;
    }
}

// The compute warp: for each live item, in order, waits for its buffer, runs
// the tap table over the staged input and weights, and leaves the raw sums
// [i][oc][64] over the input it has consumed.
template <int BR>
__device__ __forceinline__ void compute_warp(const GwParams& P, int64_t i0, int64_t i1, float* buf0,
                                             float* buf1, uint32_t bc0, uint32_t bc1, uint32_t bf0,
                                             uint32_t bf1, volatile int* abort, int lane) {
    int k = 0;  // live items seen
    Item m = decode(P, i0);
    for (int64_t it = i0; it < i1; ++it, advance(P, m)) {
        if (!live(P, m)) continue;
        const int x = k & 1;
        float* bx = x ? buf1 : buf0;
        const float4* wsm4 = reinterpret_cast<const float4*>(bx + P.in_floats);
        const int2* tab = reinterpret_cast<const int2*>(bx + P.in_floats + (size_t)P.taps * kWC * kWC);
        const int nt = m.nd * P.ntap[1][m.rh] * P.ntap[2][m.rw];
        if (!wait_all(x ? bc1 : bc0, (uint32_t)(k >> 1) & 1u, kErrWarpCopy, abort, P.wait_ns)) return;
        // acc[i][u][c]: row i, position q0 + lane + 32u, output channels 2c, 2c + 1
        float2 acc[kWRows][2][kWC / 2];
#pragma unroll
        for (int i = 0; i < kWRows; ++i)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int c = 0; c < kWC / 2; ++c) acc[i][u][c] = make_float2(0.f, 0.f);
        const float* xb = bx + lane;
        for (int t = 0; t < nt; ++t) {
            const int2 e = tab[t];
            const float* xp = xb + e.x;
            const float4* wp = wsm4 + e.y;
#pragma unroll
            for (int ic = 0; ic < kWC; ++ic) {
                float xv[kWRows][2];
#pragma unroll
                for (int i = 0; i < kWRows; ++i) {
                    xv[i][0] = xp[(ic * BR + i) * kWBW];
                    xv[i][1] = xp[(ic * BR + i) * kWBW + 32];
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 wq = wp[ic * 2 + h];  // output channels 4h .. 4h + 3
                    const float2 wa = make_float2(wq.x, wq.y), wb = make_float2(wq.z, wq.w);
#pragma unroll
                    for (int i = 0; i < kWRows; ++i)
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const float2 xd = make_float2(xv[i][u], xv[i][u]);
                            acc[i][u][2 * h] = __ffma2_rn(xd, wa, acc[i][u][2 * h]);
                            acc[i][u][2 * h + 1] = __ffma2_rn(xd, wb, acc[i][u][2 * h + 1]);
                        }
                }
            }
        }
        // over the consumed input, for the memory warp
        __syncwarp();
#pragma unroll
        for (int i = 0; i < kWRows; ++i)
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int c = 0; c < kWC / 2; ++c) {
                    bx[(i * kWC + 2 * c) * kWBW + lane + 32 * u] = acc[i][u][c].x;
                    bx[(i * kWC + 2 * c + 1) * kWBW + lane + 32 * u] = acc[i][u][c].y;
                }
        __syncwarp();
        if (lane == 0) tcg::mbar_arrive(x ? bf1 : bf0);
        ++k;
    }
}

template <int BR, bool ACT>
__global__ void __launch_bounds__(2 * kWMaxPairs * 32, 1) grouped_warp_kernel(const __grid_constant__ GwParams P) {
    extern __shared__ __align__(128) float smw[];
    __shared__ __align__(8) uint64_t bar_copy[kWMaxPairs][2];
    __shared__ __align__(8) uint64_t bar_full[kWMaxPairs][2];
    __shared__ int abort_pair[kWMaxPairs];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int npairs = blockDim.x >> 6;
    const bool mem = warp >= npairs;
    const int pr = mem ? warp - npairs : warp;
    if (threadIdx.x == 0) {
        for (int j = 0; j < npairs; ++j) {
            tcg::mbar_init(smem_u32(&bar_copy[j][0]), 1);
            tcg::mbar_init(smem_u32(&bar_copy[j][1]), 1);
            tcg::mbar_init(smem_u32(&bar_full[j][0]), 1);
            tcg::mbar_init(smem_u32(&bar_full[j][1]), 1);
            abort_pair[j] = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();  // the only block-wide barrier: pairs are independent below

    const int64_t gp = (int64_t)blockIdx.x * npairs + pr;
    const int64_t NP = (int64_t)gridDim.x * npairs;
    const int64_t i0 = gp * P.n_items / NP, i1 = (gp + 1) * P.n_items / NP;
    if (i0 >= i1) return;

    // the pair's two buffers: input (later the results), weights, tap table
    const uint32_t s_raw = smem_u32(smw);
    float* base = smw + (((s_raw + 127u) & ~127u) - s_raw) / 4;
    float* buf0 = base + (size_t)pr * 2 * P.buf_floats;
    float* buf1 = buf0 + P.buf_floats;
    const uint32_t bc0 = smem_u32(&bar_copy[pr][0]), bc1 = smem_u32(&bar_copy[pr][1]);
    const uint32_t bf0 = smem_u32(&bar_full[pr][0]), bf1 = smem_u32(&bar_full[pr][1]);
    volatile int* abort = &abort_pair[pr];
    if (mem)
        memory_warp<BR, ACT>(P, i0, i1, buf0, buf1, bc0, bc1, bf0, bf1, abort, lane);
    else
        compute_warp<BR>(P, i0, i1, buf0, buf1, bc0, bc1, bf0, bf1, abort, lane);
}

struct GwPlan {
    AxisPlan ax[3];
    int offmin_h, wmin, span_h, span_w, nd_box, Q, pairs;
    size_t in_floats, buf_floats, pair_bytes, smem;
};

bool make_gw_plan(const Problem& p, GwPlan* pl) {
    if (p.dtype != CT_F32) return false;
    if (p.Cig < 5 || p.Cig > kWC || p.Cog < 5 || p.Cog > kWC) return false;
    if (p.S[2] > kWMaxSW || p.S[0] > kWMaxSA || p.S[1] > kWMaxSA) return false;
    if (p.I[2] % 4 != 0) return false;  // 16-byte row pitch for the tensor map
    if (p.B * p.C_in >= (1ll << 31) || p.I[0] * p.I[1] * p.I[2] >= (1ll << 31)) return false;
    if (p.O[0] * (int64_t)p.O[1] * p.O[2] >= (1ll << 31)) return false;
    for (int a = 0; a < 3; ++a) {
        plan_axis(p, a, &pl->ax[a]);
        for (int r = 0; r < p.S[a]; ++r)
            if (pl->ax[a].ntaps[r] > kWMaxTaps) return false;
    }
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
    pl->span_h = hmax - hmin;
    pl->span_w = wmax - wmin;
    if (pl->span_h > 3) return false;   // boxes of 3..6 rows (BR instantiations)
    if (pl->span_w > 29) return false;  // chunks of at least 32 positions
    // valid lanes read staged columns q - q0 + (off - wmin) + sh <= Q - 1 + span_w + 3 < 64
    pl->Q = 61 - pl->span_w;
    pl->offmin_h = hmin;
    pl->wmin = wmin;
    pl->nd_box = std::max(ndmax, 1);
    const int BR = kWRows + pl->span_h;
    const size_t buf_floats = (size_t)pl->nd_box * kWC * BR * kWBW + kWPad;
    // + the tap table (an int2 per tap), rounded to 128 bytes
    // two buffers, each: the input (later an item's results, [3][8][64]), the
    // weights [tap][ic][oc] and the tap table (an int2 per tap), each part a
    // multiple of 128 bytes
    pl->in_floats = buf_floats;
    pl->buf_floats = buf_floats + (size_t)p.taps() * kWC * kWC + ((size_t)p.taps() * 2 + 31) / 32 * 32;
    const size_t pair_floats = 2 * pl->buf_floats;
    pl->pair_bytes = pair_floats * sizeof(float);
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return false;
    const size_t budget = di.smem_optin > 2048 ? di.smem_optin - 2048 : 0;  // static barriers, slack
    pl->pairs = (int)std::min<size_t>(kWMaxPairs, budget / pl->pair_bytes);
    if (pl->pairs < kWMinPairs) return false;
    pl->smem = (size_t)pl->pairs * pl->pair_bytes + 128;  // + alignment slack
    return true;
}

template <int BR, bool ACT>
cudaError_t launch_br(const GwParams& P, int ctas, int pairs, size_t smem, int dev, cudaStream_t stream) {
    auto kern = grouped_warp_kernel<BR, ACT>;
    // the dynamic shared memory limit is raised once per device (to the most any
    // problem asks for: it only allows, never reserves)
    static std::mutex mu;
    static size_t raised[64] = {};
    {
        std::lock_guard<std::mutex> lock(mu);
        size_t& r = raised[dev >= 0 && dev < 64 ? dev : 0];
        if (dev < 0 || dev >= 64 || r < smem) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            r = smem;
        }
    }
    kern<<<ctas, pairs * 64, smem, stream>>>(P);
    return cudaGetLastError();
}

template <bool ACT>
cudaError_t launch_act(int BR, const GwParams& P, int ctas, int pairs, size_t smem, int dev,
                       cudaStream_t s) {
    switch (BR) {
        case 3: return launch_br<3, ACT>(P, ctas, pairs, smem, dev, s);
        case 4: return launch_br<4, ACT>(P, ctas, pairs, smem, dev, s);
        case 5: return launch_br<5, ACT>(P, ctas, pairs, smem, dev, s);
        default: return launch_br<6, ACT>(P, ctas, pairs, smem, dev, s);
    }
}

}  // namespace

bool grouped_warp_supports(const Problem& p, const void* x) {
    GwPlan pl;
    return ((uintptr_t)x % 16) == 0 && tcg::encode_fn() != nullptr && make_gw_plan(p, &pl);
}

cudaError_t launch_grouped_warp(const Problem& p, const void* x, const void* w, const void* bias,
                                void* y, cudaStream_t stream) {
    GwPlan pl;
    if (!make_gw_plan(p, &pl) || ((uintptr_t)x % 16) != 0) return cudaErrorInvalidValue;
    auto enc = tcg::encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int BR = kWRows + pl.span_h;
    GwParams P;
    std::memset(&P, 0, sizeof(P));
    {
        const cuuint64_t dims[4] = {(cuuint64_t)p.I[2], (cuuint64_t)p.I[1], (cuuint64_t)p.I[0],
                                    (cuuint64_t)(p.B * p.C_in)};
        const cuuint64_t row = (cuuint64_t)p.I[2] * 4;
        const cuuint64_t strides[3] = {row, row * p.I[1], row * p.I[1] * p.I[0]};
        const cuuint32_t box[4] = {(cuuint32_t)kWBW, (cuuint32_t)BR, 1, (cuuint32_t)kWC};
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
    P.Q = pl.Q;
    P.n_band = (int)((pl.ax[1].q_extent[0] + kWRows - 1) / kWRows);
    P.n_chunk = (int)((pl.ax[2].q_extent[0] + pl.Q - 1) / pl.Q);
    P.offmin_h = pl.offmin_h;
    P.wmin = pl.wmin;
    const bool y2 = (p.O[2] % 2) == 0 && ((uintptr_t)y % 8) == 0;
    P.n_lh = P.n_lw = 0;
    for (int r = 0; r < p.S[1]; ++r)
        if (pl.ax[1].ntaps[r] > 0) P.live_h[P.n_lh++] = r;
    for (int r = 0; r < p.S[2]; ++r)
        if (pl.ax[2].ntaps[r] > 0) P.live_w[P.n_lw++] = r;
    P.vec2 = y2 && p.S[2] == 2 && P.n_lw == 1;
    P.dense = P.vec2 && P.n_lh == 1 && P.n_chunk == 1;
    P.n_items = p.B * (int64_t)p.G * p.O[0] * P.n_band * P.n_chunk * P.n_lh * P.n_lw;
    P.box_floats = (uint32_t)(kWC * BR * kWBW);
    P.in_floats = (uint32_t)pl.in_floats;
    P.buf_floats = (uint32_t)pl.buf_floats;
    P.wait_ns = wait_limit_ns();
    P.act = p.act;
    P.act_alpha = p.act_alpha;
    if (P.n_items == 0) return cudaSuccess;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int64_t need = (P.n_items + pl.pairs - 1) / pl.pairs;
    const int ctas = (int)std::min<int64_t>(di.sm_count, need);
    if (p.act != 0) return launch_act<true>(BR, P, ctas, pl.pairs, pl.smem, di.device, stream);
    return launch_act<false>(BR, P, ctas, pl.pairs, pl.smem, di.device, stream);
}

cudaError_t grouped_warp_error_word(unsigned int* v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_device_error, sizeof(*v));
    if (e == cudaSuccess && clear && *v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace ct
