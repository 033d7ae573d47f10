// ct_tc32.cu -- fp32 stride-phase implicit GEMM on tcgen05 tensor cores with
// error-compensated TF32 ("3xTF32").
//
// Method.  The same stride-phase decomposition as the bf16/fp16 route: within
// phase (r_d, r_h, r_w) every output o = r + s*q receives the taps T_r, each
// reading input i = q + off(r, t), so the phase is the dense GEMM
//     Y_r[b, oc, q] = sum_{t in T_r, ic} W[t][oc][ic] * X[b, q + off(r,t), ic]
// (the ONNX page's implicit-gather GEMM with tap-reversed weights,
// ai.onnx.ConvTranspose variant ncdhw3d_implicit_sgmat, per stride phase).
//
// fp32 on TF32 tensor cores.  Every fp32 operand v is split into two TF32
// values, hi = v rounded to TF32 (10 explicit mantissa bits, round to nearest
// even) and lo = (v - hi) rounded to TF32; v - hi is exact in fp32 and
// |v - hi - lo| <= 2^-22 |v|.  A product is then accumulated as
//     x*w ~= xh*wh + xh*wl + xl*wh
// with three kind::tf32 MMAs into one fp32 TMEM accumulator; each TF32 x TF32
// product is exact in fp32 and the dropped xl*wl is below 2^-22 |x w|, so a
// sum of K products carries about the same error as an fp32 FMA chain.
//
// Kernels:
//   1. tc32_prepare         : one launch, two kinds of blocks:
//        w [C_in, C_out, taps] -> W'' [2][taps][N_pad][C_pad]
//                             (plane 0 = hi, plane 1 = lo; K-major A operand)
//        x [B, C, D*H*W] -> X'' [2][B][D*H*W][C_pad]
//                             (hi, lo; K-major B operand, channels innermost so
//                             that TMA boxes shift along the spatial axes only)
//   2. tc32_phase_gemm      : persistent, warp-specialised, one CTA per SM.
//        A tile is one stride phase x 128 output channels x NP positions.
//        warp 0      TMA producer: per k-block (one tap, 16 input channels)
//                    the hi and lo boxes of W'' and of X'' into a ring of
//                    64-byte-swizzled stages (48 KiB each, four in flight)
//        warp 1      TMEM allocator and single-thread MMA issuer: 6
//                    kind::tf32 MMAs per k-block (2 K-steps of 8 x 3 terms),
//                    M = 128, N = NP.  The reduction runs in chunks of
//                    kChunkKB k-blocks (128 channels of one tap), each into a
//                    fresh accumulator; two accumulators of NP columns
//                    alternate between chunks
//        warps 2..9  epilogue: warp w reads TMEM lane quarter w % 4 (32 output
//                    channels) and half of the NP positions; it adds each
//                    chunk's partial sums into fp32 registers (round to
//                    nearest) and, after a tile's last chunk, adds the bias
//                    and writes 32 x 32 blocks (channels x positions) through
//                    shared memory so that each warp store covers 32
//                    consecutive q of one output row (outputs s_w apart).
//      Why chunks: the tensor core's fp32 accumulation loses up to about an
//      ulp of the running sum per MMA, an error that grows with the reduction
//      depth times |y| (measured: 1.6e-5 of max|y| at 2048 products, above
//      fp32 accuracy).  Restarting the accumulator every 128 channels bounds
//      the running sum it rounds, and the chunk partials are summed with
//      round-to-nearest fp32 adds in registers.
//      Every mbarrier wait is bounded: on time-out the kernel records a code
//      in its device error word, stops issuing work, drains its outstanding
//      copies and MMAs (bounded too), frees TMEM and returns.
#include <algorithm>
#include <cstring>

#include "ct_routes.h"
#include "ct_tcgen05.cuh"
#include "ct_types.cuh"

namespace ct {

namespace {

using namespace tcg;

constexpr int kMaxS = 8;          // stride per axis on this route
constexpr int kMaxTaps = 8;       // taps per axis and phase on this route
constexpr int kMaxClasses = 64;   // stride phases (r_d, r_h, r_w)
constexpr int kBlockM = 128;      // output channels per tile (TMEM lanes)
constexpr int kBlockK = 16;       // fp32 channels per k-block (one 64-byte swizzled row)
constexpr int kCAlign = 32;       // C_in padding (the layout pass moves 32-channel tiles)
constexpr int kNP = 256;          // positions per tile (MMA N)
constexpr int kChunkKB = 8;       // k-blocks per TMEM accumulation chunk (128 channels)
constexpr int kEpiWarps = 8;      // epilogue warps (two per TMEM lane quarter)
constexpr int kEpiCols = kNP / 2; // positions per epilogue warp
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kPlaneA = kBlockM * kBlockK * 4;  // one A plane of a stage (8 KiB)

struct Tc32Class {
    int rd, rh, rw;         // residues on D, H, W
    int count;              // tiles of this phase
    int n_qd, n_qh_blk, n_qw_blk;
    int qd_ext, qh_ext, qw_ext;
    int taps;               // taps of this phase (product over the axes)
};

struct Tc32Params {
    CUtensorMap tmap_w;     // W'' as 3-D (C_pad, N_pad, 2 * taps)
    CUtensorMap tmap_x;     // X'' as 5-D (C_pad, W, H, D, 2 * B)
    const float* bias;
    float* y;
    int B, C_out, n_kblk, n_oc_tiles, taps;
    int O[3];
    int S[3];
    int Kdims[3];
    int WC, MR;             // tile positions = MR rows of WC positions along W
    int ntap[3][kMaxS];
    int tap[3][kMaxS][kMaxTaps];
    int off[3][kMaxS][kMaxTaps];
    int cmul[3];            // X'' coordinate of tile position q on each axis: q * cmul + tap offset
    int nwbox;              // X'' boxes per k-block and plane along W (one row of WC positions, MR = 1)
    int wbox_step;          // W coordinate step between them
    uint32_t wbox_bytes;    // shared-memory bytes of one
    int n_classes, total_tiles;
    int n_full, total_slots;  // tiles run whole; work slots (the rest run as two halves)
    int g_qd, g_qh, g_qw;   // spatial tile grid (largest over the phases)
    Tc32Class cls[kMaxClasses];
    int stages;
    uint32_t stage_bytes;
    uint32_t idesc;         // N = kNP positions
    uint32_t idesc_half;    // N = kNP / 2 (half tiles)
    uint32_t tmem_cols;
    uint32_t epi_off;       // offset of the epilogue blocks from the ring
    uint64_t wait_ns;       // limit of each bounded wait (0: give up at the first incomplete probe)
    int act;                // epilogue activation and its parameter
    float act_alpha;
};

struct Tile {
    int cls, b, qd, qh0, qw0, oc0;
    int half;   // -1: the whole tile; 0 / 1: its first / second half of positions
    bool valid;
};

// Tile order: spatial block (b, qd, qh block, qw block) outermost, then stride
// phase, then output-channel tile, so that the tiles that read the same rows
// of X'' (every phase's taps shift the same block by a few positions) run at
// about the same time and find them in L2.  The spatial grid is the largest
// over the phases; a phase with fewer blocks on an axis leaves empty slots,
// which every role skips alike.
__device__ __forceinline__ Tile decode_tile(const Tc32Params& P, int t) {
    int local = t;
    Tile T;
    const int oc_t = local % P.n_oc_tiles; local /= P.n_oc_tiles;
    T.cls = local % P.n_classes; local /= P.n_classes;
    const int qw_b = local % P.g_qw; local /= P.g_qw;
    const int qh_b = local % P.g_qh; local /= P.g_qh;
    T.qd = local % P.g_qd;
    T.b = local / P.g_qd;
    const Tc32Class& C = P.cls[T.cls];
    T.valid = qw_b < C.n_qw_blk && qh_b < C.n_qh_blk && T.qd < C.n_qd;
    T.qh0 = qh_b * P.MR;
    T.qw0 = qw_b * P.WC;
    T.oc0 = oc_t * kBlockM;
    T.half = -1;
    return T;
}

// Work slot s: slots below n_full are whole tiles; the tiles after them (the
// last, partial round of a whole-tile schedule) run as two halves of kNP / 2
// positions each, so that the last round takes half as long.  A half tile
// shifts the tile's origin by half its rows (or half its width when it is
// one row) and uses the first kNP / 2 positions of the box loaded there.
__device__ __forceinline__ Tile decode_slot(const Tc32Params& P, int s) {
    if (s < P.n_full) return decode_tile(P, s);
    const int hs = s - P.n_full;
    Tile T = decode_tile(P, P.n_full + hs / 2);
    T.half = hs & 1;
    if (P.MR >= 2) T.qh0 += T.half * (P.MR / 2);
    else T.qw0 += T.half * (P.WC / 2);
    const Tc32Class& C = P.cls[T.cls];
    T.valid = T.valid && T.qh0 < C.qh_ext && T.qw0 < C.qw_ext;
    return T;
}

// The persistent CTAs take the tiles round by round (round k covers tiles
// [k * grid, (k + 1) * grid)), each CTA one tile per round, rotated by one
// per round: a CTA then cycles through the stride classes instead of always
// landing on the same one when the grid is a multiple of their period.
__device__ __forceinline__ int tile_at(int k) {
    return k * (int)gridDim.x + (int)((blockIdx.x + (unsigned)k) % gridDim.x);
}

// ---------------------------------------------------------------------------
// the GEMM kernel
// ---------------------------------------------------------------------------

// The epilogue's activation is a compile-time choice (ACT): the plain kernel
// carries no trace of it.
template <bool ACT>
__global__ void __launch_bounds__(kThreads, 1) tc32_phase_gemm(const __grid_constant__ Tc32Params P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[8], empty_bar[8], sfull_bar[2], sempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t planeB = (uint32_t)kNP * kBlockK * 4;  // one B plane of a stage

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < P.stages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sfull_bar[b]), 1);
            mbar_init(smem_u32(&sempty_bar[b]), kEpiWarps * 32);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_w))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_x))
                     : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_slot)),
                     "r"(P.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;
    // X'' and W'' come from the preceding prepare kernel (launched as its
    // programmatic dependent): wait for its writes before any operand load.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0;
        bool ok = true;
        for (int k = 0; (int64_t)k * gridDim.x < P.total_slots && ok; ++k) {
            const int t = tile_at(k);
            if (t >= P.total_slots) continue;
            const Tile tl = decode_slot(P, t);
            if (!tl.valid) continue;
            const Tc32Class& C = P.cls[tl.cls];
            const int nd_ = P.ntap[0][C.rd], nh_ = P.ntap[1][C.rh], nw_ = P.ntap[2][C.rw];
            for (int jd = 0; jd < nd_ && ok; ++jd)
                for (int jh = 0; jh < nh_ && ok; ++jh)
                    for (int jw = 0; jw < nw_ && ok; ++jw) {
                        const int tap =
                            (P.tap[0][C.rd][jd] * P.Kdims[1] + P.tap[1][C.rh][jh]) * P.Kdims[2] +
                            P.tap[2][C.rw][jw];
                        const int id = tl.qd * P.cmul[0] + P.off[0][C.rd][jd];
                        const int ih = tl.qh0 * P.cmul[1] + P.off[1][C.rh][jh];
                        const int iw = tl.qw0 * P.cmul[2] + P.off[2][C.rw][jw];
                        for (int kb = 0; kb < P.n_kblk; ++kb) {
                            ok = issued < (uint32_t)P.stages ||  // a fresh slot is free
                                 __all_sync(0xffffffffu,
                                            mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1,
                                                      kErrProducer, &abort_flag, P.wait_ns));
                            if (!ok) break;
                            if (lane == 0) {
                                const uint32_t fb = smem_u32(&full_bar[stage]);
                                const uint32_t sa = ring + stage * P.stage_bytes;
                                mbar_expect_tx(fb, P.stage_bytes);
                                tma_load_3d(sa, &P.tmap_w, fb, kb * kBlockK, tl.oc0, tap);
                                tma_load_3d(sa + kPlaneA, &P.tmap_w, fb, kb * kBlockK, tl.oc0,
                                            P.taps + tap);
                                for (int xb = 0; xb < P.nwbox; ++xb) {
                                    const uint32_t o = 2 * kPlaneA + xb * P.wbox_bytes;
                                    tma_load_5d(sa + o, &P.tmap_x, fb, kb * kBlockK, iw + xb * P.wbox_step,
                                                ih, id, tl.b);
                                    tma_load_5d(sa + o + planeB, &P.tmap_x, fb, kb * kBlockK,
                                                iw + xb * P.wbox_step, ih, id, P.B + tl.b);
                                }
                            }
                            __syncwarp();
                            ++issued;
                            if (++stage == P.stages) {
                                stage = 0;
                                phase ^= 1;
                            }
                        }
                    }
        }
        if (!ok && lane == 0) {
            // every copy issued so far must land before the CTA exits
            const uint32_t first = issued > (uint32_t)P.stages ? issued - P.stages : 0;
            for (uint32_t k = first; k < issued; ++k)
                mbar_drain(smem_u32(&full_bar[k % P.stages]), (k / P.stages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, chunk_iter = 0;
            bool ok = true;
            for (int k = 0; (int64_t)k * gridDim.x < P.total_slots && ok; ++k) {
                const int t = tile_at(k);
                if (t >= P.total_slots) continue;
                const Tile tl = decode_slot(P, t);
                if (!tl.valid) continue;
                const Tc32Class& C = P.cls[tl.cls];
                const int nk = C.taps * P.n_kblk;
                for (int k0 = 0; k0 < nk && ok; k0 += kChunkKB) {
                    const int slot = (int)(chunk_iter & 1);
                    const uint32_t use = chunk_iter >> 1;
                    // a slot's first use finds it free
                    if (use > 0 && !mbar_wait(smem_u32(&sempty_bar[slot]), (use & 1) ^ 1, kErrMma,
                                   &abort_flag, P.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + slot * kNP;
                    const uint32_t idesc = tl.half < 0 ? P.idesc : P.idesc_half;
                    const int k1 = min(nk, k0 + kChunkKB);
                    for (int j = k0; j < k1; ++j) {
                        if (!mbar_wait(smem_u32(&full_bar[stage]), phase, kErrMma, &abort_flag, P.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sa = ring + stage * P.stage_bytes;
                        const uint64_t ah = smem_desc_sw64(sa);
                        const uint64_t al = smem_desc_sw64(sa + kPlaneA);
                        const uint64_t bh = smem_desc_sw64(sa + 2 * kPlaneA);
                        const uint64_t bl = smem_desc_sw64(sa + 2 * kPlaneA + planeB);
#pragma unroll
                        for (int k = 0; k < kBlockK / 8; ++k) {
                            // K-step of 8 TF32 elements = 32 bytes (encoded >> 4: 2)
                            const uint64_t o = 2 * k;
                            mma_tf32(d, al + o, bh + o, idesc, (j > k0 || k > 0) ? 1u : 0u);
                            mma_tf32(d, ah + o, bl + o, idesc, 1u);
                            mma_tf32(d, ah + o, bh + o, idesc, 1u);
                        }
                        mma_commit(smem_u32(&empty_bar[stage]));
                        if (++stage == P.stages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&sfull_bar[slot]));
                    ++chunk_iter;
                }
            }
            // no MMA may be in flight when TMEM is released
            mma_commit(smem_u32(&drain_bar));
            mbar_drain(smem_u32(&drain_bar), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp w reads TMEM lane quarter q = w % 4 (output channels
        // oc0 + 32q .. +31, one per lane) and positions [h * 128, h * 128 + 128)
        // of the tile, h = (w - 2) / 4.
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        // 32 x 32 block, column index XOR-swizzled by row: conflict-free both
        // when a lane writes its row and when a lane reads a column
        float* stg = reinterpret_cast<float*>(smem_raw + (P.epi_off + (ring - smem_u32(smem_raw)))) +
                     (warp - 2) * 32 * 32;
        uint32_t chunk_iter = 0;
        bool ok = true;
        for (int k = 0; (int64_t)k * gridDim.x < P.total_slots && ok; ++k) {
            const int t = tile_at(k);
            if (t >= P.total_slots) continue;
            const Tile tl = decode_slot(P, t);
            if (!tl.valid) continue;
            const Tc32Class& C = P.cls[tl.cls];
            const int nk = C.taps * P.n_kblk;
            const int od = C.rd + P.S[0] * tl.qd;
            const bool d_ok = tl.qd < C.qd_ext;
            // a half tile has positions [0, kNP / 2) only: the h = 1 warps keep
            // the chunk handshakes and store nothing
            const bool idle = tl.half >= 0 && h == 1;
            // column group c (32 positions) of this warp lies in one output row
            auto group_valid = [&](int c, int& qh, int& qwb) {
                const int p0 = h * kEpiCols + c * 32;
                qh = tl.qh0 + p0 / P.WC;
                qwb = tl.qw0 + (p0 % P.WC);
                return d_ok && qh < C.qh_ext && qwb < C.qw_ext;
            };
            float acc[kEpiCols];
#pragma unroll
            for (int i = 0; i < kEpiCols; ++i) acc[i] = 0.f;
            for (int k0 = 0; k0 < nk; k0 += kChunkKB) {
                const int slot = (int)(chunk_iter & 1);
                const uint32_t use = chunk_iter >> 1;
                ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sfull_bar[slot]), use & 1,
                                                       kErrEpilogue, &abort_flag, P.wait_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t col0 = tmem_base + ((uint32_t)(q * 32) << 16) + slot * kNP + h * kEpiCols;
                // every column is read (columns past the output only feed
                // sums that are never stored); 16 per load keeps acc in registers
                if (!idle) {
#pragma unroll
                    for (int c = 0; c < kEpiCols / 16; ++c) {
                        float v[16];
                        tmem_ld16(col0 + c * 16, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) acc[c * 16 + i] += v[i];
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&sempty_bar[slot]));
                ++chunk_iter;
            }
            if (!ok) break;
            if (idle) continue;
            const int oc_lane = tl.oc0 + q * 32 + lane;
            const float bv = (P.bias != nullptr && oc_lane < P.C_out) ? P.bias[oc_lane] : 0.f;
            const int64_t plane = (int64_t)P.O[0] * P.O[1];
            const int n_oc = min(32, P.C_out - (tl.oc0 + q * 32));
#pragma unroll
            for (int c = 0; c < kEpiCols / 32; ++c) {
                int qh, qwb;
                if (!group_valid(c, qh, qwb)) continue;  // warp-uniform
                // lane = channel: row `lane` of the block
#pragma unroll
                for (int i = 0; i < 32; ++i) stg[lane * 32 + (i ^ lane)] = (ACT ? act_f32(acc[c * 32 + i] + bv, P.act, P.act_alpha) : acc[c * 32 + i] + bv);
                __syncwarp();
                // lane = position: column `lane`, one output row per channel
                const int oh = C.rh + P.S[1] * qh;
                const int qw = qwb + lane;
                const int64_t ow = (int64_t)C.rw + (int64_t)P.S[2] * qw;
                if (qw < C.qw_ext) {
                    float* dst = P.y +
                                 ((((int64_t)tl.b * P.C_out + tl.oc0 + q * 32) * P.O[0] + od) * P.O[1] + oh) *
                                     P.O[2] + ow;
                    const int64_t step = plane * P.O[2];
                    for (int i = 0; i < n_oc; ++i, dst += step) *dst = stg[i * 32 + (lane ^ i)];
                }
                __syncwarp();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(P.tmem_cols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// operand split and layout kernels
// ---------------------------------------------------------------------------

// v rounded to TF32 (10 explicit mantissa bits), round to nearest even; a
// value that would round up past the largest finite float is truncated
// instead, and inf / NaN pass through.
__device__ __forceinline__ float tf32_rne(float v) {
    const uint32_t u = __float_as_uint(v);
    if ((u & 0x7F800000u) == 0x7F800000u) return v;
    uint32_t r = (u + 0x0FFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
    if ((r & 0x7F800000u) == 0x7F800000u) r = u & 0xFFFFE000u;
    return __uint_as_float(r);
}

__device__ __forceinline__ void split_tf32(float v, float& hi, float& lo) {
    hi = tf32_rne(v);
    lo = tf32_rne(v - hi);
}

// W''[p][t][n][c] (p = 0 hi, 1 lo) from w[c][n][t]; zero for n >= C_out or
// c >= C_in.  With j = n * taps + t, w is a [C_in][C_out * taps] matrix; one
// block moves 32 channels x 64 consecutive j through a padded shared tile,
// reading rows of w along j and writing W'' rows along c (128 bytes), every
// load of a thread in flight before its stores.
__device__ __forceinline__ void tc32_weight_tile(const float* __restrict__ w, float* __restrict__ wp,
                                                 int C_in, int C_out, int taps, int N_pad, int C_pad,
                                                 int c0, int64_t j0) {
    __shared__ float tile[32][65];
    const int64_t jn = (int64_t)C_out * taps;  // j of real output channels
    const int64_t jt = (int64_t)N_pad * taps;  // j including the padded ones
    const int t = threadIdx.x;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = t / 64 + 4 * i, jj = t % 64;
        const int64_t j = j0 + jj;
        v[i] = (c0 + c < C_in && j < jn) ? __ldg(w + (int64_t)(c0 + c) * jn + j) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) tile[t / 64 + 4 * i][t % 64] = v[i];
    __syncthreads();
    const int64_t plane = (int64_t)taps * N_pad * C_pad;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = t % 32, jj = t / 32 + 8 * i;
        const int64_t j = j0 + jj;
        if (j >= jt) continue;
        const int64_t n = j / taps, tp = j % taps;
        float hi, lo;
        split_tf32(tile[c][jj], hi, lo);
        const int64_t o = (tp * N_pad + n) * C_pad + c0 + c;
        wp[o] = hi;
        wp[plane + o] = lo;
    }
}

// X''[p][b][s][c] (p = 0 hi, 1 lo) from x[b][c][s]; zero for C <= c < C_pad.
// One block moves 32 channels x 64 positions through a shared tile of odd
// row pitch: 16-byte loads along s (when S % 4 == 0 and x is 16-byte
// aligned), 16-byte stores of four channels along c; the column reads of
// the tile fall on distinct banks.
__device__ __forceinline__ void tc32_x_tile(const float* __restrict__ x, float* __restrict__ xc, int C,
                                            int C_pad, int64_t S, int B, bool vec, int64_t s0, int c0,
                                            int64_t b) {
    __shared__ float tile[32][65];
    const int t = threadIdx.x;
    float4 v[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int c = t / 16 + 16 * i, s4 = t % 16;
        const int64_t s = s0 + 4 * s4;
        const float* src = x + (b * C + c0 + c) * S + s;
        if (c0 + c < C && vec && s + 4 <= S) {
            v[i] = __ldg(reinterpret_cast<const float4*>(src));
        } else {
            v[i].x = (c0 + c < C && s + 0 < S) ? src[0] : 0.f;
            v[i].y = (c0 + c < C && s + 1 < S) ? src[1] : 0.f;
            v[i].z = (c0 + c < C && s + 2 < S) ? src[2] : 0.f;
            v[i].w = (c0 + c < C && s + 3 < S) ? src[3] : 0.f;
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float* d = &tile[t / 16 + 16 * i][4 * (t % 16)];
        d[0] = v[i].x; d[1] = v[i].y; d[2] = v[i].z; d[3] = v[i].w;
    }
    __syncthreads();
    const int64_t plane = (int64_t)B * S * C_pad;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int c4 = t % 8, sl = t / 8 + 32 * i;
        const int64_t s = s0 + sl;
        if (s >= S) continue;
        float4 hi, lo;
        split_tf32(tile[4 * c4 + 0][sl], hi.x, lo.x);
        split_tf32(tile[4 * c4 + 1][sl], hi.y, lo.y);
        split_tf32(tile[4 * c4 + 2][sl], hi.z, lo.z);
        split_tf32(tile[4 * c4 + 3][sl], hi.w, lo.w);
        const int64_t o = (b * S + s) * C_pad + c0 + 4 * c4;
        *reinterpret_cast<float4*>(xc + o) = hi;
        *reinterpret_cast<float4*>(xc + plane + o) = lo;
    }
}

// One launch prepares both GEMM operands: blocks [0, n_wb) move W'' tiles
// (first, so that they overlap the x tiles), the remaining blocks X'' tiles
// (s-tile fastest, then c-tile, then batch).
struct Tc32Prep {
    const float* x; float* xc; const float* w; float* wp;
    int C, C_pad, B, C_out, taps, N_pad;
    int64_t S;
    int n_st, n_ct, n_jt;  // x tiles along s and c; weight tiles along j
    int64_t n_wb;          // weight blocks (first blocks of the grid)
    bool vec;
    bool w_gather;         // W''[p][tap][n][c] from w[n][c][tap] (input gradient), 256 elements per block
};

__global__ void __launch_bounds__(256) tc32_prepare(const __grid_constant__ Tc32Prep Q) {
    // the GEMM that follows may begin its prologue now
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t bid = blockIdx.x;
    if (bid < Q.n_wb && Q.w_gather) {
        // input gradient: W''[tap][n][c] = w[n][c][tap] (n < C_out, c < C, else 0), hi and lo planes
        const int64_t e = bid * 256 + threadIdx.x;
        const int64_t plane = (int64_t)Q.taps * Q.N_pad * Q.C_pad;
        if (e < plane) {
            const int tp = (int)(e / ((int64_t)Q.N_pad * Q.C_pad));
            const int n = (int)((e / Q.C_pad) % Q.N_pad), c = (int)(e % Q.C_pad);
            const float v = n < Q.C_out && c < Q.C ? __ldg(Q.w + ((int64_t)n * Q.C + c) * Q.taps + tp) : 0.f;
            float hi, lo;
            split_tf32(v, hi, lo);
            Q.wp[e] = hi;
            Q.wp[plane + e] = lo;
        }
    } else if (bid < Q.n_wb) {
        const int64_t wb = bid;
        const int jt = (int)(wb % Q.n_jt), ct = (int)(wb / Q.n_jt);
        tc32_weight_tile(Q.w, Q.wp, Q.C, Q.C_out, Q.taps, Q.N_pad, Q.C_pad, ct * 32, (int64_t)jt * 64);
    } else {
        const int64_t xb = bid - Q.n_wb;
        const int64_t st = xb % Q.n_st, rest = xb / Q.n_st;
        const int ct = (int)(rest % Q.n_ct);
        const int64_t b = rest / Q.n_ct;
        tc32_x_tile(Q.x, Q.xc, Q.C, Q.C_pad, Q.S, Q.B, Q.vec, st * 64, ct * 32, b);
    }
}

// ---------------------------------------------------------------------------
// host planning
// ---------------------------------------------------------------------------

struct Tc32Plan {
    int C_pad, N_pad, n_oc_tiles, WC, MR, stages;
    int nwbox = 1;          // X'' boxes per row of a tile (input gradient, strided W)
    size_t x_bytes, w_bytes, stage_bytes, epi_bytes;
    AxisPlan ax[3];
};

constexpr size_t kSmemLimit = 232448;  // opt-in shared memory per block (227 KiB)

bool make_plan(const Problem& p, Tc32Plan* pl) {
    if (p.dtype != CT_F32) return false;
    if (p.G != 1) return false;
    for (int a = 0; a < 3; ++a) {
        if (p.S[a] > kMaxS) return false;
        plan_axis(p, a, &pl->ax[a]);
        for (int r = 0; r < p.S[a]; ++r)
            if (pl->ax[a].ntaps[r] > kMaxTaps) return false;
    }
    if (p.S[0] * p.S[1] * p.S[2] > kMaxClasses) return false;
    pl->N_pad = (int)((p.C_out + kBlockM - 1) / kBlockM * kBlockM);
    pl->n_oc_tiles = pl->N_pad / kBlockM;
    pl->C_pad = (int)((p.C_in + kCAlign - 1) / kCAlign * kCAlign);
    int64_t qw_max = 0;
    for (int r = 0; r < p.S[2]; ++r) qw_max = std::max(qw_max, pl->ax[2].q_extent[r]);
    int wc = 32;  // an epilogue block (32 positions) stays within one row
    while (wc < qw_max && wc < kNP) wc *= 2;
    pl->WC = wc;
    pl->MR = kNP / wc;
    pl->stage_bytes = 2 * (size_t)kPlaneA + 2 * (size_t)kNP * kBlockK * 4;
    pl->epi_bytes = (size_t)kEpiWarps * 32 * 32 * 4;
    const size_t room = kSmemLimit - 1024 - 1024 - pl->epi_bytes;
    pl->stages = (int)std::min<size_t>(8, room / pl->stage_bytes);
    if (pl->stages < 2) return false;
    pl->x_bytes = 2 * (size_t)p.B * p.in_spatial() * pl->C_pad * 4;
    pl->w_bytes = 2 * (size_t)p.taps() * pl->N_pad * pl->C_pad * 4;
    // TMA limits: strides < 2^40, extents < 2^32; tile and class counts < 2^31
    if ((double)p.in_spatial() * pl->C_pad * 4 * p.B >= 1e12) return false;
    if (2 * p.B >= (1ll << 31) || 2 * p.taps() >= (1ll << 31)) return false;
    return true;
}

// How the GEMM reads its operands when it computes an input gradient (see
// make_plan_dx): X'' coordinates q * cmul + offset, X'' boxes that take every
// es-th position on W and H (TMA element strides), W'' gathered as w[n][c][tap].
struct Tc32Operands {
    int cmul[3];
    int es_w, es_h;
    bool w_gather;
};

cudaError_t launch_tc32_impl(const Problem& p, const Tc32Plan& pl, const void* x, const void* w,
                             const void* bias, void* y, void* workspace, cudaStream_t stream,
                             Profile* prof, const Tc32Operands* ops = nullptr) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    char* ws = static_cast<char*>(workspace);
    float* xc = reinterpret_cast<float*>(ws);
    float* wp = reinterpret_cast<float*>(ws + round256(pl.x_bytes));

    Tc32Params P;
    std::memset(&P, 0, sizeof(P));
    P.bias = static_cast<const float*>(bias);
    P.y = static_cast<float*>(y);
    P.B = (int)p.B;
    P.C_out = (int)p.C_out;
    P.n_kblk = pl.C_pad / kBlockK;
    P.n_oc_tiles = pl.n_oc_tiles;
    P.taps = (int)p.taps();
    for (int a = 0; a < 3; ++a) P.cmul[a] = ops ? ops->cmul[a] : 1;
    P.nwbox = pl.nwbox;
    P.wbox_step = (pl.WC / pl.nwbox) * (ops ? ops->es_w : 1);
    P.wbox_bytes = (uint32_t)(pl.WC / pl.nwbox) * kBlockK * 4;
    for (int a = 0; a < 3; ++a) {
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
    P.WC = pl.WC;
    P.MR = pl.MR;
    P.stages = pl.stages;
    P.stage_bytes = (uint32_t)pl.stage_bytes;
    P.tmem_cols = 2 * kNP;
    P.act = p.act;
    P.wait_ns = wait_limit_ns();
    P.act_alpha = p.act_alpha;
    P.idesc = (1u << 4)                              // D = f32
              | (2u << 7)                            // A = tf32
              | (2u << 10)                           // B = tf32
              | ((uint32_t)(kNP >> 3) << 17)         // N = positions
              | ((uint32_t)(kBlockM >> 4) << 24);    // M = output channels
    P.idesc_half = (P.idesc & ~(0x3Fu << 17)) | ((uint32_t)((kNP / 2) >> 3) << 17);
    P.epi_off = (uint32_t)(pl.stages * pl.stage_bytes);

    // ---- tile classes (one per stride phase), heaviest first within each spatial block
    Tc32Class hc[kMaxClasses];
    int n = 0;
    for (int rd = 0; rd < p.S[0]; ++rd)
        for (int rh = 0; rh < p.S[1]; ++rh)
            for (int rw = 0; rw < p.S[2]; ++rw) {
                const int64_t qd = pl.ax[0].q_extent[rd], qh = pl.ax[1].q_extent[rh],
                              qw = pl.ax[2].q_extent[rw];
                if (qd == 0 || qh == 0 || qw == 0) continue;
                Tc32Class c{};
                c.rd = rd;
                c.rh = rh;
                c.rw = rw;
                c.n_qd = (int)qd;
                c.n_qh_blk = (int)((qh + pl.MR - 1) / pl.MR);
                c.n_qw_blk = (int)((qw + pl.WC - 1) / pl.WC);
                c.qd_ext = (int)qd;
                c.qh_ext = (int)qh;
                c.qw_ext = (int)qw;
                c.taps = pl.ax[0].ntaps[rd] * pl.ax[1].ntaps[rh] * pl.ax[2].ntaps[rw];
                const int64_t cnt =
                    p.B * c.n_qd * (int64_t)c.n_qh_blk * c.n_qw_blk * pl.n_oc_tiles;
                if (cnt >= (1ll << 31)) return cudaErrorInvalidValue;
                c.count = (int)cnt;
                hc[n++] = c;
            }
    std::stable_sort(hc, hc + n, [](const Tc32Class& a, const Tc32Class& b) { return a.taps > b.taps; });
    int g_qd = 1, g_qh = 1, g_qw = 1;
    for (int i = 0; i < n; ++i) {
        g_qd = std::max(g_qd, hc[i].n_qd);
        g_qh = std::max(g_qh, hc[i].n_qh_blk);
        g_qw = std::max(g_qw, hc[i].n_qw_blk);
    }
    const int64_t total = p.B * (int64_t)g_qd * g_qh * g_qw * std::max(n, 1) * pl.n_oc_tiles;
    if (total >= (1ll << 31)) return cudaErrorInvalidValue;
    P.n_classes = n;
    P.total_tiles = n > 0 ? (int)total : 0;
    {
        // tiles of a last, partial round run as halves when they then fit in
        // one round of the grid
        const int64_t G = dev.sm_count;
        const int64_t rem = P.total_tiles % G;
        const int64_t R = (rem != 0 && 2 * rem <= G) ? rem : 0;
        P.n_full = (int)(P.total_tiles - R);
        P.total_slots = (int)(P.total_tiles + R);
    }
    P.g_qd = g_qd;
    P.g_qh = g_qh;
    P.g_qw = g_qw;
    for (int i = 0; i < n; ++i) P.cls[i] = hc[i];

    // ---- tensor maps
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)pl.C_pad, (cuuint64_t)pl.N_pad,
                                    (cuuint64_t)(2 * p.taps())};
        const cuuint64_t strides[2] = {(cuuint64_t)pl.C_pad * 4,
                                       (cuuint64_t)pl.C_pad * 4 * pl.N_pad};
        const cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)kBlockM, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        CUresult r = enc(&P.tmap_w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, wp, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[5] = {(cuuint64_t)pl.C_pad, (cuuint64_t)p.I[2], (cuuint64_t)p.I[1],
                                    (cuuint64_t)p.I[0], (cuuint64_t)(2 * p.B)};
        const cuuint64_t row = (cuuint64_t)pl.C_pad * 4;
        const cuuint64_t strides[4] = {row, row * p.I[2], row * p.I[2] * p.I[1],
                                       row * p.I[2] * p.I[1] * p.I[0]};
        // with element strides the box spans es x the positions it loads
        const cuuint32_t esw = ops ? (cuuint32_t)ops->es_w : 1u, esh = ops ? (cuuint32_t)ops->es_h : 1u;
        const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)(pl.WC / pl.nwbox) * esw,
                                   (cuuint32_t)pl.MR * esh, 1, 1};
        const cuuint32_t es[5] = {1, esw, esh, 1, 1};
        CUresult r = enc(&P.tmap_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 5, xc, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }

    // ---- launches
    {
        Tc32Prep Q;
        Q.x = static_cast<const float*>(x); Q.xc = xc; Q.w = static_cast<const float*>(w); Q.wp = wp;
        Q.C = (int)p.C_in; Q.C_pad = pl.C_pad; Q.B = (int)p.B; Q.C_out = (int)p.C_out;
        Q.taps = (int)p.taps(); Q.N_pad = pl.N_pad;
        Q.S = p.in_spatial();
        Q.n_st = (int)((Q.S + 63) / 64);
        Q.n_ct = pl.C_pad / 32;
        Q.n_jt = (int)(((int64_t)pl.N_pad * p.taps() + 63) / 64);
        Q.n_wb = (int64_t)Q.n_jt * Q.n_ct;
        Q.w_gather = ops && ops->w_gather;
        if (Q.w_gather) Q.n_wb = ((int64_t)p.taps() * pl.N_pad * pl.C_pad + 255) / 256;
        Q.vec = (Q.S % 4) == 0 && ((uintptr_t)x % 16) == 0;
        const int64_t blocks = Q.n_wb + (int64_t)Q.n_st * Q.n_ct * p.B;
        if ((Q.S + 63) / 64 >= (1ll << 31) || blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
        tc32_prepare<<<(unsigned)blocks, 256, 0, stream>>>(Q);
        prof_count(prof);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const size_t smem = (size_t)P.stages * P.stage_bytes + pl.epi_bytes + 1024;
    const int grid = std::max(1, std::min(P.total_slots, dev.sm_count));
    e = cudaFuncSetAttribute(P.act != 0 ? tc32_phase_gemm<true> : tc32_phase_gemm<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_begin(prof, stream);
    {
        // Programmatic dependent launch: the GEMM's CTAs may start (barrier
        // init, TMEM allocation, tensor-map prefetch) while the prepare
        // kernel finishes; they wait for its results before the first
        // operand load.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = P.act != 0 ? cudaLaunchKernelEx(&cfg, tc32_phase_gemm<true>, P)
                       : cudaLaunchKernelEx(&cfg, tc32_phase_gemm<false>, P);
    }
    prof_end(prof, stream);
    prof_count(prof);
    return e;
}

// The input gradient as a GEMM on this kernel (fp32, groups of 1; see the
// bf16/fp16 route's make_plan_dx for the mapping): one output phase of
// stride 1, dy's channels as the reduction, all taps at X'' offsets
// t * d - pad_lo, tile position q read at X'' coordinate q * s through TMA
// element strides on W and H.
bool make_plan_dx(const Problem& p, Tc32Plan* pl, Problem* pd, Tc32Operands* ops) {
    if (p.dtype != CT_F32 || p.G != 1) return false;
    for (int a = 0; a < 3; ++a)
        if (p.K[a] > kMaxTaps || p.S[a] > kMaxS) return false;
    *pd = p;
    pd->C_in = p.C_out;
    pd->C_out = p.C_in;
    pd->Cig = (int)pd->C_in;
    pd->Cog = (int)pd->C_out;
    pd->act = 0;
    for (int a = 0; a < 3; ++a) {
        pd->I[a] = p.O[a];
        pd->O[a] = p.I[a];
        pd->S[a] = 1;
        AxisPlan& ax = pl->ax[a];
        std::memset(&ax, 0, sizeof(ax));
        ax.s = 1;
        ax.q_extent[0] = p.I[a];
        ax.ntaps[0] = (int)p.K[a];
        for (int j = 0; j < p.K[a]; ++j) {
            ax.tap[0][j] = j;
            ax.off[0][j] = j * p.DL[a] - p.PL[a];
        }
        ops->cmul[a] = p.S[a];
    }
    ops->es_w = p.S[2];
    ops->es_h = p.S[1];
    ops->w_gather = true;
    pl->N_pad = (int)((pd->C_out + kBlockM - 1) / kBlockM * kBlockM);
    pl->n_oc_tiles = pl->N_pad / kBlockM;
    pl->C_pad = (int)((pd->C_in + kCAlign - 1) / kCAlign * kCAlign);
    // a box spans at most 256 traversed positions (256 / s_W loaded); a tile
    // row of more positions takes several boxes, when it is the tile's only row
    int wbox = 32;  // an epilogue block (32 positions) stays within one row
    while (wbox < p.I[2] && wbox < kNP && wbox * 2 * p.S[2] <= 256) wbox *= 2;
    int wc = wbox;
    while (wc < p.I[2] && wc < kNP) wc *= 2;
    if (wc > wbox && wc != kNP) wc = wbox;  // several boxes only for a one-row tile
    pl->WC = wc;
    pl->MR = kNP / wc;
    pl->nwbox = wc / wbox;
    if (wbox * p.S[2] > 256 || pl->MR * p.S[1] > 256) return false;  // TMA box extents
    pl->stage_bytes = 2 * (size_t)kPlaneA + 2 * (size_t)kNP * kBlockK * 4;
    pl->epi_bytes = (size_t)kEpiWarps * 32 * 32 * 4;
    const size_t room = kSmemLimit - 1024 - 1024 - pl->epi_bytes;
    pl->stages = (int)std::min<size_t>(8, room / pl->stage_bytes);
    if (pl->stages < 2) return false;
    pl->x_bytes = 2 * (size_t)p.B * p.out_spatial() * pl->C_pad * 4;
    pl->w_bytes = 2 * (size_t)p.taps() * pl->N_pad * pl->C_pad * 4;
    if ((double)p.out_spatial() * pl->C_pad * 4 * p.B >= 1e12) return false;
    if (2 * p.B >= (1ll << 31) || 2 * p.taps() >= (1ll << 31)) return false;
    return true;
}

}  // namespace

bool tc32_dx_supports(const Problem& p) {
    Tc32Plan pl;
    Problem pd;
    Tc32Operands ops;
    if (!make_plan_dx(p, &pl, &pd, &ops)) return false;
    if (p.C_in < 32 || p.C_out < 32) return false;  // small channel counts: the CUDA-core kernel
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess) return false;
    return d.cc_major == 10 && d.cc_minor == 3;
}

size_t tc32_dx_workspace_bytes(const Problem& p) {
    Tc32Plan pl;
    Problem pd;
    Tc32Operands ops;
    if (!make_plan_dx(p, &pl, &pd, &ops)) return 0;
    return round256(pl.x_bytes) + round256(pl.w_bytes);
}

cudaError_t launch_tc32_dx(const Problem& p, const void* dy, const void* w, void* dx, void* workspace,
                           cudaStream_t stream) {
    Tc32Plan pl;
    Problem pd;
    Tc32Operands ops;
    if (!make_plan_dx(p, &pl, &pd, &ops)) return cudaErrorInvalidValue;
    return launch_tc32_impl(pd, pl, dy, w, nullptr, dx, workspace, stream, nullptr, &ops);
}

bool tc32_supports(const Problem& p) {
    Tc32Plan pl;
    if (!make_plan(p, &pl)) return false;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess) return false;
    return d.cc_major == 10 && d.cc_minor == 3;
}

bool tc32_preferred(const Problem& p) { return p.C_in >= 32 && p.C_out >= 32; }

size_t tc32_workspace_bytes(const Problem& p) {
    Tc32Plan pl;
    if (!make_plan(p, &pl)) return 0;
    return round256(pl.x_bytes) + round256(pl.w_bytes);
}

cudaError_t launch_tc32(const Problem& p, const void* x, const void* w, const void* bias, void* y,
                        void* workspace, cudaStream_t stream, Profile* prof) {
    Tc32Plan pl;
    if (!make_plan(p, &pl)) return cudaErrorInvalidValue;
    return launch_tc32_impl(p, pl, x, w, bias, y, workspace, stream, prof);
}

cudaError_t tc32_error_word(unsigned int* v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_device_error, sizeof(*v));
    if (e == cudaSuccess && clear && *v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace ct
