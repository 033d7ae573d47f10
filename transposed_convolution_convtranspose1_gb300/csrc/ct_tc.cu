// ct_tc.cu -- bf16/fp16 stride-phase implicit GEMM on tcgen05 tensor cores.
//
// Method.  Output positions are split by their residue r_a = o_a mod s_a on
// every axis (stride phases).  Within a phase every output o = r + s*q
// receives the same set of taps T_r, each reading input i = q + off(r, t), so
// the phase is a dense GEMM
//     Y_r[b, oc, q] = sum_{t in T_r, ic} W[t][oc][ic] * X[b, q + off(r,t), ic]
// over C_in x |T_r| -- the ONNX page's implicit-gather GEMM with tap-reversed
// weights (ai.onnx.ConvTranspose, variant ncdhw3d_implicit_sgmat: no column
// matrix, no scatter pass, reduction over the full in-channel-by-tap depth),
// generalised from stride 1 to every stride phase.  Two kernels run:
//   1. tc_prepare        : one launch, two kinds of blocks:
//        x [B, C, D*H*W] -> X' [B, D, H, W, C_pad]
//                          (K-major B operand; TMA boxes then shift along the
//                          spatial axes only, so every box starts on a
//                          128-byte boundary of the channel axis)
//        w [C_in, C_out, taps] -> W' [taps][N_pad][C_pad]
//                          (K-major A operand, zero padded; taps indexed in the
//                          pages' unflipped order, visited per phase in
//                          reversed order, i.e. increasing input offset)
//   2. tc_phase_gemm     : persistent, warp-specialised, one CTA per SM:
//        warp 0      TMA producer: per k-block (one tap, 64 input channels)
//                    a box of W' (128 output channels) and a 5-D box of X'
//                    (NP output positions, shifted by the tap's input
//                    offsets; rows outside the input are zero-filled by TMA)
//                    into a ring of 128-byte-swizzled stages
//        warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//                    D[oc, position] += W'[oc, k] X'[position, k], M = 128
//                    output channels, N = NP positions (256 for strides 1-2),
//                    K = 16 per instruction, fp32 accumulators in TMEM
//        warps 2..9  epilogue (two per TMEM lane quarter): tcgen05.ld of each W
//                    phase's accumulator
//                    (one lane per output channel), + bias in fp32, one RNE
//                    rounding, the W phases of a position interleaved in
//                    registers so that each lane writes runs of consecutive
//                    outputs of its channel's row with 16-byte stores.
//      Why N = positions: one thread issues every MMA and each barrier wait
//      costs it a few hundred cycles, so an MMA must carry enough work
//      (M = 128, N = 256: 128 tensor cycles) for four of them to cover a wait.
//      Accumulators are double-buffered when they fit (stride 1), so the
//      epilogue of one tile overlaps the MMAs of the next.  Every mbarrier
//      wait is bounded: on time-out the kernel records a code in
//      g_device_error, stops issuing work, drains its outstanding copies and
//      MMAs (bounded too), frees TMEM and returns.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "ct_routes.h"
#include "ct_tcgen05.cuh"
#include "ct_types.cuh"

namespace ct {

namespace {

using namespace tcg;

constexpr int kTcMaxS = 8;        // D / H stride on this route
constexpr int kTcMaxSW = 4;       // W stride on this route (W phases per tile)
constexpr int kTcMaxTaps = 8;     // taps per axis and phase on this route
constexpr int kTcMaxClasses = 32; // (D residue, H residue) classes
constexpr int kBlockM = 128;      // output channels per tile (TMEM lanes)
constexpr int kBlockK = 64;       // channels per k-block (one 128-byte row)
constexpr int kEpiWarps = 8;      // epilogue warps (two per TMEM lane quarter)
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer + MMA + epilogue warps

struct TcClass {
    int rd, rh;           // D and H residues
    int count;            // tiles of this class
    int n_qd, n_qh_blk, n_qw_blk;
    int qd_ext, qh_ext;   // q extents of this class on D and H
};

struct TcParams {
    CUtensorMap tmap_w;   // W' [taps][N_pad][C_pad] as 3-D (C_pad, N_pad, taps)
    CUtensorMap tmap_x;   // X' [B, D, H, W, C_pad] as 5-D (C_pad, W, H, D, B)
    CUtensorMap tmap_y;   // y [B, C_out, O_d, O_h, O_w] as 5-D (O_w, O_h, O_d, C_out, B)
    const void* bias;
    void* y;
    int C_out, n_kblk, n_oc_tiles;
    int O[3];
    int S[3];
    int Kdims[3];         // kD, kH, kW (for the flat tap index)
    int NP;               // output positions per tile (MMA N)
    int WC, MR;           // tile positions = MR rows of WC positions along W
    int qw_ext[kTcMaxSW]; // q extent of each W residue
    int ntap[3][kTcMaxS];
    int tap[3][kTcMaxS][kTcMaxTaps];
    int off[3][kTcMaxS][kTcMaxTaps];
    int cmul[3];          // X' coordinate of tile position q on each axis: q * cmul + tap offset
    int n_classes, total_tiles;
    int g_qd, g_qh, g_qw;   // spatial tile grid (largest over the classes)
    TcClass cls[kTcMaxClasses];
    int stages;
    uint32_t stage_bytes, a_bytes;
    uint32_t idesc;
    uint32_t tmem_cols;
    int vec_store;        // 16-byte output stores allowed (O_w % 8 == 0, y aligned)
    int tma_store;        // SW = 2: epilogue writes 32 channels x 64 outputs per tensor store
    uint32_t epi_off;     // offset of the per-warp 4 KiB staging buffers from the ring
    uint64_t wait_ns;     // limit of each bounded wait (0: give up at the first incomplete probe)
    int act;              // epilogue activation and its parameter
    float act_alpha;
};

// ---------------------------------------------------------------------------
// tile decode (identical in every role)
// ---------------------------------------------------------------------------

struct Tile {
    int cls, rd, rh, b, qd, qh0, qw0, oc0;
    bool valid;
};

// Tile order: spatial block (b, qd, qh block, qw block) outermost, then
// (D, H) stride class, then output-channel tile, so that the tiles that read
// the same rows of X' run at about the same time and find them in L2.  The
// spatial grid is the largest over the classes; a class with fewer blocks on
// an axis leaves empty slots, which every role skips alike.
__device__ __forceinline__ Tile decode_tile(const TcParams& P, int t) {
    int local = t;
    Tile T;
    const int oc_t = local % P.n_oc_tiles; local /= P.n_oc_tiles;
    T.cls = local % P.n_classes; local /= P.n_classes;
    const int qw_b = local % P.g_qw; local /= P.g_qw;
    const int qh_b = local % P.g_qh; local /= P.g_qh;
    T.qd = local % P.g_qd;
    T.b = local / P.g_qd;
    const TcClass& C = P.cls[T.cls];
    T.rd = C.rd;
    T.rh = C.rh;
    T.valid = qw_b < C.n_qw_blk && qh_b < C.n_qh_blk && T.qd < C.n_qd;
    T.qh0 = qh_b * P.MR;
    T.qw0 = qw_b * P.WC;
    T.oc0 = oc_t * kBlockM;
    return T;
}

// The persistent CTAs take the tiles round by round (round k covers tiles
// [k * grid, (k + 1) * grid)), each CTA one tile per round, rotated by one
// per round: a CTA then cycles through the stride classes instead of always
// landing on the same one when the grid is a multiple of their period.
__device__ __forceinline__ int tile_at(int k) {
    return k * (int)gridDim.x + (int)((blockIdx.x + (unsigned)k) % gridDim.x);
}

template <int SW>
__device__ __forceinline__ int phase_taps(const TcParams& P, const Tile& T, int rw) {
    return P.ntap[0][T.rd] * P.ntap[1][T.rh] * P.ntap[2][rw];
}

template <int SW>
__device__ __forceinline__ bool tile_has_work(const TcParams& P, const Tile& T) {
#pragma unroll
    for (int rw = 0; rw < SW; ++rw)
        if (phase_taps<SW>(P, T, rw) > 0) return true;
    return false;
}

// W residue processed at step k of a tile.  For SW = 2 the phase with more
// taps goes first, so that its MMAs (the longer window) overlap the previous
// tile's final epilogue; otherwise phases run in residue order.
template <int SW>
__device__ __forceinline__ int phase_of(const TcParams& P, const Tile& T, int k) {
    if constexpr (SW == 2) {
        const bool swap = phase_taps<SW>(P, T, 1) > phase_taps<SW>(P, T, 0);
        return swap ? 1 - k : k;
    }
    return k;
}

// Tile shape as a function of the W stride SW.
template <int SW>
struct TcShape {
    static constexpr int NP = SW <= 2 ? 256 : 128;     // positions per tile (MMA N)
    static constexpr int NSLOT = SW == 1 ? 2 : SW;     // accumulator slots of NP columns
    static constexpr int NPW = NP / 2;                 // positions per epilogue warp
    static constexpr int CQ = 32;                      // positions per TMEM load
    static constexpr int NCH = NPW / CQ;               // chunks per epilogue warp
};

__device__ __forceinline__ uint32_t bits16(__nv_bfloat16 v) {
    return *reinterpret_cast<const uint16_t*>(&v);
}
__device__ __forceinline__ uint32_t bits16(__half v) { return *reinterpret_cast<const uint16_t*>(&v); }

// ---------------------------------------------------------------------------
// the GEMM kernel; SW = W stride (W phases per tile)
//
// TMEM holds TcShape<SW>::NSLOT accumulator slots of NP columns.  For SW = 1
// the two slots alternate between tiles (double buffering).  For SW >= 2 slot
// rw holds W phase rw of the current tile; the MMA warp fills the slots in
// phase order and the epilogue converts phases 0..SW-2 to packed 16-bit
// outputs held in registers as soon as each is complete, releasing its slot
// while the later phases' MMAs run; the last phase is combined with them and
// stored while the next tile's first phases run.
// ---------------------------------------------------------------------------

// The epilogue's activation is a compile-time choice (ACT): the plain kernel
// carries no trace of it.
template <bool ACT>
__device__ __forceinline__ float epi_act(float v, const TcParams& P) {
    if constexpr (ACT) return act_f32(v, P.act, P.act_alpha);
    else return v;
}

template <typename T, int SW, bool ACT>
__global__ void __launch_bounds__(kThreads, 1) tc_phase_gemm(const __grid_constant__ TcParams P) {
    using Sh = TcShape<SW>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[8], empty_bar[8], sfull_bar[4], sempty_bar[4], drain_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // 1024-byte aligned stage ring (SW128 atoms need the alignment)
    const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < P.stages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 4; ++b) {
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
    // X' and W' come from the preceding prepare kernel (launched as its
    // programmatic dependent): wait for its writes before any operand load.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp walks the schedule; lane 0 issues the copies.
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0;
        bool ok = true;
        for (int k = 0; (int64_t)k * gridDim.x < P.total_tiles && ok; ++k) {
            const int t = tile_at(k);
            if (t >= P.total_tiles) continue;
            const Tile tl = decode_tile(P, t);
            if (!tl.valid) continue;
            for (int step = 0; step < SW && ok; ++step) {
                const int rw = phase_of<SW>(P, tl, step);
                const int nd_ = P.ntap[0][tl.rd], nh_ = P.ntap[1][tl.rh], nw_ = P.ntap[2][rw];
                for (int jd = 0; jd < nd_ && ok; ++jd)
                    for (int jh = 0; jh < nh_ && ok; ++jh)
                        for (int jw = 0; jw < nw_ && ok; ++jw) {
                            const int tap = (P.tap[0][tl.rd][jd] * P.Kdims[1] + P.tap[1][tl.rh][jh]) *
                                                P.Kdims[2] +
                                            P.tap[2][rw][jw];
                            const int id = tl.qd * P.cmul[0] + P.off[0][tl.rd][jd];
                            const int ih = tl.qh0 * P.cmul[1] + P.off[1][tl.rh][jh];
                            const int iw = tl.qw0 * P.cmul[2] + P.off[2][rw][jw];
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
                                    tma_load_5d(sa + P.a_bytes, &P.tmap_x, fb, kb * kBlockK, iw, ih,
                                                id, tl.b);
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
        // Lane 0 waits and issues; the other lanes wait at the final barrier.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, work_iter = 0;
            bool ok = true;
            for (int k = 0; (int64_t)k * gridDim.x < P.total_tiles && ok; ++k) {
                const int t = tile_at(k);
                if (t >= P.total_tiles) continue;
                const Tile tl = decode_tile(P, t);
                if (!tl.valid) continue;
                if (!tile_has_work<SW>(P, tl)) continue;
                for (int step = 0; step < SW && ok; ++step) {
                    const int rw = phase_of<SW>(P, tl, step);
                    const int slot = SW == 1 ? (int)(work_iter & 1) : step;
                    const uint32_t use = SW == 1 ? (work_iter >> 1) : work_iter;
                    // a slot's first use finds it free
                    if (use > 0 && !mbar_wait(smem_u32(&sempty_bar[slot]), (use & 1) ^ 1, kErrMma,
                                   &abort_flag, P.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nk = phase_taps<SW>(P, tl, rw) * P.n_kblk;
                    const uint32_t d = tmem_base + slot * Sh::NP;
                    for (int j = 0; j < nk; ++j) {
                        if (!mbar_wait(smem_u32(&full_bar[stage]), phase, kErrMma, &abort_flag, P.wait_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sa = ring + stage * P.stage_bytes;
                        const uint64_t ad = smem_desc_sw128(sa);
                        const uint64_t bd = smem_desc_sw128(sa + P.a_bytes);
#pragma unroll
                        for (int k = 0; k < kBlockK / 16; ++k) {
                            // advance along K by 16 elements = 32 bytes (encoded >> 4: 2)
                            mma_f16(d, ad + 2 * k, bd + 2 * k, P.idesc, (j > 0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&empty_bar[stage]));
                        if (++stage == P.stages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&sfull_bar[slot]));
                }
                ++work_iter;
            }
            // no MMA may be in flight when TMEM is released
            mma_commit(smem_u32(&drain_bar));
            mbar_drain(smem_u32(&drain_bar), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp e = warp - 2 reads TMEM lane quarter q = warp % 4 (output
        // channels oc0 + 32q .. +31, one per lane) and positions
        // [h * NPW, (h + 1) * NPW) of the tile, h = e / 4.
        const int q = warp & 3;
        const int base = ((warp - 2) >> 2) * Sh::NPW;
        const T* __restrict__ bias = static_cast<const T*>(P.bias);
        T* __restrict__ y = static_cast<T*>(P.y);
        uint32_t work_iter = 0;
        bool ok = true;
        for (int k = 0; (int64_t)k * gridDim.x < P.total_tiles && ok; ++k) {
            const int t = tile_at(k);
            if (t >= P.total_tiles) continue;
            const Tile Tl = decode_tile(P, t);
            if (!Tl.valid) continue;
            const TcClass& C = P.cls[Tl.cls];
            const bool work = tile_has_work<SW>(P, Tl);
            const int oc = Tl.oc0 + q * 32 + lane;
            const bool oc_ok = oc < P.C_out;
            const float bv = (bias != nullptr && oc_ok) ? to_f32(bias[oc]) : 0.f;
            const int od = Tl.rd + P.S[0] * Tl.qd;
            const bool d_ok = Tl.qd < C.qd_ext;
            const int64_t chan_base = ((int64_t)Tl.b * P.C_out + oc) * P.O[0] + od;
            const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
            // chunk c covers positions base + 32c .. +31 of one output row
            auto chunk_valid = [&](int c, int& oh, int& qwb) {
                const int p0 = base + c * Sh::CQ;
                const int qh = Tl.qh0 + p0 / P.WC;
                qwb = Tl.qw0 + (p0 % P.WC);
                oh = Tl.rh + P.S[1] * qh;
                return d_ok && qh < C.qh_ext && qwb < P.qw_ext[0];
            };

            uint32_t held[SW > 1 ? SW - 1 : 1][Sh::NPW / 2];  // packed 16-bit outputs
            // steps 0 .. SW-2 (SW >= 2): convert the step's phase, hold it, release
            // its slot (slot = step)
#pragma unroll
            for (int st = 0; st < SW - 1; ++st) {
                const int rw = phase_of<SW>(P, Tl, st);
                const bool has = work && phase_taps<SW>(P, Tl, rw) > 0;
                if (work) {
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sfull_bar[st]), work_iter & 1,
                                                           kErrEpilogue, &abort_flag, P.wait_ns));
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int c = 0; c < Sh::NCH; ++c) {
                    int oh, qwb;
                    float v[Sh::CQ];
                    if (has && chunk_valid(c, oh, qwb)) {
                        tmem_ld32(lane_addr + (uint32_t)(st * Sh::NP + base + c * Sh::CQ), v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int i = 0; i < Sh::CQ; ++i) v[i] = 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < Sh::CQ / 2; ++i)
                        held[st][c * (Sh::CQ / 2) + i] = bits16(from_f32<T>(epi_act<ACT>(v[2 * i] + bv, P))) |
                                                         (bits16(from_f32<T>(epi_act<ACT>(v[2 * i + 1] + bv, P))) << 16);
                }
                if (work) {
                    tc_fence_before();
                    mbar_arrive(smem_u32(&sempty_bar[st]));
                }
            }
            if (!ok) break;
            // last phase (all of it for SW = 1): combine and store
            {
                const int rl = phase_of<SW>(P, Tl, SW - 1);  // W residue of the last step
                const int slot = SW == 1 ? (int)(work_iter & 1) : SW - 1;
                const uint32_t use = SW == 1 ? (work_iter >> 1) : work_iter;
                const bool has = work && phase_taps<SW>(P, Tl, rl) > 0;
                if (work) {
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sfull_bar[slot]), use & 1,
                                                           kErrEpilogue, &abort_flag, P.wait_ns));
                    if (!ok) break;
                    tc_fence_after();
                }
#pragma unroll
                for (int c = 0; c < Sh::NCH; ++c) {
                    int oh, qwb;
                    if (!chunk_valid(c, oh, qwb)) continue;  // warp-uniform
                    float v[Sh::CQ];
                    if (has) {
                        tmem_ld32(lane_addr + (uint32_t)(slot * Sh::NP + base + c * Sh::CQ), v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int i = 0; i < Sh::CQ; ++i) v[i] = 0.f;
                    }
                    const int ow0 = SW * qwb;
                    if constexpr (SW == 2) {
                        if (P.tma_store) {
                            // stage 32 channels x 64 outputs (128-byte rows, 128-byte
                            // swizzle) and write them with one tensor store, which
                            // clips outputs outside y
                            const uint32_t sbuf = ring + P.epi_off + (uint32_t)(warp - 2) * 4096u;
                            if (lane == 0) bulk_wait_read_all();  // previous store left sbuf
                            __syncwarp();
#pragma unroll
                            for (int pc = 0; pc < 8; ++pc) {
                                uint32_t wv[4];
#pragma unroll
                                for (int hh = 0; hh < 4; ++hh) {
                                    const int qi = pc * 4 + hh;  // outputs 2qi (phase 0), 2qi+1
                                    const uint32_t w2 = held[0][c * (Sh::CQ / 2) + qi / 2];
                                    const uint32_t h16 = (qi & 1) ? (w2 >> 16) : (w2 & 0xFFFFu);
                                    const uint32_t v16 = bits16(from_f32<T>(epi_act<ACT>(v[qi] + bv, P)));
                                    wv[hh] = rl == 1 ? (h16 | (v16 << 16)) : (v16 | (h16 << 16));
                                }
                                const uint32_t a = sbuf + lane * 128 + ((pc ^ (lane & 7)) << 4);
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                                             "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                                             : "memory");
                            }
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                            __syncwarp();
                            if (lane == 0 && Tl.oc0 + q * 32 < P.C_out)  // starts inside y
                                tma_store_5d(&P.tmap_y, sbuf, ow0, oh, od, Tl.oc0 + q * 32, Tl.b);
                            continue;
                        }
                    }
                    if (!oc_ok) continue;
                    T* dst = y + (chan_base * P.O[1] + oh) * (int64_t)P.O[2] + ow0;
                    // outputs j = qi * SW + r of this chunk, 8 per 16-byte piece
#pragma unroll
                    for (int pc = 0; pc < SW * Sh::CQ / 8; ++pc) {
                        uint32_t wv[4];
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh) {
                            uint32_t two[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int j = pc * 8 + hh * 2 + e;
                                const int qi = j / SW, r = j % SW;
                                if (r == rl) {
                                    two[e] = bits16(from_f32<T>(epi_act<ACT>(v[qi] + bv, P)));
                                } else {
                                    // held step of residue r: 0 for SW = 2, r otherwise
                                    const int hs = SW == 2 ? 0 : (r < SW - 1 ? r : 0);
                                    const uint32_t w2 = held[hs][c * (Sh::CQ / 2) + qi / 2];
                                    two[e] = (qi & 1) ? (w2 >> 16) : (w2 & 0xFFFFu);
                                }
                            }
                            wv[hh] = two[0] | (two[1] << 16);
                        }
                        const int ow = ow0 + pc * 8;
                        if (P.vec_store && ow + 8 <= P.O[2]) {
                            *reinterpret_cast<uint4*>(dst + pc * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        } else {
                            uint16_t* d16 = reinterpret_cast<uint16_t*>(dst + pc * 8);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                if (ow + i < P.O[2]) d16[i] = (uint16_t)(wv[i >> 1] >> (16 * (i & 1)));
                        }
                    }
                }
                if (work) {
                    tc_fence_before();
                    mbar_arrive(smem_u32(&sempty_bar[slot]));
                    ++work_iter;
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // tensor stores complete before the CTA exits
        __syncwarp();
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
// layout kernels
// ---------------------------------------------------------------------------

// W'[tap][n][c] = w[c][n][tap] for n < C_out, c < C_in, else 0.  With
// j = n * taps + tap, w is a [C_in][C_out * taps] matrix; one block moves a
// 64 (c) x 64 (j) tile through shared memory, reading rows of w along j and
// writing rows of W' along c (128 bytes each), every load of a thread in
// flight before its stores.
template <typename T>
__device__ __forceinline__ void tc_weight_tile(const T* __restrict__ w, T* __restrict__ wp, int C_in,
                                               int C_out, int taps, int N_pad, int C_pad, int c0,
                                               int64_t j0) {
    __shared__ uint16_t tile[64][66];
    const uint16_t* ws = reinterpret_cast<const uint16_t*>(w);
    uint16_t* wd = reinterpret_cast<uint16_t*>(wp);
    const int64_t jn = (int64_t)C_out * taps;  // j of real output channels
    const int64_t jt = (int64_t)N_pad * taps;  // j including the padded ones
    const int t = threadIdx.x;
    uint16_t v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int c = t / 64 + 4 * i, jj = t % 64;
        const int64_t j = j0 + jj;
        v[i] = (c0 + c < C_in && j < jn) ? ws[(int64_t)(c0 + c) * jn + j] : (uint16_t)0;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) tile[t / 64 + 4 * i][t % 64] = v[i];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int c = t % 64, jj = t / 64 + 4 * i;
        const int64_t j = j0 + jj;
        if (j >= jt) continue;
        const int64_t n = j / taps, tp = j % taps;
        wd[(tp * N_pad + n) * C_pad + c0 + c] = tile[c][jj];
    }
}

// X'[b][s][c] = x[b][c][s] for c < C, 0 for C <= c < C_pad.  One block moves
// a 64 (c) x 64 (s) tile through shared memory:
// 16-byte loads along s (when S % 8 == 0 and x is 16-byte aligned; 2-byte
// loads otherwise) and 16-byte stores along c; the tile is stored with
// its 8-element column chunks XOR-swizzled by row so that both the scattered
// 2-byte writes and the 16-byte row reads avoid bank conflicts.
template <typename T>
__device__ __forceinline__ void tc_x_tile(const T* __restrict__ x, T* __restrict__ xc, int C, int C_pad,
                                          int64_t S, bool vec, int64_t s0, int c0, int64_t b) {
    __shared__ __align__(16) uint16_t tile[64][64];
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(x);
    uint16_t* xd = reinterpret_cast<uint16_t*>(xc);
    const int t = threadIdx.x;
    // load: thread -> (c = t/8 + 32*i, s chunk = t%8)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int c = t / 8 + 32 * i;
        const int sv = t % 8;
        uint16_t v[8];
        const int64_t s = s0 + sv * 8;
        if (c0 + c < C && vec && s + 8 <= S) {
            const uint4 u = *reinterpret_cast<const uint4*>(xs + (b * C + c0 + c) * S + s);
            const uint16_t* h = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = h[j];
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = (c0 + c < C && s + j < S) ? xs[(b * C + c0 + c) * S + s + j] : 0;
        }
        // element (s_local = sv*8 + j, c) -> row s_local, chunk (c/8) ^ (j ^ sv)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            tile[sv * 8 + j][(((c >> 3) ^ j ^ sv) << 3) | (c & 7)] = v[j];
    }
    __syncthreads();
    // store: thread -> (s = t/8 + 32*i, c chunk = t%8)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int sl = t / 8 + 32 * i;
        const int cv = t % 8;
        const int64_t s = s0 + sl;
        if (s >= S) continue;
        const int key = (sl & 7) ^ (sl >> 3);
        const uint4 u = *reinterpret_cast<const uint4*>(&tile[sl][(cv ^ key) << 3]);
        *reinterpret_cast<uint4*>(xd + (b * S + s) * C_pad + c0 + cv * 8) = u;
    }
}

// One launch prepares both GEMM operands: blocks [0, n_wb) move W' tiles
// (first, so that they overlap the x tiles), the remaining blocks X' tiles
// (s-tile fastest, then c-tile, then batch).
struct TcPrep {
    const void* x; void* xc; const void* w; void* wp;
    int C, C_pad, B, C_out, taps, N_pad;
    int64_t S;
    int n_st, n_ct, n_jt;  // x tiles along s and c; weight tiles along j
    int64_t n_wb;          // weight blocks (first blocks of the grid)
    bool vec;
    bool w_gather;         // W'[tap][n][c] = w[n][c][tap] (input gradient), 256 elements per block
};

template <typename T>
__global__ void __launch_bounds__(256) tc_prepare(const __grid_constant__ TcPrep Q) {
    // the GEMM that follows may begin its prologue now
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t bid = blockIdx.x;
    if (bid < Q.n_wb && Q.w_gather) {
        // input gradient: W'[tap][n][c] = w[n][c][tap] (n < C_out, c < C, else 0); w is small
        const int64_t e = bid * 256 + threadIdx.x;
        const int64_t plane = (int64_t)Q.N_pad * Q.C_pad;
        if (e < plane * Q.taps) {
            const int tp = (int)(e / plane);
            const int n = (int)((e / Q.C_pad) % Q.N_pad), c = (int)(e % Q.C_pad);
            const uint16_t* ws = static_cast<const uint16_t*>(Q.w);
            static_cast<uint16_t*>(Q.wp)[e] =
                n < Q.C_out && c < Q.C ? ws[((int64_t)n * Q.C + c) * Q.taps + tp] : (uint16_t)0;
        }
    } else if (bid < Q.n_wb) {
        const int64_t wb = bid;
        const int jt = (int)(wb % Q.n_jt), ct = (int)(wb / Q.n_jt);
        tc_weight_tile<T>(static_cast<const T*>(Q.w), static_cast<T*>(Q.wp), Q.C, Q.C_out, Q.taps,
                          Q.N_pad, Q.C_pad, ct * 64, (int64_t)jt * 64);
    } else {
        const int64_t xb = bid - Q.n_wb;
        const int64_t st = xb % Q.n_st, rest = xb / Q.n_st;
        const int ct = (int)(rest % Q.n_ct);
        const int64_t b = rest / Q.n_ct;
        tc_x_tile<T>(static_cast<const T*>(Q.x), static_cast<T*>(Q.xc), Q.C, Q.C_pad, Q.S, Q.vec,
                     st * 64, ct * 64, b);
    }
}

// ---------------------------------------------------------------------------
// the weight gradient as a GEMM (16-bit types, groups of 1)
//
// Per tap t, dw_t[ic, oc] = sum over (b, i) of x[b, ic, i] * dy[b, oc, i * s +
// t * d - pad_lo]: M = 128 input channels, N = 128 output channels, K = input
// positions, 64 per k-block (one run of an input row).  A (x) is K-major
// straight from x's layout; B (dy at the tap's positions) is MN-major, from
// dy's channels-last copy: a box of 64 output channels x 64 positions taken
// with element stride s_W (so a tap's shift lands on a non-innermost
// coordinate, as TMA requires), two boxes for the 128 channels.  A tile
// keeps kDwNT taps in TMEM so that each A block serves them all.  The k-blocks
// are split over about one wave of CTAs; each writes fp32 partials
// [split][tap][ic][oc] and tc_dw_reduce adds the splits in order.
// ---------------------------------------------------------------------------

constexpr int kDwNT = 2;          // taps per tile
constexpr int kDwThreads = 192;   // producer, MMA, four epilogue warps

struct TcDwParams {
    CUtensorMap tmap_x;   // x [B, C_in, I_D, I_H, I_W] as 5-D (I_W, I_H, I_D, C_in, B)
    CUtensorMap tmap_dy;  // dy' [B, O_D, O_H, O_W, C_pad] as 5-D (C_pad, O_W, O_H, O_D, B)
    float* part;          // [split][tap][C_in][C_out]
    int C_in, C_out, taps;
    int I[3], K[3], S[3], PL[3], DL[3];
    int n_icb, n_ocb, n_tg;   // tiles: input-channel blocks, output-channel blocks, tap groups
    int n_wblk;               // 64-position blocks per input row
    int64_t n_kb;             // k-blocks: B * I_D * I_H * n_wblk
    int n_split;
    int stages;
    uint32_t idesc;
    uint64_t wait_ns;
};

// Shared-memory matrix descriptor: MN-major, 128-byte swizzle: rows of 64
// MN elements (128 bytes) per K index, 8-row groups 1024 bytes apart along K
// (SBO), 64-element MN blocks 8192 bytes apart (LBO), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);       // start address
    d |= (uint64_t)(8192u >> 4) << 16;             // leading byte offset: next 64 MN elements
    d |= (uint64_t)(1024u >> 4) << 32;             // stride byte offset: next 8 K rows
    d |= (uint64_t)1 << 46;                        // version
    d |= (uint64_t)2 << 61;                        // SWIZZLE_128B
    return d;
}

template <typename T>
__global__ void __launch_bounds__(kDwThreads, 1) tc_dw_gemm(const __grid_constant__ TcDwParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[8], empty_bar[8], done_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ volatile int abort_flag;
    constexpr uint32_t kA = 128 * 128;        // A block: 128 channels x 64 positions x 2 bytes
    constexpr uint32_t kB = 128 * 128;        // B block of one tap: two 64 x 64 boxes
    constexpr uint32_t kStage = kA + kDwNT * kB;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int n_tiles = P.n_icb * P.n_ocb * P.n_tg;
    const int tile = (int)(blockIdx.x % n_tiles), split = (int)(blockIdx.x / n_tiles);
    const int tg = tile % P.n_tg, ocb = (tile / P.n_tg) % P.n_ocb, icb = tile / (P.n_tg * P.n_ocb);
    const int64_t kb0 = (int64_t)split * P.n_kb / P.n_split, kb1 = (int64_t)(split + 1) * P.n_kb / P.n_split;
    const int t0 = tg * kDwNT, nt = min(kDwNT, P.taps - t0);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < P.stages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&done_bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.tmap_dy)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_slot)),
                     "r"(kDwNT * 128u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;
    // dy' comes from the preceding prepare kernel (launched as its programmatic dependent)
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        bool ok = true;
        for (int64_t kb = kb0; kb < kb1 && ok; ++kb) {
            ok = issued < (uint32_t)P.stages ||
                 __all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1, kErrProducer,
                                                   &abort_flag, P.wait_ns));
            if (!ok) break;
            if (lane == 0) {
                int64_t r = kb;
                const int wb = (int)(r % P.n_wblk); r /= P.n_wblk;
                const int i1 = (int)(r % P.I[1]); r /= P.I[1];
                const int i0 = (int)(r % P.I[0]);
                const int b = (int)(r / P.I[0]);
                const uint32_t fb = smem_u32(&full_bar[stage]);
                const uint32_t sa = ring + stage * kStage;
                mbar_expect_tx(fb, kA + nt * kB);
                tma_load_5d(sa, &P.tmap_x, fb, wb * 64, i1, i0, icb * 128, b);
                for (int j = 0; j < nt; ++j) {
                    const int t = t0 + j;
                    const int td = t / (P.K[1] * P.K[2]), th = (t / P.K[2]) % P.K[1], tw = t % P.K[2];
                    const int cw = wb * 64 * P.S[2] + tw * P.DL[2] - P.PL[2];
                    const int ch = i1 * P.S[1] + th * P.DL[1] - P.PL[1];
                    const int cd = i0 * P.S[0] + td * P.DL[0] - P.PL[0];
                    for (int h = 0; h < 2; ++h)
                        tma_load_5d(sa + kA + j * kB + h * 8192u, &P.tmap_dy, fb, ocb * 128 + h * 64, cw, ch, cd,
                                    b);
                }
            }
            __syncwarp();
            ++issued;
            if (++stage == P.stages) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (!ok && lane == 0) {
            const uint32_t first = issued > (uint32_t)P.stages ? issued - P.stages : 0;
            for (uint32_t k = first; k < issued; ++k)
                mbar_drain(smem_u32(&full_bar[k % P.stages]), (k / P.stages) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t kb = kb0; kb < kb1 && ok; ++kb) {
                if (!mbar_wait(smem_u32(&full_bar[stage]), phase, kErrMma, &abort_flag, P.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = ring + stage * kStage;
                const uint64_t ad = smem_desc_sw128(sa);
                for (int j = 0; j < nt; ++j) {
                    const uint64_t bd = smem_desc_mn_sw128(sa + kA + j * kB);
#pragma unroll
                    for (int k = 0; k < 4; ++k)  // K = 16 per MMA: A +32 bytes, B +16 rows (2048 bytes)
                        mma_f16(tmem_base + j * 128, ad + 2 * k, bd + 128 * k, P.idesc,
                                (kb > kb0 || k > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&empty_bar[stage]));
                if (++stage == P.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            mma_commit(smem_u32(&done_bar));  // every MMA issued has completed when it fires
            mbar_drain(smem_u32(&done_bar), 0);  // none may be in flight when TMEM is released
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // warp w reads TMEM lane quarter q = w % 4: input channels icb*128 + 32q + lane
        const int q = warp & 3;
        const bool ok = __all_sync(0xffffffffu,
                                   mbar_wait(smem_u32(&done_bar), 0, kErrEpilogue, &abort_flag, P.wait_ns));
        if (ok) {
            tc_fence_after();
            const int ic = icb * 128 + q * 32 + lane;
            const bool any = kb1 > kb0;  // an empty k range leaves TMEM unwritten: its partial is 0
            for (int j = 0; j < nt; ++j) {
                float* dst = P.part + (((int64_t)split * P.taps + t0 + j) * P.C_in + ic) * P.C_out;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[32];
                    if (any) {
                        tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(j * 128 + c * 32), v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    }
                    const int oc0 = ocb * 128 + c * 32;
                    if (ic < P.C_in)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (oc0 + i < P.C_out) dst[oc0 + i] = v[i];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kDwNT * 128u)
                     : "memory");
    }
}

// dw[ic][oc][t] = sum over splits (in order) of part[split][t][ic][oc], one rounding.
template <typename T>
__global__ void __launch_bounds__(256) tc_dw_reduce(const float* __restrict__ part, T* __restrict__ dw, int C_in,
                                                     int C_out, int taps, int n_split) {
    const int64_t n = (int64_t)taps * C_in * C_out;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
#pragma unroll 4
        for (int k = 0; k < n_split; ++k) s += part[(int64_t)k * n + e];
        const int oc = (int)(e % C_out);
        const int64_t r = e / C_out;
        const int ic = (int)(r % C_in), t = (int)(r / C_in);
        dw[((int64_t)ic * C_out + oc) * taps + t] = from_f32<T>(s);
    }
}

// ---------------------------------------------------------------------------
// host planning
// ---------------------------------------------------------------------------

struct TcPlan {
    int C_pad, N_pad, n_oc_tiles, sw, NP, WC, MR, stages, nslot;
    size_t x_bytes, w_bytes, stage_bytes, epi_bytes;
    AxisPlan ax[3];
};

constexpr size_t kSmemLimit = 232448;  // opt-in shared memory per block (227 KiB)

bool make_plan(const Problem& p, TcPlan* pl) {
    if (p.dtype != CT_BF16 && p.dtype != CT_F16) return false;
    if (p.G != 1) return false;
    if (p.S[0] > kTcMaxS || p.S[1] > kTcMaxS || p.S[2] > kTcMaxSW) return false;
    for (int a = 0; a < 3; ++a) {
        plan_axis(p, a, &pl->ax[a]);
        for (int r = 0; r < p.S[a]; ++r)
            if (pl->ax[a].ntaps[r] > kTcMaxTaps) return false;
    }
    if (p.S[0] * p.S[1] > kTcMaxClasses) return false;
    pl->sw = p.S[2];
    pl->NP = pl->sw <= 2 ? 256 : 128;      // TcShape<SW>::NP
    pl->nslot = pl->sw == 1 ? 2 : pl->sw;  // TcShape<SW>::NSLOT
    pl->N_pad = (int)((p.C_out + kBlockM - 1) / kBlockM * kBlockM);
    pl->n_oc_tiles = pl->N_pad / kBlockM;
    pl->C_pad = (int)((p.C_in + kBlockK - 1) / kBlockK * kBlockK);
    const int64_t qw0 = pl->ax[2].q_extent[0];
    int wc = 32;  // an epilogue chunk (up to 32 positions) stays within one row
    while (wc < qw0 && wc < pl->NP) wc *= 2;
    pl->WC = wc;
    pl->MR = pl->NP / wc;
    pl->stage_bytes = (size_t)kBlockM * 128 + (size_t)pl->NP * 128;
    // SW = 2 epilogue: one 4 KiB tensor-store staging buffer per epilogue warp
    pl->epi_bytes = pl->sw == 2 ? (size_t)kEpiWarps * 4096 : 0;
    const size_t room = kSmemLimit - 1024 - 1024 - pl->epi_bytes;
    pl->stages = (int)std::min<size_t>(8, room / pl->stage_bytes);
    if (pl->stages < 2) return false;
    pl->x_bytes = (size_t)p.B * p.in_spatial() * pl->C_pad * 2;
    pl->w_bytes = (size_t)p.taps() * pl->N_pad * pl->C_pad * 2;
    // TMA limits: strides < 2^40, extents < 2^32
    if ((double)p.in_spatial() * pl->C_pad * 2 * p.B >= 1e12) return false;
    return true;
}

template <typename T, int SW, bool ACT>
cudaError_t launch_gemm_t(const TcParams& P, int grid, size_t smem, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(tc_phase_gemm<T, SW, ACT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the GEMM's CTAs may start (barrier
    // init, TMEM allocation, tensor-map prefetch) while the prepare kernel
    // finishes; they wait for its results before the first operand load.
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
    return cudaLaunchKernelEx(&cfg, tc_phase_gemm<T, SW, ACT>, P);
}

template <typename T, int SW>
cudaError_t launch_gemm(const TcParams& P, int grid, size_t smem, cudaStream_t stream) {
    return P.act != 0 ? launch_gemm_t<T, SW, true>(P, grid, smem, stream)
                      : launch_gemm_t<T, SW, false>(P, grid, smem, stream);
}

// How the GEMM reads its operands when it computes an input gradient instead
// of the forward pass: X' coordinates q * cmul + offset, X' boxes that take
// every es-th position on W and H (TMA element strides), W' gathered as
// w[n][c][tap].
struct TcOperands {
    int cmul[3];
    int es_w, es_h;
    bool w_gather;
};

template <typename T>
cudaError_t launch_tc_t(const Problem& p, const TcPlan& pl, const void* x, const void* w,
                        const void* bias, void* y, void* workspace, cudaStream_t stream,
                        Profile* prof, const TcOperands* ops = nullptr) {
    DeviceInfo dev;
    cudaError_t e = device_info(&dev);
    if (e != cudaSuccess) return e;
    char* ws = static_cast<char*>(workspace);
    T* xc = reinterpret_cast<T*>(ws);
    T* wp = reinterpret_cast<T*>(ws + round256(pl.x_bytes));

    // ---- parameters
    TcParams P;
    std::memset(&P, 0, sizeof(P));
    P.bias = bias;
    P.act = p.act;
    P.wait_ns = wait_limit_ns();
    P.act_alpha = p.act_alpha;
    P.y = y;
    P.C_out = (int)p.C_out;
    for (int a = 0; a < 3; ++a) P.cmul[a] = ops ? ops->cmul[a] : 1;
    P.n_kblk = pl.C_pad / kBlockK;
    P.n_oc_tiles = pl.n_oc_tiles;
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
    P.NP = pl.NP;
    P.WC = pl.WC;
    P.MR = pl.MR;
    for (int r = 0; r < pl.sw; ++r) P.qw_ext[r] = (int)pl.ax[2].q_extent[r];
    P.stages = pl.stages;
    P.a_bytes = kBlockM * 128;
    P.stage_bytes = (uint32_t)pl.stage_bytes;
    uint32_t cols = 32;
    while (cols < (uint32_t)(pl.nslot * pl.NP)) cols *= 2;
    P.tmem_cols = cols;
    P.idesc = (1u << 4)                                   // D = f32
              | ((p.dtype == CT_BF16 ? 1u : 0u) << 7)     // A = bf16 / f16
              | ((p.dtype == CT_BF16 ? 1u : 0u) << 10)    // B = bf16 / f16
              | ((uint32_t)(pl.NP >> 3) << 17)            // N = positions
              | ((uint32_t)(kBlockM >> 4) << 24);         // M = output channels
    P.vec_store = (p.O[2] % 8 == 0) && ((uintptr_t)y % 16 == 0);
    P.tma_store = P.vec_store && pl.epi_bytes > 0;
    P.epi_off = (uint32_t)(pl.stages * pl.stage_bytes);

    // ---- tile classes, heaviest first within each spatial block
    TcClass hc[kTcMaxClasses];
    int work[kTcMaxClasses];
    int n = 0;
    const int qw_blk = (int)((pl.ax[2].q_extent[0] + pl.WC - 1) / pl.WC);
    for (int rd = 0; rd < p.S[0]; ++rd)
        for (int rh = 0; rh < p.S[1]; ++rh) {
            const int64_t qd = pl.ax[0].q_extent[rd], qh = pl.ax[1].q_extent[rh];
            if (qd == 0 || qh == 0 || qw_blk == 0) continue;
            TcClass c{};
            c.rd = rd;
            c.rh = rh;
            c.n_qd = (int)qd;
            c.n_qh_blk = (int)((qh + pl.MR - 1) / pl.MR);
            c.n_qw_blk = qw_blk;
            c.qd_ext = (int)qd;
            c.qh_ext = (int)qh;
            const int64_t cnt = p.B * c.n_qd * (int64_t)c.n_qh_blk * c.n_qw_blk * pl.n_oc_tiles;
            if (cnt >= (1ll << 31)) return cudaErrorInvalidValue;
            c.count = (int)cnt;
            int wsum = 0;
            for (int rw = 0; rw < pl.sw; ++rw)
                wsum += pl.ax[0].ntaps[rd] * pl.ax[1].ntaps[rh] * pl.ax[2].ntaps[rw];
            work[n] = wsum;
            hc[n++] = c;
        }
    for (int i = 0; i < n; ++i)  // selection sort, descending work
        for (int j = i + 1; j < n; ++j)
            if (work[j] > work[i]) {
                std::swap(work[i], work[j]);
                std::swap(hc[i], hc[j]);
            }
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
    P.g_qd = g_qd;
    P.g_qh = g_qh;
    P.g_qw = g_qw;
    for (int i = 0; i < n; ++i) P.cls[i] = hc[i];

    // ---- tensor maps
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        p.dtype == CT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)pl.C_pad, (cuuint64_t)pl.N_pad,
                                    (cuuint64_t)p.taps()};
        const cuuint64_t strides[2] = {(cuuint64_t)pl.C_pad * 2,
                                       (cuuint64_t)pl.C_pad * 2 * pl.N_pad};
        const cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)kBlockM, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        CUresult r = enc(&P.tmap_w, dt, 3, wp, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[5] = {(cuuint64_t)pl.C_pad, (cuuint64_t)p.I[2], (cuuint64_t)p.I[1],
                                    (cuuint64_t)p.I[0], (cuuint64_t)p.B};
        const cuuint64_t row = (cuuint64_t)pl.C_pad * 2;
        const cuuint64_t strides[4] = {row, row * p.I[2], row * p.I[2] * p.I[1],
                                       row * p.I[2] * p.I[1] * p.I[0]};
        // with element strides the box spans es x the positions it loads
        const cuuint32_t esw = ops ? (cuuint32_t)ops->es_w : 1u, esh = ops ? (cuuint32_t)ops->es_h : 1u;
        const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)pl.WC * esw, (cuuint32_t)pl.MR * esh, 1, 1};
        const cuuint32_t es[5] = {1, esw, esh, 1, 1};
        CUresult r = enc(&P.tmap_x, dt, 5, xc, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }

    if (P.tma_store) {
        const cuuint64_t dims[5] = {(cuuint64_t)p.O[2], (cuuint64_t)p.O[1], (cuuint64_t)p.O[0],
                                    (cuuint64_t)p.C_out, (cuuint64_t)p.B};
        const cuuint64_t row = (cuuint64_t)p.O[2] * 2;
        const cuuint64_t strides[4] = {row, row * p.O[1], row * p.O[1] * p.O[0],
                                       row * p.O[1] * p.O[0] * p.C_out};
        const cuuint32_t box[5] = {64, 1, 1, 32, 1};
        const cuuint32_t es[5] = {1, 1, 1, 1, 1};
        CUresult r = enc(&P.tmap_y, dt, 5, y, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }

    // ---- launches
    {
        TcPrep Q;
        Q.x = x; Q.xc = xc; Q.w = w; Q.wp = wp;
        Q.C = (int)p.C_in; Q.C_pad = pl.C_pad; Q.B = (int)p.B; Q.C_out = (int)p.C_out;
        Q.taps = (int)p.taps(); Q.N_pad = pl.N_pad;
        Q.S = p.in_spatial();
        Q.n_st = (int)((Q.S + 63) / 64);
        Q.n_ct = pl.C_pad / 64;
        Q.n_jt = (int)(((int64_t)pl.N_pad * p.taps() + 63) / 64);
        Q.n_wb = (int64_t)Q.n_jt * Q.n_ct;
        Q.w_gather = ops && ops->w_gather;
        if (Q.w_gather) Q.n_wb = ((int64_t)p.taps() * pl.N_pad * pl.C_pad + 255) / 256;
        // 16-byte loads need S % 8 == 0 and a 16-byte aligned x
        Q.vec = (Q.S % 8) == 0 && ((uintptr_t)x % 16) == 0;
        const int64_t blocks = Q.n_wb + (int64_t)Q.n_st * Q.n_ct * p.B;
        if ((Q.S + 63) / 64 >= (1ll << 31) || blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
        tc_prepare<T><<<(unsigned)blocks, 256, 0, stream>>>(Q);
        prof_count(prof);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const size_t smem = (size_t)P.stages * P.stage_bytes + pl.epi_bytes + 1024;
    const int grid = std::max(1, std::min(P.total_tiles, dev.sm_count));
    prof_begin(prof, stream);
    switch (pl.sw) {
        case 1: e = launch_gemm<T, 1>(P, grid, smem, stream); break;
        case 2: e = launch_gemm<T, 2>(P, grid, smem, stream); break;
        case 3: e = launch_gemm<T, 3>(P, grid, smem, stream); break;
        default: e = launch_gemm<T, 4>(P, grid, smem, stream); break;
    }
    prof_end(prof, stream);
    prof_count(prof);
    return e;
}

// The input gradient as a GEMM on this kernel (groups of 1, 16-bit types):
//     dx[b, ic, i] = sum_{oc, t} w[ic, oc, t] * dy[b, oc, i * s + t * d - pad_lo]
// is the kernel's computation with one output phase (stride 1), the input
// gradient's channels as output channels, dy's channels as the reduction, all
// taps of every axis at X' offsets t * d - pad_lo, and the tile position q of
// an axis mapped to X' coordinate q * s: X' is the channels-last copy of dy,
// read with TMA element strides s on W and H (on D a box is one position, so
// the coordinate alone does it).  W' gathers w[ic][oc][t] into [t][ic][oc].
// Fills the GEMM's problem and plan; false when the shape is off this route.
bool make_plan_dx(const Problem& p, TcPlan* pl, Problem* pd, TcOperands* ops) {
    if (p.dtype != CT_BF16 && p.dtype != CT_F16) return false;
    if (p.G != 1) return false;
    for (int a = 0; a < 3; ++a)
        if (p.K[a] > kTcMaxTaps || p.S[a] > 8) return false;
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
    pl->sw = 1;
    pl->NP = 256;
    pl->nslot = 2;
    pl->N_pad = (int)((pd->C_out + kBlockM - 1) / kBlockM * kBlockM);
    pl->n_oc_tiles = pl->N_pad / kBlockM;
    pl->C_pad = (int)((pd->C_in + kBlockK - 1) / kBlockK * kBlockK);
    int wc = 32;  // an epilogue chunk (32 positions) stays within one row
    while (wc < p.I[2] && wc < pl->NP && wc * 2 * p.S[2] <= 256) wc *= 2;
    pl->WC = wc;
    pl->MR = pl->NP / wc;
    if (wc * p.S[2] > 256 || pl->MR * p.S[1] > 256) return false;  // TMA box extents
    pl->stage_bytes = (size_t)kBlockM * 128 + (size_t)pl->NP * 128;
    pl->epi_bytes = 0;
    pl->stages = (int)std::min<size_t>(8, (kSmemLimit - 2048) / pl->stage_bytes);
    if (pl->stages < 2) return false;
    pl->x_bytes = (size_t)p.B * p.out_spatial() * pl->C_pad * 2;
    pl->w_bytes = (size_t)p.taps() * pl->N_pad * pl->C_pad * 2;
    if ((double)p.out_spatial() * pl->C_pad * 2 * p.B >= 1e12) return false;
    return true;
}

struct DwPlan {
    int C_pad, n_icb, n_ocb, n_tg, n_wblk, n_split, stages;
    int64_t n_kb;
    size_t x_bytes, part_bytes;
};

// The weight gradient's GEMM plan (16-bit types, groups of 1, at least 16
// channels each side, W stride at most 4 so a B box spans at most 256
// positions, I_W a multiple of 8 so x's rows are 16-byte strided for TMA).
// The k-blocks are split so that the tiles x splits fill about one wave of
// one CTA per SM.
bool make_plan_dw(const Problem& p, int sm_count, DwPlan* pl) {
    if (p.dtype != CT_BF16 && p.dtype != CT_F16) return false;
    if (p.G != 1 || p.C_in < 16 || p.C_out < 16) return false;
    if (p.S[2] > 4 || p.I[2] % 8 != 0) return false;
    pl->C_pad = (int)((p.C_out + kBlockK - 1) / kBlockK * kBlockK);
    pl->n_icb = (int)((p.C_in + 127) / 128);
    pl->n_ocb = (int)((p.C_out + 127) / 128);
    pl->n_tg = (int)((p.taps() + kDwNT - 1) / kDwNT);
    pl->n_wblk = (int)((p.I[2] + 63) / 64);
    pl->n_kb = p.B * p.I[0] * p.I[1] * pl->n_wblk;
    const int64_t tiles = (int64_t)pl->n_icb * pl->n_ocb * pl->n_tg;
    const int64_t split = std::max<int64_t>(1, std::min<int64_t>(std::max<int64_t>(1, pl->n_kb),
                                                                  std::max(1, sm_count) / std::max<int64_t>(1, tiles)));
    pl->n_split = (int)split;
    if (tiles * split >= (1ll << 31)) return false;
    pl->stages = (int)std::min<size_t>(8, (kSmemLimit - 2048) / (size_t)(128 * 128 * (1 + kDwNT)));
    pl->x_bytes = (size_t)p.B * p.out_spatial() * pl->C_pad * 2;
    pl->part_bytes = (size_t)split * p.taps() * p.C_in * p.C_out * sizeof(float);
    if ((double)p.out_spatial() * pl->C_pad * 2 * p.B >= 1e12) return false;
    return true;
}

template <typename T>
cudaError_t launch_tc_dw_t(const Problem& p, const DwPlan& pl, const void* x, const void* dy, void* dw,
                           void* workspace, cudaStream_t stream) {
    char* ws = static_cast<char*>(workspace);
    T* dyc = reinterpret_cast<T*>(ws);
    float* part = reinterpret_cast<float*>(ws + round256(pl.x_bytes));
    TcDwParams P;
    std::memset(&P, 0, sizeof(P));
    P.part = part;
    P.C_in = (int)p.C_in;
    P.C_out = (int)p.C_out;
    P.taps = (int)p.taps();
    for (int a = 0; a < 3; ++a) {
        P.I[a] = (int)p.I[a];
        P.K[a] = (int)p.K[a];
        P.S[a] = p.S[a];
        P.PL[a] = p.PL[a];
        P.DL[a] = p.DL[a];
    }
    P.n_icb = pl.n_icb;
    P.n_ocb = pl.n_ocb;
    P.n_tg = pl.n_tg;
    P.n_wblk = pl.n_wblk;
    P.n_kb = pl.n_kb;
    P.n_split = pl.n_split;
    P.stages = pl.stages;
    P.wait_ns = wait_limit_ns();
    P.idesc = (1u << 4)                                   // D = f32
              | ((p.dtype == CT_BF16 ? 1u : 0u) << 7)     // A = bf16 / f16
              | ((p.dtype == CT_BF16 ? 1u : 0u) << 10)    // B = bf16 / f16
              | (1u << 16)                                // B MN-major
              | ((uint32_t)(128 >> 3) << 17)              // N = 128 output channels
              | ((uint32_t)(128 >> 4) << 24);             // M = 128 input channels
    auto enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        p.dtype == CT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    {
        const cuuint64_t dims[5] = {(cuuint64_t)p.I[2], (cuuint64_t)p.I[1], (cuuint64_t)p.I[0],
                                    (cuuint64_t)p.C_in, (cuuint64_t)p.B};
        const cuuint64_t row = (cuuint64_t)p.I[2] * 2;
        const cuuint64_t strides[4] = {row, row * p.I[1], row * p.I[1] * p.I[0],
                                       row * p.I[1] * p.I[0] * p.C_in};
        const cuuint32_t box[5] = {64, 1, 1, 128, 1};
        const cuuint32_t es[5] = {1, 1, 1, 1, 1};
        CUresult r = enc(&P.tmap_x, dt, 5, const_cast<void*>(x), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[5] = {(cuuint64_t)pl.C_pad, (cuuint64_t)p.O[2], (cuuint64_t)p.O[1],
                                    (cuuint64_t)p.O[0], (cuuint64_t)p.B};
        const cuuint64_t row = (cuuint64_t)pl.C_pad * 2;
        const cuuint64_t strides[4] = {row, row * p.O[2], row * p.O[2] * p.O[1],
                                       row * p.O[2] * p.O[1] * p.O[0]};
        const cuuint32_t box[5] = {64, (cuuint32_t)(64 * p.S[2]), 1, 1, 1};
        const cuuint32_t es[5] = {1, (cuuint32_t)p.S[2], 1, 1, 1};
        CUresult r = enc(&P.tmap_dy, dt, 5, dyc, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    cudaError_t e;
    {
        // dy -> dy' (channels-last), the same layout kernel as the forward's x
        TcPrep Q;
        std::memset(&Q, 0, sizeof(Q));
        Q.x = dy;
        Q.xc = dyc;
        Q.C = (int)p.C_out;
        Q.C_pad = pl.C_pad;
        Q.B = (int)p.B;
        Q.S = p.out_spatial();
        Q.n_st = (int)((Q.S + 63) / 64);
        Q.n_ct = pl.C_pad / 64;
        Q.n_wb = 0;
        Q.vec = (Q.S % 8) == 0 && ((uintptr_t)dy % 16) == 0;
        const int64_t blocks = (int64_t)Q.n_st * Q.n_ct * p.B;
        if ((Q.S + 63) / 64 >= (1ll << 31) || blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
        tc_prepare<T><<<(unsigned)blocks, 256, 0, stream>>>(Q);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        const size_t smem = (size_t)pl.stages * 128 * 128 * (1 + kDwNT) + 1024;
        e = cudaFuncSetAttribute(tc_dw_gemm<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(pl.n_icb * pl.n_ocb * pl.n_tg * pl.n_split));
        cfg.blockDim = dim3(kDwThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, tc_dw_gemm<T>, P);
        if (e != cudaSuccess) return e;
    }
    const int64_t n = p.taps() * p.C_in * p.C_out;
    const int rb = (int)std::min<int64_t>((n + 255) / 256, 152 * 8);
    tc_dw_reduce<T><<<rb, 256, 0, stream>>>(part, static_cast<T*>(dw), (int)p.C_in, (int)p.C_out,
                                            (int)p.taps(), pl.n_split);
    return cudaGetLastError();
}

int sm_count_or_default() {
    DeviceInfo d;
    return device_info(&d) == cudaSuccess ? d.sm_count : 152;
}

}  // namespace

bool tc_dw_supports(const Problem& p) {
    DwPlan pl;
    if (!make_plan_dw(p, sm_count_or_default(), &pl)) return false;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess) return false;
    return d.cc_major == 10 && d.cc_minor == 3;
}

size_t tc_dw_workspace_bytes(const Problem& p) {
    DwPlan pl;
    if (!make_plan_dw(p, sm_count_or_default(), &pl)) return 0;
    return round256(pl.x_bytes) + round256(pl.part_bytes);
}

cudaError_t launch_tc_dw(const Problem& p, const void* x, const void* dy, void* dw, void* workspace,
                         cudaStream_t stream) {
    DwPlan pl;
    if (!make_plan_dw(p, sm_count_or_default(), &pl) || pl.n_kb == 0) return cudaErrorInvalidValue;
    if ((uintptr_t)x % 16 != 0) return cudaErrorInvalidValue;
    if (p.dtype == CT_BF16) return launch_tc_dw_t<__nv_bfloat16>(p, pl, x, dy, dw, workspace, stream);
    return launch_tc_dw_t<__half>(p, pl, x, dy, dw, workspace, stream);
}

bool tc_dx_supports(const Problem& p) {
    TcPlan pl;
    Problem pd;
    TcOperands ops;
    if (!make_plan_dx(p, &pl, &pd, &ops)) return false;
    if (p.C_in < 16 || p.C_out < 16) return false;  // tiny channel counts: the CUDA-core kernel
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess) return false;
    return d.cc_major == 10 && d.cc_minor == 3;
}

size_t tc_dx_workspace_bytes(const Problem& p) {
    TcPlan pl;
    Problem pd;
    TcOperands ops;
    if (!make_plan_dx(p, &pl, &pd, &ops)) return 0;
    return round256(pl.x_bytes) + round256(pl.w_bytes);
}

cudaError_t launch_tc_dx(const Problem& p, const void* dy, const void* w, void* dx, void* workspace,
                         cudaStream_t stream) {
    TcPlan pl;
    Problem pd;
    TcOperands ops;
    if (!make_plan_dx(p, &pl, &pd, &ops)) return cudaErrorInvalidValue;
    if (p.dtype == CT_BF16)
        return launch_tc_t<__nv_bfloat16>(pd, pl, dy, w, nullptr, dx, workspace, stream, nullptr, &ops);
    return launch_tc_t<__half>(pd, pl, dy, w, nullptr, dx, workspace, stream, nullptr, &ops);
}

bool tc_supports(const Problem& p) {
    TcPlan pl;
    if (!make_plan(p, &pl)) return false;
    DeviceInfo d;
    if (device_info(&d) != cudaSuccess) return false;
    return d.cc_major == 10 && d.cc_minor == 3;
}

bool tc_preferred(const Problem& p) { return p.C_in >= 16 && p.C_out >= 16; }

size_t tc_workspace_bytes(const Problem& p) {
    TcPlan pl;
    if (!make_plan(p, &pl)) return 0;
    return round256(pl.x_bytes) + round256(pl.w_bytes);
}

cudaError_t launch_tc(const Problem& p, const void* x, const void* w, const void* bias, void* y,
                      void* workspace, cudaStream_t stream, Profile* prof) {
    TcPlan pl;
    if (!make_plan(p, &pl)) return cudaErrorInvalidValue;
    if (p.dtype == CT_BF16)
        return launch_tc_t<__nv_bfloat16>(p, pl, x, w, bias, y, workspace, stream, prof);
    return launch_tc_t<__half>(p, pl, x, w, bias, y, workspace, stream, prof);
}

cudaError_t tc_error_word(unsigned int* v, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_device_error, sizeof(*v));
    if (e == cudaSuccess && clear && *v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace ct
