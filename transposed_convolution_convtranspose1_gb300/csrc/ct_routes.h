// ct_routes.h -- the specialised routes: which problems each one serves,
// its workspace, and its launcher.  Each route lives in its own .cu file.
#pragma once

#include "ct_internal.h"

namespace ct {

// fp32 grouped gather with TMA-staged input rows for groups of 5..8 channels
// on 2-D/3-D outputs (ct_grouped_tma.cu); launched by launch_grouped when it
// applies.
bool grouped_tma_supports(const Problem& p, const void* x);
cudaError_t launch_grouped_tma(const Problem& p, const void* x, const void* w, const void* bias,
                               void* y, cudaStream_t stream);
cudaError_t grouped_tma_error_word(unsigned int* v, bool clear);

// fp32 grouped gather for groups of 5..8 channels on 2-D/3-D outputs in
// which every warp of a persistent grid runs its own double-buffered TMA
// pipeline (ct_grouped_warp.cu); launched by launch_grouped when it applies.
// It applies Problem.act in its epilogue.
bool grouped_warp_supports(const Problem& p, const void* x);
cudaError_t launch_grouped_warp(const Problem& p, const void* x, const void* w, const void* bias,
                                void* y, cudaStream_t stream);
cudaError_t grouped_warp_error_word(unsigned int* v, bool clear);
// Error word of the backward kernels (the small-group dw kernel's staged copies).
cudaError_t backward_error_word(unsigned int* v, bool clear);

// CUDA-core grouped/depthwise stride-phase gather (ct_grouped.cu).
bool grouped_supports(const Problem& p);
// The kernel launch_grouped runs for p (x assumed 16-byte aligned).
const char* grouped_kernel_name(const Problem& p);
bool grouped_preferred(const Problem& p);
// *act_done says whether the launched kernel applied Problem.act itself.
cudaError_t launch_grouped(const Problem& p, const void* x, const void* w, const void* bias,
                           void* y, cudaStream_t stream, Profile* prof, bool* act_done);

// fp32 stride-phase implicit GEMM on CUDA cores (ct_simt.cu).
bool simt_supports(const Problem& p);
bool simt_preferred(const Problem& p);
size_t simt_workspace_bytes(const Problem& p);
cudaError_t launch_simt(const Problem& p, const void* x, const void* w, const void* bias, void* y,
                        void* workspace, cudaStream_t stream, Profile* prof);

// bf16/fp16 stride-phase implicit GEMM on tcgen05 tensor cores (ct_tc.cu).
bool tc_supports(const Problem& p);
bool tc_preferred(const Problem& p);
size_t tc_workspace_bytes(const Problem& p);
cudaError_t launch_tc(const Problem& p, const void* x, const void* w, const void* bias, void* y,
                      void* workspace, cudaStream_t stream, Profile* prof);

// fp32 stride-phase implicit GEMM on tcgen05 tensor cores, error-compensated
// TF32 (ct_tc32.cu).
bool tc32_supports(const Problem& p);
bool tc32_preferred(const Problem& p);
size_t tc32_workspace_bytes(const Problem& p);
cudaError_t launch_tc32(const Problem& p, const void* x, const void* w, const void* bias, void* y,
                        void* workspace, cudaStream_t stream, Profile* prof);

// Gradients of the transposed convolution on CUDA cores (ct_backward.cu):
// dx, dw and db, each skipped when its pointer is null.  The workspace holds
// dw's per-slice fp32 partials.  `launches` (optional) counts the kernels.
bool backward_supported(const Problem& p);
// Workspace of the backward call: the largest of the db partials, the dw
// partials (or dy's channels-last copy and the split partials) and, when dx
// runs on the tensor cores, dy's channels-last copy and the gathered weights
// (stream-ordered, so the uses share it).
size_t backward_workspace_bytes(const Problem& p);
size_t backward_workspace_bytes(const Problem& p, bool dx, bool dw, bool db);
// Kernels that take most of the device time of dx and of dw.
const char* backward_dx_kernel_name(const Problem& p);
const char* backward_dw_kernel_name(const Problem& p);
// The input gradient on the tcgen05 GEMM (16-bit types, groups of 1): ct_tc.cu.
bool tc_dx_supports(const Problem& p);
size_t tc_dx_workspace_bytes(const Problem& p);
cudaError_t launch_tc_dx(const Problem& p, const void* dy, const void* w, void* dx, void* workspace,
                         cudaStream_t stream);
// The input gradient on the error-compensated TF32 GEMM (fp32, groups of 1): ct_tc32.cu.
bool tc32_dx_supports(const Problem& p);
size_t tc32_dx_workspace_bytes(const Problem& p);
cudaError_t launch_tc32_dx(const Problem& p, const void* dy, const void* w, void* dx, void* workspace,
                           cudaStream_t stream);
// The weight gradient on the tcgen05 GEMM (16-bit types, groups of 1): ct_tc.cu.
bool tc_dw_supports(const Problem& p);
size_t tc_dw_workspace_bytes(const Problem& p);
cudaError_t launch_tc_dw(const Problem& p, const void* x, const void* dy, void* dw, void* workspace,
                         cudaStream_t stream);
cudaError_t launch_backward(const Problem& p, const void* x, const void* w, const void* dy, void* dx,
                            void* dw, void* db, void* workspace, cudaStream_t stream, int* launches);

// Device error words of the tcgen05 routes: codes recorded by bounded waits
// that timed out (0 = none); `clear` resets a non-zero word.
cudaError_t tc_error_word(unsigned int* v, bool clear);
cudaError_t tc32_error_word(unsigned int* v, bool clear);

}  // namespace ct
