/*
 * ct.h -- C ABI of the GB300 forward transposed-convolution library (libct.so).
 *
 * The operation.  y = ConvTranspose(x, w, bias): the transpose of a
 * convolution ("fractionally strided convolution", "deconvolution"), as
 * described on the ONNX page "ai.onnx.ConvTranspose" (Description) with the
 * PyTorch conventions stated in "feat(ops): implement convTranspose2d -- CPU
 * kernel, backward and StableHLO lowering" (SKaiNET #1464, Summary):
 *
 *   y[b, oc, o] = bias[oc]
 *               + sum over ic in oc's group, taps t, inputs i with
 *                 o_a = i_a*stride_a - pad_lo_a + t_a*dilation_a on every axis a
 *                 of x[b, ic, i] * w[ic, oc mod (C_out/groups), t]
 *
 * i.e. each input sample is scattered through every weight tap, and products
 * that land outside the output are dropped.  Per spatial axis the output
 * extent is
 *
 *   O_a = (I_a - 1)*stride_a - pad_lo_a - pad_hi_a + dilation_a*(k_a - 1)
 *         + output_padding_a + 1
 *
 * (SKaiNET #1464, Summary, output size; asymmetric per-side padding as in the
 * NKI page "Conv3D Transpose Kernel API Reference", conv3d_transpose
 * parameters).  output_padding extends the high end of each axis.
 *
 * Layouts (all dense, row-major, one dtype for x, w, bias and y):
 *   x    [B, C_in, I_1 .. I_nd]                 (NCL / NCHW / NCDHW)
 *   w    [C_in, C_out/groups, k_1 .. k_nd]       (PyTorch ConvTranspose layout)
 *   bias [C_out] or NULL
 *   y    [B, C_out, O_1 .. O_nd]
 * Accumulation is in fp32 for every dtype; bias is added in fp32 and the sum
 * is rounded once (round-to-nearest-even) to the output dtype.
 *
 * Conventions for every entry point:
 *   - Return value is a ct_status; CT_OK (0) on success.  On any other value
 *     ct_last_error() gives a message (thread-local, valid until the next
 *     failing call from the same thread).
 *   - Argument validation happens on the host before any device work; a
 *     rejected call launches nothing and leaves y untouched.
 *   - Arrays of per-axis values (in_spatial, k, stride, pad_lo, pad_hi,
 *     dilation, output_padding) hold nd entries each, outermost axis first.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device entry points are asynchronous on that stream.
 *   - The library holds no per-call state; calls on different streams may run
 *     concurrently provided they use distinct workspaces.
 */
#ifndef CT_H
#define CT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  Integer types are not accepted: the SKaiNET pull request
 * (#1464, Summary) rejects non-float dtypes with an error instead of
 * computing with them. */
typedef enum { CT_F32 = 0, CT_F16 = 1, CT_BF16 = 2 } ct_dtype;

typedef enum {
    CT_OK = 0,
    CT_ERR_NULL = 1,            /* a required pointer is NULL */
    CT_ERR_RANK = 2,            /* nd outside 1..3 */
    CT_ERR_SHAPE = 3,           /* negative size, or an output extent < 1 */
    CT_ERR_PARAM = 4,           /* k, stride, dilation < 1; pad < 0;
                                   output_padding outside [0, max(stride, dilation)) */
    CT_ERR_GROUPS = 5,          /* groups < 1 or not dividing C_in and C_out */
    CT_ERR_BIAS = 6,            /* bias shape is not [C_out] (binding-level check) */
    CT_ERR_DTYPE = 7,           /* dtype is not one of ct_dtype */
    CT_ERR_CUDA = 8,            /* a CUDA runtime call or launch failed */
    CT_ERR_DEVICE_TIMEOUT = 9,  /* a bounded device-side wait gave up */
    CT_ERR_WORKSPACE = 10,      /* workspace given but smaller than required */
    CT_ERR_ALIGN = 11,          /* a pointer is not aligned to its element size */
    CT_ERR_ROUTE = 12,          /* a forced route cannot run this problem */
    CT_ERR_TOO_LARGE = 13       /* a size exceeds what the kernels index */
} ct_status;

/* Kernel routes.  CT_ROUTE_AUTO lets the library choose per call from the
 * shapes and dtype, as the ONNX page's "Implementation variants" section
 * describes one variant being selected per call. */
typedef enum {
    CT_ROUTE_AUTO = -1,
    CT_ROUTE_NONE = 0,      /* y has no elements: nothing to do */
    CT_ROUTE_BIAS_FILL = 1, /* no input contributes (C_in == 0 or an input
                               extent is 0): y = bias broadcast, or 0 */
    CT_ROUTE_GATHER = 2,    /* generic CUDA-core gather, any shape and dtype */
    CT_ROUTE_GROUPED = 3,   /* CUDA-core grouped/depthwise stride-phase gather */
    CT_ROUTE_SIMT_GEMM = 4, /* fp32 stride-phase implicit GEMM on CUDA cores */
    CT_ROUTE_TC_GEMM = 5,   /* bf16/fp16 stride-phase implicit GEMM on tcgen05 */
    CT_ROUTE_TC32_GEMM = 6  /* fp32 stride-phase implicit GEMM on tcgen05 with
                               error-compensated TF32: each operand split into
                               TF32 hi + lo parts, products accumulated as
                               hi*hi + hi*lo + lo*hi in fp32 (about fp32
                               accuracy; CT_ROUTE_SIMT_GEMM is the plain fp32
                               FMA route) */
} ct_route;

/* Library version (major*10000 + minor*100 + patch). */
int ct_version(void);

/* Message for the last nonzero status returned on this thread. */
const char* ct_last_error(void);

/* Fixed text for a status code. */
const char* ct_status_string(int status);

/*
 * Output spatial extents (host only, no device work).  The shape-only
 * counterpart of the operation (SKaiNET #1464: "VoidTensorOps: shape-only
 * implementation"; ONNX page: output shapes are inferred from the inputs and
 * attributes).  Writes nd values to out_spatial.
 * Errors: CT_ERR_NULL, CT_ERR_RANK, CT_ERR_SHAPE, CT_ERR_PARAM, CT_ERR_TOO_LARGE.
 */
int ct_conv_transpose_out_shape(int nd, const int64_t* in_spatial,
                                const int64_t* k, const int* stride,
                                const int* pad_lo, const int* pad_hi,
                                const int* dilation, const int* output_padding,
                                int64_t* out_spatial);

/*
 * Bytes of device workspace ct_conv_transpose_nd needs for this problem on
 * the route it would choose (0 when the route needs none).  The workspace
 * holds the reordered (tap-reversed, per-phase, K-major) weights and, for the
 * tensor-core route, a channels-last copy of x.  Host only.
 * Errors: the validation errors of ct_conv_transpose_nd.
 */
int ct_conv_transpose_workspace_bytes(int nd, int64_t B, int64_t C_in,
                                      int64_t C_out, const int64_t* in_spatial,
                                      const int64_t* k, const int* stride,
                                      const int* pad_lo, const int* pad_hi,
                                      const int* dilation,
                                      const int* output_padding, int groups,
                                      int dtype, size_t* bytes);

/*
 * The route ct_conv_transpose_nd would take for this problem (a ct_route
 * value written to *route).  Host only; the route also depends on the current
 * device (the tensor-core route needs an sm_103 device).
 */
int ct_conv_transpose_route(int nd, int64_t B, int64_t C_in, int64_t C_out,
                            const int64_t* in_spatial, const int64_t* k,
                            const int* stride, const int* pad_lo,
                            const int* pad_hi, const int* dilation,
                            const int* output_padding, int groups, int dtype,
                            int* route);

/*
 * Name of the kernel that takes most of the device time of
 * ct_conv_transpose_nd on this problem (for example "tc_phase_gemm" or
 * "grouped_tma_kernel"; "" when the call launches nothing), written to
 * *name as a pointer to a static string.  Host only; like the route it
 * depends on the current device, and it assumes x is 16-byte aligned, as
 * device allocations are (an x that is not aligned can move a grouped fp32
 * problem from grouped_tma_kernel to grouped_staged_kernel).  Used to tie a
 * measured time to the kernel's roofline and profile.
 */
int ct_conv_transpose_kernel(int nd, int64_t B, int64_t C_in, int64_t C_out,
                             const int64_t* in_spatial, const int64_t* k,
                             const int* stride, const int* pad_lo,
                             const int* pad_hi, const int* dilation,
                             const int* output_padding, int groups, int dtype,
                             const char** name);

/*
 * Forward transposed convolution on the device.
 *
 *   x, w, bias, y : device pointers owned by the caller, layouts above; bias
 *                   may be NULL.  x, w and bias are only read; y is fully
 *                   overwritten (every element, including positions no input
 *                   reaches, which receive bias or 0).  y must not overlap
 *                   x, w, bias or the workspace.
 *   workspace     : device memory of at least ct_conv_transpose_workspace_bytes
 *                   bytes, 256-byte aligned, or NULL.  When NULL and the route
 *                   needs workspace, the call takes it from the stream-ordered
 *                   allocator (cudaMallocAsync / cudaFreeAsync on `stream`).
 *   workspace_bytes : size of `workspace` (ignored when workspace is NULL).
 *   nd            : number of spatial axes, 1..3.
 *   B, C_in, C_out, groups : batch, channels and groups; C_out = w.shape[1]*groups.
 *   dtype         : ct_dtype of x, w, bias and y.
 *   stream        : cudaStream_t (as void*).
 *
 * Pointers must be aligned to the element size (CT_ERR_ALIGN otherwise); the
 * fast routes additionally want 16-byte alignment and otherwise fall back to
 * the generic gather route.  Launch failures return CT_ERR_CUDA.  The call
 * does not synchronise.
 */
int ct_conv_transpose_nd(const void* x, const void* w, const void* bias,
                         void* y, void* workspace, size_t workspace_bytes,
                         int nd, int64_t B, int64_t C_in, int64_t C_out,
                         const int64_t* in_spatial, const int64_t* k,
                         const int* stride, const int* pad_lo,
                         const int* pad_hi, const int* dilation,
                         const int* output_padding, int groups, int dtype,
                         void* stream);

/*
 * As ct_conv_transpose_nd, with the kernel route chosen by the caller
 * (CT_ROUTE_AUTO = the library's choice).  A route that cannot run the
 * problem returns CT_ERR_ROUTE.  Used to test every route on the same inputs.
 * The workspace, when given, must be sized for the forced route
 * (ct_conv_transpose_route_workspace_bytes).
 */
int ct_conv_transpose_nd_route(const void* x, const void* w, const void* bias,
                               void* y, void* workspace, size_t workspace_bytes,
                               int nd, int64_t B, int64_t C_in, int64_t C_out,
                               const int64_t* in_spatial, const int64_t* k,
                               const int* stride, const int* pad_lo,
                               const int* pad_hi, const int* dilation,
                               const int* output_padding, int groups,
                               int dtype, int route, void* stream);

/*
 * As ct_conv_transpose_nd_route, for measurement.  main_start / main_stop
 * (cudaEvent_t as void*, either may be NULL) are recorded on `stream` just
 * before and just after the launch of the route's dominant kernel, so the
 * caller can time that kernel alone with cudaEventElapsedTime.  *launches
 * (nullable) receives the number of kernels the call launched and
 * *route_taken (nullable) the route that ran.
 */
int ct_conv_transpose_nd_profiled(const void* x, const void* w, const void* bias,
                                  void* y, void* workspace,
                                  size_t workspace_bytes, int nd, int64_t B,
                                  int64_t C_in, int64_t C_out,
                                  const int64_t* in_spatial, const int64_t* k,
                                  const int* stride, const int* pad_lo,
                                  const int* pad_hi, const int* dilation,
                                  const int* output_padding, int groups,
                                  int dtype, int route, void* stream,
                                  void* main_start, void* main_stop,
                                  int* launches, int* route_taken);

/* Workspace bytes of a given route (CT_ERR_ROUTE if it cannot run the problem). */
int ct_conv_transpose_route_workspace_bytes(int nd, int64_t B, int64_t C_in,
                                            int64_t C_out,
                                            const int64_t* in_spatial,
                                            const int64_t* k, const int* stride,
                                            const int* pad_lo, const int* pad_hi,
                                            const int* dilation,
                                            const int* output_padding,
                                            int groups, int dtype, int route,
                                            size_t* bytes);

/*
 * End-to-end call on HOST buffers: x, w, bias (nullable) and y are host
 * pointers (pinned memory gives the fastest copies).  The call takes device
 * buffers from a library-owned stream-ordered memory pool (one per device,
 * created by the first call; it keeps its memory between calls until
 * ct_host_buffers_release), copies w and bias in, then runs the batch in up
 * to 8 chunks as a pipeline: chunk c's input copy (on a library side stream),
 * its computation (on `stream`, as ct_conv_transpose_nd) and its output copy
 * (on a second side stream) overlap the neighbouring chunks' copies.  Calls
 * whose x and y together hold less than 8 MiB, or with B = 1, run as one
 * chunk.  The call synchronises `stream` before returning; concurrent calls
 * from several host threads on one device are serialised.  Same validation
 * and errors as the device call.
 */
int ct_conv_transpose_nd_host(const void* x, const void* w, const void* bias,
                              void* y, int nd, int64_t B, int64_t C_in,
                              int64_t C_out, const int64_t* in_spatial,
                              const int64_t* k, const int* stride,
                              const int* pad_lo, const int* pad_hi,
                              const int* dilation, const int* output_padding,
                              int groups, int dtype, void* stream);

/*
 * Activations of the extended call, applied to each output after the bias
 * (the NKI page's conv3d_transpose takes an optional activation function
 * run on the convolution's result; it names no particular ones, so these are
 * the common ones).  The tcgen05 routes and the bias fill apply it in fp32
 * before the one rounding to the output type; the CUDA-core routes (gather,
 * grouped, SIMT) round the convolution first and apply it in a second pass
 * over y, so a 16-bit output is then rounded twice.
 */
typedef enum {
    CT_ACT_NONE = 0,
    CT_ACT_RELU = 1,        /* max(v, 0) */
    CT_ACT_LEAKY_RELU = 2,  /* v >= 0 ? v : alpha * v */
    CT_ACT_SILU = 3,        /* v / (1 + exp(-v)) */
    CT_ACT_GELU = 4,        /* v * (1 + erf(v / sqrt(2))) / 2 */
    CT_ACT_TANH = 5,
    CT_ACT_SIGMOID = 6      /* 1 / (1 + exp(-v)) */
} ct_activation;

/* Weight layouts of the extended call (NKI page, conv3d_transpose filter_shape). */
typedef enum {
    CT_W_TORCH = 0,         /* [C_in, C_out/groups, k...] (PyTorch, ONNX) */
    CT_W_KDHW_CI_CO = 1,    /* [k..., C_in, C_out], groups 1 */
    CT_W_KDHW_CO_CI = 2     /* [k..., C_out, C_in], groups 1 */
} ct_weight_layout;

/*
 * ct_conv_transpose_nd with the options of the NKI page's conv3d_transpose:
 * w_layout (ct_weight_layout), taps_flipped (1: the stored taps are reversed
 * along every spatial axis relative to the PyTorch orientation, i.e. the
 * caller flipped them -- NKI's flip_filter_taps_in_kernel = False; 0: as
 * PyTorch stores them), activation (ct_activation) and activation_alpha (the
 * leaky-relu slope; ignored by the others).  A weight that is not in the
 * PyTorch layout, or is flipped, is first rewritten into it in the head of
 * the workspace (ct_conv_transpose_ex_workspace_bytes; NULL: allocated
 * stream-ordered); the rest of the call is ct_conv_transpose_nd's, followed
 * by the activation as described at ct_activation.  Extra errors: CT_ERR_PARAM
 * for an unknown layout, flag or activation; CT_ERR_GROUPS for layouts 1, 2
 * with groups != 1.
 */
int ct_conv_transpose_nd_ex(const void* x, const void* w, const void* bias,
                            void* y, void* workspace, size_t workspace_bytes,
                            int nd, int64_t B, int64_t C_in, int64_t C_out,
                            const int64_t* in_spatial, const int64_t* k,
                            const int* stride, const int* pad_lo,
                            const int* pad_hi, const int* dilation,
                            const int* output_padding, int groups, int dtype,
                            int w_layout, int taps_flipped, int activation,
                            float activation_alpha, void* stream);

/* Workspace bytes of ct_conv_transpose_nd_ex for the given layout options. */
int ct_conv_transpose_ex_workspace_bytes(int nd, int64_t B, int64_t C_in,
                                         int64_t C_out, const int64_t* in_spatial,
                                         const int64_t* k, const int* stride,
                                         const int* pad_lo, const int* pad_hi,
                                         const int* dilation,
                                         const int* output_padding, int groups,
                                         int dtype, int w_layout, int taps_flipped,
                                         size_t* bytes);

/*
 * Gradients of y = ConvTranspose(x, w, bias): the backward pass of the
 * SKaiNET pull request "feat(ops): implement convTranspose2d -- CPU kernel,
 * backward and StableHLO lowering" (#1464, Summary: convTranspose2dBackward,
 * the adjoint giving input, weight and bias gradients), for the same
 * problems as ct_conv_transpose_nd.  For an upstream gradient dy (y's shape
 * [B, C_out, out spatial...]):
 *   dx[b, ic, i]    = sum_{oc in ic's group, t} w[ic, oc_g, t] * dy[b, oc, o(i, t)]
 *   dw[ic, oc_g, t] = sum_{b, i}               x[b, ic, i]    * dy[b, oc, o(i, t)]
 *   db[oc]          = sum_{b, o}               dy[b, oc, o]
 * with o_a(i, t) = i_a*stride_a - pad_lo_a + t_a*dilation_a, terms whose o
 * falls outside the output dropped.  All pointers are device pointers owned
 * by the caller, dense, in the layouts of the forward call and one dtype;
 * dx ([B, C_in, in spatial...]), dw ([C_in, C_out/groups, k...]) and db
 * ([C_out]) may each be NULL (not computed); x is needed for dw, w for dx.
 * Each result is written, not accumulated into.  fp32 accumulation, one
 * rounding to the dtype, fixed summation order (bit-reproducible).
 * workspace: device buffer of ct_conv_transpose_backward_workspace_bytes
 * (256-byte aligned), or NULL to have the call allocate it stream-ordered.
 * Asynchronous on `stream`.  Errors as the forward call; CT_ERR_TOO_LARGE
 * when the kernel has more taps than the staged weight slab holds.
 */
int ct_conv_transpose_backward_nd(const void* x, const void* w, const void* dy,
                                  void* dx, void* dw, void* db, void* workspace,
                                  size_t workspace_bytes, int nd, int64_t B,
                                  int64_t C_in, int64_t C_out,
                                  const int64_t* in_spatial, const int64_t* k,
                                  const int* stride, const int* pad_lo,
                                  const int* pad_hi, const int* dilation,
                                  const int* output_padding, int groups,
                                  int dtype, void* stream);

/*
 * Workspace bytes of ct_conv_transpose_backward_nd: the largest of db's
 * per-segment partials (a few floats per output channel), dw's
 * per-slice partials (or, on the tensor cores, dy's channels-last copy and
 * the split partials) and, when dx runs on the tensor cores, dy's
 * channels-last copy (fp32: as TF32 high and low parts) and the gathered
 * weights.  Covers a call that requests any of dx, dw and db.
 */
int ct_conv_transpose_backward_workspace_bytes(int nd, int64_t B, int64_t C_in,
                                               int64_t C_out,
                                               const int64_t* in_spatial,
                                               const int64_t* k, const int* stride,
                                               const int* pad_lo, const int* pad_hi,
                                               const int* dilation,
                                               const int* output_padding,
                                               int groups, int dtype, size_t* bytes);

/*
 * Names of the kernels that take most of the device time of the input
 * gradient and of the weight gradient of ct_conv_transpose_backward_nd on
 * this problem, written to *dx_kernel and *dw_kernel as pointers to static
 * strings: "tc_phase_gemm" (dx on the tensor cores: bf16/fp16, groups of 1,
 * at least 16 channels each side), "tc32_phase_gemm" (dx on the
 * error-compensated TF32 tensor-core GEMM: fp32, groups of 1, at least 32
 * channels each side) or "bwd_dx_kernel"; "tc_dw_gemm" (dw on
 * the tensor cores: the same class with a W stride of at most 4 and an input
 * width that is a multiple of 8), "bwd_dw_grouped_kernel" (groups of at most
 * 8 input and 8 output channels, at most 27 taps) or "bwd_dw_kernel"; "" for
 * an empty gradient.  Host only; depends on the
 * current device.  Errors as ct_conv_transpose_backward_workspace_bytes.
 */
int ct_conv_transpose_backward_kernels(int nd, int64_t B, int64_t C_in,
                                       int64_t C_out, const int64_t* in_spatial,
                                       const int64_t* k, const int* stride,
                                       const int* pad_lo, const int* pad_hi,
                                       const int* dilation,
                                       const int* output_padding, int groups,
                                       int dtype, const char** dx_kernel,
                                       const char** dw_kernel);

/*
 * Returns the memory the host-buffer entry point keeps in its pool on the
 * current device to the device (the pool itself stays, empty).  The memory
 * is otherwise kept until process exit.  Host only; CT_ERR_CUDA on failure.
 */
int ct_host_buffers_release(void);

/*
 * Size of the fixed scratch array behind ct_conv_transpose_nd_noalloc.
 */
#define CT_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * Forward transposed convolution that allocates no device memory.  The pages
 * have no counterpart: this entry point exists for callers that cannot call
 * cudaMalloc or cudaMallocAsync where they run the convolution -- code
 * running under a CUDA graph capture that forbids allocation, inference-
 * engine plugins that may only use memory the engine hands them, frameworks
 * that own the whole device memory budget through their own pool, and
 * real-time callers that allow no allocation after start-up.
 *
 * Arguments, layouts, validation and results are those of
 * ct_conv_transpose_nd; x, w, bias and y are device pointers the caller owns.
 * Instead of a workspace, the call uses one static device array of
 * CT_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU which loads the library
 * holds until the process exits.  A problem whose route needs more scratch
 * than that is rejected with CT_ERR_WORKSPACE before any device work.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it with the
 * unique id of the device's context; make that first call before any stream
 * capture.  After a cudaDeviceReset the next call finds a new context id and
 * looks the address up again (make it, too, outside a capture).  All calls share the one array and
 * it keeps whatever the last call left there; the kernels overwrite every
 * byte of scratch they read, so no call depends on its contents.  Calls that
 * may overlap on the GPU (different streams, or concurrent host threads on
 * different streams) race on the array: serialise them.
 */
int ct_conv_transpose_nd_noalloc(const void* x, const void* w, const void* bias,
                                 void* y, int nd, int64_t B, int64_t C_in,
                                 int64_t C_out, const int64_t* in_spatial,
                                 const int64_t* k, const int* stride,
                                 const int* pad_lo, const int* pad_hi,
                                 const int* dilation, const int* output_padding,
                                 int groups, int dtype, void* stream);

/*
 * Device-side error word written by bounded waits in the kernels that wait on
 * asynchronous copies or MMAs (0 = none; otherwise the bits say which wait
 * gave up: 1 TMA producer, 2 MMA issuer, 4 epilogue (tensor-core routes),
 * 8 a drain after a give-up that itself ran out, 16 the grouped TMA kernel's
 * copy, 32 a grouped warp pair's input copy, 64 a grouped warp pair's results,
 * 128 a staged copy of the backward pass's small-group weight-gradient
 * kernel; the words of every kernel file are
 * OR-ed).  Synchronises the current device, writes the word to *code and
 * clears it when `clear` is nonzero.  Returns CT_ERR_DEVICE_TIMEOUT when the
 * word was set, CT_OK otherwise.  The SKaiNET pull request's rule that bad
 * states fail loudly instead of giving silent results, applied to the device:
 * a kernel whose wait gives up stops its work, lets every copy and MMA it has
 * already issued finish (bounded by a fixed 2 s), frees its tensor memory,
 * returns, and leaves its outputs unspecified; the word tells the caller.
 */
int ct_device_status(int clear, unsigned int* code);

/* Default limit of each bounded device-side wait, in nanoseconds (2 s). */
#define CT_WAIT_LIMIT_DEFAULT_NS 2000000000ull

/*
 * Sets the limit, in nanoseconds, of every bounded device-side wait in the
 * launches that follow (process-wide, all devices) and returns the previous
 * limit.  The default, CT_WAIT_LIMIT_DEFAULT_NS, is far above any wait of a
 * healthy call.  A limit of 0 makes a wait give up at the first probe that
 * finds its copy or MMA incomplete, as if it would never arrive: tests use it
 * to drive the give-up path of ct_device_status on purpose.  Host only; for
 * tests and diagnostics -- calls made while the limit is small may stop early
 * and leave y unspecified (ct_device_status then reports it).
 */
unsigned long long ct_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* CT_H */
