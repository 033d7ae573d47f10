/*
 * ct_oracle.c -- fp64 CPU oracle for the forward transposed convolution and
 * its gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) links, loads or calls this file.  Only the test suite, the
 * package smoke check and the CPU-baseline leg of the benchmark use it.  It
 * shares no code, header, table or constant with the CUDA path.
 *
 * What it computes.  The scatter-add definition of ConvTranspose given in
 * "feat(ops): implement convTranspose2d -- CPU kernel, backward and StableHLO
 * lowering" (SKaiNET pull request #1464), Summary, DefaultCpuOps paragraph:
 * every input sample is multiplied by every weight tap and added into the
 * output position  i*stride - padding + t*dilation  of each axis, and products
 * that land outside the output are dropped.  The same page states the PyTorch
 * conventions used here: weight layout [C_in, C_out/groups, k...], so the
 * output channel count is C_out = w.shape[1] * groups.  The ONNX page "ai.onnx.ConvTranspose"
 * (Description) and the NKI page "Conv3D Transpose Kernel API Reference"
 * (conv3d_transpose parameters) extend it to 1-D/3-D, asymmetric low/high
 * padding and output_padding on the high side.
 *
 * Arithmetic: every input is widened to double by the caller; the oracle does
 * all products and sums in double and never rounds to a narrower type.
 * Threading: the output is split into disjoint (b, oc) slices, one thread per
 * slice at a time, so the result does not depend on the thread count.
 *
 * Every rank 1..3 problem is handled as a 3-D one whose unused leading axes
 * have extent 1, kernel 1, stride 1, no padding and dilation 1.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_BAD_ARG 1
#define OR_BAD_SHAPE 2
#define OR_NO_MEMORY 3

/* One problem, normalised to three spatial axes (index 0 = D, 1 = H, 2 = W). */
typedef struct {
    int64_t B, C_in, C_out, groups;
    int64_t I[3], K[3], S[3], PL[3], PH[3], DL[3], OP[3], O[3];
} or_problem;

/*
 * Output extent of one axis.  The NKI page (conv3d_transpose, output shape)
 * and the SKaiNET pull request (Summary, output size) give the symmetric form
 * (in-1)*stride - 2*padding + dilation*(k-1) [+ outputPadding] + 1; with the
 * asymmetric 6-value padding of the NKI page the two pads enter separately.
 */
static int64_t or_out_extent(int64_t I, int64_t K, int64_t S, int64_t PL,
                             int64_t PH, int64_t DL, int64_t OP)
{
    return (I - 1) * S - PL - PH + DL * (K - 1) + OP + 1;
}

static int or_setup(or_problem* p, int nd, int64_t B, int64_t C_in,
                    int64_t C_out, int64_t groups, const int64_t* in_sp,
                    const int64_t* k, const int64_t* stride,
                    const int64_t* pad_lo, const int64_t* pad_hi,
                    const int64_t* dilation, const int64_t* out_pad)
{
    if (nd < 1 || nd > 3) return OR_BAD_ARG;
    if (B < 0 || C_in < 0 || C_out < 0 || groups < 1) return OR_BAD_ARG;
    if (C_in % groups != 0 || C_out % groups != 0) return OR_BAD_ARG;
    memset(p, 0, sizeof(*p));
    p->B = B; p->C_in = C_in; p->C_out = C_out; p->groups = groups;
    for (int a = 0; a < 3; ++a) {
        p->I[a] = 1; p->K[a] = 1; p->S[a] = 1; p->PL[a] = 0; p->PH[a] = 0;
        p->DL[a] = 1; p->OP[a] = 0;
    }
    for (int j = 0; j < nd; ++j) {
        int a = 3 - nd + j;
        p->I[a] = in_sp[j]; p->K[a] = k[j]; p->S[a] = stride[j];
        p->PL[a] = pad_lo[j]; p->PH[a] = pad_hi[j]; p->DL[a] = dilation[j];
        p->OP[a] = out_pad[j];
        if (p->I[a] < 0 || p->K[a] < 1 || p->S[a] < 1 || p->DL[a] < 1 ||
            p->PL[a] < 0 || p->PH[a] < 0 || p->OP[a] < 0)
            return OR_BAD_ARG;
    }
    for (int a = 0; a < 3; ++a) {
        p->O[a] = or_out_extent(p->I[a], p->K[a], p->S[a], p->PL[a], p->PH[a],
                                p->DL[a], p->OP[a]);
        if (p->O[a] < 1) return OR_BAD_SHAPE;
    }
    return OR_OK;
}

int oracle_out_shape(int nd, const int64_t* in_sp, const int64_t* k,
                     const int64_t* stride, const int64_t* pad_lo,
                     const int64_t* pad_hi, const int64_t* dilation,
                     const int64_t* out_pad, int64_t* out_sp)
{
    or_problem p;
    int rc = or_setup(&p, nd, 1, 1, 1, 1, in_sp, k, stride, pad_lo, pad_hi,
                      dilation, out_pad);
    if (rc != OR_OK) return rc;
    for (int j = 0; j < nd; ++j) out_sp[j] = p.O[3 - nd + j];
    return OR_OK;
}

typedef struct {
    const or_problem* p;
    const double* x;      /* [B, C_in, I0, I1, I2] */
    const double* w;      /* [C_in, C_out/groups, K0, K1, K2] */
    const double* bias;   /* [C_out] or NULL */
    double* y;            /* [B, C_out, O0, O1, O2] */
    int64_t next_slice;   /* shared work counter, guarded by lock */
    pthread_mutex_t lock;
} or_job;

/*
 * One output slice y[b, oc, :, :, :]: start from the bias (or zero), then add
 * x[b, ic, i] * w[ic, oc_g, t] at o_a = i_a*s_a - pad_lo_a + t_a*d_a for every
 * input channel ic of the slice's group, every input position i and every tap
 * t, dropping products whose o falls outside [0, O_a) on some axis.
 * The loops run ic, t, i so that the innermost loop walks a row of x.
 */
static void or_scatter_slice(const or_job* job, int64_t b, int64_t oc)
{
    const or_problem* p = job->p;
    const int64_t Cig = p->C_in / p->groups, Cog = p->C_out / p->groups;
    const int64_t g = oc / Cog, oc_g = oc % Cog;
    const int64_t In = p->I[0] * p->I[1] * p->I[2];
    const int64_t On = p->O[0] * p->O[1] * p->O[2];
    const int64_t Kn = p->K[0] * p->K[1] * p->K[2];
    double* ys = job->y + (b * p->C_out + oc) * On;
    const double init = job->bias ? job->bias[oc] : 0.0;
    for (int64_t o = 0; o < On; ++o) ys[o] = init;

    for (int64_t ic_g = 0; ic_g < Cig; ++ic_g) {
        const int64_t ic = g * Cig + ic_g;
        const double* xs = job->x + (b * p->C_in + ic) * In;
        const double* ws = job->w + (ic * Cog + oc_g) * Kn;
        for (int64_t t0 = 0; t0 < p->K[0]; ++t0)
        for (int64_t t1 = 0; t1 < p->K[1]; ++t1)
        for (int64_t t2 = 0; t2 < p->K[2]; ++t2) {
            const double wv = ws[(t0 * p->K[1] + t1) * p->K[2] + t2];
            for (int64_t i0 = 0; i0 < p->I[0]; ++i0) {
                const int64_t o0 = i0 * p->S[0] - p->PL[0] + t0 * p->DL[0];
                if (o0 < 0 || o0 >= p->O[0]) continue;
                for (int64_t i1 = 0; i1 < p->I[1]; ++i1) {
                    const int64_t o1 = i1 * p->S[1] - p->PL[1] + t1 * p->DL[1];
                    if (o1 < 0 || o1 >= p->O[1]) continue;
                    const double* xr = xs + (i0 * p->I[1] + i1) * p->I[2];
                    double* yr = ys + (o0 * p->O[1] + o1) * p->O[2];
                    for (int64_t i2 = 0; i2 < p->I[2]; ++i2) {
                        const int64_t o2 = i2 * p->S[2] - p->PL[2] + t2 * p->DL[2];
                        if (o2 < 0 || o2 >= p->O[2]) continue;
                        yr[o2] += xr[i2] * wv;
                    }
                }
            }
        }
    }
}

static void* or_worker(void* arg)
{
    or_job* job = (or_job*)arg;
    const int64_t nslices = job->p->B * job->p->C_out;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t s = job->next_slice++;
        pthread_mutex_unlock(&job->lock);
        if (s >= nslices) break;
        or_scatter_slice(job, s / job->p->C_out, s % job->p->C_out);
    }
    return NULL;
}

/*
 * Full forward transposed convolution, y = ConvTranspose(x, w, bias), in fp64.
 * Layouts: x [B, C_in, spatial...], w [C_in, C_out/groups, k...], bias [C_out]
 * (NULL for none), y [B, C_out, out spatial...], all dense and row-major.
 * Returns OR_OK, or a nonzero code for invalid arguments.  nthreads <= 0 uses 1.
 */
int oracle_conv_transpose_f64(const double* x, const double* w,
                              const double* bias, double* y, int nd, int64_t B,
                              int64_t C_in, int64_t C_out, int64_t groups,
                              const int64_t* in_sp, const int64_t* k,
                              const int64_t* stride, const int64_t* pad_lo,
                              const int64_t* pad_hi, const int64_t* dilation,
                              const int64_t* out_pad, int nthreads)
{
    or_problem p;
    int rc = or_setup(&p, nd, B, C_in, C_out, groups, in_sp, k, stride,
                      pad_lo, pad_hi, dilation, out_pad);
    if (rc != OR_OK) return rc;
    or_job job;
    job.p = &p; job.x = x; job.w = w; job.bias = bias; job.y = y;
    job.next_slice = 0;
    pthread_mutex_init(&job.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[started], NULL, or_worker, &job) != 0) break;
        ++started;
    }
    or_worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    pthread_mutex_destroy(&job.lock);
    return OR_OK;
}

/*
 * Point evaluation: y at a list of output coordinates, one by one, for checks
 * at sizes where the full scatter is too slow.  It sums the same products as
 * the scatter, found by inverting its index map: output o_a receives tap t_a
 * from input i_a exactly when o_a + pad_lo_a - t_a*d_a is a non-negative
 * multiple of s_a whose quotient i_a lies in [0, I_a).  The test suite checks
 * this function against the full scatter on random problems.
 * idx holds n rows of (b, oc, o_D, o_H, o_W) in the normalised 3-D indexing
 * (leading unused axes are 0).  Returns OR_OK or an error code.
 */
int oracle_points_f64(const double* x, const double* w, const double* bias,
                      int nd, int64_t B, int64_t C_in, int64_t C_out,
                      int64_t groups, const int64_t* in_sp, const int64_t* k,
                      const int64_t* stride, const int64_t* pad_lo,
                      const int64_t* pad_hi, const int64_t* dilation,
                      const int64_t* out_pad, const int64_t* idx, int64_t n,
                      double* out)
{
    or_problem p;
    int rc = or_setup(&p, nd, B, C_in, C_out, groups, in_sp, k, stride,
                      pad_lo, pad_hi, dilation, out_pad);
    if (rc != OR_OK) return rc;
    const int64_t Cig = p.C_in / p.groups, Cog = p.C_out / p.groups;
    const int64_t In = p.I[0] * p.I[1] * p.I[2];
    const int64_t Kn = p.K[0] * p.K[1] * p.K[2];
    for (int64_t e = 0; e < n; ++e) {
        const int64_t* q = idx + 5 * e;
        const int64_t b = q[0], oc = q[1];
        if (b < 0 || b >= p.B || oc < 0 || oc >= p.C_out) return OR_BAD_ARG;
        for (int a = 0; a < 3; ++a)
            if (q[2 + a] < 0 || q[2 + a] >= p.O[a]) return OR_BAD_ARG;
        const int64_t g = oc / Cog, oc_g = oc % Cog;
        double acc = bias ? bias[oc] : 0.0;
        for (int64_t ic_g = 0; ic_g < Cig; ++ic_g) {
            const int64_t ic = g * Cig + ic_g;
            for (int64_t t0 = 0; t0 < p.K[0]; ++t0) {
                const int64_t v0 = q[2] + p.PL[0] - t0 * p.DL[0];
                if (v0 < 0 || v0 % p.S[0] != 0 || v0 / p.S[0] >= p.I[0]) continue;
                for (int64_t t1 = 0; t1 < p.K[1]; ++t1) {
                    const int64_t v1 = q[3] + p.PL[1] - t1 * p.DL[1];
                    if (v1 < 0 || v1 % p.S[1] != 0 || v1 / p.S[1] >= p.I[1]) continue;
                    for (int64_t t2 = 0; t2 < p.K[2]; ++t2) {
                        const int64_t v2 = q[4] + p.PL[2] - t2 * p.DL[2];
                        if (v2 < 0 || v2 % p.S[2] != 0 || v2 / p.S[2] >= p.I[2]) continue;
                        const int64_t i0 = v0 / p.S[0], i1 = v1 / p.S[1], i2 = v2 / p.S[2];
                        const double xv = x[(b * p.C_in + ic) * In +
                                            (i0 * p.I[1] + i1) * p.I[2] + i2];
                        const double wv = w[(ic * Cog + oc_g) * Kn +
                                            (t0 * p.K[1] + t1) * p.K[2] + t2];
                        acc += xv * wv;
                    }
                }
            }
        }
        out[e] = acc;
    }
    return OR_OK;
}

/*
 * Backward pass (gradients), in fp64: the adjoint of the scatter above, as the
 * SKaiNET pull request's Summary describes its convTranspose2dBackward (input,
 * weight and bias gradients).  Every product of the forward pass,
 *     y[b, oc, o] += x[b, ic, i] * w[ic, oc_g, t]   at o_a = i_a*s_a - pad_lo_a + t_a*d_a
 * (o inside the output, ic in oc's group), contributes
 *     dx[b, ic, i]    += dy[b, oc, o] * w[ic, oc_g, t]
 *     dw[ic, oc_g, t] += dy[b, oc, o] * x[b, ic, i]
 * and every output element contributes db[oc] += dy[b, oc, o].
 * Slices: dx by (b, ic), dw by ic, db by oc; each is one thread's at a time,
 * with a fixed loop order, so the result does not depend on the thread count.
 */
typedef struct {
    const or_problem* p;
    const double* x;      /* [B, C_in, I...] */
    const double* w;      /* [C_in, C_out/groups, K...] */
    const double* dy;     /* [B, C_out, O...] */
    double* dx;           /* [B, C_in, I...] or NULL */
    double* dw;           /* [C_in, C_out/groups, K...] or NULL */
    double* db;           /* [C_out] or NULL */
    int64_t next_task;
    pthread_mutex_t lock;
} or_bjob;

/* dx[b, ic, :]: for each oc of the group and tap t, walk the input positions
 * and read dy at the output position the forward pass wrote them to. */
static void or_dx_slice(const or_bjob* j, int64_t b, int64_t ic)
{
    const or_problem* p = j->p;
    const int64_t Cig = p->C_in / p->groups, Cog = p->C_out / p->groups;
    const int64_t g = ic / Cig;
    const int64_t In = p->I[0] * p->I[1] * p->I[2];
    const int64_t On = p->O[0] * p->O[1] * p->O[2];
    const int64_t Kn = p->K[0] * p->K[1] * p->K[2];
    double* dxs = j->dx + (b * p->C_in + ic) * In;
    for (int64_t i = 0; i < In; ++i) dxs[i] = 0.0;
    for (int64_t oc_g = 0; oc_g < Cog; ++oc_g) {
        const int64_t oc = g * Cog + oc_g;
        const double* dys = j->dy + (b * p->C_out + oc) * On;
        const double* ws = j->w + (ic * Cog + oc_g) * Kn;
        for (int64_t t0 = 0; t0 < p->K[0]; ++t0)
        for (int64_t t1 = 0; t1 < p->K[1]; ++t1)
        for (int64_t t2 = 0; t2 < p->K[2]; ++t2) {
            const double wv = ws[(t0 * p->K[1] + t1) * p->K[2] + t2];
            for (int64_t i0 = 0; i0 < p->I[0]; ++i0) {
                const int64_t o0 = i0 * p->S[0] - p->PL[0] + t0 * p->DL[0];
                if (o0 < 0 || o0 >= p->O[0]) continue;
                for (int64_t i1 = 0; i1 < p->I[1]; ++i1) {
                    const int64_t o1 = i1 * p->S[1] - p->PL[1] + t1 * p->DL[1];
                    if (o1 < 0 || o1 >= p->O[1]) continue;
                    double* dxr = dxs + (i0 * p->I[1] + i1) * p->I[2];
                    const double* dyr = dys + (o0 * p->O[1] + o1) * p->O[2];
                    for (int64_t i2 = 0; i2 < p->I[2]; ++i2) {
                        const int64_t o2 = i2 * p->S[2] - p->PL[2] + t2 * p->DL[2];
                        if (o2 < 0 || o2 >= p->O[2]) continue;
                        dxr[i2] += dyr[o2] * wv;
                    }
                }
            }
        }
    }
}

/* dw[ic, :, :]: for each oc of the group and tap t, the sum over batch and
 * input positions of x times dy at the position the product landed on. */
static void or_dw_slice(const or_bjob* j, int64_t ic)
{
    const or_problem* p = j->p;
    const int64_t Cig = p->C_in / p->groups, Cog = p->C_out / p->groups;
    const int64_t g = ic / Cig;
    const int64_t In = p->I[0] * p->I[1] * p->I[2];
    const int64_t On = p->O[0] * p->O[1] * p->O[2];
    const int64_t Kn = p->K[0] * p->K[1] * p->K[2];
    for (int64_t oc_g = 0; oc_g < Cog; ++oc_g) {
        const int64_t oc = g * Cog + oc_g;
        for (int64_t t0 = 0; t0 < p->K[0]; ++t0)
        for (int64_t t1 = 0; t1 < p->K[1]; ++t1)
        for (int64_t t2 = 0; t2 < p->K[2]; ++t2) {
            double acc = 0.0;
            for (int64_t b = 0; b < p->B; ++b) {
                const double* xs = j->x + (b * p->C_in + ic) * In;
                const double* dys = j->dy + (b * p->C_out + oc) * On;
                for (int64_t i0 = 0; i0 < p->I[0]; ++i0) {
                    const int64_t o0 = i0 * p->S[0] - p->PL[0] + t0 * p->DL[0];
                    if (o0 < 0 || o0 >= p->O[0]) continue;
                    for (int64_t i1 = 0; i1 < p->I[1]; ++i1) {
                        const int64_t o1 = i1 * p->S[1] - p->PL[1] + t1 * p->DL[1];
                        if (o1 < 0 || o1 >= p->O[1]) continue;
                        const double* xr = xs + (i0 * p->I[1] + i1) * p->I[2];
                        const double* dyr = dys + (o0 * p->O[1] + o1) * p->O[2];
                        for (int64_t i2 = 0; i2 < p->I[2]; ++i2) {
                            const int64_t o2 = i2 * p->S[2] - p->PL[2] + t2 * p->DL[2];
                            if (o2 < 0 || o2 >= p->O[2]) continue;
                            acc += xr[i2] * dyr[o2];
                        }
                    }
                }
            }
            j->dw[(ic * Cog + oc_g) * Kn + (t0 * p->K[1] + t1) * p->K[2] + t2] = acc;
        }
    }
}

/* db[oc]: every output element of channel oc, batch by batch. */
static void or_db_slice(const or_bjob* j, int64_t oc)
{
    const or_problem* p = j->p;
    const int64_t On = p->O[0] * p->O[1] * p->O[2];
    double acc = 0.0;
    for (int64_t b = 0; b < p->B; ++b) {
        const double* dys = j->dy + (b * p->C_out + oc) * On;
        for (int64_t o = 0; o < On; ++o) acc += dys[o];
    }
    j->db[oc] = acc;
}

static void* or_bworker(void* arg)
{
    or_bjob* j = (or_bjob*)arg;
    const or_problem* p = j->p;
    const int64_t n_dx = j->dx ? p->B * p->C_in : 0;
    const int64_t n_dw = j->dw ? p->C_in : 0;
    const int64_t n_db = j->db ? p->C_out : 0;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int64_t s = j->next_task++;
        pthread_mutex_unlock(&j->lock);
        if (s < n_dx) { or_dx_slice(j, s / p->C_in, s % p->C_in); continue; }
        s -= n_dx;
        if (s < n_dw) { or_dw_slice(j, s); continue; }
        s -= n_dw;
        if (s < n_db) { or_db_slice(j, s); continue; }
        break;
    }
    return NULL;
}

/*
 * Gradients of y = ConvTranspose(x, w, bias) with respect to x, w and the
 * bias for an upstream gradient dy, in fp64.  Layouts as in
 * oracle_conv_transpose_f64; dy has y's shape.  dx, dw and db may each be
 * NULL (not computed).  Returns OR_OK or a nonzero code for invalid arguments.
 */
int oracle_conv_transpose_backward_f64(const double* x, const double* w,
                                       const double* dy, double* dx, double* dw,
                                       double* db, int nd, int64_t B,
                                       int64_t C_in, int64_t C_out, int64_t groups,
                                       const int64_t* in_sp, const int64_t* k,
                                       const int64_t* stride, const int64_t* pad_lo,
                                       const int64_t* pad_hi, const int64_t* dilation,
                                       const int64_t* out_pad, int nthreads)
{
    or_problem p;
    int rc = or_setup(&p, nd, B, C_in, C_out, groups, in_sp, k, stride,
                      pad_lo, pad_hi, dilation, out_pad);
    if (rc != OR_OK) return rc;
    or_bjob j;
    j.p = &p; j.x = x; j.w = w; j.dy = dy; j.dx = dx; j.dw = dw; j.db = db;
    j.next_task = 0;
    pthread_mutex_init(&j.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[started], NULL, or_bworker, &j) != 0) break;
        ++started;
    }
    or_bworker(&j);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    pthread_mutex_destroy(&j.lock);
    return OR_OK;
}

/*
 * Activation after the convolution, in fp64: the NKI page "Conv3D Transpose
 * Kernel API Reference" (conv3d_transpose, activation_fn: an optional
 * activation applied after the convolution).  The page does not list the
 * functions; these are the common ones, each from its textbook definition:
 *   0 none; 1 relu max(v, 0); 2 leaky relu v >= 0 ? v : alpha*v;
 *   3 silu v / (1 + e^-v); 4 gelu v * (1 + erf(v / sqrt 2)) / 2;
 *   5 tanh; 6 sigmoid 1 / (1 + e^-v).
 * Applied in place to n values (y includes the bias).  Returns OR_OK or
 * OR_BAD_ARG for an unknown code.
 */
#include <math.h>
int oracle_activation_f64(double* y, int64_t n, int act, double alpha)
{
    if (act < 0 || act > 6) return OR_BAD_ARG;
    for (int64_t e = 0; e < n; ++e) {
        const double v = y[e];
        double r = v;
        switch (act) {
            case 1: r = v > 0.0 ? v : 0.0; break;
            case 2: r = v >= 0.0 ? v : alpha * v; break;
            case 3: r = v / (1.0 + exp(-v)); break;
            case 4: r = 0.5 * v * (1.0 + erf(v / sqrt(2.0))); break;
            case 5: r = tanh(v); break;
            case 6: r = 1.0 / (1.0 + exp(-v)); break;
            default: break;
        }
        y[e] = r;
    }
    return OR_OK;
}
