/*
 * Plain CPU oracle for grouped-convolution backward-weight (wgrad).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file's library.  It shares no code with the CUDA
 * path: its own problem record, its own output-size rule, its own 16-bit
 * decoders, its own loops.
 *
 * What it computes is the definition of the weight gradient of a grouped
 * convolution, written out as a direct sum in fp64:
 *
 *   dW[g,k,z,y,x,c] = sum over n, od, oh, ow of
 *       dY[n,od,oh,ow,g,k] * X[n, od*sd - pld + z*dd, oh*sh - plh + y*dh,
 *                              ow*sw - plw + x*dw, g, c]
 *
 * with terms whose input position falls outside the image skipped (zero
 * padding).  Layouts follow "Composable Kernel: grouped_convolution_backward_
 * weight_kernel.hpp Source File", GroupedConvBwdWeightKernelArgs (the
 * NWGC/GKXC/NWGK, NHWGC/GKYXC/NHWGK and NDHWGC/GKZYXC/NDHWGK constructors):
 * activations are N,(D),(H),W,G,C (input) and N,(Do),(Ho),Wo,G,K (output
 * gradient), the weight gradient is G,K,(Z),(Y),X,C, and C, K are the channels
 * of one group (group strides K for dY, C for X and K*C*Z*Y*X for dW, as in the
 * group_stride_a/b/c lines of that constructor).
 *
 * The output spatial size is not given on that page (it is passed in as
 * output_spatial_lengths_); the oracle uses the standard convolution rule
 * out = floor((in + pad_l + pad_r - dil*(f-1) - 1) / stride) + 1.
 *
 * Every spatial problem is held as three dims (D, H, W), outermost first; a
 * 1-D or 2-D problem has the unused leading dims set to in = f = stride =
 * dil = 1 and pads 0.
 *
 * Besides dW the oracle returns A = sum of |dY * X| over the same terms, the
 * scale that the tolerance of a floating-point comparison is stated in.
 *
 * It also holds the forward convolution with the same geometry and the
 * backward-data gradient dX (the adjoint of the forward convolution in X),
 * each written out the same way (see orc_conv_fwd and orc_dgrad).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int G, N, C, K;
    int in[3], filt[3], stride[3], dil[3], pad_l[3], pad_r[3];
} orc_problem;

int orc_out_len(int in, int f, int s, int d, int pl, int pr)
{
    long num = (long)in + pl + pr - (long)d * (f - 1) - 1;
    if (num < 0 || s <= 0) return 0;
    return (int)(num / s) + 1;
}

static void out_dims(const orc_problem* p, int o[3])
{
    for (int i = 0; i < 3; ++i)
        o[i] = orc_out_len(p->in[i], p->filt[i], p->stride[i], p->dil[i], p->pad_l[i], p->pad_r[i]);
}

int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* bf16: the upper half of an IEEE binary32 word. */
static double dec_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp16: IEEE binary16, decoded field by field. */
static double dec_fp16(uint16_t b)
{
    int sign = (b >> 15) & 1, e = (b >> 10) & 31, m = b & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

void orc_decode16(const uint16_t* bits, long n, int is_bf16, double* out)
{
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) out[i] = is_bf16 ? dec_bf16(bits[i]) : dec_fp16(bits[i]);
}

/* Full dW (and A).  dw, absacc: G*K*Z*Y*X*C doubles each (absacc may be NULL). */
void orc_wgrad(const orc_problem* p, const double* x, const double* dy, double* dw, double* absacc)
{
    int o[3];
    out_dims(p, o);
    const int G = p->G, N = p->N, C = p->C, K = p->K;
    const int D = p->in[0], H = p->in[1], W = p->in[2];
    const int Z = p->filt[0], Y = p->filt[1], X = p->filt[2];
    const long T = (long)Z * Y * X;
    long gk;
#pragma omp parallel for schedule(dynamic, 1)
    for (gk = 0; gk < (long)G * K; ++gk) {
        const int g = (int)(gk / K), k = (int)(gk % K);
        double* acc = dw + gk * T * C;
        double* aab = absacc ? absacc + gk * T * C : 0;
        for (long i = 0; i < T * C; ++i) {
            acc[i] = 0.0;
            if (aab) aab[i] = 0.0;
        }
        for (int z = 0; z < Z; ++z)
            for (int y = 0; y < Y; ++y)
                for (int xx = 0; xx < X; ++xx) {
                    const long tap = ((long)z * Y + y) * X + xx;
                    for (int n = 0; n < N; ++n)
                        for (int od = 0; od < o[0]; ++od) {
                            const int id = od * p->stride[0] - p->pad_l[0] + z * p->dil[0];
                            if (id < 0 || id >= D) continue;
                            for (int oh = 0; oh < o[1]; ++oh) {
                                const int ih = oh * p->stride[1] - p->pad_l[1] + y * p->dil[1];
                                if (ih < 0 || ih >= H) continue;
                                for (int ow = 0; ow < o[2]; ++ow) {
                                    const int iw = ow * p->stride[2] - p->pad_l[2] + xx * p->dil[2];
                                    if (iw < 0 || iw >= W) continue;
                                    const long yo = ((((long)n * o[0] + od) * o[1] + oh) * o[2] + ow) * G + g;
                                    const double v = dy[yo * K + k];
                                    const long xo = ((((long)n * D + id) * H + ih) * W + iw) * G + g;
                                    const double* xr = x + xo * C;
                                    double* ar = acc + tap * C;
                                    for (int c = 0; c < C; ++c) ar[c] += v * xr[c];
                                    if (aab) {
                                        double* br = aab + tap * C;
                                        for (int c = 0; c < C; ++c) br[c] += fabs(v * xr[c]);
                                    }
                                }
                            }
                        }
                }
    }
}

/* Selected elements of dW only: idx[i] is a flat G,K,Z,Y,X,C index. */
void orc_wgrad_at(const orc_problem* p, const double* x, const double* dy, const int64_t* idx, long m,
                  double* out, double* absout)
{
    int o[3];
    out_dims(p, o);
    const int G = p->G, N = p->N, C = p->C, K = p->K;
    const int D = p->in[0], H = p->in[1], W = p->in[2];
    const int Z = p->filt[0], Y = p->filt[1], X = p->filt[2];
    long i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < m; ++i) {
        long r = idx[i];
        const int c = (int)(r % C); r /= C;
        const int xx = (int)(r % X); r /= X;
        const int y = (int)(r % Y); r /= Y;
        const int z = (int)(r % Z); r /= Z;
        const int k = (int)(r % K); r /= K;
        const int g = (int)r;
        double s = 0.0, a = 0.0;
        for (int n = 0; n < N; ++n)
            for (int od = 0; od < o[0]; ++od) {
                const int id = od * p->stride[0] - p->pad_l[0] + z * p->dil[0];
                if (id < 0 || id >= D) continue;
                for (int oh = 0; oh < o[1]; ++oh) {
                    const int ih = oh * p->stride[1] - p->pad_l[1] + y * p->dil[1];
                    if (ih < 0 || ih >= H) continue;
                    for (int ow = 0; ow < o[2]; ++ow) {
                        const int iw = ow * p->stride[2] - p->pad_l[2] + xx * p->dil[2];
                        if (iw < 0 || iw >= W) continue;
                        const long yo = ((((long)n * o[0] + od) * o[1] + oh) * o[2] + ow) * G + g;
                        const long xo = ((((long)n * D + id) * H + ih) * W + iw) * G + g;
                        const double t = dy[yo * K + k] * x[xo * C + c];
                        s += t;
                        a += fabs(t);
                    }
                }
            }
        out[i] = s;
        if (absout) absout[i] = a;
    }
}

/* Forward grouped convolution with the same geometry (used to check the
 * adjoint identity <dW, W'> = <dY, conv_fwd(X, W')>):
 *   y[n,od,oh,ow,g,k] = sum over z,y,x,c of w[g,k,z,y,x,c] * X[n, od*sd-pld+z*dd, ..., g, c]. */
void orc_conv_fwd(const orc_problem* p, const double* x, const double* w, double* yout)
{
    int o[3];
    out_dims(p, o);
    const int G = p->G, N = p->N, C = p->C, K = p->K;
    const int D = p->in[0], H = p->in[1], W = p->in[2];
    const int Z = p->filt[0], Y = p->filt[1], X = p->filt[2];
    long pix;
    const long P = (long)N * o[0] * o[1] * o[2];
#pragma omp parallel for schedule(static)
    for (pix = 0; pix < P; ++pix) {
        long r = pix;
        const int ow = (int)(r % o[2]); r /= o[2];
        const int oh = (int)(r % o[1]); r /= o[1];
        const int od = (int)(r % o[0]); r /= o[0];
        const int n = (int)r;
        for (int g = 0; g < G; ++g)
            for (int k = 0; k < K; ++k) {
                double s = 0.0;
                for (int z = 0; z < Z; ++z) {
                    const int id = od * p->stride[0] - p->pad_l[0] + z * p->dil[0];
                    if (id < 0 || id >= D) continue;
                    for (int y = 0; y < Y; ++y) {
                        const int ih = oh * p->stride[1] - p->pad_l[1] + y * p->dil[1];
                        if (ih < 0 || ih >= H) continue;
                        for (int xx = 0; xx < X; ++xx) {
                            const int iw = ow * p->stride[2] - p->pad_l[2] + xx * p->dil[2];
                            if (iw < 0 || iw >= W) continue;
                            const long xo = ((((long)n * D + id) * H + ih) * W + iw) * G + g;
                            const long wo = ((((long)g * K + k) * Z + z) * Y + y) * X + xx;
                            for (int c = 0; c < C; ++c) s += w[wo * C + c] * x[xo * C + c];
                        }
                    }
                }
                yout[(pix * G + g) * K + k] = s;
            }
    }
}

/* Backward-data (dgrad) of the same grouped convolution, the adjoint of
 * orc_conv_fwd in X: each input position gathers every (output position, tap)
 * pair that reads it,
 *   dX[n,id,ih,iw,g,c] = sum over k, z, y, x with
 *       od = (id + pld - z*dd) / sd, oh = (ih + plh - y*dh) / sh, ow = (iw + plw - x*dw) / sw
 *       integral and inside the output
 *   of dY[n,od,oh,ow,g,k] * W[g,k,z,y,x,c].
 * Also returns A = sum of |dY * W| over the same terms. */
void orc_dgrad(const orc_problem* p, const double* dy, const double* w, double* dx, double* absacc)
{
    int o[3];
    out_dims(p, o);
    const int G = p->G, N = p->N, C = p->C, K = p->K;
    const int D = p->in[0], H = p->in[1], W = p->in[2];
    const int Z = p->filt[0], Y = p->filt[1], X = p->filt[2];
    long pix;
    const long P = (long)N * D * H * W;
#pragma omp parallel for schedule(static)
    for (pix = 0; pix < P; ++pix) {
        long r = pix;
        const int iw = (int)(r % W); r /= W;
        const int ih = (int)(r % H); r /= H;
        const int id = (int)(r % D); r /= D;
        const int n = (int)r;
        for (int g = 0; g < G; ++g)
            for (int c = 0; c < C; ++c) {
                double s = 0.0, a = 0.0;
                for (int z = 0; z < Z; ++z) {
                    const int td = id + p->pad_l[0] - z * p->dil[0];
                    if (td < 0 || td % p->stride[0]) continue;
                    const int od = td / p->stride[0];
                    if (od >= o[0]) continue;
                    for (int y = 0; y < Y; ++y) {
                        const int th = ih + p->pad_l[1] - y * p->dil[1];
                        if (th < 0 || th % p->stride[1]) continue;
                        const int oh = th / p->stride[1];
                        if (oh >= o[1]) continue;
                        for (int xx = 0; xx < X; ++xx) {
                            const int tw = iw + p->pad_l[2] - xx * p->dil[2];
                            if (tw < 0 || tw % p->stride[2]) continue;
                            const int ow = tw / p->stride[2];
                            if (ow >= o[2]) continue;
                            const long yo = ((((long)n * o[0] + od) * o[1] + oh) * o[2] + ow) * G + g;
                            for (int k = 0; k < K; ++k) {
                                const double t = dy[yo * K + k] * w[(((((long)g * K + k) * Z + z) * Y + y) * X + xx) * C + c];
                                s += t;
                                a += fabs(t);
                            }
                        }
                    }
                }
                const long xo = ((pix * G) + g) * C + c;
                dx[xo] = s;
                absacc[xo] = a;
            }
    }
}
