/*
 * conv2d_oracle.c - plain, slow, obviously correct CPU oracle for the training
 * step of one NHWC conv2d layer (conv + bias, optional training-mode batch
 * norm, activation; analytic backward).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code with the CUDA library.
 *
 * Source of every formula: the rl-tools conv2d layer, page
 * "hyperray 0.0.1 .../rl_tools/nn/layers/conv2d/operations_generic.h"
 * (functions `forward`, `evaluate`, `backward_full`). The loops below follow
 * the definitions written there, in double precision, with two-pass batch
 * statistics. Readings of points the page leaves open:
 *   - output size OH = floor((H + 2P - KH)/S) + 1, symmetric zero padding, no
 *     dilation (loop bounds of `forward`);
 *   - cross-correlation, no kernel flip; weights laid out [OC][KH][KW][IC];
 *   - biased variance (divide by n) both for normalisation and for the
 *     running variance, running = (1-m)*running + m*batch (BN branch of
 *     `forward`);
 *   - batch-norm backward uses the mean / inv_std saved by the forward pass
 *     (training branch of `backward_full`);
 *   - activations: identity, ReLU = max(0,v), tanh, sigmoid = 1/(1+e^-v); the
 *     derivative is taken at the activation input, ReLU'(0) = 0.
 *   - dX is overwritten, dW / dBias / dGamma / dBeta are accumulated into
 *     (`backward_full` loads the existing gradients first).
 *   - `bn_eval` selects the pages' evaluation mode of batch norm inside
 *     training (`forward` / `backward_full` with mode::Evaluation).
 *   - norm 2 is layer norm: per-sample statistics over OH*OW*OC of the
 *     stored pre-activations (it keeps no running statistics), per-channel
 *     gamma / beta; mean / inv_std then have N entries.
 *   - norm 3 is group norm (WebGPU page "groupnorm_backward.wgsl"): the OC
 *     channels form `groups` groups of OC/groups consecutive channels;
 *     statistics per (image, group) over OH*OW*OC/groups stored
 *     pre-activations, per-channel gamma / beta, no running statistics;
 *     mean / inv_std have N*groups entries, index n*groups + g.
 *   - the pre-activations are stored in the layer's element type T (`forward`
 *     Phase 1 writes `(T)acc` into `pre_activations`), and the normalisation,
 *     the activation and the backward pass read that stored value. The batch
 *     statistics are taken from the conv output before that rounding (fp32
 *     batch-norm statistics from the accumulator): with a bf16 T, statistics
 *     of the rounded values cannot be reproduced to 1e-5 by any fp32
 *     accumulation, because values near a bf16 rounding midpoint round either
 *     way. The `store` field names T: fp32 (round to nearest) or bf16 (round
 *     to nearest even, through fp32); 0 keeps fp64 (the pure definition).
 * Parallelism (OpenMP) is only over independent output elements; every
 * element is the plain sum its definition states.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t N, H, W, IC, OC, KH, KW, S, P;
    int32_t norm; /* 0 none, 1 batch norm, 2 layer norm, 3 group norm */
    int32_t act;  /* 0 identity, 1 relu, 2 tanh, 3 sigmoid */
    int32_t store; /* element type T of the stored pre-activations: 0 keep fp64, 1 fp32, 2 bf16 */
    int32_t bn_eval; /* batch norm in evaluation mode: running statistics, nothing updated */
    int32_t groups;  /* group norm (norm 3): number of channel groups, dividing OC */
    double eps, momentum;
} oracle_desc;

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Round v to the storage type T of the pre-activations. */
double oracle_store_round(int store, double v) {
    if (store == 1) return (double)(float)v;
    if (store == 2) {
        float f = (float)v;
        uint32_t u;
        memcpy(&u, &f, 4);
        if ((u & 0x7f800000u) != 0x7f800000u) u += 0x7fffu + ((u >> 16) & 1u); /* nearest, ties to even */
        u &= 0xffff0000u;
        memcpy(&f, &u, 4);
        return (double)f;
    }
    return v;
}

static int out_h(const oracle_desc* d) { return (d->H + 2 * d->P - d->KH) / d->S + 1; }
static int out_w(const oracle_desc* d) { return (d->W + 2 * d->P - d->KW) / d->S + 1; }

int oracle_out_hw(const oracle_desc* d, int32_t* OH, int32_t* OW) {
    if (d->H + 2 * d->P < d->KH || d->W + 2 * d->P < d->KW || d->S < 1) return 1;
    *OH = out_h(d);
    *OW = out_w(d);
    return 0;
}

/* activation and its derivative at the activation input (operations_generic.h,
 * `activation<...>` / `d_activation_d_x<...>` call sites in forward/backward) */
double oracle_act(int act, double v) {
    switch (act) {
    case 1: return v > 0.0 ? v : 0.0;
    case 2: return tanh(v);
    case 3: return 1.0 / (1.0 + exp(-v));
    default: return v;
    }
}
double oracle_dact(int act, double v) {
    switch (act) {
    case 1: return v > 0.0 ? 1.0 : 0.0;
    case 2: { double t = tanh(v); return 1.0 - t * t; }
    case 3: { double s = 1.0 / (1.0 + exp(-v)); return s * (1.0 - s); }
    default: return 1.0;
    }
}

#define X_AT(x, n, h, w, c) (x)[(((size_t)(n) * d->H + (h)) * d->W + (w)) * d->IC + (c)]
#define W_AT(w, o, kh, kw, c) (w)[(((size_t)(o) * d->KH + (kh)) * d->KW + (kw)) * d->IC + (c)]

/* One output element of the convolution: bias plus the sum over the taps that
 * fall inside the image (forward, "Phase 1: Compute conv output"). */
double oracle_conv_point(const oracle_desc* d, const double* x, const double* w, const double* b,
                         int n, int oh, int ow, int oc) {
    double acc = b ? b[oc] : 0.0;
    for (int kh = 0; kh < d->KH; kh++) {
        int ihp = oh * d->S + kh;
        if (ihp < d->P || ihp >= d->H + d->P) continue;
        int ih = ihp - d->P;
        for (int kw = 0; kw < d->KW; kw++) {
            int iwp = ow * d->S + kw;
            if (iwp < d->P || iwp >= d->W + d->P) continue;
            int iw = iwp - d->P;
            for (int ic = 0; ic < d->IC; ic++)
                acc += W_AT(w, oc, kh, kw, ic) * X_AT(x, n, ih, iw, ic);
        }
    }
    return acc;
}

/* Ypre = conv(X, W) + b for every output element (forward, Phase 1). */
void oracle_conv_fwd(const oracle_desc* d, const double* x, const double* w, const double* b,
                     double* ypre) {
    const int OH = out_h(d), OW = out_w(d);
    const long rows = (long)d->N * OH;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; r++) {
        int n = (int)(r / OH), oh = (int)(r % OH);
        for (int ow = 0; ow < OW; ow++)
            for (int oc = 0; oc < d->OC; oc++)
                ypre[(((size_t)n * OH + oh) * OW + ow) * d->OC + oc] =
                    oracle_conv_point(d, x, w, b, n, oh, ow, oc);
    }
}

/* Per-channel batch mean and biased variance over N*OH*OW, two passes
 * (forward, BN training branch). */
void oracle_bn_batch_stats(const oracle_desc* d, const double* ypre, double* mean, double* var) {
    const long npix = (long)d->N * out_h(d) * out_w(d);
    const int C = d->OC;
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        double m = 0.0;
        for (long p = 0; p < npix; p++) m += ypre[(size_t)p * C + c];
        m /= (double)npix;
        double v = 0.0;
        for (long p = 0; p < npix; p++) {
            double t = ypre[(size_t)p * C + c] - m;
            v += t * t;
        }
        mean[c] = m;
        var[c] = v / (double)npix;
    }
}

/* Per-sample layer-norm statistics over all OH*OW*OC elements of image n, two passes, biased variance
 * (`forward` / `evaluate`, LAYER_NORM branch). */
void oracle_ln_stats(const oracle_desc* d, const double* ypre, double* mean, double* inv_std) {
    const long per = (long)out_h(d) * out_w(d) * d->OC;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < d->N; n++) {
        const double* v = ypre + (size_t)n * per;
        double m = 0.0;
        for (long i = 0; i < per; i++) m += v[i];
        m /= (double)per;
        double var = 0.0;
        for (long i = 0; i < per; i++) var += (v[i] - m) * (v[i] - m);
        var /= (double)per;
        mean[n] = m;
        inv_std[n] = 1.0 / sqrt(var + d->eps);
    }
}

/* Group-norm statistics per (image n, group g) over the OH*OW*(OC/groups) stored values of the
 * group's channels, two passes, biased variance ("groupnorm_backward.wgsl" Phase 1 recomputes the same
 * mean and variance from its input; its E[x^2] - mean^2 form is not reproduced). */
void oracle_gn_stats(const oracle_desc* d, const double* ypre, double* mean, double* inv_std) {
    const long hw = (long)out_h(d) * out_w(d);
    const int C = d->OC, G = d->groups, cpg = C / G;
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < d->N; n++)
        for (int g = 0; g < G; g++) {
            const double* v = ypre + (size_t)n * hw * C;
            double m = 0.0;
            for (long p = 0; p < hw; p++)
                for (int c = g * cpg; c < (g + 1) * cpg; c++) m += v[p * C + c];
            m /= (double)(hw * cpg);
            double var = 0.0;
            for (long p = 0; p < hw; p++)
                for (int c = g * cpg; c < (g + 1) * cpg; c++) var += (v[p * C + c] - m) * (v[p * C + c] - m);
            var /= (double)(hw * cpg);
            mean[n * G + g] = m;
            inv_std[n * G + g] = 1.0 / sqrt(var + d->eps);
        }
}

/* Training forward: Ypre, batch stats, running-stat EMA, normalise + affine +
 * activation (forward, all phases). rm / rv are updated in place. */
void oracle_fwd_train(const oracle_desc* d, const double* x, const double* w, const double* b,
                      const double* gamma, const double* beta, double* rm, double* rv,
                      double* ypre, double* mean, double* inv_std, double* y) {
    const long npix = (long)d->N * out_h(d) * out_w(d);
    const int C = d->OC;
    oracle_conv_fwd(d, x, w, b, ypre);
    double* var = NULL;
    if (d->norm == 1 && d->bn_eval) {
        /* `forward` with mode::Evaluation: the cached statistics are the running ones, no update */
        for (int c = 0; c < C; c++) {
            mean[c] = rm[c];
            inv_std[c] = 1.0 / sqrt(rv[c] + d->eps);
        }
    } else if (d->norm == 1) {
        /* batch statistics of the conv output before it is stored in T */
        var = (double*)malloc(sizeof(double) * C);
        oracle_bn_batch_stats(d, ypre, mean, var);
    }
    if (d->store)
        for (long i = 0; i < npix * C; i++) ypre[i] = oracle_store_round(d->store, ypre[i]);
    if (d->norm == 0) {
        for (long i = 0; i < npix * C; i++) y[i] = oracle_act(d->act, ypre[i]);
        return;
    }
    if (d->norm == 3) {
        /* group norm: statistics of the stored pre-activations per (image, group), then normalise,
         * per-channel affine and activation */
        oracle_gn_stats(d, ypre, mean, inv_std);
        const long per = npix / d->N;
        const int cpg = C / d->groups;
#pragma omp parallel for schedule(static)
        for (long p = 0; p < npix; p++) {
            const int n = (int)(p / per);
            for (int c = 0; c < C; c++) {
                size_t i = (size_t)p * C + c;
                const int s = n * d->groups + c / cpg;
                double z = (ypre[i] - mean[s]) * inv_std[s];
                y[i] = oracle_act(d->act, gamma[c] * z + beta[c]);
            }
        }
        return;
    }
    if (d->norm == 2) {
        /* layer norm (`forward`, LAYER_NORM branch): per-sample two-pass statistics over OH*OW*OC of
         * the stored pre-activations; mean / inv_std have N entries; per-channel gamma, beta */
        oracle_ln_stats(d, ypre, mean, inv_std);
        const long per = npix / d->N;
#pragma omp parallel for schedule(static)
        for (long p = 0; p < npix; p++) {
            const int n = (int)(p / per);
            for (int c = 0; c < C; c++) {
                size_t i = (size_t)p * C + c;
                double z = (ypre[i] - mean[n]) * inv_std[n];
                y[i] = oracle_act(d->act, gamma[c] * z + beta[c]);
            }
        }
        return;
    }
    if (!d->bn_eval) {
        for (int c = 0; c < C; c++) {
            inv_std[c] = 1.0 / sqrt(var[c] + d->eps);
            rm[c] = (1.0 - d->momentum) * rm[c] + d->momentum * mean[c];
            rv[c] = (1.0 - d->momentum) * rv[c] + d->momentum * var[c];
        }
        free(var);
    }
#pragma omp parallel for schedule(static)
    for (long p = 0; p < npix; p++)
        for (int c = 0; c < C; c++) {
            size_t i = (size_t)p * C + c;
            double z = (ypre[i] - mean[c]) * inv_std[c];
            y[i] = oracle_act(d->act, gamma[c] * z + beta[c]);
        }
}

/* Inference forward: conv + bias, then (BN) normalise with the running
 * statistics, then activation; no state is written (`evaluate`). */
void oracle_fwd_infer(const oracle_desc* d, const double* x, const double* w, const double* b,
                      const double* gamma, const double* beta, const double* rm,
                      const double* rv, double* y) {
    const long npix = (long)d->N * out_h(d) * out_w(d);
    const int C = d->OC;
    oracle_conv_fwd(d, x, w, b, y);
#pragma omp parallel for schedule(static)
    for (long p = 0; p < npix; p++)
        for (int c = 0; c < C; c++) {
            size_t i = (size_t)p * C + c;
            double v = y[i];
            if (d->norm >= 2) continue; /* layer / group norm: below, per sample */
            if (d->norm == 1) {
                /* `evaluate` BN branch: the conv output is stored as T first */
                v = oracle_store_round(d->store, v);
                double is = 1.0 / sqrt(rv[c] + d->eps);
                v = gamma[c] * ((v - rm[c]) * is) + beta[c];
            }
            y[i] = oracle_act(d->act, v);
        }
    if (d->norm == 2) {
        /* `evaluate`, LAYER_NORM branch: the conv output is stored as T, per-sample statistics on the fly */
        for (long i = 0; i < npix * C; i++) y[i] = oracle_store_round(d->store, y[i]);
        double* m = (double*)malloc(sizeof(double) * d->N);
        double* is = (double*)malloc(sizeof(double) * d->N);
        oracle_ln_stats(d, y, m, is);
        const long per = npix / d->N;
        for (long p = 0; p < npix; p++) {
            const int n = (int)(p / per);
            for (int c = 0; c < C; c++) {
                size_t i = (size_t)p * C + c;
                y[i] = oracle_act(d->act, gamma[c] * ((y[i] - m[n]) * is[n]) + beta[c]);
            }
        }
        free(m);
        free(is);
    }
    if (d->norm == 3) {
        /* group norm at inference: the same per-(image, group) statistics of the stored conv output */
        for (long i = 0; i < npix * C; i++) y[i] = oracle_store_round(d->store, y[i]);
        const int G = d->groups, cpg = C / G;
        double* m = (double*)malloc(sizeof(double) * d->N * G);
        double* is = (double*)malloc(sizeof(double) * d->N * G);
        oracle_gn_stats(d, y, m, is);
        const long per = npix / d->N;
        for (long p = 0; p < npix; p++) {
            const int n = (int)(p / per);
            for (int c = 0; c < C; c++) {
                size_t i = (size_t)p * C + c;
                const int s = n * G + c / cpg;
                y[i] = oracle_act(d->act, gamma[c] * ((y[i] - m[s]) * is[s]) + beta[c]);
            }
        }
        free(m);
        free(is);
    }
}

/* Gradient at the conv output (backward_full, before the scatter loops):
 *   none: d_conv = act'(Ypre) * dY
 *   batch norm (training): z = (Ypre-mean)*inv_std, bn = gamma*z+beta,
 *     d_norm = act'(bn)*dY, dgamma += sum d_norm*z, dbeta += sum d_norm,
 *     d_conv = inv_std/n * (n*dz - sum dz - z*sum dz*z), dz = gamma*d_norm.
 * dgamma / dbeta may be NULL (not accumulated). */
void oracle_dconv(const oracle_desc* d, const double* gamma, const double* beta,
                  const double* ypre, const double* mean, const double* inv_std,
                  const double* dy, double* dconv, double* dgamma, double* dbeta) {
    const long npix = (long)d->N * out_h(d) * out_w(d);
    const int C = d->OC;
    if (d->norm == 0) {
#pragma omp parallel for schedule(static)
        for (long i = 0; i < npix * C; i++) dconv[i] = oracle_dact(d->act, ypre[i]) * dy[i];
        return;
    }
    if (d->norm == 3) {
        /* group norm backward ("groupnorm_backward.wgsl", Phases 2 and 3, with the activation derivative
         * in front and the per-channel dgamma / dbeta sums the shader leaves out): with w = gamma[c] and
         * g_out = d_norm the gradient at the norm output, per (image, group) of n_g elements
         *   term1 = sum g_out*w,   term2 = sum g_out*w*(x - mean) * inv_std^2,
         *   d_conv = inv_std * (g_out*w - (term1 + (x - mean)*term2) / n_g). */
        const int G = d->groups, cpg = C / G;
        const long per = npix / d->N;
        const double ng = (double)(per * cpg);
        double* t1 = (double*)calloc((size_t)d->N * G, sizeof(double));
        double* t2 = (double*)calloc((size_t)d->N * G, sizeof(double));
        for (long p = 0; p < npix; p++) {
            const int n = (int)(p / per);
            for (int c = 0; c < C; c++) {
                size_t i = (size_t)p * C + c;
                const int s = n * G + c / cpg;
                const double xm = ypre[i] - mean[s];
                const double z = xm * inv_std[s];
                const double gout = oracle_dact(d->act, gamma[c] * z + beta[c]) * dy[i];
                if (dgamma) dgamma[c] += gout * z;
                if (dbeta) dbeta[c] += gout;
                t1[s] += gout * gamma[c];
                t2[s] += gout * gamma[c] * xm;
            }
        }
        for (int s2 = 0; s2 < d->N * G; s2++) t2[s2] *= inv_std[s2] * inv_std[s2];
#pragma omp parallel for schedule(static)
        for (long p = 0; p < npix; p++) {
            const int n = (int)(p / per);
            for (int c = 0; c < C; c++) {
                size_t i = (size_t)p * C + c;
                const int s = n * G + c / cpg;
                const double xm = ypre[i] - mean[s];
                const double gout = oracle_dact(d->act, gamma[c] * (xm * inv_std[s]) + beta[c]) * dy[i];
                dconv[i] = inv_std[s] * (gout * gamma[c] - (t1[s] + xm * t2[s]) / ng);
            }
        }
        free(t1);
        free(t2);
        return;
    }
    if (d->norm == 2) {
        /* `backward_full` training branch with NORM_DIM = batch: the sums of dz and dz*z run over the
         * OH*OW*OC elements of each image (M of them); dgamma / dbeta stay per channel */
        const long per_pix = npix / d->N;
        const double M = (double)(per_pix * C);
        double* sdz = (double*)calloc(d->N, sizeof(double));
        double* sdzz = (double*)calloc(d->N, sizeof(double));
        for (int n = 0; n < d->N; n++)
            for (long p = n * per_pix; p < (n + 1) * per_pix; p++)
                for (int c = 0; c < C; c++) {
                    size_t i = (size_t)p * C + c;
                    double z = (ypre[i] - mean[n]) * inv_std[n];
                    double dn = oracle_dact(d->act, gamma[c] * z + beta[c]) * dy[i];
                    double dz = dn * gamma[c];
                    if (dgamma) dgamma[c] += dn * z;
                    if (dbeta) dbeta[c] += dn;
                    sdz[n] += dz;
                    sdzz[n] += dz * z;
                }
#pragma omp parallel for schedule(static)
        for (long p = 0; p < npix; p++) {
            const int n = (int)(p / per_pix);
            for (int c = 0; c < C; c++) {
                size_t i = (size_t)p * C + c;
                double z = (ypre[i] - mean[n]) * inv_std[n];
                double dz = oracle_dact(d->act, gamma[c] * z + beta[c]) * dy[i] * gamma[c];
                dconv[i] = inv_std[n] * (1.0 / M) * (M * dz - sdz[n] - z * sdzz[n]);
            }
        }
        free(sdz);
        free(sdzz);
        return;
    }
    if (d->bn_eval) {
        /* `backward_full` evaluation branch: frozen statistics, d_conv = d_norm * gamma * inv_std */
#pragma omp parallel for schedule(static)
        for (int c = 0; c < C; c++) {
            double s_g = 0.0, s_b = 0.0;
            for (long p = 0; p < npix; p++) {
                size_t i = (size_t)p * C + c;
                double z = (ypre[i] - mean[c]) * inv_std[c];
                double dn = oracle_dact(d->act, gamma[c] * z + beta[c]) * dy[i];
                s_g += dn * z;
                s_b += dn;
                dconv[i] = dn * gamma[c] * inv_std[c];
            }
            if (dgamma) dgamma[c] += s_g;
            if (dbeta) dbeta[c] += s_b;
        }
        return;
    }
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        double s_dz = 0.0, s_dzz = 0.0, s_g = 0.0, s_b = 0.0;
        for (long p = 0; p < npix; p++) {
            size_t i = (size_t)p * C + c;
            double z = (ypre[i] - mean[c]) * inv_std[c];
            double dn = oracle_dact(d->act, gamma[c] * z + beta[c]) * dy[i];
            double dz = dn * gamma[c];
            s_g += dn * z;
            s_b += dn;
            s_dz += dz;
            s_dzz += dz * z;
        }
        if (dgamma) dgamma[c] += s_g;
        if (dbeta) dbeta[c] += s_b;
        const double n = (double)npix;
        for (long p = 0; p < npix; p++) {
            size_t i = (size_t)p * C + c;
            double z = (ypre[i] - mean[c]) * inv_std[c];
            double dn = oracle_dact(d->act, gamma[c] * z + beta[c]) * dy[i];
            double dz = dn * gamma[c];
            dconv[i] = inv_std[c] * (1.0 / n) * (n * dz - s_dz - z * s_dzz);
        }
    }
}

/* dBias[oc] += sum over pixels of d_conv (backward_full, `d_biases_acc`). */
void oracle_dbias(const oracle_desc* d, const double* dconv, double* db) {
    const long npix = (long)d->N * out_h(d) * out_w(d);
    for (int c = 0; c < d->OC; c++) {
        double s = 0.0;
        for (long p = 0; p < npix; p++) s += dconv[(size_t)p * d->OC + c];
        db[c] += s;
    }
}

/* dX[n,ih,iw,ic] = sum over (kh,kw,oc) with ih = oh*S+kh-P, iw = ow*S+kw-P of
 * W[oc,kh,kw,ic] * d_conv[n,oh,ow,oc]; overwritten (backward_full,
 * `d_input_acc`, written per input element instead of scattered). */
void oracle_dgrad(const oracle_desc* d, const double* dconv, const double* w, double* dx) {
    const int OH = out_h(d), OW = out_w(d);
    const long rows = (long)d->N * d->H;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; r++) {
        int n = (int)(r / d->H), ih = (int)(r % d->H);
        for (int iw = 0; iw < d->W; iw++)
            for (int ic = 0; ic < d->IC; ic++) {
                double acc = 0.0;
                for (int kh = 0; kh < d->KH; kh++) {
                    int th = ih + d->P - kh;
                    if (th < 0 || th % d->S) continue;
                    int oh = th / d->S;
                    if (oh >= OH) continue;
                    for (int kw = 0; kw < d->KW; kw++) {
                        int tw = iw + d->P - kw;
                        if (tw < 0 || tw % d->S) continue;
                        int ow = tw / d->S;
                        if (ow >= OW) continue;
                        const double* g = dconv + (((size_t)n * OH + oh) * OW + ow) * d->OC;
                        for (int oc = 0; oc < d->OC; oc++) acc += W_AT(w, oc, kh, kw, ic) * g[oc];
                    }
                }
                X_AT(dx, n, ih, iw, ic) = acc;
            }
    }
}

/* One input-gradient element (the sum of `oracle_dgrad` for one (n,ih,iw,ic)). */
double oracle_dgrad_point(const oracle_desc* d, const double* dconv, const double* w, int n, int ih, int iw,
                          int ic) {
    const int OH = out_h(d), OW = out_w(d);
    double acc = 0.0;
    for (int kh = 0; kh < d->KH; kh++) {
        int th = ih + d->P - kh;
        if (th < 0 || th % d->S) continue;
        int oh = th / d->S;
        if (oh >= OH) continue;
        for (int kw = 0; kw < d->KW; kw++) {
            int tw = iw + d->P - kw;
            if (tw < 0 || tw % d->S) continue;
            int ow = tw / d->S;
            if (ow >= OW) continue;
            const double* g = dconv + (((size_t)n * OH + oh) * OW + ow) * d->OC;
            for (int oc = 0; oc < d->OC; oc++) acc += W_AT(w, oc, kh, kw, ic) * g[oc];
        }
    }
    return acc;
}

/* One weight-gradient element, sum over batch and output pixels of
 * d_conv[n,oh,ow,oc] * X[n, oh*S+kh-P, ow*S+kw-P, ic] (backward_full,
 * `d_weights_acc`); not accumulated into anything. */
double oracle_wgrad_point(const oracle_desc* d, const double* x, const double* dconv,
                          int oc, int kh, int kw, int ic) {
    const int OH = out_h(d), OW = out_w(d);
    double acc = 0.0;
    for (int n = 0; n < d->N; n++)
        for (int oh = 0; oh < OH; oh++) {
            int ihp = oh * d->S + kh;
            if (ihp < d->P || ihp >= d->H + d->P) continue;
            for (int ow = 0; ow < OW; ow++) {
                int iwp = ow * d->S + kw;
                if (iwp < d->P || iwp >= d->W + d->P) continue;
                acc += dconv[(((size_t)n * OH + oh) * OW + ow) * d->OC + oc] *
                       X_AT(x, n, ihp - d->P, iwp - d->P, ic);
            }
        }
    return acc;
}

/* dW += weight gradient, every element. */
void oracle_wgrad(const oracle_desc* d, const double* x, const double* dconv, double* dw) {
    const long total = (long)d->OC * d->KH * d->KW;
#pragma omp parallel for schedule(dynamic)
    for (long t = 0; t < total; t++) {
        int oc = (int)(t / (d->KH * d->KW));
        int kh = (int)((t / d->KW) % d->KH);
        int kw = (int)(t % d->KW);
        for (int ic = 0; ic < d->IC; ic++)
            W_AT(dw, oc, kh, kw, ic) += oracle_wgrad_point(d, x, dconv, oc, kh, kw, ic);
    }
}

/* Full backward (backward_full): d_conv, then dBias, dX (if dx != NULL,
 * overwritten), dW (if dw != NULL, accumulated). dconv_out, if given,
 * receives d_conv. */
void oracle_bwd(const oracle_desc* d, const double* x, const double* w, const double* gamma,
                const double* beta, const double* ypre, const double* mean,
                const double* inv_std, const double* dy, double* dx, double* dw, double* db,
                double* dgamma, double* dbeta, double* dconv_out) {
    const long ny = (long)d->N * out_h(d) * out_w(d) * d->OC;
    double* dconv = dconv_out ? dconv_out : (double*)malloc(sizeof(double) * (size_t)ny);
    oracle_dconv(d, gamma, beta, ypre, mean, inv_std, dy, dconv, dgamma, dbeta);
    if (db) oracle_dbias(d, dconv, db);
    if (dx) oracle_dgrad(d, dconv, w, dx);
    if (dw) oracle_wgrad(d, x, dconv, dw);
    if (!dconv_out) free(dconv);
}
