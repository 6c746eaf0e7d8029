/*
 * Plain CPU oracle of the streaming codec-to-waveform decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py load this code.  It shares nothing with the CUDA
 * library: not a header, not a helper, not a table.  The two meet only in the
 * flat fp32 weight blob and its tensor order, which both read independently.
 *
 * What it computes (vllm-omni "Edge TTS design", section 1.3, and the
 * readings listed in the design notes):
 *   RVQ embedding sum -> causal Conv1d -> L x pre-norm sliding-window
 *   transformer -> final RMSNorm -> two causal ConvTranspose1d (k=4, s=2) ->
 *   4 BigVGAN stages [Snake -> causal ConvT(k=2s, s) -> MRF of Snake-dilated
 *   residual convs] -> Snake -> causal conv -> tanh.
 *
 * Arithmetic: tensors are stored in fp32 (the page gives the decoder as fp32).
 * Every dot product, norm, softmax and transcendental is evaluated in double
 * in a fixed order and rounded to fp32 once per op output.  The one exception
 * is the codebook sum, which is an fp32 running sum with q ascending, so that
 * its bits are defined exactly.  Products and sums are kept separate
 * (built with -ffp-contract=off): "double products, double sums, in the order
 * written".
 *
 * Streaming: each causal op concatenates its carried history rows in front of
 * the chunk, computes the chunk rows, and keeps the last rows of that
 * concatenation as the new history (blixt/phonon "Speed" item 7: each stage's
 * left context; the attention keeps the keys and values of the last W-1
 * positions).  Every output element therefore sees exactly the same operation
 * sequence whatever the chunking, and chunked decoding equals a full decode
 * bit for bit.
 *
 * Latent-input variant (blixt/phonon "Weights" and "Speed" item 7: the
 * codec's latents are denormalised, projected by a 1x1 convolution without
 * bias and upsampled x16 by a depthwise transposed convolution; the codec
 * transformer then runs at the upsampled rate, 200 Hz, with a 251-position
 * window): in place of the codebook sum and the pre-conv, latent frames
 * [n][L] go through z = x sigma + mu, p = Wp z, and a causal depthwise
 * ConvTranspose1d (kernel 2 s, stride s = tf_up, its own taps per channel),
 * giving n s rows of d channels; the transformer's positions and window count
 * those rows.  The oracle computes the three steps one after the other, as
 * written; the GPU folds the projection into the upsampling weights.
 *
 * Loops parallelise over output rows with OpenMP; within a row, the sum over
 * (tap, input channel) runs in ascending order for every output channel, with
 * the output channels as the innermost (vectorisable) loop.  That order is
 * the definition's order for each individual output.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OC_EXPORT __attribute__((visibility("default")))
#define OC_ERR_BAD_CODE 1u

typedef struct oc_config {
    int32_t Q, V, E, pre_k, d, heads, ffn, layers, window;
    int32_t n_up, up_k, up_s;
    int32_t up_ch[4];
    int32_t n_stages;
    int32_t strides[8];
    int32_t ch[8];
    int32_t n_rb;
    int32_t rb_k[4];
    int32_t n_dil;
    int32_t dil[4];
    int32_t final_k;
    float rms_eps;
    int32_t latent_dim;   /* 0: RVQ code input; L > 0: latent frames of L channels */
    int32_t tf_up;        /* latent input: depthwise upsampling stride before the transformer */
} oc_config;

/* ------------------------------------------------------------------ ops -- */

/* Snake, x + sin(alpha x)^2 / alpha, per channel; double, rounded to fp32. */
static void snake_rows(const float* x, int64_t rows, int C, const float* alpha, float* y)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++)
        for (int c = 0; c < C; c++) {
            double a = alpha[c], v = x[r * C + c];
            double s = sin(a * v);
            y[r * C + c] = (float)(v + s * s / a);
        }
}

/* Weight transposes: the stored PyTorch layouts to [tap][in][out]. */
static float* conv_w_t(const float* w, int Cout, int Cin, int k)
{   /* w[co][ci][j] -> t[j][ci][co] */
    float* t = (float*)malloc(sizeof(float) * (size_t)Cout * Cin * k);
    for (int co = 0; co < Cout; co++)
        for (int ci = 0; ci < Cin; ci++)
            for (int j = 0; j < k; j++)
                t[((size_t)j * Cin + ci) * Cout + co] = w[((size_t)co * Cin + ci) * k + j];
    return t;
}

static float* convt_w_t(const float* w, int Cin, int Cout, int k)
{   /* w[ci][co][j] -> t[j][ci][co] */
    float* t = (float*)malloc(sizeof(float) * (size_t)Cout * Cin * k);
    for (int ci = 0; ci < Cin; ci++)
        for (int co = 0; co < Cout; co++)
            for (int j = 0; j < k; j++)
                t[((size_t)j * Cin + ci) * Cout + co] = w[((size_t)ci * Cout + co) * k + j];
    return t;
}

static float* linear_w_t(const float* w, int Cout, int Cin)
{   /* w[o][i] -> t[i][o] */
    float* t = (float*)malloc(sizeof(float) * (size_t)Cout * Cin);
    for (int o = 0; o < Cout; o++)
        for (int i = 0; i < Cin; i++)
            t[(size_t)i * Cout + o] = w[(size_t)o * Cin + i];
    return t;
}

/*
 * Causal dilated Conv1d over a chunk: a holds H + T rows [row][Cin], the
 * first H = (k-1)*dil being history.  For t in [0, T):
 *   y[t][co] = (res[t][co]) + b[co] + sum_{j=0}^{k-1} sum_ci W[co][ci][j] a[H + t - (k-1-j) dil][ci]
 * wt is W transposed to [j][ci][co].
 */
static void conv_core(const float* a, int T, int Cin, const float* wt, const float* b,
                      int Cout, int k, int dil, const float* res, float* y)
{
    const int H = (k - 1) * dil;
    #pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)Cout);
        #pragma omp for schedule(static)
        for (int t = 0; t < T; t++) {
            for (int co = 0; co < Cout; co++) acc[co] = 0.0;
            for (int j = 0; j < k; j++) {
                const float* xr = a + (size_t)(H + t - (k - 1 - j) * dil) * Cin;
                const float* wj = wt + (size_t)j * Cin * Cout;
                for (int ci = 0; ci < Cin; ci++) {
                    const double xv = xr[ci];
                    const float* w = wj + (size_t)ci * Cout;
                    for (int co = 0; co < Cout; co++) acc[co] += (double)w[co] * xv;
                }
            }
            for (int co = 0; co < Cout; co++) {
                double v = acc[co] + (double)b[co];
                if (res) v += (double)res[(size_t)t * Cout + co];
                y[(size_t)t * Cout + co] = (float)v;
            }
        }
        free(acc);
    }
}

/*
 * Causal ConvTranspose1d with kernel 2s and stride s over a chunk: a holds
 * 1 + T rows, the first being the previous chunk's last input row.  Output row
 * m = n s + p receives the two inputs whose scatter reaches it:
 *   y[n s + p][co] = b[co] + sum_ci W[ci][co][p + s] a[n-1][ci] + sum_ci W[ci][co][p] a[n][ci]
 * i.e. conv_transpose1d with the last k - s outputs left for the next chunk.
 * wt is W transposed to [j][ci][co].
 */
static void convt_core(const float* a, int T, int Cin, const float* wt, const float* b,
                       int Cout, int s, float* y)
{
    #pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)Cout);
        #pragma omp for schedule(static)
        for (int64_t m = 0; m < (int64_t)T * s; m++) {
            const int n = (int)(m / s), p = (int)(m % s);
            for (int co = 0; co < Cout; co++) acc[co] = 0.0;
            const float* prev = a + (size_t)n * Cin;          /* a[n-1] */
            const float* cur = a + (size_t)(n + 1) * Cin;     /* a[n] */
            const float* w1 = wt + (size_t)(p + s) * Cin * Cout;
            const float* w0 = wt + (size_t)p * Cin * Cout;
            for (int ci = 0; ci < Cin; ci++) {
                const double xv = prev[ci];
                const float* w = w1 + (size_t)ci * Cout;
                for (int co = 0; co < Cout; co++) acc[co] += (double)w[co] * xv;
            }
            for (int ci = 0; ci < Cin; ci++) {
                const double xv = cur[ci];
                const float* w = w0 + (size_t)ci * Cout;
                for (int co = 0; co < Cout; co++) acc[co] += (double)w[co] * xv;
            }
            for (int co = 0; co < Cout; co++)
                y[(size_t)m * Cout + co] = (float)(acc[co] + (double)b[co]);
        }
        free(acc);
    }
}

/*
 * Causal depthwise ConvTranspose1d, kernel 2s, stride s: a holds 1 + T rows
 * of C channels, the first being the previous chunk's last input row; each
 * channel has its own taps u[c][0 .. 2s-1] (PyTorch ConvTranspose1d with
 * groups = C, weight [C][1][2s]):
 *   y[n s + p][c] = b[c] + u[c][p + s] a[n-1][c] + u[c][p] a[n][c].
 */
static void dwconvt_core(const float* a, int T, int C, const float* u, const float* b, int s, float* y)
{
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < (int64_t)T * s; m++) {
        const int n = (int)(m / s), p = (int)(m % s);
        const float* prev = a + (size_t)n * C;
        const float* cur = a + (size_t)(n + 1) * C;
        for (int c = 0; c < C; c++) {
            double v = (double)u[(size_t)c * 2 * s + p + s] * (double)prev[c];
            v += (double)u[(size_t)c * 2 * s + p] * (double)cur[c];
            y[(size_t)m * C + c] = (float)(v + (double)b[c]);
        }
    }
}

/* y[t][o] = (res[t][o]) + sum_i W[o][i] x[t][i]; wt = W^T [i][o]. */
static void linear_core(const float* x, int T, int Cin, const float* wt, int Cout,
                        const float* res, float* y)
{
    #pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)Cout);
        #pragma omp for schedule(static)
        for (int t = 0; t < T; t++) {
            for (int o = 0; o < Cout; o++) acc[o] = 0.0;
            const float* xr = x + (size_t)t * Cin;
            for (int i = 0; i < Cin; i++) {
                const double xv = xr[i];
                const float* w = wt + (size_t)i * Cout;
                for (int o = 0; o < Cout; o++) acc[o] += (double)w[o] * xv;
            }
            for (int o = 0; o < Cout; o++) {
                double v = acc[o];
                if (res) v += (double)res[(size_t)t * Cout + o];
                y[(size_t)t * Cout + o] = (float)v;
            }
        }
        free(acc);
    }
}

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g. */
static void rms_norm_core(const float* x, int T, int d, const float* g, float eps, float* y)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        const float* xr = x + (size_t)t * d;
        double ss = 0.0;
        for (int c = 0; c < d; c++) ss += (double)xr[c] * (double)xr[c];
        const double r = 1.0 / sqrt(ss / d + (double)eps);
        for (int c = 0; c < d; c++) y[(size_t)t * d + c] = (float)((double)xr[c] * r * (double)g[c]);
    }
}

/* GELU, erf form: 0.5 x (1 + erf(x / sqrt 2)). */
static void gelu_core(const float* x, int64_t n, float* y)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        double v = x[i];
        y[i] = (float)(0.5 * v * (1.0 + erf(v / sqrt(2.0))));
    }
}

/*
 * Sliding-window attention over a chunk.  q is [T][d]; k and v hold
 * Hk + T rows, the first Hk being carried keys/values of the previous
 * positions, of which the rows before index `first` do not exist (positions
 * before the stream start).  Query t sits at row Hk + t and attends rows
 * i with Hk + t - window < i <= Hk + t and i >= first: window keys,
 * itself included.  Per head: softmax(q k^T / sqrt(dh)) v, max-subtracted.
 */
static void swa_core(const float* q, const float* k, const float* v, int T, int Hk, int first,
                     int d, int heads, int window, float* o)
{
    const int dh = d / heads;
    const double scale = 1.0 / sqrt((double)dh);
    #pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)window);
        double* acc = (double*)malloc(sizeof(double) * (size_t)dh);
        #pragma omp for schedule(static) collapse(2)
        for (int t = 0; t < T; t++)
            for (int h = 0; h < heads; h++) {
                const int qi = Hk + t;
                int lo = qi - window + 1;
                if (lo < first) lo = first;
                const float* qr = q + (size_t)t * d + h * dh;
                double m = -INFINITY;
                for (int i = lo; i <= qi; i++) {
                    const float* kr = k + (size_t)i * d + h * dh;
                    double dot = 0.0;
                    for (int c = 0; c < dh; c++) dot += (double)qr[c] * (double)kr[c];
                    s[i - lo] = dot * scale;
                    if (s[i - lo] > m) m = s[i - lo];
                }
                double z = 0.0;
                for (int i = lo; i <= qi; i++) { s[i - lo] = exp(s[i - lo] - m); z += s[i - lo]; }
                for (int c = 0; c < dh; c++) acc[c] = 0.0;
                for (int i = lo; i <= qi; i++) {
                    const float* vr = v + (size_t)i * d + h * dh;
                    const double p = s[i - lo];
                    for (int c = 0; c < dh; c++) acc[c] += p * (double)vr[c];
                }
                for (int c = 0; c < dh; c++) o[(size_t)t * d + h * dh + c] = (float)(acc[c] / z);
            }
        free(s);
        free(acc);
    }
}

/* Codebook sum, fp32 running sum with q ascending; an out-of-range code
 * zeroes the whole row and raises the bad-code bit. */
static uint32_t rvq_core(const float* const* cb, int Q, int V, int E, const int32_t* codes,
                         int64_t ld, int T, float* e)
{
    uint32_t err = 0;
    for (int t = 0; t < T; t++) {
        int bad = 0;
        for (int q = 0; q < Q; q++) {
            int32_t c = codes[(size_t)q * ld + t];
            if (c < 0 || c >= V) bad = 1;
        }
        float* row = e + (size_t)t * E;
        if (bad) {
            for (int c = 0; c < E; c++) row[c] = 0.0f;
            err |= OC_ERR_BAD_CODE;
            continue;
        }
        for (int c = 0; c < E; c++) {
            float acc = 0.0f;
            for (int q = 0; q < Q; q++) acc += cb[q][(size_t)codes[(size_t)q * ld + t] * E + c];
            row[c] = acc;
        }
    }
    return err;
}

/* ---------------------------------------------------- exported single ops -- */
/* Op-level entry points take PyTorch weight layouts; tests pin each one. */

OC_EXPORT void oc_op_snake(const float* x, int64_t rows, int C, const float* alpha, float* y)
{
    snake_rows(x, rows, C, alpha, y);
}

/* x: [(k-1)*dil + T][Cin] (history first); w: [Cout][Cin][k]. alpha may be NULL. */
OC_EXPORT void oc_op_causal_conv(const float* x, int T, int Cin, const float* w, const float* b,
                                 int Cout, int k, int dil, const float* alpha, const float* res,
                                 float* y)
{
    const int H = (k - 1) * dil;
    float* wt = conv_w_t(w, Cout, Cin, k);
    const float* a = x;
    float* tmp = NULL;
    if (alpha) {
        tmp = (float*)malloc(sizeof(float) * (size_t)(H + T) * Cin);
        snake_rows(x, H + T, Cin, alpha, tmp);
        a = tmp;
    }
    conv_core(a, T, Cin, wt, b, Cout, k, dil, res, y);
    free(tmp);
    free(wt);
}

/* x: [1 + T][Cin] (history row first); w: [Cin][Cout][2s]. */
OC_EXPORT void oc_op_causal_conv_t(const float* x, int T, int Cin, const float* w, const float* b,
                                   int Cout, int s, const float* alpha, float* y)
{
    float* wt = convt_w_t(w, Cin, Cout, 2 * s);
    const float* a = x;
    float* tmp = NULL;
    if (alpha) {
        tmp = (float*)malloc(sizeof(float) * (size_t)(1 + T) * Cin);
        snake_rows(x, 1 + T, Cin, alpha, tmp);
        a = tmp;
    }
    convt_core(a, T, Cin, wt, b, Cout, s, y);
    free(tmp);
    free(wt);
}

/* x: [1 + T][C] (history row first); u: [C][1][2s]. */
OC_EXPORT void oc_op_dw_conv_t(const float* x, int T, int C, const float* u, const float* b, int s, float* y)
{
    dwconvt_core(x, T, C, u, b, s, y);
}

/* w: [Cout][Cin]. */
OC_EXPORT void oc_op_linear(const float* x, int T, int Cin, const float* w, int Cout,
                            const float* res, float* y)
{
    float* wt = linear_w_t(w, Cout, Cin);
    linear_core(x, T, Cin, wt, Cout, res, y);
    free(wt);
}

OC_EXPORT void oc_op_rms_norm(const float* x, int T, int d, const float* g, float eps, float* y)
{
    rms_norm_core(x, T, d, g, eps, y);
}

OC_EXPORT void oc_op_gelu(const float* x, int64_t n, float* y) { gelu_core(x, n, y); }

OC_EXPORT void oc_op_swa(const float* q, const float* k, const float* v, int T, int Hk, int first,
                         int d, int heads, int window, float* o)
{
    swa_core(q, k, v, T, Hk, first, d, heads, window, o);
}

/* cb: [Q][V][E] contiguous; codes: [Q][ld]. Returns the error bits. */
OC_EXPORT uint32_t oc_op_rvq_sum(const float* cb, int Q, int V, int E, const int32_t* codes,
                                 int64_t ld, int T, float* e)
{
    const float** tabs = (const float**)malloc(sizeof(float*) * (size_t)Q);
    for (int q = 0; q < Q; q++) tabs[q] = cb + (size_t)q * V * E;
    uint32_t err = rvq_core(tabs, Q, V, E, codes, ld, T, e);
    free(tabs);
    return err;
}

/* ---------------------------------------------------------------- model -- */

typedef struct oc_layer {
    const float *n1, *n2;
    float *wq, *wk, *wv, *wo, *w1, *w2;   /* transposed [in][out] */
} oc_layer;

typedef struct oc_conv {
    const float *alpha, *b;   /* alpha NULL: no Snake on the input */
    float* wt;                /* [k][Cin][Cout] */
    int Cin, Cout, k, dil;
} oc_conv;

typedef struct oc_model {
    oc_config cfg;
    float* blob;              /* private copy of the caller's blob */
    const float* cb[64];
    oc_conv pre;
    const float *lat_mu, *lat_sigma, *lat_up_u, *lat_up_b;   /* latent input */
    float* lat_proj;          /* [L][d] transposed */
    oc_layer* layer;
    const float* tf_norm;
    oc_conv up[4];            /* ConvT: k = up_k, dil unused */
    oc_conv st[8];            /* stage ConvT with Snake alpha */
    oc_conv* rb;              /* [stage][j][i] */
    oc_conv out;
} oc_model;

typedef struct oc_state {
    const oc_model* m;
    float* h_pre;             /* [pre_k-1][E] */
    float* h_lat;             /* latent input: [1][d], the last projected row */
    float** kh;               /* per layer [window-1][d] */
    float** vh;
    float* h_up[4];           /* [1][Cin] */
    float* h_st[8];           /* [1][Cin], raw (pre-Snake) */
    float** h_rb;             /* [stage][j][i] : [(k-1)dil][C] raw */
    float* h_out;             /* [final_k-1][C4] raw */
    int64_t frames;
    uint32_t err;
} oc_state;

static int cfg_ok(const oc_config* c)
{
    if (c->latent_dim == 0 && (c->Q < 1 || c->Q > 64 || c->V < 1 || c->E < 1 || c->pre_k < 1)) return 0;
    if (c->d < 1) return 0;
    if (c->heads < 1 || c->d % c->heads || c->ffn < 1 || c->layers < 0 || c->window < 1) return 0;
    if (c->latent_dim < 0 || (c->latent_dim > 0 && c->tf_up < 1)) return 0;
    if (c->n_up < (c->latent_dim > 0 ? 0 : 1) || c->n_up > 4 || c->up_s < 1 || c->up_k != 2 * c->up_s) return 0;
    if (c->n_stages < 1 || c->n_stages > 8 || c->n_rb < 1 || c->n_rb > 4) return 0;
    if (c->n_dil < 1 || c->n_dil > 4 || c->final_k < 1) return 0;
    return 1;
}

static int64_t model_blob_floats(const oc_config* c)
{
    int64_t n;
    if (c->latent_dim > 0)   /* mu, sigma, projection [d][L], depthwise taps [d][1][2 s], bias [d] */
        n = 2 * (int64_t)c->latent_dim + (int64_t)c->d * c->latent_dim + (int64_t)c->d * 2 * c->tf_up + c->d;
    else
        n = (int64_t)c->Q * c->V * c->E + (int64_t)c->d * c->E * c->pre_k + c->d;
    n += (int64_t)c->layers * (2 * c->d + 4 * (int64_t)c->d * c->d + 2 * (int64_t)c->ffn * c->d);
    n += c->d;
    int cin = c->d;
    for (int u = 0; u < c->n_up; u++) {
        n += (int64_t)cin * c->up_ch[u] * c->up_k + c->up_ch[u];
        cin = c->up_ch[u];
    }
    for (int s = 0; s < c->n_stages; s++) {
        int co = c->ch[s];
        n += cin + (int64_t)cin * co * 2 * c->strides[s] + co;
        for (int j = 0; j < c->n_rb; j++)
            n += (int64_t)c->n_dil * (co + (int64_t)co * co * c->rb_k[j] + co);
        cin = co;
    }
    n += cin + (int64_t)cin * c->final_k + 1;
    return n;
}

OC_EXPORT int64_t oc_blob_floats(const oc_config* cfg) { return model_blob_floats(cfg); }

OC_EXPORT oc_model* oc_model_create(const oc_config* cfg, const float* blob, int64_t n_floats)
{
    if (!cfg_ok(cfg) || n_floats != model_blob_floats(cfg)) return NULL;
    oc_model* m = (oc_model*)calloc(1, sizeof(oc_model));
    m->cfg = *cfg;
    const oc_config* c = &m->cfg;
    m->blob = (float*)malloc(sizeof(float) * (size_t)n_floats);
    memcpy(m->blob, blob, sizeof(float) * (size_t)n_floats);
    const float* p = m->blob;
#define TAKE(n) (p += (n), p - (n))
    if (c->latent_dim > 0) {
        m->lat_mu = TAKE(c->latent_dim);
        m->lat_sigma = TAKE(c->latent_dim);
        m->lat_proj = linear_w_t(TAKE((int64_t)c->d * c->latent_dim), c->d, c->latent_dim);
        m->lat_up_u = TAKE((int64_t)c->d * 2 * c->tf_up);
        m->lat_up_b = TAKE(c->d);
    } else {
        for (int q = 0; q < c->Q; q++) m->cb[q] = TAKE((int64_t)c->V * c->E);
        const float* w = TAKE((int64_t)c->d * c->E * c->pre_k);
        m->pre.wt = conv_w_t(w, c->d, c->E, c->pre_k);
        m->pre.b = TAKE(c->d);
        m->pre.alpha = NULL;
        m->pre.Cin = c->E; m->pre.Cout = c->d; m->pre.k = c->pre_k; m->pre.dil = 1;
    }
    m->layer = (oc_layer*)calloc((size_t)(c->layers > 0 ? c->layers : 1), sizeof(oc_layer));
    for (int l = 0; l < c->layers; l++) {
        oc_layer* L = &m->layer[l];
        L->n1 = TAKE(c->d);
        L->wq = linear_w_t(TAKE((int64_t)c->d * c->d), c->d, c->d);
        L->wk = linear_w_t(TAKE((int64_t)c->d * c->d), c->d, c->d);
        L->wv = linear_w_t(TAKE((int64_t)c->d * c->d), c->d, c->d);
        L->wo = linear_w_t(TAKE((int64_t)c->d * c->d), c->d, c->d);
        L->n2 = TAKE(c->d);
        L->w1 = linear_w_t(TAKE((int64_t)c->ffn * c->d), c->ffn, c->d);
        L->w2 = linear_w_t(TAKE((int64_t)c->d * c->ffn), c->d, c->ffn);
    }
    m->tf_norm = TAKE(c->d);
    int cin = c->d;
    for (int u = 0; u < c->n_up; u++) {
        oc_conv* U = &m->up[u];
        U->Cin = cin; U->Cout = c->up_ch[u]; U->k = c->up_k; U->dil = 1; U->alpha = NULL;
        U->wt = convt_w_t(TAKE((int64_t)cin * U->Cout * U->k), cin, U->Cout, U->k);
        U->b = TAKE(U->Cout);
        cin = U->Cout;
    }
    m->rb = (oc_conv*)calloc((size_t)c->n_stages * c->n_rb * c->n_dil, sizeof(oc_conv));
    for (int s = 0; s < c->n_stages; s++) {
        oc_conv* S = &m->st[s];
        const int co = c->ch[s];
        S->Cin = cin; S->Cout = co; S->k = 2 * c->strides[s]; S->dil = 1;
        S->alpha = TAKE(cin);
        S->wt = convt_w_t(TAKE((int64_t)cin * co * S->k), cin, co, S->k);
        S->b = TAKE(co);
        for (int j = 0; j < c->n_rb; j++)
            for (int i = 0; i < c->n_dil; i++) {
                oc_conv* R = &m->rb[((size_t)s * c->n_rb + j) * c->n_dil + i];
                R->Cin = co; R->Cout = co; R->k = c->rb_k[j]; R->dil = c->dil[i];
                R->alpha = TAKE(co);
                R->wt = conv_w_t(TAKE((int64_t)co * co * R->k), co, co, R->k);
                R->b = TAKE(co);
            }
        cin = co;
    }
    m->out.Cin = cin; m->out.Cout = 1; m->out.k = c->final_k; m->out.dil = 1;
    m->out.alpha = TAKE(cin);
    m->out.wt = conv_w_t(TAKE((int64_t)cin * c->final_k), 1, cin, c->final_k);
    m->out.b = TAKE(1);
#undef TAKE
    return m;
}

OC_EXPORT void oc_model_destroy(oc_model* m)
{
    if (!m) return;
    const oc_config* c = &m->cfg;
    free(m->pre.wt);
    free(m->lat_proj);
    for (int l = 0; l < c->layers; l++) {
        oc_layer* L = &m->layer[l];
        free(L->wq); free(L->wk); free(L->wv); free(L->wo); free(L->w1); free(L->w2);
    }
    free(m->layer);
    for (int u = 0; u < c->n_up; u++) free(m->up[u].wt);
    for (int s = 0; s < c->n_stages; s++) free(m->st[s].wt);
    for (int i = 0; i < c->n_stages * c->n_rb * c->n_dil; i++) free(m->rb[i].wt);
    free(m->rb);
    free(m->out.wt);
    free(m->blob);
    free(m);
}

static int64_t samples_per_frame(const oc_config* c)
{
    int64_t r = c->latent_dim > 0 ? c->tf_up : 1;
    for (int u = 0; u < c->n_up; u++) r *= c->up_s;
    for (int s = 0; s < c->n_stages; s++) r *= c->strides[s];
    return r;
}

OC_EXPORT int64_t oc_samples_per_frame(const oc_model* m) { return samples_per_frame(&m->cfg); }

OC_EXPORT oc_state* oc_state_create(const oc_model* m)
{
    const oc_config* c = &m->cfg;
    oc_state* st = (oc_state*)calloc(1, sizeof(oc_state));
    st->m = m;
    st->h_pre = (float*)calloc((size_t)(c->pre_k - 1) * c->E + 1, sizeof(float));
    st->h_lat = (float*)calloc((size_t)c->d, sizeof(float));
    st->kh = (float**)calloc((size_t)(c->layers + 1), sizeof(float*));
    st->vh = (float**)calloc((size_t)(c->layers + 1), sizeof(float*));
    for (int l = 0; l < c->layers; l++) {
        st->kh[l] = (float*)calloc((size_t)(c->window - 1) * c->d + 1, sizeof(float));
        st->vh[l] = (float*)calloc((size_t)(c->window - 1) * c->d + 1, sizeof(float));
    }
    for (int u = 0; u < c->n_up; u++) st->h_up[u] = (float*)calloc((size_t)m->up[u].Cin, sizeof(float));
    for (int s = 0; s < c->n_stages; s++) st->h_st[s] = (float*)calloc((size_t)m->st[s].Cin, sizeof(float));
    const int nrb = c->n_stages * c->n_rb * c->n_dil;
    st->h_rb = (float**)calloc((size_t)nrb, sizeof(float*));
    for (int i = 0; i < nrb; i++) {
        const oc_conv* R = &m->rb[i];
        st->h_rb[i] = (float*)calloc((size_t)(R->k - 1) * R->dil * R->Cin + 1, sizeof(float));
    }
    st->h_out = (float*)calloc((size_t)(c->final_k - 1) * m->out.Cin + 1, sizeof(float));
    return st;
}

OC_EXPORT void oc_state_reset(oc_state* st)
{
    const oc_model* m = st->m;
    const oc_config* c = &m->cfg;
    memset(st->h_pre, 0, sizeof(float) * (size_t)(c->pre_k - 1) * c->E);
    memset(st->h_lat, 0, sizeof(float) * (size_t)c->d);
    for (int l = 0; l < c->layers; l++) {
        memset(st->kh[l], 0, sizeof(float) * (size_t)(c->window - 1) * c->d);
        memset(st->vh[l], 0, sizeof(float) * (size_t)(c->window - 1) * c->d);
    }
    for (int u = 0; u < c->n_up; u++) memset(st->h_up[u], 0, sizeof(float) * (size_t)m->up[u].Cin);
    for (int s = 0; s < c->n_stages; s++) memset(st->h_st[s], 0, sizeof(float) * (size_t)m->st[s].Cin);
    for (int i = 0; i < c->n_stages * c->n_rb * c->n_dil; i++) {
        const oc_conv* R = &m->rb[i];
        memset(st->h_rb[i], 0, sizeof(float) * (size_t)(R->k - 1) * R->dil * R->Cin);
    }
    memset(st->h_out, 0, sizeof(float) * (size_t)(c->final_k - 1) * m->out.Cin);
    st->frames = 0;
    st->err = 0;
}

OC_EXPORT void oc_state_destroy(oc_state* st)
{
    if (!st) return;
    const oc_config* c = &st->m->cfg;
    free(st->h_pre);
    free(st->h_lat);
    for (int l = 0; l < c->layers; l++) { free(st->kh[l]); free(st->vh[l]); }
    free(st->kh); free(st->vh);
    for (int u = 0; u < c->n_up; u++) free(st->h_up[u]);
    for (int s = 0; s < c->n_stages; s++) free(st->h_st[s]);
    for (int i = 0; i < c->n_stages * c->n_rb * c->n_dil; i++) free(st->h_rb[i]);
    free(st->h_rb);
    free(st->h_out);
    free(st);
}

OC_EXPORT int64_t oc_state_frames(const oc_state* st) { return st->frames; }
OC_EXPORT uint32_t oc_state_error(const oc_state* st) { return st->err; }

/* [hist (H rows) | x (n rows)] -> new buffer; hist <- its last H rows. */
static float* with_history(float* hist, int H, const float* x, int64_t n, int C)
{
    float* ext = (float*)malloc(sizeof(float) * (size_t)(H + n) * C + sizeof(float));
    if (H) memcpy(ext, hist, sizeof(float) * (size_t)H * C);
    memcpy(ext + (size_t)H * C, x, sizeof(float) * (size_t)n * C);
    if (H) memcpy(hist, ext + (size_t)n * C, sizeof(float) * (size_t)H * C);
    return ext;
}

/* One causal conv with carried input history (raw input kept, Snake applied
 * to history and chunk alike).  y = conv(snake(x)) (+ res). */
static void conv_step(const oc_conv* cv, float* hist, const float* x, int64_t n, const float* res,
                      float* y)
{
    const int H = (cv->k - 1) * cv->dil;
    float* ext = with_history(hist, H, x, n, cv->Cin);
    if (cv->alpha) snake_rows(ext, H + n, cv->Cin, cv->alpha, ext);
    conv_core(ext, (int)n, cv->Cin, cv->wt, cv->b, cv->Cout, cv->k, cv->dil, res, y);
    free(ext);
}

static void convt_step(const oc_conv* cv, float* hist, const float* x, int64_t n, float* y)
{
    float* ext = with_history(hist, 1, x, n, cv->Cin);
    if (cv->alpha) snake_rows(ext, 1 + n, cv->Cin, cv->alpha, ext);
    convt_core(ext, (int)n, cv->Cin, cv->wt, cv->b, cv->Cout, cv->k / 2, y);
    free(ext);
}

/*
 * The decoder after its front end: h holds `rows` transformer rows [rows][d]
 * (one per frame for code input, tf_up per frame for latent input), `seen`
 * the transformer positions the stream had before them.  Runs the
 * transformer, the latent ConvTs, the stages and the final Snake-conv-tanh,
 * writing rows * (remaining upsampling) samples.  Takes ownership of h.
 */
static void decode_body(oc_state* st, float* h, int n, int64_t seen, float* audio, float* pre_tanh)
{
    const oc_model* m = st->m;
    const oc_config* c = &m->cfg;
    const int d = c->d;

    /* transformer */
    const int W = c->window, Hk = W - 1;
    float* u = (float*)malloc(sizeof(float) * (size_t)n * (c->ffn > d ? c->ffn : d));
    float* q = (float*)malloc(sizeof(float) * (size_t)n * d);
    float* k = (float*)malloc(sizeof(float) * (size_t)n * d);
    float* v = (float*)malloc(sizeof(float) * (size_t)n * d);
    float* o = (float*)malloc(sizeof(float) * (size_t)n * d);
    float* f = (float*)malloc(sizeof(float) * (size_t)n * c->ffn);
    const int first = (seen >= Hk) ? 0 : (int)(Hk - seen);
    for (int l = 0; l < c->layers; l++) {
        const oc_layer* L = &m->layer[l];
        rms_norm_core(h, n, d, L->n1, c->rms_eps, u);
        linear_core(u, n, d, L->wq, d, NULL, q);
        linear_core(u, n, d, L->wk, d, NULL, k);
        linear_core(u, n, d, L->wv, d, NULL, v);
        float* kx = with_history(st->kh[l], Hk, k, n, d);
        float* vx = with_history(st->vh[l], Hk, v, n, d);
        swa_core(q, kx, vx, n, Hk, first, d, c->heads, W, o);
        free(kx);
        free(vx);
        linear_core(o, n, d, L->wo, d, h, h);
        rms_norm_core(h, n, d, L->n2, c->rms_eps, u);
        linear_core(u, n, d, L->w1, c->ffn, NULL, f);
        gelu_core(f, (int64_t)n * c->ffn, f);
        linear_core(f, n, c->ffn, L->w2, d, h, h);
    }
    rms_norm_core(h, n, d, m->tf_norm, c->rms_eps, h);
    free(u); free(q); free(k); free(v); free(o); free(f);

    /* latent ConvT x2 */
    float* x = h;
    int64_t rows = n;
    for (int uu = 0; uu < c->n_up; uu++) {
        const oc_conv* U = &m->up[uu];
        float* y = (float*)malloc(sizeof(float) * (size_t)rows * c->up_s * U->Cout);
        convt_step(U, st->h_up[uu], x, rows, y);
        free(x);
        x = y;
        rows *= c->up_s;
    }

    /* BigVGAN stages */
    for (int s = 0; s < c->n_stages; s++) {
        const oc_conv* S = &m->st[s];
        const int stride = c->strides[s], C = S->Cout;
        float* x0 = (float*)malloc(sizeof(float) * (size_t)rows * stride * C);
        convt_step(S, st->h_st[s], x, rows, x0);
        free(x);
        rows *= stride;
        const size_t nel = (size_t)rows * C;
        float* mrf = (float*)malloc(sizeof(float) * nel);
        float* r = (float*)malloc(sizeof(float) * nel);
        float* r2 = (float*)malloc(sizeof(float) * nel);
        double* sum = (c->n_rb > 1) ? (double*)calloc(nel, sizeof(double)) : NULL;
        for (int j = 0; j < c->n_rb; j++) {
            memcpy(r, x0, sizeof(float) * nel);
            for (int i = 0; i < c->n_dil; i++) {
                const size_t idx = ((size_t)s * c->n_rb + j) * c->n_dil + i;
                conv_step(&m->rb[idx], st->h_rb[idx], r, rows, r, r2);  /* r2 = r + conv(snake(r)) + b */
                float* t = r; r = r2; r2 = t;
            }
            if (sum) {
                for (size_t e2 = 0; e2 < nel; e2++) sum[e2] += (double)r[e2];
            } else {
                memcpy(mrf, r, sizeof(float) * nel);
            }
        }
        if (sum) {
            for (size_t e2 = 0; e2 < nel; e2++) mrf[e2] = (float)(sum[e2] / c->n_rb);
            free(sum);
        }
        free(r); free(r2); free(x0);
        x = mrf;
    }

    /* Snake -> conv -> tanh */
    float* y = (float*)malloc(sizeof(float) * (size_t)rows);
    conv_step(&m->out, st->h_out, x, rows, NULL, y);
    free(x);
    for (int64_t i = 0; i < rows; i++) {
        if (pre_tanh) pre_tanh[i] = y[i];
        audio[i] = (float)tanh((double)y[i]);
    }
    free(y);
}

/*
 * Decode n frames continuing the stream: codes [Q][ld] (columns 0..n-1 used),
 * audio [n * samples_per_frame].  pre_tanh, if not NULL, receives the final
 * conv output before tanh.  Returns the stream's sticky error bits.
 */
OC_EXPORT uint32_t oc_decode(oc_state* st, const int32_t* codes, int64_t ld, int n, float* audio,
                             float* pre_tanh)
{
    const oc_model* m = st->m;
    const oc_config* c = &m->cfg;
    if (n <= 0 || c->latent_dim > 0) return st->err;

    /* RVQ embedding sum */
    float* e = (float*)malloc(sizeof(float) * (size_t)n * c->E);
    st->err |= rvq_core(m->cb, c->Q, c->V, c->E, codes, ld, n, e);

    /* causal pre-conv */
    float* h = (float*)malloc(sizeof(float) * (size_t)n * c->d);
    conv_step(&m->pre, st->h_pre, e, n, NULL, h);
    free(e);

    decode_body(st, h, n, st->frames, audio, pre_tanh);
    st->frames += n;
    return st->err;
}

/*
 * Latent-input decoder: n frames of latents [n][L] continuing the stream.
 *   z = x sigma + mu (per channel), p = Wp z (1x1, no bias), then the causal
 *   depthwise ConvTranspose1d (stride s = tf_up) with the last projected row of
 *   the previous chunk as its history: n s rows for the transformer.
 */
OC_EXPORT uint32_t oc_decode_latents(oc_state* st, const float* x, int n, float* audio, float* pre_tanh)
{
    const oc_model* m = st->m;
    const oc_config* c = &m->cfg;
    if (n <= 0 || c->latent_dim <= 0) return st->err;
    const int L = c->latent_dim, d = c->d, s = c->tf_up;
    float* z = (float*)malloc(sizeof(float) * (size_t)n * L);
    for (int64_t i = 0; i < (int64_t)n * L; i++) {
        const int l = (int)(i % L);
        z[i] = (float)((double)x[i] * (double)m->lat_sigma[l] + (double)m->lat_mu[l]);
    }
    float* pr = (float*)malloc(sizeof(float) * (size_t)n * d);
    linear_core(z, n, L, m->lat_proj, d, NULL, pr);
    free(z);
    float* ext = with_history(st->h_lat, 1, pr, n, d);
    free(pr);
    float* h = (float*)malloc(sizeof(float) * (size_t)n * s * d);
    dwconvt_core(ext, n, d, m->lat_up_u, m->lat_up_b, s, h);
    free(ext);
    decode_body(st, h, n * s, st->frames * s, audio, pre_tanh);
    st->frames += n;
    return st->err;
}

OC_EXPORT int oc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

OC_EXPORT void oc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
