/*
 * gpt2_oracle.c -- plain, slow, double-precision CPU reference of one GPT-2
 * training step (forward, backward, AdamW) and of the fused
 * Linear+bias+GELU(tanh)+row-softmax operator.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg. Nothing in the GPU product path links it.
 *
 * Every function is the textbook definition of the step it names, written as
 * naive loops with double accumulators. OpenMP (when enabled) only splits the
 * outer loop of independent output rows, so each output element is always
 * computed by one thread in one fixed order and results do not depend on the
 * thread count.
 *
 * Sources (page titles; sections are the kernels/functions named there):
 *   [P1] llm.c "train_gpt2.cu" (mixed-precision CUDA training step)
 *   [P2] llm.c "train_gpt2_fp32.cu" (fp32 CUDA training step)
 *   [P3] POPCORNBENCH transcript "fused Linear + GELU + Softmax"
 */
#include "gpt2_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define LN_EPS 1e-5

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* [P1] fill_in_parameter_sizes: the 16 parameter tensors, in order. */
size_t oracle_param_sizes(const oracle_config* cfg, size_t s[ORACLE_NUM_PARAM_TENSORS]) {
    size_t C = (size_t)cfg->C, L = (size_t)cfg->L;
    s[0] = (size_t)cfg->Vp * C;   /* wte */
    s[1] = (size_t)cfg->maxT * C; /* wpe */
    s[2] = L * C;                 /* ln1w */
    s[3] = L * C;                 /* ln1b */
    s[4] = L * 3 * C * C;         /* qkvw */
    s[5] = L * 3 * C;             /* qkvb */
    s[6] = L * C * C;             /* attprojw */
    s[7] = L * C;                 /* attprojb */
    s[8] = L * C;                 /* ln2w */
    s[9] = L * C;                 /* ln2b */
    s[10] = L * 4 * C * C;        /* fcw */
    s[11] = L * 4 * C;            /* fcb */
    s[12] = L * C * 4 * C;        /* fcprojw */
    s[13] = L * C;                /* fcprojb */
    s[14] = C;                    /* lnfw */
    s[15] = C;                    /* lnfb */
    size_t total = 0;
    for (int i = 0; i < ORACLE_NUM_PARAM_TENSORS; i++) total += s[i];
    return total;
}

/* ------------------------------------------------------------------------ */
/* Single operations                                                          */
/* ------------------------------------------------------------------------ */

/* [P1] encoder_forward_kernel2, [P2] encoder_forward_kernel3:
 * token embedding row plus position embedding row. */
void oracle_encoder_forward(double* out, const int* tokens, const double* wte, const double* wpe,
                            int B, int T, int C) {
    for (int b = 0; b < B; b++) {
        for (int t = 0; t < T; t++) {
            const double* we = wte + (size_t)tokens[b * T + t] * C;
            const double* pe = wpe + (size_t)t * C;
            double* o = out + ((size_t)b * T + t) * C;
            for (int c = 0; c < C; c++) o[c] = we[c] + pe[c];
        }
    }
}

/* [P1] encoder_backward_kernel: dwte[token] += dout, dwpe[t] += dout. */
static void encoder_backward(double* dwte, double* dwpe, const double* dout, const int* tokens,
                             int B, int T, int C) {
    for (int b = 0; b < B; b++) {
        for (int t = 0; t < T; t++) {
            const double* d = dout + ((size_t)b * T + t) * C;
            double* dw = dwte + (size_t)tokens[b * T + t] * C;
            double* dp = dwpe + (size_t)t * C;
            for (int c = 0; c < C; c++) {
                dw[c] += d[c];
                dp[c] += d[c];
            }
        }
    }
}

/* [P1] layernorm_forward_kernel3: mean, biased variance over C,
 * rstd = 1/sqrt(var + 1e-5), y = (x - mean) * rstd * w + b. */
void oracle_layernorm_forward(double* out, double* mean, double* rstd, const double* inp,
                              const double* w, const double* b, int N, int C) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const double* x = inp + (size_t)n * C;
        double m = 0.0;
        for (int c = 0; c < C; c++) m += x[c];
        m /= C;
        double v = 0.0;
        for (int c = 0; c < C; c++) v += (x[c] - m) * (x[c] - m);
        v /= C;
        double s = 1.0 / sqrt(v + LN_EPS);
        double* y = out + (size_t)n * C;
        for (int c = 0; c < C; c++) y[c] = (x[c] - m) * s * w[c] + b[c];
        if (mean) mean[n] = m;
        if (rstd) rstd[n] = s;
    }
}

/* [P1] layernorm_backward_kernel6 (read with += for every output, the
 * accumulation the page's header note prescribes for parameters and for the
 * residual stream):
 *   nhat = (x - mean) * rstd,  g = w * dy
 *   dx += rstd * (g - mean(g) - nhat * mean(g * nhat))
 *   dw += sum_rows nhat * dy,  db += sum_rows dy */
void oracle_layernorm_backward(double* dinp, double* dw, double* db, const double* dout,
                               const double* inp, const double* w, const double* mean,
                               const double* rstd, int N, int C) {
    /* input gradient: rows are independent */
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const double* x = inp + (size_t)n * C;
        const double* dy = dout + (size_t)n * C;
        double* dx = dinp + (size_t)n * C;
        double g_mean = 0.0, gn_mean = 0.0;
        for (int c = 0; c < C; c++) {
            double nh = (x[c] - mean[n]) * rstd[n];
            double g = w[c] * dy[c];
            g_mean += g;
            gn_mean += g * nh;
        }
        g_mean /= C;
        gn_mean /= C;
        for (int c = 0; c < C; c++) {
            double nh = (x[c] - mean[n]) * rstd[n];
            double g = w[c] * dy[c];
            dx[c] += rstd[n] * (g - g_mean - nh * gn_mean);
        }
    }
    /* parameter gradients: sum over rows in row order */
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; c++) {
        double sw = 0.0, sb = 0.0;
        for (int n = 0; n < N; n++) {
            double nh = (inp[(size_t)n * C + c] - mean[n]) * rstd[n];
            double dy = dout[(size_t)n * C + c];
            sw += nh * dy;
            sb += dy;
        }
        dw[c] += sw;
        db[c] += sb;
    }
}

/* [P1] matmul_forward_cublaslt: out = inp . w^T + bias with w stored (OC, C). */
void oracle_matmul_forward(double* out, const double* inp, const double* w, const double* bias,
                           int N, int Cin, int Cout) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const double* x = inp + (size_t)n * Cin;
        double* y = out + (size_t)n * Cout;
        for (int o = 0; o < Cout; o++) {
            const double* wr = w + (size_t)o * Cin;
            double acc = bias ? bias[o] : 0.0;
            for (int c = 0; c < Cin; c++) acc += x[c] * wr[c];
            y[o] = acc;
        }
    }
}

/* [P1] matmul_backward: dinp = dout . w (written), dw += dout^T . inp,
 * dbias += column sums of dout. */
void oracle_matmul_backward(double* dinp, double* dw, double* dbias, const double* dout,
                            const double* inp, const double* w, int N, int Cin, int Cout) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; n++) {
        const double* dy = dout + (size_t)n * Cout;
        double* dx = dinp + (size_t)n * Cin;
        for (int c = 0; c < Cin; c++) dx[c] = 0.0;
        for (int o = 0; o < Cout; o++) {
            const double* wr = w + (size_t)o * Cin;
            double d = dy[o];
            for (int c = 0; c < Cin; c++) dx[c] += d * wr[c];
        }
    }
#pragma omp parallel for schedule(static)
    for (int o = 0; o < Cout; o++) {
        double* dwr = dw + (size_t)o * Cin;
        double sb = 0.0;
        for (int n = 0; n < N; n++) {
            double d = dout[(size_t)n * Cout + o];
            const double* x = inp + (size_t)n * Cin;
            for (int c = 0; c < Cin; c++) dwr[c] += d * x[c];
            sb += d;
        }
        if (dbias) dbias[o] += sb;
    }
}

/* [P1] gelu_forward_kernel2: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
static double gelu_tanh(double x) {
    double u = sqrt(2.0 / M_PI) * (x + 0.044715 * x * x * x);
    return 0.5 * x * (1.0 + tanh(u));
}

void oracle_gelu_forward(double* out, const double* inp, size_t n) {
    for (size_t i = 0; i < n; i++) out[i] = gelu_tanh(inp[i]);
}

/* [P1] gelu_backward_kernel: derivative of the tanh form,
 * 0.5 (1 + tanh u) + 0.5 x sech^2(u) sqrt(2/pi) (1 + 3 * 0.044715 x^2). */
void oracle_gelu_backward(double* dinp, const double* inp, const double* dout, size_t n) {
    const double s = sqrt(2.0 / M_PI);
    for (size_t i = 0; i < n; i++) {
        double x = inp[i];
        double u = s * (x + 0.044715 * x * x * x);
        double th = tanh(u);
        double ch = cosh(u);
        double sech2 = 1.0 / (ch * ch);
        double local = 0.5 * (1.0 + th) + 0.5 * x * sech2 * s * (1.0 + 3.0 * 0.044715 * x * x);
        dinp[i] = local * dout[i];
    }
}

/* [P1] attention_forward (permute, Q K^T, softmax_forward_kernel5 with the
 * 1/sqrt(HS) scale, att . V, unpermute): for every (b, h, i)
 *   s_ij = (q_i . k_j) / sqrt(HS) for j <= i,
 *   p_ij = exp(s_ij - max_j s_ij) / sum_j exp(...),  p_ij = 0 for j > i,
 *   out_i = sum_j p_ij v_j. */
void oracle_attention_forward(double* out, double* att, const double* qkv,
                              int B, int T, int C, int NH) {
    int HS = C / NH;
    double scale = 1.0 / sqrt((double)HS);
    size_t C3 = 3 * (size_t)C;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < NH; h++) {
            double* p = (double*)malloc(sizeof(double) * (size_t)T);
            for (int i = 0; i < T; i++) {
                const double* q = qkv + ((size_t)b * T + i) * C3 + (size_t)h * HS;
                double mx = -INFINITY;
                for (int j = 0; j <= i; j++) {
                    const double* k = qkv + ((size_t)b * T + j) * C3 + C + (size_t)h * HS;
                    double s = 0.0;
                    for (int d = 0; d < HS; d++) s += q[d] * k[d];
                    s *= scale;
                    p[j] = s;
                    if (s > mx) mx = s;
                }
                double sum = 0.0;
                for (int j = 0; j <= i; j++) {
                    p[j] = exp(p[j] - mx);
                    sum += p[j];
                }
                for (int j = 0; j <= i; j++) p[j] /= sum;
                for (int j = i + 1; j < T; j++) p[j] = 0.0;
                double* o = out + ((size_t)b * T + i) * C + (size_t)h * HS;
                for (int d = 0; d < HS; d++) o[d] = 0.0;
                for (int j = 0; j <= i; j++) {
                    const double* v = qkv + ((size_t)b * T + j) * C3 + 2 * (size_t)C + (size_t)h * HS;
                    for (int d = 0; d < HS; d++) o[d] += p[j] * v[d];
                }
                if (att) {
                    double* a = att + (((size_t)b * NH + h) * T + i) * T;
                    for (int j = 0; j < T; j++) a[j] = p[j];
                }
            }
            free(p);
        }
    }
}

/* [P1] attention_backward with softmax_autoregressive_backward_kernel: for
 * every (b, h, i), with p the forward probabilities,
 *   dp_ij = do_i . v_j,           dv_j += p_ij do_i,
 *   ds_ij = p_ij (dp_ij - sum_k p_ik dp_ik)   (softmax Jacobian),
 *   dq_i += ds_ij k_j / sqrt(HS), dk_j += ds_ij q_i / sqrt(HS). */
void oracle_attention_backward(double* dqkv, const double* dout, const double* qkv,
                               const double* att, int B, int T, int C, int NH) {
    int HS = C / NH;
    double scale = 1.0 / sqrt((double)HS);
    size_t C3 = 3 * (size_t)C;
    memset(dqkv, 0, sizeof(double) * (size_t)B * T * C3);
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < NH; h++) {
            double* dp = (double*)malloc(sizeof(double) * (size_t)T);
            for (int i = 0; i < T; i++) {
                const double* p = att + (((size_t)b * NH + h) * T + i) * T;
                const double* dO = dout + ((size_t)b * T + i) * C + (size_t)h * HS;
                double dot = 0.0;
                for (int j = 0; j <= i; j++) {
                    const double* v = qkv + ((size_t)b * T + j) * C3 + 2 * (size_t)C + (size_t)h * HS;
                    double* dv = dqkv + ((size_t)b * T + j) * C3 + 2 * (size_t)C + (size_t)h * HS;
                    double s = 0.0;
                    for (int d = 0; d < HS; d++) {
                        s += dO[d] * v[d];
                        dv[d] += p[j] * dO[d];
                    }
                    dp[j] = s;
                    dot += p[j] * s;
                }
                const double* q = qkv + ((size_t)b * T + i) * C3 + (size_t)h * HS;
                double* dq = dqkv + ((size_t)b * T + i) * C3 + (size_t)h * HS;
                for (int j = 0; j <= i; j++) {
                    double ds = p[j] * (dp[j] - dot) * scale;
                    const double* k = qkv + ((size_t)b * T + j) * C3 + C + (size_t)h * HS;
                    double* dk = dqkv + ((size_t)b * T + j) * C3 + C + (size_t)h * HS;
                    for (int d = 0; d < HS; d++) {
                        dq[d] += ds * k[d];
                        dk[d] += ds * q[d];
                    }
                }
            }
            free(dp);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Whole model                                                                */
/* ------------------------------------------------------------------------ */

struct oracle_model {
    oracle_config cfg;
    int B, T;
    int have_targets;
    int grad_accum_k;
    int* tokens;
    int* targets;
    /* activations ([P1] ActivationTensors, with att holding probabilities) */
    double *encoded;                          /* (B,T,C) */
    double *ln1, *ln1_mean, *ln1_rstd;        /* (L,B,T,C), (L,B,T) */
    double *qkv;                              /* (L,B,T,3C) */
    double *att;                              /* (L,B,NH,T,T) */
    double *atty;                             /* (L,B,T,C) */
    double *attproj;                          /* (L,B,T,C) */
    double *residual2;                        /* (L,B,T,C) */
    double *ln2, *ln2_mean, *ln2_rstd;        /* (L,B,T,C), (L,B,T) */
    double *fch, *fch_gelu;                   /* (L,B,T,4C) */
    double *fcproj;                           /* (L,B,T,C) */
    double *residual3;                        /* (L,B,T,C) */
    double *lnf, *lnf_mean, *lnf_rstd;        /* (B,T,C), (B,T) */
    double *logits;                           /* (B,T,Vp) */
    double *probs;                            /* (B,T,Vp) */
    double *dlogits;                          /* (B,T,Vp) */
    double *losses;                           /* (B,T) */
};

static double* dalloc(size_t n) { return (double*)calloc(n ? n : 1, sizeof(double)); }

oracle_model* oracle_create(const oracle_config* cfg, int B, int T) {
    if (B <= 0 || T <= 0 || T > cfg->maxT || cfg->C % cfg->NH != 0) return NULL;
    oracle_model* m = (oracle_model*)calloc(1, sizeof(oracle_model));
    if (!m) return NULL;
    m->cfg = *cfg;
    m->B = B;
    m->T = T;
    size_t L = (size_t)cfg->L, C = (size_t)cfg->C, NH = (size_t)cfg->NH, Vp = (size_t)cfg->Vp;
    size_t BT = (size_t)B * T;
    m->tokens = (int*)calloc(BT, sizeof(int));
    m->targets = (int*)calloc(BT, sizeof(int));
    m->encoded = dalloc(BT * C);
    m->ln1 = dalloc(L * BT * C);
    m->ln1_mean = dalloc(L * BT);
    m->ln1_rstd = dalloc(L * BT);
    m->qkv = dalloc(L * BT * 3 * C);
    m->att = dalloc(L * (size_t)B * NH * T * T);
    m->atty = dalloc(L * BT * C);
    m->attproj = dalloc(L * BT * C);
    m->residual2 = dalloc(L * BT * C);
    m->ln2 = dalloc(L * BT * C);
    m->ln2_mean = dalloc(L * BT);
    m->ln2_rstd = dalloc(L * BT);
    m->fch = dalloc(L * BT * 4 * C);
    m->fch_gelu = dalloc(L * BT * 4 * C);
    m->fcproj = dalloc(L * BT * C);
    m->residual3 = dalloc(L * BT * C);
    m->lnf = dalloc(BT * C);
    m->lnf_mean = dalloc(BT);
    m->lnf_rstd = dalloc(BT);
    m->logits = dalloc(BT * Vp);
    m->probs = dalloc(BT * Vp);
    m->dlogits = dalloc(BT * Vp);
    m->losses = dalloc(BT);
    if (!m->tokens || !m->targets || !m->encoded || !m->ln1 || !m->qkv || !m->att || !m->atty ||
        !m->attproj || !m->residual2 || !m->ln2 || !m->fch || !m->fch_gelu || !m->fcproj ||
        !m->residual3 || !m->lnf || !m->logits || !m->probs || !m->dlogits || !m->losses) {
        oracle_destroy(m);
        return NULL;
    }
    return m;
}

void oracle_destroy(oracle_model* m) {
    if (!m) return;
    free(m->tokens); free(m->targets);
    free(m->encoded); free(m->ln1); free(m->ln1_mean); free(m->ln1_rstd); free(m->qkv);
    free(m->att); free(m->atty); free(m->attproj); free(m->residual2); free(m->ln2);
    free(m->ln2_mean); free(m->ln2_rstd); free(m->fch); free(m->fch_gelu); free(m->fcproj);
    free(m->residual3); free(m->lnf); free(m->lnf_mean); free(m->lnf_rstd); free(m->logits);
    free(m->probs); free(m->dlogits); free(m->losses);
    free(m);
}

/* pointers to the 16 parameter tensors inside a flat array */
typedef struct {
    double *wte, *wpe, *ln1w, *ln1b, *qkvw, *qkvb, *attprojw, *attprojb, *ln2w, *ln2b, *fcw, *fcb,
        *fcprojw, *fcprojb, *lnfw, *lnfb;
} ptensors;

static ptensors point_params(const oracle_config* cfg, const double* base) {
    size_t s[ORACLE_NUM_PARAM_TENSORS];
    oracle_param_sizes(cfg, s);
    double* p = (double*)base;
    double** slots[ORACLE_NUM_PARAM_TENSORS];
    ptensors t;
    slots[0] = &t.wte; slots[1] = &t.wpe; slots[2] = &t.ln1w; slots[3] = &t.ln1b;
    slots[4] = &t.qkvw; slots[5] = &t.qkvb; slots[6] = &t.attprojw; slots[7] = &t.attprojb;
    slots[8] = &t.ln2w; slots[9] = &t.ln2b; slots[10] = &t.fcw; slots[11] = &t.fcb;
    slots[12] = &t.fcprojw; slots[13] = &t.fcprojb; slots[14] = &t.lnfw; slots[15] = &t.lnfb;
    for (int i = 0; i < ORACLE_NUM_PARAM_TENSORS; i++) {
        *slots[i] = p;
        p += s[i];
    }
    return t;
}

/* [P1] gpt2_forward: encoder, then per layer
 *   ln1 -> qkv -> attention -> attproj -> residual2 = residual + attproj
 *   -> ln2 -> fc -> gelu -> fcproj -> residual3 = residual2 + fcproj,
 * then lnf, the tied classifier over Vp columns, and fused_classifier_kernel3:
 * softmax over the first V columns, loss = -log p[target], and
 * dlogits = (p - 1[target]) * dloss with dloss = 1/(k*B*T), zero on [V, Vp). */
double oracle_forward(oracle_model* m, const double* params, const int* tokens,
                      const int* targets, int grad_accum_k) {
    const oracle_config* cfg = &m->cfg;
    int B = m->B, T = m->T, C = cfg->C, NH = cfg->NH, V = cfg->V, Vp = cfg->Vp, L = cfg->L;
    size_t BT = (size_t)B * T;
    ptensors p = point_params(cfg, params);
    memcpy(m->tokens, tokens, BT * sizeof(int));
    m->have_targets = targets != NULL;
    m->grad_accum_k = grad_accum_k > 0 ? grad_accum_k : 1;
    if (targets) memcpy(m->targets, targets, BT * sizeof(int));

    oracle_encoder_forward(m->encoded, tokens, p.wte, p.wpe, B, T, C);
    const double* residual = m->encoded;
    for (int l = 0; l < L; l++) {
        size_t oC = (size_t)l * BT * C, oS = (size_t)l * BT;
        double* ln1 = m->ln1 + oC;
        double* qkv = m->qkv + 3 * oC;
        double* att = m->att + (size_t)l * B * NH * T * T;
        double* atty = m->atty + oC;
        double* attproj = m->attproj + oC;
        double* res2 = m->residual2 + oC;
        double* ln2 = m->ln2 + oC;
        double* fch = m->fch + 4 * oC;
        double* fchg = m->fch_gelu + 4 * oC;
        double* fcproj = m->fcproj + oC;
        double* res3 = m->residual3 + oC;
        oracle_layernorm_forward(ln1, m->ln1_mean + oS, m->ln1_rstd + oS, residual,
                                 p.ln1w + (size_t)l * C, p.ln1b + (size_t)l * C, (int)BT, C);
        oracle_matmul_forward(qkv, ln1, p.qkvw + (size_t)l * 3 * C * C, p.qkvb + (size_t)l * 3 * C,
                              (int)BT, C, 3 * C);
        oracle_attention_forward(atty, att, qkv, B, T, C, NH);
        oracle_matmul_forward(attproj, atty, p.attprojw + (size_t)l * C * C,
                              p.attprojb + (size_t)l * C, (int)BT, C, C);
        for (size_t i = 0; i < BT * C; i++) res2[i] = residual[i] + attproj[i];
        oracle_layernorm_forward(ln2, m->ln2_mean + oS, m->ln2_rstd + oS, res2,
                                 p.ln2w + (size_t)l * C, p.ln2b + (size_t)l * C, (int)BT, C);
        oracle_matmul_forward(fch, ln2, p.fcw + (size_t)l * 4 * C * C, p.fcb + (size_t)l * 4 * C,
                              (int)BT, C, 4 * C);
        oracle_gelu_forward(fchg, fch, BT * 4 * C);
        oracle_matmul_forward(fcproj, fchg, p.fcprojw + (size_t)l * C * 4 * C,
                              p.fcprojb + (size_t)l * C, (int)BT, 4 * C, C);
        for (size_t i = 0; i < BT * C; i++) res3[i] = res2[i] + fcproj[i];
        residual = res3;
    }
    oracle_layernorm_forward(m->lnf, m->lnf_mean, m->lnf_rstd, residual, p.lnfw, p.lnfb, (int)BT, C);
    oracle_matmul_forward(m->logits, m->lnf, p.wte, NULL, (int)BT, C, Vp);

    /* softmax over the real vocabulary; the padded columns get probability 0 */
    for (size_t n = 0; n < BT; n++) {
        const double* lg = m->logits + n * Vp;
        double* pr = m->probs + n * Vp;
        double mx = -INFINITY;
        for (int v = 0; v < V; v++) if (lg[v] > mx) mx = lg[v];
        double sum = 0.0;
        for (int v = 0; v < V; v++) {
            pr[v] = exp(lg[v] - mx);
            sum += pr[v];
        }
        for (int v = 0; v < V; v++) pr[v] /= sum;
        for (int v = V; v < Vp; v++) pr[v] = 0.0;
    }
    if (!targets) return -1.0;

    double dloss = 1.0 / ((double)m->grad_accum_k * (double)BT);
    double mean = 0.0;
    for (size_t n = 0; n < BT; n++) {
        int tg = targets[n];
        const double* lg = m->logits + n * Vp;
        /* -log p[target] computed as logsumexp - logit[target] */
        double mx = -INFINITY;
        for (int v = 0; v < V; v++) if (lg[v] > mx) mx = lg[v];
        double sum = 0.0;
        for (int v = 0; v < V; v++) sum += exp(lg[v] - mx);
        m->losses[n] = (mx + log(sum)) - lg[tg];
        mean += m->losses[n];
        double* dl = m->dlogits + n * Vp;
        const double* pr = m->probs + n * Vp;
        for (int v = 0; v < V; v++) dl[v] = (pr[v] - (v == tg ? 1.0 : 0.0)) * dloss;
        for (int v = V; v < Vp; v++) dl[v] = 0.0;
    }
    return mean / (double)BT;
}

/* [P1] gpt2_backward: classifier matmul backward, lnf backward into the
 * residual-stream gradient, then for each layer from the last:
 *   fcproj backward, gelu backward, fc backward, ln2 backward (+= residual grad),
 *   attproj backward, attention backward, qkv backward, ln1 backward (+=),
 * and finally the encoder backward. Parameter gradients accumulate. */
int oracle_backward(oracle_model* m, const double* params, double* grads) {
    if (!m->have_targets) return -1;
    const oracle_config* cfg = &m->cfg;
    int B = m->B, T = m->T, C = cfg->C, NH = cfg->NH, Vp = cfg->Vp, L = cfg->L;
    size_t BT = (size_t)B * T;
    ptensors p = point_params(cfg, params);
    ptensors g = point_params(cfg, grads);

    double* dresidual = dalloc(BT * C);  /* the residual-stream gradient, accumulated */
    double* dbtc = dalloc(BT * C);
    double* dbtc2 = dalloc(BT * C);
    double* dbt4c = dalloc(BT * 4 * C);
    double* dbt4c2 = dalloc(BT * 4 * C);
    double* dqkv = dalloc(BT * 3 * C);

    /* logits = lnf . wte^T  ->  dlnf = dlogits . wte,  dwte += dlogits^T . lnf */
    oracle_matmul_backward(dbtc, g.wte, NULL, m->dlogits, m->lnf, p.wte, (int)BT, C, Vp);
    const double* residual = m->residual3 + (size_t)(L - 1) * BT * C;
    oracle_layernorm_backward(dresidual, g.lnfw, g.lnfb, dbtc, residual, p.lnfw, m->lnf_mean,
                              m->lnf_rstd, (int)BT, C);

    for (int l = L - 1; l >= 0; l--) {
        size_t oC = (size_t)l * BT * C, oS = (size_t)l * BT;
        residual = l == 0 ? m->encoded : m->residual3 + (size_t)(l - 1) * BT * C;
        /* residual3 = residual2 + fcproj(gelu(fc(ln2(residual2)))) */
        oracle_matmul_backward(dbt4c, g.fcprojw + (size_t)l * C * 4 * C, g.fcprojb + (size_t)l * C,
                               dresidual, m->fch_gelu + 4 * oC, p.fcprojw + (size_t)l * C * 4 * C,
                               (int)BT, 4 * C, C);
        oracle_gelu_backward(dbt4c2, m->fch + 4 * oC, dbt4c, BT * 4 * C);
        oracle_matmul_backward(dbtc, g.fcw + (size_t)l * 4 * C * C, g.fcb + (size_t)l * 4 * C,
                               dbt4c2, m->ln2 + oC, p.fcw + (size_t)l * 4 * C * C, (int)BT, C, 4 * C);
        oracle_layernorm_backward(dresidual, g.ln2w + (size_t)l * C, g.ln2b + (size_t)l * C, dbtc,
                                  m->residual2 + oC, p.ln2w + (size_t)l * C, m->ln2_mean + oS,
                                  m->ln2_rstd + oS, (int)BT, C);
        /* residual2 = residual + attproj(attention(qkv(ln1(residual)))) */
        oracle_matmul_backward(dbtc2, g.attprojw + (size_t)l * C * C, g.attprojb + (size_t)l * C,
                               dresidual, m->atty + oC, p.attprojw + (size_t)l * C * C, (int)BT, C, C);
        oracle_attention_backward(dqkv, dbtc2, m->qkv + 3 * oC, m->att + (size_t)l * B * NH * T * T,
                                  B, T, C, NH);
        oracle_matmul_backward(dbtc, g.qkvw + (size_t)l * 3 * C * C, g.qkvb + (size_t)l * 3 * C, dqkv,
                               m->ln1 + oC, p.qkvw + (size_t)l * 3 * C * C, (int)BT, C, 3 * C);
        oracle_layernorm_backward(dresidual, g.ln1w + (size_t)l * C, g.ln1b + (size_t)l * C, dbtc,
                                  residual, p.ln1w + (size_t)l * C, m->ln1_mean + oS,
                                  m->ln1_rstd + oS, (int)BT, C);
    }
    encoder_backward(g.wte, g.wpe, dresidual, m->tokens, B, T, C);

    free(dresidual); free(dbtc); free(dbtc2); free(dbt4c); free(dbt4c2); free(dqkv);
    return 0;
}

size_t oracle_get_act(const oracle_model* m, int which, int layer, double* out) {
    const oracle_config* cfg = &m->cfg;
    size_t BT = (size_t)m->B * m->T, C = (size_t)cfg->C, Vp = (size_t)cfg->Vp;
    size_t l = (size_t)(layer < 0 ? 0 : layer);
    if (layer < 0 || layer >= cfg->L) l = 0;
    const double* src = NULL;
    size_t n = 0;
    switch (which) {
        case ORACLE_ACT_ENCODED: src = m->encoded; n = BT * C; break;
        case ORACLE_ACT_LN1: src = m->ln1 + l * BT * C; n = BT * C; break;
        case ORACLE_ACT_QKV: src = m->qkv + l * BT * 3 * C; n = BT * 3 * C; break;
        case ORACLE_ACT_ATT: n = (size_t)m->B * cfg->NH * m->T * m->T; src = m->att + l * n; break;
        case ORACLE_ACT_ATTY: src = m->atty + l * BT * C; n = BT * C; break;
        case ORACLE_ACT_RESIDUAL2: src = m->residual2 + l * BT * C; n = BT * C; break;
        case ORACLE_ACT_LN2: src = m->ln2 + l * BT * C; n = BT * C; break;
        case ORACLE_ACT_FCH: src = m->fch + l * BT * 4 * C; n = BT * 4 * C; break;
        case ORACLE_ACT_FCH_GELU: src = m->fch_gelu + l * BT * 4 * C; n = BT * 4 * C; break;
        case ORACLE_ACT_RESIDUAL3: src = m->residual3 + l * BT * C; n = BT * C; break;
        case ORACLE_ACT_LNF: src = m->lnf; n = BT * C; break;
        case ORACLE_ACT_LOGITS: src = m->logits; n = BT * Vp; break;
        case ORACLE_ACT_PROBS: src = m->probs; n = BT * Vp; break;
        case ORACLE_ACT_LOSSES: src = m->losses; n = BT; break;
        case ORACLE_ACT_DLOGITS: src = m->dlogits; n = BT * Vp; break;
        case ORACLE_ACT_LN1_MEAN: src = m->ln1_mean + l * BT; n = BT; break;
        case ORACLE_ACT_LN1_RSTD: src = m->ln1_rstd + l * BT; n = BT; break;
        default: return 0;
    }
    memcpy(out, src, n * sizeof(double));
    return n;
}

/* [P1] adamw_kernel3 / gpt2_update (master-weight path), [P2] adamw_kernel2:
 *   m = b1 m + (1-b1) g,  v = b2 v + (1-b2) g^2,
 *   mhat = m / (1 - b1^t), vhat = v / (1 - b2^t),
 *   theta -= lr * (mhat / (sqrt(vhat) + eps) + wd * theta). */
void oracle_adamw(double* params, const double* grads, double* mstate, double* vstate, size_t n,
                  double lr, double beta1, double beta2, double eps, double wd, int t) {
    double c1 = 1.0 - pow(beta1, t);
    double c2 = 1.0 - pow(beta2, t);
#pragma omp parallel for schedule(static)
    for (size_t i = 0; i < n; i++) {
        double g = grads[i];
        double mm = beta1 * mstate[i] + (1.0 - beta1) * g;
        double vv = beta2 * vstate[i] + (1.0 - beta2) * g * g;
        mstate[i] = mm;
        vstate[i] = vv;
        double mhat = mm / c1;
        double vhat = vv / c2;
        double th = params[i];
        params[i] = th - lr * (mhat / (sqrt(vhat) + eps) + wd * th);
    }
}

/* [P3] problem statement: y = softmax over dim 1 of gelu(x . W^T + b), with
 * the tanh form of GELU. One row at a time: linear, bias, GELU, then the
 * max-subtracted softmax of the row. */
void oracle_fused_linear_bias_gelu_softmax(const double* x, const double* W, const double* b,
                                           double* y, int M, int K, int N) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; i++) {
        double* row = y + (size_t)i * N;
        const double* xr = x + (size_t)i * K;
        for (int j = 0; j < N; j++) {
            const double* wr = W + (size_t)j * K;
            double acc = b[j];
            for (int k = 0; k < K; k++) acc += xr[k] * wr[k];
            row[j] = gelu_tanh(acc);
        }
        double mx = -INFINITY;
        for (int j = 0; j < N; j++) if (row[j] > mx) mx = row[j];
        double sum = 0.0;
        for (int j = 0; j < N; j++) {
            row[j] = exp(row[j] - mx);
            sum += row[j];
        }
        for (int j = 0; j < N; j++) row[j] /= sum;
    }
}

/* ------------------------------------------------------------------------
 * Random numbers, stochastic rounding and sampling ([P1]).
 * These follow the page's fixed-width integer and float arithmetic: the
 * stochastic-rounding decision depends on the float bits of the update, so
 * the AdamW update below is computed in float (the page's precision), with
 * each operation written out (no contraction: the oracle is built with
 * -ffp-contract=off) and the page's two-FMA lerp.
 * ------------------------------------------------------------------------ */

/* [P1] random_u32: xorshift* (Vigna) -- three xorshifts of the 64-bit state,
 * then the top 32 bits of the state times 0x2545F4914F6CDD1D. */
unsigned int oracle_random_u32(unsigned long long* state) {
    unsigned long long x = *state;
    x ^= x >> 12;
    x ^= x << 25;
    x ^= x >> 27;
    *state = x;
    return (unsigned int)((x * 0x2545F4914F6CDD1DULL) >> 32);
}

/* [P1] random_f32: the top 24 of those 32 bits as a float in [0, 1). */
float oracle_random_f32(unsigned long long* state) {
    return (float)(oracle_random_u32(state) >> 8) / 16777216.0f;
}

/* [P1] SquirrelNoise5 (Squirrel Eiserloh's position hash, version 5): the
 * position times a constant, plus the seed, then four rounds of
 * xorshift-right / add-or-multiply by a constant, and a last xorshift.
 * All arithmetic is modulo 2^32. Parity unpinned for the exact values (the
 * page prints none to check against). */
unsigned int oracle_squirrel_noise5(unsigned int position, unsigned int seed) {
    unsigned int b = position;
    b *= 0xd2a80a3fu;
    b += seed;
    b ^= b >> 9;
    b += 0xa884f197u;
    b ^= b >> 11;
    b *= 0x6C736F4Bu;
    b ^= b >> 13;
    b += 0xB79F3ABBu;
    b ^= b >> 15;
    b *= 0x1b56c4f5u;
    b ^= b >> 17;
    return b;
}

/* [P1] Get2dNoiseUint: the 2-D position (x, y) hashed as x + 198491317 y
 * (modulo 2^32). */
unsigned int oracle_noise_2d(unsigned int x, unsigned int y, unsigned int seed) {
    return oracle_squirrel_noise5(x + 198491317u * y, seed);
}

static unsigned int f32_bits(float f) {
    unsigned int u;
    memcpy(&u, &f, 4);
    return u;
}
static float bits_f32(unsigned int u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE round-to-nearest-even of a float to bfloat16 (the upper 16 bits of
 * the float format); a NaN stays a (quiet) NaN. */
unsigned short oracle_bf16_rne(float x) {
    unsigned int u = f32_bits(x);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu))
        return (unsigned short)((u >> 16) | 0x0040u);
    unsigned int lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (unsigned short)(u >> 16);
}

/* [P1] stochastic_rounding, bf16 form: the low 16 bits of the float are
 * compared with the low 16 bits of `random`; above them the float is pushed
 * to the top of its bf16 interval (low bits all ones), else to the bottom
 * (low bits cleared), and the result is converted with round-to-nearest. */
unsigned short oracle_stochastic_round_bf16(float x, unsigned int random) {
    unsigned int threshold = random & 0xFFFFu;
    unsigned int u = f32_bits(x);
    unsigned int low = u & 0xFFFFu;
    u = low > threshold ? (u | 0xFFFFu) : (u & ~0xFFFFu);
    return oracle_bf16_rne(bits_f32(u));
}

/* [P1] adamw_kernel3 without master weights: bf16 parameters and gradients,
 * float moments. With g = grad, lerp(a, b, w) = fma(w, b, fma(-w, a, a)):
 *   m = lerp(g, m, b1); v = lerp(g*g, v, b2);
 *   mhat = m / (1 - b1^t); vhat = v / (1 - b2^t);
 *   p = p - lr * (mhat / (sqrt(vhat) + eps) + wd * p)     (all in float)
 * and the new bf16 parameter is p stochastically rounded. Element i of the
 * flat buffer is the page's thread (i mod 512) of block (i / 512); its random
 * word is Get2dNoiseUint of that position under the step's seed, and the
 * page's bf16 rounding routine hashes the same position again with that word
 * as the seed. Parameters and gradients are passed as bf16 bit patterns. */
void oracle_adamw_bf16_sr(unsigned short* params, const unsigned short* grads, float* mstate,
                          float* vstate, size_t n, float lr, float beta1, float beta2, float eps,
                          float wd, int t, unsigned int seed) {
    const float c1 = 1.0f - powf(beta1, (float)t);
    const float c2 = 1.0f - powf(beta2, (float)t);
    for (size_t i = 0; i < n; i++) {
        float g = bits_f32((unsigned int)grads[i] << 16);
        float m = fmaf(beta1, mstate[i], fmaf(-beta1, g, g));
        float gg = g * g;
        float v = fmaf(beta2, vstate[i], fmaf(-beta2, gg, gg));
        mstate[i] = m;
        vstate[i] = v;
        float mhat = m / c1;
        float vhat = v / c2;
        float old = bits_f32((unsigned int)params[i] << 16);
        float den = sqrtf(vhat) + eps;
        float upd = mhat / den + wd * old;
        float p = old - lr * upd;
        unsigned int x = (unsigned int)(i % 512), y = (unsigned int)(i / 512);
        unsigned int random = oracle_noise_2d(x, y, seed);
        params[i] = oracle_stochastic_round_bf16(p, oracle_noise_2d(x, y, random));
    }
}

/* [P1] sample_softmax: the index drawn from softmax(logits[0..n)) with a
 * coin in [0, 1): the first i whose cumulative probability exceeds the coin
 * (n - 1 when rounding leaves none). In double precision, with the row max
 * subtracted before exponentiating (the probabilities are unchanged). */
int oracle_sample_softmax(const double* logits, int n, double coin) {
    double mx = -INFINITY;
    for (int i = 0; i < n; i++) if (logits[i] > mx) mx = logits[i];
    double norm = 0.0;
    for (int i = 0; i < n; i++) norm += exp(logits[i] - mx);
    double target = coin * norm;
    double cdf = 0.0;
    for (int i = 0; i < n; i++) {
        cdf += exp(logits[i] - mx);
        if (target < cdf) return i;
    }
    return n - 1;
}
