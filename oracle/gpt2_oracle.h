/*
 * gpt2_oracle.h -- plain, slow CPU reference of one GPT-2 training step and of
 * the fused Linear+bias+GELU+row-softmax operator.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this library. The GPU product
 * path never links, loads or calls it, and shares no code with it.
 *
 * Everything is computed in double precision. Parameters are one flat array in
 * the order of llm.c train_gpt2.cu, "ParameterTensors" / fill_in_parameter_sizes:
 *   wte(Vp,C) wpe(maxT,C) ln1w(L,C) ln1b(L,C) qkvw(L,3C,C) qkvb(L,3C)
 *   attprojw(L,C,C) attprojb(L,C) ln2w(L,C) ln2b(L,C) fcw(L,4C,C) fcb(L,4C)
 *   fcprojw(L,C,4C) fcprojb(L,C) lnfw(C) lnfb(C)
 * Activations use the (B,T,C) row-major layout of the same page; the fused
 * QKV activation is (B,T,3,NH,HS).
 *
 * Every function is pinned by a test against something other than itself,
 * except the exact values of the SquirrelNoise5 hash: parity unpinned there.
 */
#ifndef GPT2_ORACLE_H
#define GPT2_ORACLE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_NUM_PARAM_TENSORS 16

typedef struct {
    int L;     /* layers */
    int C;     /* channels */
    int NH;    /* heads */
    int V;     /* vocabulary size */
    int Vp;    /* padded vocabulary size (rows of wte) */
    int maxT;  /* rows of wpe */
} oracle_config;

/* Fills sizes[16] (elements per tensor) and returns the total element count. */
size_t oracle_param_sizes(const oracle_config* cfg, size_t sizes[ORACLE_NUM_PARAM_TENSORS]);

/* ---- single operations (each is the plain definition) ---- */

/* out[n,c] = wte[tok[n],c] + wpe[n % T, c] for n in [0, B*T). */
void oracle_encoder_forward(double* out, const int* tokens, const double* wte, const double* wpe,
                            int B, int T, int C);

/* Row-wise LayerNorm over C with biased variance and eps = 1e-5.
 * mean/rstd may be NULL. */
void oracle_layernorm_forward(double* out, double* mean, double* rstd, const double* inp,
                              const double* w, const double* b, int N, int C);

/* dinp += ..., dw += ..., db += ... (textbook LayerNorm derivative). */
void oracle_layernorm_backward(double* dinp, double* dw, double* db, const double* dout,
                               const double* inp, const double* w, const double* mean,
                               const double* rstd, int N, int C);

/* out[n,o] = bias[o] + sum_c inp[n,c] * w[o,c]; bias may be NULL. */
void oracle_matmul_forward(double* out, const double* inp, const double* w, const double* bias,
                           int N, int Cin, int Cout);

/* dinp = dout . w (overwrite); dw += dout^T . inp; dbias += column sums (dbias may be NULL). */
void oracle_matmul_backward(double* dinp, double* dw, double* dbias, const double* dout,
                            const double* inp, const double* w, int N, int Cin, int Cout);

/* tanh-approximate GELU and its derivative applied to dout. */
void oracle_gelu_forward(double* out, const double* inp, size_t n);
void oracle_gelu_backward(double* dinp, const double* inp, const double* dout, size_t n);

/* Causal multi-head attention by the materialised definition.
 * qkv (B,T,3C) -> out (B,T,C); att (B,NH,T,T) receives the probabilities
 * (zero above the diagonal). att may be NULL. */
void oracle_attention_forward(double* out, double* att, const double* qkv,
                              int B, int T, int C, int NH);

/* dqkv = d(attention)/d(qkv) . dout (overwrite). att must be the forward's output. */
void oracle_attention_backward(double* dqkv, const double* dout, const double* qkv,
                               const double* att, int B, int T, int C, int NH);

/* ---- whole model ---- */

typedef struct oracle_model oracle_model;

/* Allocates the activations for a (B,T) batch. Returns NULL on failure. */
oracle_model* oracle_create(const oracle_config* cfg, int B, int T);
void oracle_destroy(oracle_model* m);

/* Forward pass. targets may be NULL (then returns -1 and computes no loss).
 * grad_accum_k sets dloss = 1 / (k*B*T) for the following backward.
 * Returns the mean loss over the B*T positions. */
double oracle_forward(oracle_model* m, const double* params, const int* tokens,
                      const int* targets, int grad_accum_k);

/* Backward pass of the last forward. grads (flat, same layout as params) are
 * ACCUMULATED (+=). Returns 0 on success, -1 if the last forward had no targets. */
int oracle_backward(oracle_model* m, const double* params, double* grads);

/* Activation read-out for tests. which: see ORACLE_ACT_* below; layer ignored
 * for non-layer tensors. Returns the element count copied, or 0 if unknown. */
enum {
    ORACLE_ACT_ENCODED = 0, ORACLE_ACT_LN1 = 1, ORACLE_ACT_QKV = 2, ORACLE_ACT_ATT = 3,
    ORACLE_ACT_ATTY = 4, ORACLE_ACT_RESIDUAL2 = 5, ORACLE_ACT_LN2 = 6, ORACLE_ACT_FCH = 7,
    ORACLE_ACT_FCH_GELU = 8, ORACLE_ACT_RESIDUAL3 = 9, ORACLE_ACT_LNF = 10,
    ORACLE_ACT_LOGITS = 11, ORACLE_ACT_PROBS = 12, ORACLE_ACT_LOSSES = 13,
    ORACLE_ACT_DLOGITS = 14, ORACLE_ACT_LN1_MEAN = 15, ORACLE_ACT_LN1_RSTD = 16
};
size_t oracle_get_act(const oracle_model* m, int which, int layer, double* out);

/* AdamW with decoupled weight decay applied to every parameter; t >= 1. */
void oracle_adamw(double* params, const double* grads, double* mstate, double* vstate, size_t n,
                  double lr, double beta1, double beta2, double eps, double wd, int t);

/* ---- standalone fused operator ----
 * y[m,:] = softmax_row( gelu_tanh( x[m,:] . W^T + b ) ), W is (N,K) row-major. */
void oracle_fused_linear_bias_gelu_softmax(const double* x, const double* W, const double* b,
                                           double* y, int M, int K, int N);

/* ---- random numbers, stochastic rounding, sampling ---- */
/* xorshift* step of the 64-bit state; a float in [0, 1) from its top 24 bits. */
unsigned int oracle_random_u32(unsigned long long* state);
float oracle_random_f32(unsigned long long* state);
/* SquirrelNoise5 position hash, and its 2-D form (x + 198491317 y).
 * Parity unpinned for the exact output values: the page prints no worked
 * values, so only statistical properties are checked (balanced bits, seed
 * sensitivity, uncorrelated neighbours); a wrong constant would pass them. */
unsigned int oracle_squirrel_noise5(unsigned int position, unsigned int seed);
unsigned int oracle_noise_2d(unsigned int x, unsigned int y, unsigned int seed);
/* float -> bf16 bits, round to nearest even. */
unsigned short oracle_bf16_rne(float x);
/* float -> bf16 bits, stochastic rounding with the low 16 bits of random. */
unsigned short oracle_stochastic_round_bf16(float x, unsigned int random);
/* AdamW without master weights: bf16 params (bit patterns, updated in place)
 * and grads, float moments; the update in float, the result stochastically
 * rounded with the step's seed. */
void oracle_adamw_bf16_sr(unsigned short* params, const unsigned short* grads, float* mstate,
                          float* vstate, size_t n, float lr, float beta1, float beta2, float eps,
                          float wd, int t, unsigned int seed);
/* Index sampled from softmax(logits[0..n)) with coin in [0, 1). */
int oracle_sample_softmax(const double* logits, int n, double coin);

/* Number of OpenMP threads the oracle uses (1 when built without OpenMP). */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif

#endif
