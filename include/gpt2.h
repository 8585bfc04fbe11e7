/*
 * gpt2.h -- C ABI of the GB300 (sm_103a) GPT-2 training-step library (libgpt2.so).
 *
 * One process-global model instance (the llm.c pages drive a single
 * `GPT2 model` from main; these calls follow that page's gpt2_build /
 * gpt2_forward / gpt2_zero_grad / gpt2_backward / gpt2_update / gpt2_free
 * sequence, llm.c "train_gpt2.cu", sections gpt2_forward .. gpt2_free).
 *
 * Conventions for every call:
 *  - Integer-returning calls return GPT2_OK (0) or a negative GPT2_ERR_* code;
 *    gpt2_last_error() then holds a one-line description. No call exits the
 *    process or prints.
 *  - The library owns all model memory (parameters, gradients, AdamW state,
 *    activations) on the current CUDA device, and allocates nothing per step.
 *  - Work is enqueued on the library's stream (gpt2_set_stream); calls that
 *    return host values synchronise that stream, the others are asynchronous.
 *  - Parameter layout: one flat array of 16 tensors in the order
 *      wte(Vp,C) wpe(maxT,C) ln1w(L,C) ln1b(L,C) qkvw(L,3C,C) qkvb(L,3C)
 *      attprojw(L,C,C) attprojb(L,C) ln2w(L,C) ln2b(L,C) fcw(L,4C,C) fcb(L,4C)
 *      fcprojw(L,C,4C) fcprojb(L,C) lnfw(C) lnfb(C)
 *    (llm.c "train_gpt2.cu", ParameterTensors / fill_in_parameter_sizes).
 *    Weight matrices are (out, in) row-major, as nn.Linear stores them.
 */
#ifndef GPT2_GB300_H
#define GPT2_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define GPT2_OK 0
#define GPT2_ERR_CONFIG (-1)         /* invalid model dimensions or unsupported mode */
#define GPT2_ERR_STATE (-2)          /* call out of order (no model, backward before forward, ...) */
#define GPT2_ERR_SHAPE (-3)          /* B or T differs from the first forward, or T > maxT */
#define GPT2_ERR_TOKEN (-4)          /* a token or target id outside [0, V) */
#define GPT2_ERR_ALIGN (-5)          /* pointer, leading dimension or size not aligned as the call requires */
#define GPT2_ERR_CUDA (-6)           /* a CUDA runtime/driver call failed */
#define GPT2_ERR_NOMEM (-7)          /* device or pinned-host allocation failed */
#define GPT2_ERR_ARG (-8)            /* NULL pointer or out-of-range scalar argument */
#define GPT2_ERR_DEVICE_TIMEOUT (-9) /* a bounded in-kernel wait gave up; results are invalid */

/* precision modes for gpt2_init_ex */
#define GPT2_FP32 0 /* fp32 parameters, gradients and activations (llm.c train_gpt2_fp32.cu) */
#define GPT2_BF16 1 /* bf16 parameters, gradients and activations; fp32 master weights and AdamW
                       moments (llm.c train_gpt2.cu, default floatX and use_master_weights) */
#define GPT2_FP16 2 /* fp16 parameters, gradients and activations, fp32 master weights and AdamW
                       moments (llm.c train_gpt2.cu, the ENABLE_FP16 build: floatX = half), with
                       dynamic loss scaling (gpt2_set_loss_scaling), which that page lacks */

/* Create the model with seeded random initial weights in bf16 mixed precision on
 * the tensor cores (the llm.c page's default build). Equivalent to
 * gpt2_init_ex(L, C, NH, V, Vp, maxT, seed, GPT2_BF16, 1).
 *  L >= 0 layers, C channels (C % NH == 0, head size C/NH in {16, 32, 64, 128}, C % 8 == 0),
 *  V <= Vp vocabulary (Vp % 8 == 0), maxT >= 1 positions.
 * Initial weights: wte, wpe, qkvw, fcw ~ N(0, 0.02); attprojw, fcprojw ~ N(0, 0.02/sqrt(2L));
 * biases 0; LayerNorm gains 1, shifts 0; wte rows [V, Vp) are 0. Replaces any
 * previous model. Errors: GPT2_ERR_CONFIG, GPT2_ERR_NOMEM, GPT2_ERR_CUDA. */
int gpt2_init(int L, int C, int NH, int V, int Vp, int maxT, unsigned long long seed);

/* As gpt2_init with an explicit precision (GPT2_FP32 / GPT2_BF16 / GPT2_FP16)
 * and tensor_cores: 1 = tcgen05 tensor-core GEMMs and attention (bf16 or fp16
 * operands), 0 = SIMT FP32-FMA kernels ("-f 0", TF32 off, in llm.c
 * train_gpt2.cu main). */
int gpt2_init_ex(int L, int C, int NH, int V, int Vp, int maxT, unsigned long long seed,
                 int precision, int tensor_cores);

/* Use `stream` (a cudaStream_t, e.g. torch.cuda.current_stream().cuda_stream)
 * for all further work; NULL selects the library's own stream. */
int gpt2_set_stream(void* stream);

/* Forward pass (llm.c "train_gpt2.cu", gpt2_forward). tokens/targets are HOST
 * int32 arrays of B*T ids in [0, V); targets may be NULL (then no loss and the
 * call returns -1.0f, as on the page). The first forward fixes B and T
 * (later calls must use the same B, T <= maxT). Returns the mean loss over
 * the B*T positions (synchronises the stream), or NaN on error (see
 * gpt2_last_error). Ids are validated on the host before any work is enqueued. */
float gpt2_forward(const int* tokens, const int* targets, int B, int T);

/* Forward pass on DEVICE-resident int32 tokens/targets (B*T each; targets may
 * be NULL). Fully asynchronous: the mean loss is written to the device float
 * *d_mean_loss (may be NULL). Ids outside [0, V) are clamped to 0 on the device
 * and reported as GPT2_ERR_TOKEN by the next gpt2_sync(). */
int gpt2_forward_device(const int* d_tokens, const int* d_targets, int B, int T,
                        float* d_mean_loss);

/* Set every parameter gradient to zero (llm.c gpt2_zero_grad). */
int gpt2_zero_grad(void);

/* Gradient accumulation over k >= 1 micro-steps: the next forwards seed the
 * backward with dloss = 1/(k*B*T) instead of the page's 1/(B*T). */
int gpt2_set_grad_accum(int k);

/* The current accumulation count k (>= 1), or GPT2_ERR_STATE without a model. */
int gpt2_get_grad_accum(void);

/* Backward pass of the last forward (llm.c gpt2_backward). Parameter
 * gradients ACCUMULATE (+=); activation gradients are overwritten, except the
 * residual-stream gradient to which each LayerNorm backward adds.
 * GPT2_ERR_STATE if the last forward had no targets. */
int gpt2_backward(void);

/* AdamW update of every parameter (llm.c gpt2_update / adamw_kernel3):
 * m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; mhat = m/(1-b1^step); vhat = v/(1-b2^step);
 * theta -= lr (mhat/(sqrt(vhat)+eps) + wd theta). step >= 1. In GPT2_BF16 the fp32
 * master copy is updated and rounded (nearest-even) into the bf16 parameters;
 * without master weights (gpt2_set_master_weights(0)) the bf16 parameters are
 * updated in place: the update is computed in fp32 as the page writes it and
 * rounded to bf16 stochastically (adamw_kernel3's stochastic_rounding branch). */
int gpt2_adamw(float lr, float beta1, float beta2, float eps, float weight_decay, int step);

/* Keep (1, the default) or drop (0) the fp32 master copy of the bf16
 * parameters (llm.c "train_gpt2.cu", use_master_weights / the -w flag).
 * Without it AdamW reads and writes the bf16 parameters directly and rounds
 * each new value stochastically: with the low 16 bits of the fp32 value
 * compared against 16 random bits, it goes to the upper bf16 neighbour with
 * probability (low bits) / 65536, so the rounding is unbiased. The random
 * bits of element i come from the page's SquirrelNoise5 hash of the position
 * (i mod 512, i / 512) under a per-update seed drawn from the model's
 * xorshift* stream (state 13371337 at gpt2_init, as on the page). This saves
 * 4 bytes per parameter of memory and of AdamW traffic. Turning it back on
 * copies the current bf16 parameters into a new master copy. bf16 models
 * only (GPT2_ERR_CONFIG otherwise, except enabled = 1, which is a no-op);
 * discards a recorded gpt2_train_step graph. */
int gpt2_set_master_weights(int enabled);

/* One whole training step on DEVICE-resident int32 tokens and targets:
 * gpt2_zero_grad, then for each of the k = gpt2_set_grad_accum micro-steps
 * gpt2_forward_device and gpt2_backward on the next B*T ids (the buffers hold
 * k*B*T each), then gpt2_adamw, with the same results as those calls. The
 * mean loss of micro-step i goes to d_mean_loss[i] (may be NULL). The first call for a given (d_tokens,
 * d_targets, d_mean_loss, B, T, grad-accumulation k) runs eagerly and records
 * the step's launches into a CUDA graph; later calls with the same set replay
 * the graph (the AdamW arguments may change from call to call), which removes
 * the per-launch host cost and most of the gaps between kernels. The buffers
 * are read at replay time, so refill them in place between calls. Fully
 * asynchronous on the model's stream. With gpt2_timing_begin active every call
 * runs eagerly. */
int gpt2_train_step(const int* d_tokens, const int* d_targets, int B, int T, float lr, float beta1,
                    float beta2, float eps, float weight_decay, int step, float* d_mean_loss);

/* The same whole step on HOST int32 tokens and targets (k*B*T ids each, k =
 * gpt2_set_grad_accum), the training loop of llm.c "train_gpt2.cu" (main:
 * a batch from the loader, gpt2_forward, gpt2_zero_grad, gpt2_backward,
 * gpt2_update, the loss printed). The ids are checked on the host (any id
 * outside [0, V) returns GPT2_ERR_TOKEN before any work is enqueued), staged
 * in a pinned buffer the library keeps, copied to the device in one transfer,
 * the step runs as gpt2_train_step does (a CUDA-graph replay after the first
 * call), and the k micro-step mean losses are copied back to the HOST array
 * mean_loss (k floats; may be NULL). The call synchronises the model's stream
 * and reports device errors (GPT2_ERR_DEVICE_TIMEOUT, GPT2_ERR_TOKEN) like
 * gpt2_sync. The caller keeps ownership of all three host arrays. */
int gpt2_train_step_host(const int* tokens, const int* targets, int B, int T, float lr, float beta1,
                         float beta2, float eps, float weight_decay, int step, float* mean_loss);

/* Time limit (nanoseconds) of every bounded in-kernel wait of the library's
 * tensor-core and bulk-copy kernels on the current device (0 restores the
 * default, 2 s). A kernel whose wait runs out sets GPT2_ERR_DEVICE_TIMEOUT in
 * its error word, waits (up to 2 s, whatever this limit) for the copies and
 * MMAs it has in flight, frees its tensor memory and returns; the results of
 * that launch are undefined. Applies to launches made after the call. */
int gpt2_set_wait_limit(unsigned long long ns);

/* Wait for the stream; report GPT2_ERR_DEVICE_TIMEOUT / GPT2_ERR_TOKEN raised by kernels. */
int gpt2_sync(void);

/* Introspection (host fp32 copies, flat order above; all synchronise). */
size_t gpt2_num_params(void);
int gpt2_param_sizes(size_t out[16]);
int gpt2_get_params(float* host);       /* current parameters (bf16 widened to fp32) */
int gpt2_set_params(const float* host); /* also resets the fp32 master copy and AdamW moments */
int gpt2_get_grads(float* host);
int gpt2_set_grads(const float* host);  /* overwrite the gradients (e.g. to drive gpt2_adamw alone) */
int gpt2_get_master(float* host);       /* fp32 master weights (GPT2_BF16 only) */
int gpt2_get_losses(float* host);       /* per-position losses of the last forward, B*T */

/* Activation read-out for tests: which = GPT2_ACT_*, layer in [0, L) where it applies.
 * Copies the tensor (widened to fp32) to host and returns its element count
 * through *n (may be NULL). */
#define GPT2_ACT_ENCODED 0   /* (B,T,C) */
#define GPT2_ACT_LN1 1       /* (L,B,T,C) */
#define GPT2_ACT_QKV 2       /* (L,B,T,3C) */
#define GPT2_ACT_ATTY 4      /* (L,B,T,C) */
#define GPT2_ACT_RESIDUAL2 5 /* (L,B,T,C) */
#define GPT2_ACT_LN2 6       /* (L,B,T,C) */
#define GPT2_ACT_FCH 7       /* (L,B,T,4C) */
#define GPT2_ACT_FCH_GELU 8  /* (L,B,T,4C) */
#define GPT2_ACT_RESIDUAL3 9 /* (L,B,T,C) */
#define GPT2_ACT_LNF 10      /* (B,T,C) */
#define GPT2_ACT_LOGITS 11   /* (B,T,Vp): logits after forward without targets, dlogits after one with targets */
#define GPT2_ACT_LSE 18      /* (L,B,NH,T) fp32 attention log-sum-exp */
#define GPT2_ACT_PROBS 12    /* (B,T,Vp) fp32 softmax over the first V logits, 0 on the padding,
                                after a forward without targets (the probs output of llm.c
                                fused_classifier_kernel3); computed on the device at the call */
int gpt2_get_activation(int which, int layer, float* host, size_t* n);

/* ---- inference (llm.c "train_gpt2.cu": sample_softmax and the generation
 * block of main) ----
 * gpt2_sample: after a forward without targets, draw one token per sequence
 * b in [0, B) from the model's distribution at position t (softmax over the
 * first V logits of row (b, t)), following sample_softmax: the first index
 * whose cumulative probability exceeds coins[b]. coins: HOST, B floats in
 * [0, 1) (e.g. from the page's random_f32); out: HOST, B ints. Runs on the
 * device (one block per sequence) and synchronises. GPT2_ERR_STATE without
 * a preceding target-less forward; GPT2_ERR_ARG for t outside [0, T) or a
 * coin outside [0, 1). */
int gpt2_sample(int t, const float* coins, int* out);

/* gpt2_generate: autoregressive sampling on the device. tokens: HOST int32
 * (B, T), read and written; positions [t_begin, t_end) are generated, each
 * from a forward over the whole (B, T) window (the page's generation loop,
 * which also recomputes the full forward per token) and gpt2_sample at
 * position t - 1 with one coin per sequence drawn from *rng_state by the
 * page's xorshift* random_f32 (for t, then for b). Tokens stay on the device
 * between positions (one upload, one download, no synchronisation per
 * token). *rng_state is advanced as the draws did. 1 <= t_begin <= t_end <= T;
 * B, T as for gpt2_forward. */
int gpt2_generate(int* tokens, int B, int T, int t_begin, int t_end, unsigned long long* rng_state);

/* ---- loss scaling (GPT2_FP16 only) ----
 * fp16 keeps 5 exponent bits, so small gradients underflow and large ones
 * overflow. The backward is seeded with dloss = scale / (k B T) (the loss
 * itself and its value are unscaled); gradients are stored scaled. Before
 * each AdamW update a kernel checks every gradient: if any is inf or NaN the
 * update is skipped (parameters and moments unchanged) and the scale halves;
 * otherwise AdamW uses gradient / scale and, after growth_interval updates in
 * a row without overflow, the scale doubles. The state lives in device memory,
 * so CUDA-graph replays of gpt2_train_step keep it current. Defaults: scale
 * 65536 (2^16), growth_interval 2000. gpt2_get_grads / gpt2_set_grads work in
 * unscaled values.
 * gpt2_set_loss_scaling: restart with init_scale (a power of two) and
 * growth_interval >= 1; GPT2_ERR_CONFIG outside GPT2_FP16.
 * gpt2_get_loss_scale: the current scale (1 outside GPT2_FP16) and the number
 * of updates skipped so far (either pointer may be NULL); synchronises. */
int gpt2_set_loss_scaling(float init_scale, int growth_interval);
int gpt2_get_loss_scale(float* scale, long long* skipped);

/* Release all device memory held by the model. */
int gpt2_free(void);

/* Text of the last error (static storage, never NULL). */
const char* gpt2_last_error(void);

/* Code (GPT2_ERR_*) of the last error; lets callers of gpt2_forward, which
 * signals failure with NaN, tell the causes apart. */
int gpt2_last_status(void);

/* ---- kernel timing (CUDA events around each launch, for roofline reporting) ----
 * family: 0 GEMM, 1 attention forward, 2 attention backward, 3 LayerNorm forward,
 * 4 LayerNorm backward, 5 classifier softmax-CE, 6 AdamW, 7 encoder, 8 other.
 * gpt2_timing_begin(max_launches) starts recording (events are preallocated);
 * gpt2_timing_end() synchronises and totals; gpt2_timing_get returns, per family,
 * total milliseconds, launch count and algorithmic work (FLOPs for GEMM and
 * attention families, bytes for the others). */
int gpt2_timing_begin(int max_launches);
int gpt2_timing_end(void);
int gpt2_timing_get(int family, double* total_ms, long long* launches, double* work);

/* Number of CUDA kernels this library has launched in this process (all entry
 * points, counted on the host at launch). */
long long gpt2_launch_count(void);

/* ---- standalone fused operator ----
 * out = softmax_row( gelu_tanh( x . W^T + b ) ) (POPCORNBENCH "fused Linear +
 * GELU + Softmax" problem statement: nn.Linear then GELU then softmax over dim 1).
 * x: DEVICE fp32 (M,K) row-major; W: DEVICE fp32 (N,K) row-major (nn.Linear
 * layout); b: DEVICE fp32 (N); out: DEVICE fp32 (M,N) row-major, caller-owned.
 * The product kernel splits each fp32 operand into bf16 halves (hi, lo) in
 * shared memory as its tiles arrive and runs hi.hi + hi.lo + lo.hi on the bf16
 * tensor cores with fp32 accumulation (about 2^-16 relative per product;
 * outputs within 1e-3 relative of fp64). x, W, b and out must be 16-byte
 * aligned with K % 4 == 0 and N % 4 == 0 (else GPT2_ERR_ALIGN); M, K, N >= 1
 * (else GPT2_ERR_ARG). Asynchronous on `stream` (a cudaStream_t, NULL = legacy
 * default stream). The first call on a device allocates its scratch (the
 * per-row softmax partials, 8 bytes per row and column tile: tiles of 256
 * columns, or of 224 where those fill the GPU's CTA pairs better; grown as
 * needed and kept until exit). The output is undefined when gpt2_device_status() then
 * reports GPT2_ERR_DEVICE_TIMEOUT. */
int fused_linear_bias_gelu_softmax(const float* x, const float* W, const float* b, float* out,
                                   int M, int K, int N, void* stream);

/* Allocation-free variant of fused_linear_bias_gelu_softmax (an addition to the
 * operator's problem statement: it exists for callers that cannot let a library allocate device
 * memory -- processes whose own pool allocator owns all device memory, where a
 * cudaMalloc behind its back can fail or fragment the pool, and loops that
 * cannot take the device-wide synchronisation a cudaMalloc may imply).
 * Same arguments, errors and arithmetic as fused_linear_bias_gelu_softmax (the
 * same kernels, so the same output bit for bit, within 1e-3 relative of fp64);
 * it calls no cudaMalloc/cudaFree or other allocating routine. Its per-row
 * softmax partials live in a static device array of 1 MiB that every GPU
 * loading the library holds until exit, which limits M * ceil(N/256) to
 * 131072 (e.g. M = 1024 rows with N up to 32768); larger sizes return
 * GPT2_ERR_ARG with a message in gpt2_last_error(). Every call shares that
 * array and leaves its contents behind (nothing needs clearing: each call
 * writes every partial it reads); calls whose GPU work overlaps race on it.
 * The first call on a device (with that device current) looks up the array's
 * device address; make that first call before any stream capture. An expired
 * in-kernel wait is reported by gpt2_device_status(), and the output of that
 * call is then undefined. */
int fused_linear_bias_gelu_softmax_noalloc(const float* x, const float* W, const float* b,
                                           float* out, int M, int K, int N, void* stream);

/* ---- kernel-level entry points (DEVICE pointers, asynchronous on `stream`) ----
 * gpt2_gemm: D[M,N] = A[M,K] . B[N,K]^T with the step's fused epilogues.
 *  dtype GPT2_FP32 / GPT2_BF16 / GPT2_FP16 is the element type of A, B, D, bias,
 *  aux, D2; tensor_cores = 1 selects the tcgen05 kernel (bf16 and fp16:
 *  kind::f16; fp32: kind::tf32, K-major operands only), 0 the SIMT FP32-FMA kernel.
 *  Storage: a_kmajor ? A(m,k) = A[m*lda + k] : A[k*lda + m];
 *           b_kmajor ? B(n,k) = B[n*ldb + k] : B[k*ldb + n];  D(m,n) = D[m*ldd + n].
 *  epilogue: 0 D = acc (+ bias[n]); 1 D = acc + bias[n], D2 = gelu(D) (same ldd);
 *            2 D = acc + bias[n] + aux(m,n); 3 D = acc * gelu'(aux(m,n)); 4 D += acc.
 *  (llm.c "train_gpt2.cu": matmul_forward_cublaslt, matmul_backward, gelu_forward,
 *  gelu_backward, residual_forward.) bias may be NULL. Tensor-core path needs
 *  16-byte aligned pointers and leading dimensions and N % (16/elem) == 0, else
 *  GPT2_ERR_ALIGN.
 *  Errors: GPT2_ERR_ARG for A, B or D NULL, M, N or K < 1, an unknown epilogue,
 *  epilogues 2 and 3 without aux or 1 without D2; GPT2_ERR_CONFIG for an unknown
 *  dtype or an fp32 tensor-core product with an MN-major operand.
 *  ws / ws_floats: optional DEVICE fp32 scratch, caller-owned, 16-byte aligned
 *  (NULL or 0 = none). With epilogue 4, bf16 and tensor cores, a product with
 *  fewer output tiles than the GPU has CTA slots (a weight gradient: small
 *  M x N, long K) may split K into ranges whose fp32 partial sums go to ws
 *  (at most ws_floats of them) and are then added to D in range order, so the
 *  result stays deterministic. Nothing else may use ws until the call's work
 *  on `stream` has finished. */
int gpt2_gemm(int dtype, int tensor_cores, int epilogue, const void* A, long long lda, int a_kmajor,
              const void* B, long long ldb, int b_kmajor, void* D, long long ldd, const void* bias,
              const void* aux, long long ldaux, void* D2, int M, int N, int K, float* ws,
              size_t ws_floats, void* stream);

/* Causal attention forward over a fused (B,T,3,NH,HS) qkv: out (B,T,NH*HS) and
 * lse (B,NH,T) fp32 natural-log sum of exp of the scaled scores (llm.c
 * attention_forward with softmax_forward_kernel5, scale 1/sqrt(HS)).
 * HS = C/NH in {16,32,64,128}; bf16 or fp16 with tensor_cores and HS == 64 uses the
 * tensor-core flash kernel (operands its tensor maps cannot address take a kernel
 * without them instead), everything else the SIMT kernel. Errors: GPT2_ERR_ARG for a NULL
 * pointer, B, T or NH < 1 or C % NH != 0; GPT2_ERR_CONFIG for another head size or an
 * unknown dtype. */
int gpt2_attention_forward(int dtype, int tensor_cores, const void* qkv, void* out, float* lse,
                           int B, int T, int C, int NH, void* stream);

/* Its backward: dqkv (B,T,3C) is written (llm.c attention_backward with
 * softmax_autoregressive_backward_kernel); scratch_D is B*NH*T floats. Same
 * size rules and errors as the forward. */
int gpt2_attention_backward(int dtype, int tensor_cores, const void* dout, const void* qkv,
                            const void* out, const float* lse, void* dqkv, float* scratch_D, int B,
                            int T, int C, int NH, void* stream);

/* LayerNorm over the last dimension C of N rows (llm.c "train_gpt2.cu",
 * layernorm_forward_kernel3): biased variance, eps 1e-5; out (N,C), mean and
 * rstd (N) fp32. N >= 1, C % 8 == 0, 8 <= C <= 2048 (16-bit) / 1024 (fp32), else
 * GPT2_ERR_ARG (also for a NULL pointer); GPT2_ERR_CONFIG for an unknown dtype. */
int gpt2_layernorm_forward(int dtype, void* out, float* mean, float* rstd, const void* inp,
                           const void* w, const void* b, int N, int C, void* stream);

/* Its backward (layernorm_backward_kernel6 with += for every output): dinp +=
 * (or = when accumulate == 0), dw += and db += sums over the N rows, computed
 * deterministically through `scratch` (fp32, gpt2_layernorm_backward_scratch_floats(C)
 * floats, caller-owned). Same size rules and errors as the forward. */
size_t gpt2_layernorm_backward_scratch_floats(int C);
int gpt2_layernorm_backward(int dtype, void* dinp, void* dw, void* db, const void* dout,
                            const void* inp, const void* w, const float* mean, const float* rstd,
                            int N, int C, int accumulate, float* scratch, void* stream);

/* Synchronise the device and report (then clear) the error word of the
 * stand-alone entry points: GPT2_ERR_DEVICE_TIMEOUT if a bounded wait expired. */
int gpt2_device_status(void);

#ifdef __cplusplus
}
#endif

#endif
